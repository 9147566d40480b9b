"""Pins for the oracle's fp16 / bf16 rounding (brute force and library)."""
import numpy as np
import pytest
import torch

from oracle import fp


def all_finite_fp16():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    h = bits.view(np.float16)
    v = h[np.isfinite(h)].astype(np.float64)
    return np.unique(v)  # sorted, -0 and +0 merge


def sample_values(rng, n):
    mags = 10.0 ** rng.uniform(-9, 5.2, n)
    v = mags * rng.choice([-1.0, 1.0], n)
    fin = all_finite_fp16()
    exact = rng.choice(fin, n // 4)
    return np.concatenate([v, exact, [0.0, 65504.0, -65504.0, 65519.0,
                                      -65519.0, 6e-8, -6e-8, 1e-10]])


def test_fp16_directed_rounding_brute_force():
    rng = np.random.default_rng(0)
    fin = all_finite_fp16()
    v = sample_values(rng, 20000)
    rd = fp.fp16_rd(v).astype(np.float64)
    ru = fp.fp16_ru(v).astype(np.float64)
    # brute force: largest finite fp16 <= v, smallest >= v
    i = np.searchsorted(fin, v, side="right") - 1
    exp_rd = np.where(i >= 0, fin[np.clip(i, 0, None)], -np.inf)
    j = np.searchsorted(fin, v, side="left")
    exp_ru = np.where(j < fin.size, fin[np.clip(j, None, fin.size - 1)],
                      np.inf)
    np.testing.assert_array_equal(rd, exp_rd)
    np.testing.assert_array_equal(ru, exp_ru)


def test_fp16_nearest_brute_force():
    rng = np.random.default_rng(1)
    fin = all_finite_fp16()
    v = rng.uniform(-60000, 60000, 5000)
    v = np.concatenate([v, (fin[:-1] + fin[1:]) / 2])  # exact ties
    v = v[np.abs(v) < 65504]
    got = fp.fp16_rne(v).astype(np.float64)
    j = np.searchsorted(fin, v)
    lo, hi = fin[j - 1], fin[np.clip(j, None, fin.size - 1)]
    lo = np.where(fin[j] == v, v, lo)
    dlo, dhi = v - lo, hi - v
    even_lo = (fp.fp16_bits(fp.fp16_rne(lo)) & 1) == 0
    exp = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi,
                                           np.where(even_lo, lo, hi)))
    np.testing.assert_array_equal(got, exp)


def test_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(100000) * 10.0 ** rng.uniform(-30, 30, 100000)
         ).astype(np.float32)
    # include exact ties between bf16 neighbours
    b = rng.integers(0, 0x7F7F, 1000, dtype=np.uint32) << 16 | (1 << 15)
    x = np.concatenate([x, b.view(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy()
    got = fp.bf16_rne_bits(x.astype(np.float64))
    np.testing.assert_array_equal(got, ref.view(np.uint16))


def test_bf16_single_rounding_from_fp64():
    """fp64 values just above a bf16 tie must round up, although the fp32
    detour would land exactly on the tie and round to even."""
    base = np.float64(1.0)          # bf16 neighbours 1 and 1 + 2^-7
    tie = base + 2.0 ** -8
    v = np.array([tie + 2.0 ** -40, tie - 2.0 ** -40, tie])
    got = fp.bf16_rne_value(v)
    np.testing.assert_array_equal(got, [1 + 2.0 ** -7, 1.0, 1.0])
    # subnormal range: quantum 2^-133
    q = 2.0 ** -133
    v = np.array([3.4 * q, 2.5 * q, 3.5 * q])
    np.testing.assert_array_equal(fp.bf16_rne_value(v), [3 * q, 2 * q, 4 * q])


def test_fp16_bit_views_against_the_format():
    """fp16_from_bits decodes every finite binary16 pattern to the value the
    format defines (sign, 5-bit biased exponent, 10-bit fraction, subnormals
    at 2^-14 * f/1024), and fp16_bits gives the pattern back."""
    b = np.arange(1 << 16, dtype=np.uint32)
    sign = np.where(b >> 15, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    f = (b & 0x3FF).astype(np.float64)
    finite = e != 0x1F
    want = np.where(e == 0, sign * np.ldexp(f / 1024.0, -14),
                    sign * np.ldexp(1.0 + f / 1024.0, e.astype(np.int64) - 15))
    got = fp.fp16_from_bits(b.astype(np.uint16)).astype(np.float64)
    np.testing.assert_array_equal(got[finite], want[finite])
    back = fp.fp16_bits(fp.fp16_from_bits(b[finite].astype(np.uint16)))
    np.testing.assert_array_equal(back, b[finite].astype(np.uint16))
    assert np.all(np.isinf(got[(e == 0x1F) & ((b & 0x3FF) == 0)]))
