"""Edge cases of the quantiser driven through the CUDA path (needs a GB300).

The calibration here is built by hand: mu = 0 and V = I, so the
coefficients are the rows themselves and every case of the kvtc page's
microscaled quantiser (technical summary 2A, shared fp16 scale and shift per
16-component group; 2B, quantisation) can be reached on purpose:

  * constant groups: max = min, so scale = 0, every code is 0 and the
    reconstruction is the shift exactly;
  * exact half-way ties: (c - shift) / scale = q + 1/2 with a power-of-two
    scale, which round up;
  * full-range codes: width-8 groups whose codes cover 0 .. 255;
  * a coefficient beyond the fp16 range (a bf16 input of 1e5), which must
    raise KVTC_FLAG_RANGE and leave that token's record unwritten, with no
    fault.

With an identity basis the projection is exact in fp32 (one nonzero term
per output), so the GPU's records must equal the oracle's byte for byte on
the crafted rows, and the restore of the oracle's records must equal the
oracle's bf16 rows bit for bit.
"""
import numpy as np
import pytest

import synth
from oracle import calibrate, codec, fp

from _parity import check_decompress, check_records, record

pytestmark = pytest.mark.gpu

D = 128
WIDTHS = np.array([8, 8, 4, 2, 1, 3, 5, 7])        # 8 groups, all active
BUDGET = 1024                                       # 864 bits used, R = 128
SINK, WINDOW = 4, 16


@pytest.fixture(scope="module")
def kv():
    from kv_cache_transform_gb300 import _build
    _build.build()
    import kv_cache_transform_gb300 as kv
    return kv


@pytest.fixture(scope="module")
def torch():
    import torch
    assert torch.cuda.is_available()
    return torch


def identity_blob():
    mu = np.zeros(D)
    V = np.eye(D)
    return calibrate.write_blob([(0, 0, mu, V, np.ones(D), WIDTHS)], SINK,
                                WINDOW, BUDGET)


def crafted_group(rng, b, kind):
    """16 values of one group of width b, exact in bf16 and in fp16."""
    lev = (1 << b) - 1
    if kind == "const":
        v = rng.choice([0.0, 1.5, -3.25, 0.0078125, 1000.0, -0.5, 96.0])
        return np.full(16, v)
    if kind == "ties":
        # shift 0 or -lev s, scale s = 2^e, eight values at q + 1/2
        e = int(rng.integers(-6, 3))
        s = 2.0 ** e
        qmax = min(lev - 1, 127)
        q = rng.integers(0, qmax + 1, 16).astype(float) + 0.5
        q[0], q[1] = 0.0, float(lev)      # pin min and max
        v = q * s
        if lev <= 127 and rng.random() < 0.5:   # (2q + 1 - 2 lev) fits 8 bits
            v = v - lev * s
        return v
    if kind == "grid":
        # every code of the width, min and max included
        e = int(rng.integers(-8, 2))
        q = rng.integers(0, lev + 1, 16).astype(float)
        q[0], q[1] = 0.0, float(lev)
        return q * 2.0 ** e
    raise ValueError(kind)


def crafted_rows(n, seed):
    rng = np.random.default_rng(seed)
    x = np.zeros((n, D))
    kinds = ["const", "ties", "grid"]
    for t in range(n):
        for g, b in enumerate(WIDTHS):
            x[t, 16 * g:16 * g + 16] = crafted_group(
                rng, int(b), kinds[(t + g) % 3])
    # full code range at width 8: group 0 of the first 256 rows counts up
    for t in range(min(n, 256)):
        v = np.full(16, 0.0)
        v[1] = 255.0 / 256
        v[2] = t / 256.0
        x[t, 0:16] = v
    bits = synth.f32_to_bf16_bits(x)
    assert np.array_equal(fp.bf16_bits_to_f64(bits), x), "not bf16-exact"
    assert np.array_equal(fp.fp16_rne(x).astype(np.float64), x), \
        "not fp16-exact"
    return bits


def to_dev(torch, bits):
    return torch.from_numpy(bits.view(np.int16).copy()).cuda()


def stream_calib(basis):
    b = calibrate.read_blob(identity_blob())
    return calibrate.stream_calib(b["streams"][0], SINK, WINDOW, BUDGET,
                                  basis=basis)


def test_identity_basis_records_and_restore_bit_exact(kv, torch):
    n = 300
    T = SINK + WINDOW + n
    rng = np.random.default_rng(17)
    raw = synth.f32_to_bf16_bits(rng.standard_normal((T, D)))
    x = raw.copy()
    x[SINK:SINK + n] = crafted_rows(n, 3)
    sc_enc, sc_dec = stream_calib("bf16"), stream_calib("fp16")
    calib = kv.kvtc_calib_load(identity_blob(), 0)
    nbytes = calib.stream_bytes(0, 0, T)
    dst = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device="cuda")
    kv.kvtc_compress(calib, 0, 1, 1, [to_dev(torch, x), None], D, T, dst,
                     nbytes)
    assert kv.kvtc_device_status(calib) == 0
    got = dst.cpu().numpy().tobytes()
    ref = codec.compress_stream(x, sc_enc)
    assert got == ref, "records differ from the oracle's"
    # the parity rule agrees, and the cases were reached
    R = sc_enc.R
    off = (SINK + WINDOW) * D * 2
    rec = np.frombuffer(ref, np.uint8, n * R, off).reshape(n, R)
    st = check_records(rec, x[SINK:SINK + n], sc_enc)
    record("identity basis, crafted rows", st=st)
    assert st["bad"] == 0 and st["field_flips"] == 0 and st["code_flips"] == 0
    shift, scale, q = codec.unpack(rec, sc_enc.bits)
    assert np.sum(scale == 0) > 100                    # constant groups
    assert set(np.unique(q[:, :16])) == set(range(256))  # width 8, 0..255
    c = fp.bf16_bits_to_f64(x[SINK:SINK + n])
    u = (c.reshape(n, 8, 16) - shift.astype(float)[:, :, None]) / \
        np.where(scale > 0, scale, 1).astype(float)[:, :, None]
    ties = (u - np.floor(u)) == 0.5
    assert ties.sum() > 1000                           # exact half-way ties
    # half rounds up
    assert np.all(q.reshape(n, 8, 16)[ties] == np.floor(u[ties]) + 1)
    # restore of the oracle's records
    out = torch.full((T, D), 0x7FC0, dtype=torch.int16, device="cuda")
    srcd = torch.from_numpy(np.frombuffer(ref, np.uint8).copy()).cuda()
    kv.kvtc_decompress(calib, 0, 1, 1, srcd, len(ref), T, [out, None], D)
    assert kv.kvtc_device_status(calib) == 0
    xg = out.cpu().numpy().view(np.uint16)
    xo = codec.decompress_stream(ref, T, sc_dec)
    assert np.array_equal(xg, xo)
    # constant groups come back exactly as they went in
    cst = (scale == 0)
    rows, groups = np.nonzero(cst)
    for t, g in zip(rows[:200], groups[:200]):
        assert np.array_equal(xg[SINK + t, 16 * g:16 * g + 16],
                              x[SINK + t, 16 * g:16 * g + 16])
    calib.free()


def test_fp16_overflow_sets_range_flag_and_skips_the_record(kv, torch):
    n = 300
    T = SINK + WINDOW + n
    x = np.zeros((T, D), dtype=np.uint16)
    x[SINK:SINK + n] = crafted_rows(n, 4)
    huge = synth.f32_to_bf16_bits(np.array([1e5, -1e5]))
    # token 7 (and 200): a width-1 group's max beyond 65504 makes the scale
    # overflow; token 100: a minimum below -65504 makes the shift overflow
    bad_rows = {7: (4, huge[0]), 100: (2, huge[1]), 200: (4, huge[0])}
    for t, (g, v) in bad_rows.items():
        x[SINK + t, 16 * g + 5] = v
    calib = kv.kvtc_calib_load(identity_blob(), 0)
    nbytes = calib.stream_bytes(0, 0, T)
    dst = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device="cuda")
    kv.kvtc_compress(calib, 0, 1, 1, [to_dev(torch, x), None], D, T, dst,
                     nbytes)
    flags = kv.kvtc_device_status(calib)
    assert flags == kv.KVTC_FLAG_RANGE
    got = dst.cpu().numpy()
    sc_enc = stream_calib("bf16")
    ref = np.frombuffer(codec.compress_stream(x, sc_enc), np.uint8)
    R = sc_enc.R
    off = (SINK + WINDOW) * D * 2
    g_rec = got[off:off + n * R].reshape(n, R)
    o_rec = ref[off:off + n * R].reshape(n, R)
    for t in range(n):
        if t in bad_rows:
            assert np.all(g_rec[t] == 0xAB), f"record {t} was written"
        else:
            assert np.array_equal(g_rec[t], o_rec[t]), f"record {t} differs"
    assert np.array_equal(got[:off], ref[:off])
    # the flag is cleared by reading it, and the context still works
    assert kv.kvtc_device_status(calib) == 0
    calib.free()


def test_random_rows_through_identity_basis(kv, torch):
    """General rows (not exact in any sense) on the identity basis: the
    parity rule holds and the restore is within its tolerance."""
    rng = np.random.default_rng(23)
    T = 1100
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, D)) *
                               np.exp(rng.uniform(-4, 4, (T, 1))))
    sc_enc, sc_dec = stream_calib("bf16"), stream_calib("fp16")
    calib = kv.kvtc_calib_load(identity_blob(), 0)
    nbytes = calib.stream_bytes(0, 0, T)
    dst = torch.zeros((nbytes,), dtype=torch.uint8, device="cuda")
    kv.kvtc_compress(calib, 0, 1, 1, [to_dev(torch, x), None], D, T, dst,
                     nbytes)
    assert kv.kvtc_device_status(calib) == 0
    got = dst.cpu().numpy()
    s_, w_, tc = codec.split_tokens(T, SINK, WINDOW)
    R = sc_enc.R
    off = (s_ + w_) * D * 2
    st = check_records(got[off:off + tc * R].reshape(tc, R),
                       x[s_:s_ + tc], sc_enc)
    record("identity basis, random rows", st=st)
    assert st["bad"] == 0, st
    ref = codec.compress_stream(x, sc_enc)
    out = torch.zeros((T, D), dtype=torch.int16, device="cuda")
    srcd = torch.from_numpy(np.frombuffer(ref, np.uint8).copy()).cuda()
    kv.kvtc_decompress(calib, 0, 1, 1, srcd, len(ref), T, [out, None], D)
    xo = codec.decompress_stream(ref, T, sc_dec)
    ds = check_decompress(out.cpu().numpy().view(np.uint16)[s_:T - w_],
                          xo[s_:T - w_])
    record("identity basis, random rows", dst=ds)
    assert ds["ok"], ds
    calib.free()
