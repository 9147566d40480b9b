"""Pins for the parity checker used by the GPU tests: records made by the
oracle pass, and records with a planted mistake (made on the CPU, in the
oracle's output) are caught."""
import numpy as np
import pytest

import synth
from oracle import calibrate, codec, fp

from _parity import check_decompress, check_records


@pytest.fixture(scope="module")
def case():
    w = synth.WORKLOADS["llama31_8b_8k"]
    cb = synth.calib_tokens(w, 2, 0)
    mu, V, evals, widths, _ = calibrate.calibrate_stream(cb, w.budget_bits)
    blob = calibrate.write_blob([(2, 0, mu, V, evals, widths)], w.sink,
                                w.window, w.budget_bits)
    e = calibrate.read_blob(blob)["streams"][0]
    sc = calibrate.stream_calib(e, w.sink, w.window, w.budget_bits, "bf16")
    x = synth.eval_tokens(w, 2, 0, T=300)
    c = codec.coefficients(x, sc)
    qz = codec.quantise(c, sc.bits)
    rec = codec.pack(qz.shift, qz.scale, qz.q, sc.bits, sc.R)
    return sc, x, c, qz, rec


def test_oracle_records_pass(case):
    sc, x, c, qz, rec = case
    st = check_records(rec, x, sc)
    assert st["bad"] == 0 and st["code_flips"] == 0 and st["field_flips"] == 0


def far_from_boundary(c, qz, sc):
    """(token, component) whose code is at least 0.3 steps from a rounding
    boundary and not at either end of its range."""
    n = c.shape[0]
    ga = sc.bits.size
    s = np.repeat(qz.shift.astype(float), 16, axis=1)
    d = np.repeat(qz.scale.astype(float), 16, axis=1)
    u = (c - s) / np.where(d > 0, d, 1)
    frac = u + 0.5 - np.floor(u + 0.5)
    lev = np.repeat(2 ** sc.bits - 1, 16)[None, :]
    ok = (np.minimum(frac, 1 - frac) > 0.3) & (qz.q > 0) & (qz.q < lev) & \
        (d > 0)
    t, j = np.argwhere(ok)[0]
    return int(t), int(j)


def test_planted_code_flip_is_caught(case):
    sc, x, c, qz, rec = case
    t, j = far_from_boundary(c, qz, sc)
    q = qz.q.copy()
    q[t, j] += 1
    bad = codec.pack(qz.shift, qz.scale, q, sc.bits, sc.R)
    assert check_records(bad, x, sc)["code_bad"] >= 1


def step16(h, n, direction):
    for _ in range(n):
        h = np.nextafter(h, np.float16(direction))
    return h


def test_planted_field_change_is_caught(case):
    """A field moved by 32 fp16 steps (far outside any window: the window
    is at most the fp32 accumulation bound, a few fp16 steps for this K
    stream with outlier channels)."""
    sc, x, c, qz, rec = case
    shift = qz.shift.copy()
    shift[5, 0] = step16(shift[5, 0], 32, -np.inf)
    bad = codec.pack(shift, qz.scale, qz.q, sc.bits, sc.R)
    assert check_records(bad, x, sc)["field_bad"] >= 1
    scale = qz.scale.copy()
    scale[7, 1] = step16(scale[7, 1], 32, np.inf)
    bad = codec.pack(qz.shift, scale, qz.q, sc.bits, sc.R)
    assert check_records(bad, x, sc)["field_bad"] >= 1


def test_planted_two_step_code_error_is_caught(case):
    sc, x, c, qz, rec = case
    q = qz.q.copy()
    lev = np.repeat(2 ** sc.bits - 1, 16)
    t, j = np.argwhere((q >= 2) & (q <= lev[None, :]))[0]
    q[t, j] -= 2
    bad = codec.pack(qz.shift, qz.scale, q, sc.bits, sc.R)
    assert check_records(bad, x, sc)["code_bad"] >= 1


def test_decompress_rule():
    o = fp.bf16_rne_bits(np.linspace(-3, 3, 1000))
    assert check_decompress(o, o)["ok"]
    g = o.copy()
    g[10] += 3  # three bf16 ulps
    assert not check_decompress(g, o)["ok"]
