"""Pins for the oracle's quantiser, record packing and stream codec."""
import json
import os

import numpy as np
import pytest

import synth
from oracle import calibrate, codec, fp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------- golden record
def test_golden_record_pack_and_unpack():
    g = load("record_example.json")
    c = np.array(g["coefficients"], dtype=np.float64)[None, :]
    bits = np.array(g["widths"])
    qz = codec.quantise(c, bits)
    np.testing.assert_array_equal(qz.q[0], g["codes"])
    rec = codec.pack(qz.shift, qz.scale, qz.q, bits,
                     codec.record_bytes(g["budget_bits"]))
    assert rec.tobytes().hex() == g["record_hex"]
    shift, scale, q = codec.unpack(rec, bits)
    np.testing.assert_array_equal(q[0], g["codes"])
    chat = codec.dequantise(shift, scale, q)
    np.testing.assert_array_equal(chat, c)


def test_golden_record_decompress_identity_basis():
    g = load("record_example.json")
    D = 32
    sc = codec.StreamCalib(mu=np.zeros(D), basis=np.eye(D),
                           widths=np.array(g["widths"]), sink=0, window=0,
                           budget_bits=g["budget_bits"])
    buf = bytes.fromhex(g["record_hex"])
    buf = buf + bytes(codec.stream_bytes(1, D, 0, 0, g["budget_bits"])
                      - len(buf))
    out = codec.decompress_stream(buf, 1, sc)
    exp = np.array([int(h, 16) for h in g["identity_basis_bf16_hex"]],
                   dtype=np.uint16)
    np.testing.assert_array_equal(out[0], exp)


def test_page_facts():
    f = load("page_facts.json")
    w = synth.WORKLOADS["llama31_8b_8k"]
    per_token = len(w.streams()) * w.D * 2
    assert per_token * 1024 == f["kv_bytes_per_1k_tokens_llama31_8b"]["value"]
    # 1 bit per coefficient -> one record is 1/16 of the bf16 row
    assert w.D * 2 // codec.record_bytes(w.budget_bits) == \
        f["pre_deflate_ratio_at_1_bit"]["value"]
    assert w.sink == f["attention_sinks"]["value"]


# --------------------------------------------------------------- quantiser
@pytest.mark.parametrize("b", range(1, 9))
def test_quantiser_half_step_bound(b):
    rng = np.random.default_rng(10 + b)
    n, ga = 500, 3
    scale_mag = 10.0 ** rng.uniform(-4, 2, (n, ga, 1))
    c = (rng.standard_normal((n, ga, 16)) * scale_mag).reshape(n, ga * 16)
    bits = np.full(ga, b)
    qz = codec.quantise(c, bits)
    assert not qz.range_error
    assert qz.q.max() <= 2 ** b - 1
    chat = codec.dequantise(qz.shift, qz.scale, qz.q)
    step = np.repeat(qz.scale.astype(np.float64), 16, axis=1)
    err = np.abs(c - chat)
    assert np.all(err <= step / 2 * (1 + 1e-12) + 1e-300)
    # fields bracket the group's range
    cg = c.reshape(n, ga, 16)
    s64 = qz.shift.astype(np.float64)
    assert np.all(s64 <= cg.min(axis=2))
    assert np.all(s64 + (2 ** b - 1) * qz.scale.astype(np.float64)
                  >= cg.max(axis=2))
    # the fields are the tightest fp16 values with that property
    assert np.all(np.nextafter(qz.shift, np.float16(np.inf)).astype(
        np.float64) > cg.min(axis=2))


def test_quantiser_constant_group_and_rounding_rule():
    # exactly representable constant: scale 0, codes 0, exact reconstruction
    c = np.full((2, 16), 0.375)
    c[1] = -7.0
    qz = codec.quantise(c, np.array([3]))
    assert np.all(qz.scale.astype(np.float64) == 0)
    assert np.all(qz.q == 0)
    np.testing.assert_array_equal(
        codec.dequantise(qz.shift, qz.scale, qz.q), c)
    # half-way values round up: shift 0, scale 1, values k + 1/2
    c = np.array([[0.0, 0.5, 1.5, 2.5, 3.0] + [0.0] * 11])
    qz = codec.quantise(c, np.array([2]))
    assert qz.shift[0, 0] == 0 and qz.scale[0, 0] == 1.0
    np.testing.assert_array_equal(qz.q[0, :5], [0, 1, 2, 3, 3])


def test_quantiser_flags_fp16_overflow():
    c = np.zeros((1, 16))
    c[0, 3] = -70000.0
    assert codec.quantise(c, np.array([4])).range_error
    c = np.zeros((1, 16))
    c[0, 3] = 65504.0
    c[0, 4] = -65504.0
    assert codec.quantise(c, np.array([1])).range_error  # scale > max


# ----------------------------------------------------------------- packing
def test_pack_unpack_round_trip_random_widths():
    rng = np.random.default_rng(3)
    for trial in range(50):
        ga = int(rng.integers(1, 9))
        bits = rng.integers(1, 9, ga)
        used = int((32 + 16 * bits).sum())
        R = codec.record_bytes(used + int(rng.integers(0, 300)))
        n = 17
        q = np.concatenate([rng.integers(0, 2 ** b, (n, 16)) for b in bits],
                           axis=1).astype(np.uint16)
        shift = rng.standard_normal((n, ga)).astype(np.float16)
        scale = np.abs(rng.standard_normal((n, ga))).astype(np.float16)
        rec = codec.pack(shift, scale, q, bits, R)
        assert rec.shape == (n, R)
        _, _, nbytes = codec.record_layout(bits)
        assert nbytes * 8 == used
        assert np.all(rec[:, nbytes:] == 0)  # zero padding
        s2, d2, q2 = codec.unpack(rec, bits)
        np.testing.assert_array_equal(q2, q)
        np.testing.assert_array_equal(fp.fp16_bits(s2), fp.fp16_bits(shift))
        np.testing.assert_array_equal(fp.fp16_bits(d2), fp.fp16_bits(scale))


# ------------------------------------------------------- stream: raw tokens
@pytest.fixture(scope="module")
def tiny_calib():
    w = synth.WORKLOADS["tiny"]
    cb = synth.calib_tokens(w, 0, 0)
    mu, V, evals, widths, E = calibrate.calibrate_stream(cb, w.budget_bits)
    return w, mu, V, evals, widths, E


@pytest.mark.parametrize("T", [0, 1, 3, 4, 5, 19, 20, 21, 147, 256])
def test_sink_window_pass_through(tiny_calib, T):
    w, mu, V, evals, widths, E = tiny_calib
    cols = codec.active_columns(widths)
    sc = codec.StreamCalib(mu, V[:, cols], widths, w.sink, w.window,
                           w.budget_bits)
    x = synth.eval_tokens(w, 0, 0, T=T)
    buf = codec.compress_stream(x, sc)
    assert len(buf) == codec.stream_bytes(T, w.D, w.sink, w.window,
                                          w.budget_bits)
    assert len(buf) % codec.STREAM_ALIGN == 0
    out = codec.decompress_stream(buf, T, sc)
    s_, w_, tc = codec.split_tokens(T, w.sink, w.window)
    assert s_ + w_ + tc == T and tc >= 0
    np.testing.assert_array_equal(out[:s_], x[:s_])
    np.testing.assert_array_equal(out[T - w_:], x[T - w_:])
    if tc:
        # compressed rows are not copies
        assert not np.array_equal(out[s_:T - w_], x[s_:T - w_])


# ------------------------------------------------------------ Parseval etc.
def test_parseval_full_and_dropped(tiny_calib):
    w, mu, V, evals, widths, E = tiny_calib
    x_bits = synth.eval_tokens(w, 0, 0)
    x = fp.bf16_bits_to_f64(x_bits)
    for wd in (np.full(w.D // 16, 8), widths):
        cols = codec.active_columns(wd)
        sc = codec.StreamCalib(mu, V[:, cols], wd, 0, 0, w.budget_bits * 8)
        c_all = (x - mu) @ V
        c = c_all[:, cols]
        qz = codec.quantise(c, sc.bits)
        rec = codec.pack(qz.shift, qz.scale, qz.q, sc.bits, sc.R)
        xh = codec.reconstruct(rec, sc)
        chat = codec.dequantise(qz.shift, qz.scale, qz.q)
        lhs = ((x - xh) ** 2).sum()
        dropped = np.setdiff1d(np.arange(w.D), cols)
        rhs = ((c - chat) ** 2).sum() + (c_all[:, dropped] ** 2).sum()
        assert abs(lhs - rhs) <= 1e-9 * rhs
        # each coefficient within half a step
        step = np.repeat(qz.scale.astype(np.float64), 16, axis=1)
        assert np.all(np.abs(c - chat) <= step / 2 * (1 + 1e-12))


def test_all_eight_bits_full_rank_is_accurate(tiny_calib):
    w, mu, V, evals, widths, E = tiny_calib
    wd = np.full(w.D // 16, 8)
    sc = codec.StreamCalib(mu, V, wd, w.sink, w.window, w.D * 16)
    x = synth.eval_tokens(w, 0, 0)
    out = codec.decompress_stream(codec.compress_stream(x, sc), 256, sc,
                                  exact=True)
    xf = fp.bf16_bits_to_f64(x)
    c = (xf - mu) @ V
    rng_g = (c.reshape(256, -1, 16).max(2) - c.reshape(256, -1, 16).min(2))
    err = np.abs(out - xf)[w.sink:256 - w.window]
    # error norm is at most half a step per coefficient (Parseval)
    bound = np.sqrt(((rng_g / 255 / 2) ** 2 * 16).sum(1))[w.sink:256 - w.window]
    assert np.all(np.sqrt((err ** 2).sum(1)) <= bound * 1.01 + 1e-3)


# --------------------------------------------------------------- paged write
def test_paged_write_identity_table_is_a_reshape():
    """With block table 0, 1, 2, ... the pool is the rows cut into blocks."""
    rng = np.random.default_rng(9)
    T, bs, D = 50, 16, 8
    rows = rng.integers(0, 2 ** 16, (T, D)).astype(np.uint16)
    nb = -(-T // bs)
    pool = np.full((nb, bs, D), 0xFFFF, dtype=np.uint16)
    codec.paged_write(pool, rows, np.arange(nb), bs)
    flat = pool.reshape(nb * bs, D)
    np.testing.assert_array_equal(flat[:T], rows)
    assert np.all(flat[T:] == 0xFFFF)          # the ragged block's tail


def test_paged_write_permuted_table_inverse():
    """Every pool row holds the token its block and slot name; blocks the
    table does not name are untouched."""
    rng = np.random.default_rng(10)
    T, bs, D = 77, 16, 4
    rows = np.arange(T * D, dtype=np.uint16).reshape(T, D)
    nb_used = -(-T // bs)
    table = rng.permutation(12)[:nb_used]
    pool = np.full((12, bs, D), 0xFFFF, dtype=np.uint16)
    codec.paged_write(pool, rows, table, bs)
    for j, blk in enumerate(table):
        for slot in range(bs):
            t = j * bs + slot
            if t < T:
                np.testing.assert_array_equal(pool[blk, slot], rows[t])
            else:
                assert np.all(pool[blk, slot] == 0xFFFF)
    for blk in set(range(12)) - set(table.tolist()):
        assert np.all(pool[blk] == 0xFFFF)
