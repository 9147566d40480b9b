"""Pins for the oracle's lossless field packing (oracle/fieldpack.py).

The stage is lossless, so its first pin is the identity it must satisfy:
unpacking gives back every byte of the compressed stream.  The packed bytes
themselves are pinned by a hand-worked example (tests/golden) and by a
brute-force construction of each token's code bits as a character string,
written independently of the oracle's array arithmetic.
"""
import json
import os

import numpy as np
import pytest

import synth
from oracle import calibrate, codec, fieldpack

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_golden_example_pack_unpack():
    g = load("fieldpack_example.json")
    bits = np.array([b for b in g["widths"] if b > 0])
    R = codec.record_bytes(g["budget_bits"])
    rec = np.array([list(bytes.fromhex(h)) for h in g["records_hex"]],
                   dtype=np.uint8)
    assert rec.shape == (2, R)
    vmin, dbits, packed = fieldpack.pack_records(rec, bits)
    assert list(vmin) == g["vmin"] and list(dbits) == g["dbits"]
    assert packed.shape[1] == g["packed_record_bytes"]
    assert [r.tobytes().hex() for r in packed] == g["packed_records_hex"]
    back = fieldpack.unpack_records(packed, bits, vmin, dbits, R)
    np.testing.assert_array_equal(back, rec)


def test_golden_example_stream():
    g = load("fieldpack_example.json")
    D = 32
    sc = codec.StreamCalib(mu=np.zeros(D), basis=np.eye(D),
                           widths=np.array(g["widths"]), sink=0, window=0,
                           budget_bits=g["budget_bits"])
    buf = b"".join(bytes.fromhex(h) for h in g["records_hex"])
    buf += bytes(codec.stream_bytes(2, D, 0, 0, g["budget_bits"]) - len(buf))
    pbuf = fieldpack.pack_stream(buf, 2, sc)
    assert len(pbuf) == g["stream_bytes"]
    pre = bytes.fromhex(g["stream_prefix_hex"])
    assert pbuf[:len(pre)] == pre
    assert pbuf[len(pre):] == bytes(len(pbuf) - len(pre))
    assert fieldpack.unpack_stream(pbuf, 2, sc) == buf


def _brute_codes(rec_row, bits, vmin, dbits):
    """Code bytes of one token built as a string of '0'/'1' characters:
    per slot the two low bits of the high byte, then its sign/exponent
    offset from the slot's minimum, least significant bit first."""
    ga = len(bits)
    s = ""
    for a in range(ga):
        for byte in (4 * a + 1, 4 * a + 3):          # shift, scale high bytes
            slot = 2 * a + (byte - 4 * a - 1) // 2
            h = int(rec_row[byte])
            u = h // 4 - int(vmin[slot])
            assert 0 <= u < 2 ** int(dbits[slot]) or (u == 0 and
                                                      dbits[slot] == 0)
            s += format(h % 4, "02b")[::-1]
            s += format(u, "b").zfill(int(dbits[slot]))[::-1] \
                if dbits[slot] else ""
    while len(s) % 16:
        s += "0"
    return bytes(int(s[i:i + 8][::-1], 2) for i in range(0, len(s), 8))


def _random_records(rng, n, bits, R, spread):
    """Records with random fields whose sign/exponent span `spread` values."""
    ga = len(bits)
    _, _, used = codec.record_layout(bits)
    rec = np.zeros((n, R), dtype=np.uint8)
    rec[:, :used] = rng.integers(0, 256, (n, used))
    for a in range(ga):
        for byte in (4 * a + 1, 4 * a + 3):
            base = int(rng.integers(0, 64 - spread + 1))
            v = base + rng.integers(0, spread, n)
            rec[:, byte] = (v << 2) | rng.integers(0, 4, n)
    return rec


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_codes_and_layout(seed):
    rng = np.random.default_rng(seed)
    for _ in range(8):
        ga = int(rng.integers(1, 16))
        bits = rng.integers(1, 9, ga)
        _, _, used = codec.record_layout(bits)
        R = 16 * -(-used // 16)
        n = int(rng.integers(1, 9))
        spread = int(rng.choice([1, 2, 3, 5, 17, 64]))
        rec = _random_records(rng, n, bits, R, spread)
        vmin, dbits, packed = fieldpack.pack_records(rec, bits)
        for s in range(2 * ga):
            col = rec[:, 4 * (s // 2) + 1 + 2 * (s % 2)] // 4
            assert vmin[s] == col.min()
            assert dbits[s] == int(col.max() - col.min()).bit_length()
        hb = len(_brute_codes(rec[0], bits, vmin, dbits))
        body = 2 * ga + hb + used - 4 * ga
        assert packed.shape[1] == body + (-body) % 4
        for t in range(n):
            row = packed[t]
            lo = bytes(rec[t, [4 * (s // 2) + 2 * (s % 2)
                               for s in range(2 * ga)]])
            assert row[:2 * ga].tobytes() == lo
            assert row[2 * ga:2 * ga + hb].tobytes() == \
                _brute_codes(rec[t], bits, vmin, dbits)
            assert row[2 * ga + hb:body].tobytes() == \
                rec[t, 4 * ga:used].tobytes()
            assert not row[body:].any()
        back = fieldpack.unpack_records(packed, bits, vmin, dbits, R)
        np.testing.assert_array_equal(back, rec)


def test_packed_record_never_larger_and_word_sized():
    rng = np.random.default_rng(11)
    for _ in range(200):
        ga = int(rng.integers(1, 16))
        bits = rng.integers(1, 9, ga)
        dbits = rng.integers(0, 7, 2 * ga)
        _, _, used = codec.record_layout(bits)
        rp = fieldpack.packed_record_bytes(bits, dbits)
        assert rp % 4 == 0 and rp <= used + (-used) % 4
        assert rp <= 16 * -(-used // 16)           # never longer than R
    # worst case: every slot's sign/exponent spans all 64 values; used is
    # 4 * 3 + 2 * 6 = 24 bytes
    bits = np.array([1, 2, 3])
    assert fieldpack.packed_record_bytes(bits, np.full(6, 6)) == 24
    # used = 4 + 2 = 6 bytes, codes of 2 slots x 8 bits: 2 + 2 + 2 -> 8
    assert fieldpack.packed_record_bytes(np.array([1]), np.full(2, 6)) == 8


def test_constant_fields_cost_two_bits_per_slot():
    bits = np.array([2, 2, 2, 2])
    rec = np.zeros((5, 48), dtype=np.uint8)
    rec[:, 1::2][:, :8] = 0x3C           # every high byte equal
    _, dbits, packed = fieldpack.pack_records(rec, bits)
    assert dbits.sum() == 0
    assert fieldpack.code_bytes(dbits) == 2   # 8 slots x 2 bits
    assert packed.shape[1] == 8 + 2 + 16 + 2  # padded to a multiple of 4


@pytest.fixture(scope="module")
def tiny_sc():
    w = synth.WORKLOADS["tiny"]
    cb = synth.calib_tokens(w, 0, 0)
    mu, V, _, widths, _ = calibrate.calibrate_stream(cb, w.budget_bits)
    cols = codec.active_columns(widths)
    return w, codec.StreamCalib(mu, V[:, cols], widths, w.sink, w.window,
                                w.budget_bits)


@pytest.mark.parametrize("T", [0, 1, 4, 20, 21, 147, 256])
def test_stream_round_trip_is_lossless(tiny_sc, T):
    w, sc = tiny_sc
    x = synth.eval_tokens(w, 0, 0, T=T)
    buf = codec.compress_stream(x, sc)
    pbuf = fieldpack.pack_stream(buf, T, sc)
    assert len(pbuf) % codec.STREAM_ALIGN == 0
    assert pbuf[:4] == fieldpack.MAGIC
    rp = int(np.frombuffer(pbuf, "<u2", 1, 8)[0])
    assert len(pbuf) == fieldpack.packed_stream_bytes(T, sc, rp)
    assert fieldpack.unpack_stream(pbuf, T, sc) == buf
    s_, w_, tc = codec.split_tokens(T, sc.sink, sc.window)
    off = 128 * -(-(16 + 4 * len(sc.bits)) // 128)   # header + table
    assert off % 128 == 0
    assert pbuf[off:off + (s_ + w_) * sc.D * 2] == buf[:(s_ + w_) * sc.D * 2]


def test_real_stream_gets_smaller():
    """A Llama-3.1-8B-shaped stream (D = 1024, 128-byte records): the
    sign/exponent of every field spans at most 16 values over 512 tokens, so
    the packed record is shorter than the used bytes."""
    w = synth.WORKLOADS["llama31_8b_8k"]
    cb = synth.calib_tokens(w, 0, 0)
    mu, V, _, widths, _ = calibrate.calibrate_stream(cb, w.budget_bits)
    sc = codec.StreamCalib(mu, V[:, codec.active_columns(widths)], widths,
                           w.sink, w.window, w.budget_bits)
    T = 512
    buf = codec.compress_stream(synth.eval_tokens(w, 0, 0, T=T), sc)
    rec = codec.stream_records(buf, T, sc)
    _, dbits, packed = fieldpack.pack_records(rec, sc.bits)
    _, _, used = codec.record_layout(sc.bits)
    assert dbits.max() <= 4
    assert packed.shape[1] < used <= sc.R
    pbuf = fieldpack.pack_stream(buf, T, sc)
    assert len(pbuf) < len(buf)
    assert fieldpack.unpack_stream(pbuf, T, sc) == buf
