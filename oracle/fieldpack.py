"""Lossless field packing of kvtc records (oracle; test infrastructure).

The kvtc page ("KV Cache Transform Coding for Compact Storage in LLM
Inference", technical summary 2B) follows quantisation and bit-packing with
a lossless entropy stage (DEFLATE through nvCOMP).  This module is a
lossless stage of our own, aimed at the part of a record that carries
redundancy: the high byte of each fp16 field (sign, exponent and the two top
mantissa bits).  Within one field slot -- the shift or the scale of one
active group -- the sign and exponent of a stream's tokens span a narrow
range, so each is stored as a fixed-width offset from the slot's minimum over
the stream.  Everything else in the record is kept bit for bit, and the
record's zero padding is dropped.

Packed stream of one (layer, K|V), little-endian:
  header      b"KVFP", u32 T_c, u16 Rp (packed record bytes),
              u16 nslot (= 2 G_a), u32 0                          16 bytes
  slot table  per slot s: u8 vmin_s, u8 dbits_s; zero-padded so that
              header and table together fill a multiple of 128 bytes
  raw rows    the sink and window rows, unchanged ((s'+w') x 2D bytes)
  records     T_c packed records of Rp bytes
  padding     zeros to a multiple of 256 bytes
Slot s = 2a is the shift of active group a (record byte 4a + 1 holds its
high byte), s = 2a + 1 its scale (byte 4a + 3).  With h the high byte,
v = h >> 2 (sign and exponent), vmin_s / vmax_s the least / greatest v of
slot s over the stream's tokens and dbits_s the bit length of
vmax_s - vmin_s (0 when T_c = 0).
Packed record of one token:
  the low bytes of its fields in slot order                       2 G_a B
  the high-byte codes: for s = 0 .. nslot - 1, h - 4 vmin_s in
  dbits_s + 2 bits (its low 2 bits are h & 3, the others v - vmin_s),
  packed least significant bit first into 2 ceil(sum_s (dbits_s + 2) / 16)
  bytes (unused high bits zero)
  the bit-planes, record bytes [4 G_a, used)
  zero bytes to a multiple of 4
Every part has an even number of bytes, so a packed record keeps the
16-bit alignment of the bit-planes, and its length is a multiple of 4.
Before that last padding it never exceeds the used bytes of a record
(dbits_s <= 6, so the codes take at most 16 G_a bits), so Rp <= R.  The
128-byte prefix and the 4-byte record length are layout choices of this
format: a stream's records start on a 128-byte boundary of the stream and
32 consecutive records span whole 128-byte lines.
"""
from __future__ import annotations

from typing import Tuple

import numpy as np

from . import codec

MAGIC = b"KVFP"
HEADER = 16


def _hi_lo(records: np.ndarray, ga: int) -> Tuple[np.ndarray, np.ndarray]:
    """High and low bytes of the 2 G_a fields, slot order: [n][2 G_a]."""
    idx = np.empty(2 * ga, dtype=np.int64)
    idx[0::2] = 4 * np.arange(ga)        # shift
    idx[1::2] = 4 * np.arange(ga) + 2    # scale
    return records[:, idx + 1], records[:, idx]


def slot_table(records: np.ndarray, ga: int) -> Tuple[np.ndarray, np.ndarray]:
    """(vmin, dbits) per slot over the stream's tokens."""
    if records.shape[0] == 0:
        z = np.zeros(2 * ga, dtype=np.int64)
        return z, z.copy()
    hi, _ = _hi_lo(records, ga)
    v = hi.astype(np.int64) >> 2
    vmin, vmax = v.min(axis=0), v.max(axis=0)
    dbits = np.array([int(d).bit_length() for d in vmax - vmin],
                     dtype=np.int64)
    return vmin, dbits


def code_bytes(dbits: np.ndarray) -> int:
    """Bytes of the high-byte codes of one token (a multiple of 2)."""
    hbits = int((np.asarray(dbits) + 2).sum())
    return 2 * (-(-hbits // 16))


def packed_record_bytes(bits: np.ndarray, dbits: np.ndarray) -> int:
    ga = len(bits)
    _, _, used = codec.record_layout(bits)
    n = 2 * ga + code_bytes(dbits) + (used - 4 * ga)
    return -(-n // 4) * 4


def pack_records(records: np.ndarray, bits: np.ndarray):
    """records uint8 [n][R] -> (vmin, dbits, packed uint8 [n][Rp])."""
    n = records.shape[0]
    ga = len(bits)
    _, _, used = codec.record_layout(bits)
    vmin, dbits = slot_table(records, ga)
    rp = packed_record_bytes(bits, dbits)
    out = np.zeros((n, rp), dtype=np.uint8)
    if n == 0:
        return vmin, dbits, out
    hi, lo = _hi_lo(records, ga)
    out[:, :2 * ga] = lo
    # code bits of every token, least significant first, slot after slot
    cols = []
    for s in range(2 * ga):
        c = hi[:, s].astype(np.int64) - 4 * vmin[s]
        for b in range(int(dbits[s]) + 2):
            cols.append((c >> b) & 1)
    hbytes = code_bytes(dbits)
    bitmat = np.zeros((n, 8 * hbytes), dtype=np.uint8)
    if cols:
        bitmat[:, :len(cols)] = np.stack(cols, axis=1)
    hb = np.packbits(bitmat, axis=1, bitorder="little")
    out[:, 2 * ga:2 * ga + hbytes] = hb
    out[:, 2 * ga + hbytes:2 * ga + hbytes + used - 4 * ga] = \
        records[:, 4 * ga:used]
    return vmin, dbits, out


def unpack_records(packed: np.ndarray, bits: np.ndarray, vmin: np.ndarray,
                   dbits: np.ndarray, R: int) -> np.ndarray:
    """Inverse of :func:`pack_records`: uint8 [n][R] with zero padding."""
    n = packed.shape[0]
    ga = len(bits)
    _, _, used = codec.record_layout(bits)
    rec = np.zeros((n, R), dtype=np.uint8)
    if n == 0:
        return rec
    hbits = int((np.asarray(dbits) + 2).sum())
    hbytes = code_bytes(dbits)
    bitmat = np.unpackbits(packed[:, 2 * ga:2 * ga + hbytes], axis=1,
                           bitorder="little")[:, :hbits].astype(np.int64)
    pos = 0
    for s in range(2 * ga):
        c = np.zeros(n, dtype=np.int64)
        for b in range(int(dbits[s]) + 2):
            c |= bitmat[:, pos] << b
            pos += 1
        h = c + 4 * vmin[s]
        a, which = divmod(s, 2)
        rec[:, 4 * a + 2 * which + 1] = h.astype(np.uint8)
        rec[:, 4 * a + 2 * which] = packed[:, s]
    rec[:, 4 * ga:used] = \
        packed[:, 2 * ga + hbytes:2 * ga + hbytes + used - 4 * ga]
    return rec


def _table_bytes(nslot: int) -> int:
    """Slot table bytes: header and table fill a multiple of 128 bytes."""
    return -(-(HEADER + 2 * nslot) // 128) * 128 - HEADER


def pack_stream(buf: bytes, T: int, sc: codec.StreamCalib) -> bytes:
    """One compressed stream -> its packed form."""
    s_, w_, tc = codec.split_tokens(T, sc.sink, sc.window)
    raw = (s_ + w_) * sc.D * 2
    rec = codec.stream_records(buf, T, sc)
    vmin, dbits, packed = pack_records(rec, sc.bits)
    rp = packed_record_bytes(sc.bits, dbits)
    nslot = 2 * len(sc.bits)
    head = MAGIC + np.array([tc], "<u4").tobytes() + \
        np.array([rp, nslot], "<u2").tobytes() + bytes(4)
    table = np.zeros(_table_bytes(nslot), dtype=np.uint8)
    table[0:2 * nslot:2] = vmin
    table[1:2 * nslot:2] = dbits
    body = head + table.tobytes() + buf[:raw] + packed.tobytes()
    n = -(-len(body) // codec.STREAM_ALIGN) * codec.STREAM_ALIGN
    return body + bytes(n - len(body))


def unpack_stream(pbuf: bytes, T: int, sc: codec.StreamCalib) -> bytes:
    """Packed stream -> the compressed stream it came from."""
    assert pbuf[:4] == MAGIC
    tc = int(np.frombuffer(pbuf, "<u4", 1, 4)[0])
    rp, nslot = (int(v) for v in np.frombuffer(pbuf, "<u2", 2, 8))
    s_, w_, tc2 = codec.split_tokens(T, sc.sink, sc.window)
    assert tc == tc2 and nslot == 2 * len(sc.bits)
    table = np.frombuffer(pbuf, np.uint8, 2 * nslot, HEADER)
    vmin = table[0::2].astype(np.int64)
    dbits = table[1::2].astype(np.int64)
    raw = (s_ + w_) * sc.D * 2
    off = HEADER + _table_bytes(nslot)
    packed = np.frombuffer(pbuf, np.uint8, tc * rp, off + raw).reshape(tc, rp)
    rec = unpack_records(packed, sc.bits, vmin, dbits, sc.R)
    out = bytearray(codec.stream_bytes(T, sc.D, sc.sink, sc.window,
                                       sc.budget_bits))
    out[:raw] = pbuf[off:off + raw]
    out[raw:raw + rec.size] = rec.tobytes()
    return bytes(out)


def packed_stream_bytes(T: int, sc: codec.StreamCalib, rp: int) -> int:
    s_, w_, tc = codec.split_tokens(T, sc.sink, sc.window)
    n = HEADER + _table_bytes(2 * len(sc.bits)) + (s_ + w_) * sc.D * 2 + \
        tc * rp
    return -(-n // codec.STREAM_ALIGN) * codec.STREAM_ALIGN
