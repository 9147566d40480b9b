"""kvtc transform codec in fp64 (oracle).

Follows the kvtc page ("KV Cache Transform Coding for Compact Storage in LLM
Inference"), Technical summary section 2:
  A  calibration -- tokens [0, s) (attention sinks) and the last w tokens
     (sliding window) are not compressed; components share a scale and a
     shift per group ("microscaling");
  B  compression -- subtract the mean, multiply by the basis V, quantise the
     coefficients with the DP-chosen widths, pack the integers;
  C  decompression -- dequantise, multiply by V^T, add the mean back.
The DEFLATE stage of part B/C is not part of this path.

Readings where the page is silent (all listed in the design notes):
  * one width per 16-component group (the group shares its fields, so it
    shares its width); width 0 drops the group (reconstructs as 0, the mean of
    a centred coefficient);
  * shift = fp16 round-down of the group minimum, scale = fp16 round-up of
    (max - shift) / (2^b - 1); code q = clamp(floor((c - shift)/scale + 1/2),
    0, 2^b - 1), q = 0 when scale = 0; reconstruction shift + q * scale;
  * record of one token: for each active group in ascending order its fp16
    shift then fp16 scale (2 x u16), then for each active group in ascending
    order its b bit-planes (u16 each; bit i of plane j is bit j of the code of
    the group's i-th component), then zero padding to R = 16 * ceil(B / 128)
    bytes; little-endian;
  * stream of one (request, layer, K|V): sink rows, then window rows (raw
    bf16), then the T_c records in token order; each stream starts on a
    256-byte boundary.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Tuple

import numpy as np

from . import fp

GROUP = 16
STREAM_ALIGN = 256


# ---------------------------------------------------------------- geometry
def split_tokens(T: int, s: int, w: int) -> Tuple[int, int, int]:
    """(s', w', T_c): sink rows kept, window rows kept, compressed rows."""
    s_ = min(s, T)
    w_ = min(w, T - s_)
    return s_, w_, T - s_ - w_


def record_bytes(budget_bits: int) -> int:
    return 16 * (-(-budget_bits // 128))


def stream_bytes(T: int, D: int, s: int, w: int, budget_bits: int) -> int:
    """Bytes of one stream, rounded up to the stream alignment."""
    s_, w_, tc = split_tokens(T, s, w)
    n = (s_ + w_) * D * 2 + tc * record_bytes(budget_bits)
    return -(-n // STREAM_ALIGN) * STREAM_ALIGN


def active_groups(widths: np.ndarray) -> np.ndarray:
    return np.nonzero(np.asarray(widths) > 0)[0]


def active_columns(widths: np.ndarray, group: int = GROUP) -> np.ndarray:
    """Component indices kept (ascending): all members of active groups."""
    g = active_groups(widths)
    return (g[:, None] * group + np.arange(group)[None, :]).reshape(-1)


# --------------------------------------------------------------- quantiser
@dataclasses.dataclass
class Quantised:
    shift: np.ndarray   # fp16 [n][Ga]
    scale: np.ndarray   # fp16 [n][Ga]
    q: np.ndarray       # uint16 codes [n][Ga*16]
    range_error: bool   # a field left the finite fp16 range


def quantise(c: np.ndarray, bits: np.ndarray, group: int = GROUP) -> Quantised:
    """Microscaled quantisation of active coefficients.

    c: fp64 [n][Ga*group], the coefficients of the active groups only, in
    ascending group order; bits: widths (>= 1) of those groups."""
    c = np.asarray(c, dtype=np.float64)
    bits = np.asarray(bits, dtype=np.int64)
    n = c.shape[0]
    ga = bits.shape[0]
    cg = c.reshape(n, ga, group)
    lo = cg.min(axis=2)
    hi = cg.max(axis=2)
    levels = (2.0 ** bits - 1.0)[None, :]
    shift = fp.fp16_rd(lo)
    with np.errstate(over="ignore", invalid="ignore"):
        scale = fp.fp16_ru((hi - shift.astype(np.float64)) / levels)
    bad = bool(np.any(~np.isfinite(shift)) or np.any(~np.isfinite(scale)))
    s64 = shift.astype(np.float64)[:, :, None]
    d64 = scale.astype(np.float64)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        u = (cg - s64) / d64
    q = np.floor(u + 0.5)
    q = np.where(d64 > 0, q, 0.0)
    q = np.clip(q, 0.0, levels[:, :, None])
    q = np.nan_to_num(q, nan=0.0)
    return Quantised(shift, scale, q.astype(np.uint16).reshape(n, ga * group),
                     bad)


def dequantise(shift: np.ndarray, scale: np.ndarray, q: np.ndarray,
               group: int = GROUP) -> np.ndarray:
    """c_hat = shift + q * scale (exact in fp64) for the active groups."""
    n, ga = shift.shape
    qg = np.asarray(q, dtype=np.float64).reshape(n, ga, group)
    r = (shift.astype(np.float64)[:, :, None]
         + qg * scale.astype(np.float64)[:, :, None])
    return r.reshape(n, ga * group)


# ----------------------------------------------------------------- packing
def record_layout(bits: np.ndarray) -> Tuple[np.ndarray, np.ndarray, int]:
    """Byte offsets of each active group's (shift, scale) pair and of its
    first bit-plane, and the number of bytes used."""
    bits = np.asarray(bits, dtype=np.int64)
    ga = bits.shape[0]
    field_off = 4 * np.arange(ga)
    plane_off = 4 * ga + 2 * np.concatenate([[0], np.cumsum(bits)[:-1]])
    used = 4 * ga + 2 * int(bits.sum())
    return field_off, plane_off.astype(np.int64), used


def pack(shift: np.ndarray, scale: np.ndarray, q: np.ndarray,
         bits: np.ndarray, R: int, group: int = GROUP) -> np.ndarray:
    """Token records, uint8 [n][R]."""
    assert group == 16, "bit-planes are 16-bit words"
    n, ga = shift.shape
    field_off, plane_off, used = record_layout(bits)
    assert used <= R
    words = np.zeros((n, R // 2), dtype=np.uint16)
    words[:, field_off // 2] = fp.fp16_bits(shift)
    words[:, field_off // 2 + 1] = fp.fp16_bits(scale)
    qg = np.asarray(q, dtype=np.uint32).reshape(n, ga, group)
    lane = np.arange(group, dtype=np.uint32)
    for a in range(ga):
        for j in range(int(bits[a])):
            plane = (((qg[:, a, :] >> np.uint32(j)) & np.uint32(1))
                     << lane[None, :]).sum(axis=1)
            words[:, plane_off[a] // 2 + j] = plane.astype(np.uint16)
    return words.astype("<u2").view(np.uint8).reshape(n, R)


def unpack(records: np.ndarray, bits: np.ndarray, group: int = GROUP):
    """Inverse of :func:`pack`: (shift fp16, scale fp16, q uint16)."""
    n, R = records.shape
    bits = np.asarray(bits, dtype=np.int64)
    ga = bits.shape[0]
    field_off, plane_off, _ = record_layout(bits)
    words = np.ascontiguousarray(records).view("<u2").reshape(n, R // 2)
    shift = fp.fp16_from_bits(words[:, field_off // 2])
    scale = fp.fp16_from_bits(words[:, field_off // 2 + 1])
    q = np.zeros((n, ga, group), dtype=np.uint32)
    lane = np.arange(group, dtype=np.uint32)
    for a in range(ga):
        for j in range(int(bits[a])):
            plane = words[:, plane_off[a] // 2 + j].astype(np.uint32)
            q[:, a, :] |= ((plane[:, None] >> lane[None, :]) & np.uint32(1)) \
                << np.uint32(j)
    return shift, scale, q.reshape(n, ga * group).astype(np.uint16)


# ------------------------------------------------------------------ stream
@dataclasses.dataclass
class StreamCalib:
    """What the codec needs for one (layer, K|V) stream.

    basis: fp64 [D][k], columns = kept principal components (ascending);
    mu: fp64 [D]; widths: int [G] (0..8), active groups are the nonzero ones.
    """
    mu: np.ndarray
    basis: np.ndarray
    widths: np.ndarray
    sink: int
    window: int
    budget_bits: int

    @property
    def D(self) -> int:
        return self.mu.shape[0]

    @property
    def bits(self) -> np.ndarray:
        w = np.asarray(self.widths)
        return w[w > 0].astype(np.int64)

    @property
    def R(self) -> int:
        return record_bytes(self.budget_bits)


def coefficients(x_bits: np.ndarray, sc: StreamCalib) -> np.ndarray:
    """c = (x - mu) V for the given bf16 rows (page section 2B)."""
    x = fp.bf16_bits_to_f64(x_bits)
    return (x - sc.mu[None, :]) @ sc.basis


def compress_stream(x_bits: np.ndarray, sc: StreamCalib,
                    range_errors: Optional[list] = None) -> bytes:
    """One stream: x bf16 bits [T][D] -> bytes (sink, window, records)."""
    T, D = x_bits.shape
    s_, w_, tc = split_tokens(T, sc.sink, sc.window)
    out = bytearray(stream_bytes(T, D, sc.sink, sc.window, sc.budget_bits))
    raw = np.concatenate([x_bits[:s_], x_bits[T - w_:]], axis=0)
    raw_b = np.ascontiguousarray(raw.astype("<u2")).view(np.uint8).reshape(-1)
    out[:raw_b.size] = raw_b.tobytes()
    if tc > 0:
        c = coefficients(x_bits[s_:T - w_], sc)
        qz = quantise(c, sc.bits)
        if range_errors is not None and qz.range_error:
            range_errors.append(True)
        rec = pack(qz.shift, qz.scale, qz.q, sc.bits, sc.R)
        off = raw_b.size
        out[off:off + rec.size] = rec.reshape(-1).tobytes()
    return bytes(out)


def stream_records(buf: bytes, T: int, sc: StreamCalib) -> np.ndarray:
    s_, w_, tc = split_tokens(T, sc.sink, sc.window)
    off = (s_ + w_) * sc.D * 2
    return np.frombuffer(buf, dtype=np.uint8, count=tc * sc.R,
                         offset=off).reshape(tc, sc.R)


def reconstruct(records: np.ndarray, sc: StreamCalib) -> np.ndarray:
    """Exact fp64 x_hat = mu + V c_hat for records (page section 2C)."""
    shift, scale, q = unpack(records, sc.bits)
    chat = dequantise(shift, scale, q)
    return sc.mu[None, :] + chat @ sc.basis.T


def decompress_stream(buf: bytes, T: int, sc: StreamCalib,
                      exact: bool = False) -> np.ndarray:
    """bytes -> bf16 bits [T][D] (or fp64 values when ``exact``)."""
    D = sc.D
    s_, w_, tc = split_tokens(T, sc.sink, sc.window)
    raw = np.frombuffer(buf, dtype="<u2", count=(s_ + w_) * D).reshape(
        s_ + w_, D)
    out = np.zeros((T, D), dtype=np.float64 if exact else np.uint16)
    conv = fp.bf16_bits_to_f64 if exact else (lambda b: b)
    out[:s_] = conv(raw[:s_])
    out[T - w_:] = conv(raw[s_:])
    if tc > 0:
        xh = reconstruct(stream_records(buf, T, sc), sc)
        out[s_:T - w_] = xh if exact else fp.bf16_rne_bits(xh)
    return out


def paged_write(pool: np.ndarray, rows: np.ndarray, table_row: np.ndarray,
                block_size: int) -> None:
    """Token t of a request goes to pool[table_row[t // bs], t % bs]."""
    for t in range(rows.shape[0]):
        pool[table_row[t // block_size], t % block_size] = rows[t]
