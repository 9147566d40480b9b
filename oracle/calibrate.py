"""Calibration in fp64 (oracle): PCA basis, distortion table, DP allocation.

kvtc page ("KV Cache Transform Coding for Compact Storage in LLM
Inference"), Technical summary section 2A Calibration:
  * KV from a calibration set is decorrelated by PCA; the orthonormal basis V
    comes from an SVD of the centred data (here: eigenvectors of the sample
    covariance, the same right singular vectors), computed once and reused
    for every request;
  * a dynamic program picks a bit width per principal component so that the
    reconstruction error is smallest under a bit budget; high-variance
    components get more bits, low-variance ones may get 0 (dropped);
  * groups of components share a scale and a shift (microscaling).

Readings (the page is silent on them):
  * sign of each eigenvector: its largest-magnitude entry is positive (first
    index on ties); eigenvalues sorted descending;
  * the distortion of width b on group g is measured on the calibration
    coefficients with the codec's own quantiser; width 0 costs the group's
    energy.  Because V is orthonormal these per-group errors add up to the
    squared reconstruction error, so the objective is separable;
  * a group of width b >= 1 costs its two fp16 fields plus b 16-bit planes,
    32 + 16 b bits per token; the budget is the stored size per token;
  * DP over budget units of 16 bits, F[g][u] = least error of the first g
    groups within u units; ties go to the smaller width.
"""
from __future__ import annotations

import struct
import zlib
from typing import Iterable, List, Tuple

import numpy as np

from . import codec, fp

BLOB_MAGIC = b"KVTC"
BLOB_VERSION = 1


def pca(calib_bits: np.ndarray):
    """mu [D], eigenvalues [D] (descending), V [D][D] (columns)."""
    x = fp.bf16_bits_to_f64(calib_bits)
    n = x.shape[0]
    mu = x.mean(axis=0)
    xc = x - mu[None, :]
    cov = (xc.T @ xc) / n
    evals, evecs = np.linalg.eigh(cov)
    order = np.argsort(-evals, kind="stable")
    evals = evals[order]
    V = evecs[:, order]
    idx = np.argmax(np.abs(V), axis=0)
    sign = np.where(V[idx, np.arange(V.shape[1])] < 0, -1.0, 1.0)
    return mu, evals, V * sign[None, :]


def distortion_table(c: np.ndarray, bmax: int = 8,
                     group: int = codec.GROUP) -> np.ndarray:
    """E[g][b]: summed squared coefficient error of group g at width b."""
    n, D = c.shape
    G = D // group
    cg = c.reshape(n, G, group)
    E = np.zeros((G, bmax + 1))
    E[:, 0] = (cg ** 2).sum(axis=(0, 2))
    for b in range(1, bmax + 1):
        qz = codec.quantise(c, np.full(G, b), group)
        chat = codec.dequantise(qz.shift, qz.scale, qz.q, group)
        E[:, b] = ((c - chat) ** 2).reshape(n, G, group).sum(axis=(0, 2))
    return E


def width_cost_units(b: int) -> int:
    """Cost of one group at width b in 16-bit units (fields + planes)."""
    return 0 if b == 0 else 2 + b


def allocate_bits(E: np.ndarray, budget_bits: int) -> np.ndarray:
    """DP bit allocation: widths [G] minimising sum_g E[g][b_g] subject to
    sum_g cost(b_g) <= budget."""
    G, nb = E.shape
    U = budget_bits // 16
    F = np.zeros((G + 1, U + 1))
    choice = np.zeros((G + 1, U + 1), dtype=np.int64)
    for g in range(1, G + 1):
        for u in range(U + 1):
            best = np.inf
            bb = 0
            for b in range(nb):
                cu = width_cost_units(b)
                if cu > u:
                    break
                v = F[g - 1, u - cu] + E[g - 1, b]
                if v < best:
                    best = v
                    bb = b
            F[g, u] = best
            choice[g, u] = bb
    widths = np.zeros(G, dtype=np.int64)
    u = U
    for g in range(G, 0, -1):
        b = int(choice[g, u])
        widths[g - 1] = b
        u -= width_cost_units(b)
    return widths


def calibrate_stream(calib_bits: np.ndarray, budget_bits: int,
                     bmax: int = 8, group: int = codec.GROUP):
    """mu, V (all D columns), eigenvalues, widths for one stream."""
    mu, evals, V = pca(calib_bits)
    c = (fp.bf16_bits_to_f64(calib_bits) - mu[None, :]) @ V
    E = distortion_table(c, bmax, group)
    widths = allocate_bits(E, budget_bits)
    return mu, V, evals, widths, E


# -------------------------------------------------------------------- blob
def write_blob(entries: Iterable[Tuple[int, int, np.ndarray, np.ndarray,
                                       np.ndarray, np.ndarray]],
               sink: int, window: int, budget_bits: int, bmax: int = 8,
               group: int = codec.GROUP) -> bytes:
    """Calibration blob, version 1 (little-endian):

    header  "KVTC" u32 version, u32 n_streams, u32 group, u32 bmax,
            u32 sink, u32 window, u32 budget_bits
    stream  u32 layer, u32 kv, u32 D, u32 k, u8 widths[G] (zero-padded to a
            multiple of 8 bytes), f64 mu[D], f64 V_kept[k][D] (row a = the
            a-th kept principal vector), f64 eigenvalues[D]
    trailer u32 CRC-32 (IEEE 802.3, as zlib) of everything before it,
            u32 zero.

    entries: (layer, kv, mu, V_full [D][D], eigenvalues, widths)."""
    entries = list(entries)
    parts: List[bytes] = [BLOB_MAGIC, struct.pack(
        "<7I", BLOB_VERSION, len(entries), group, bmax, sink, window,
        budget_bits)]
    for layer, kv, mu, V, evals, widths in entries:
        D = mu.shape[0]
        widths = np.asarray(widths, dtype=np.uint8)
        cols = codec.active_columns(widths, group)
        k = cols.size
        parts.append(struct.pack("<4I", layer, kv, D, k))
        G = D // group
        wpad = np.zeros(-(-G // 8) * 8, dtype=np.uint8)
        wpad[:G] = widths
        parts.append(wpad.tobytes())
        parts.append(np.ascontiguousarray(mu, dtype="<f8").tobytes())
        parts.append(np.ascontiguousarray(V[:, cols].T, dtype="<f8").tobytes())
        parts.append(np.ascontiguousarray(evals, dtype="<f8").tobytes())
    body = b"".join(parts)
    return body + struct.pack("<2I", zlib.crc32(body) & 0xFFFFFFFF, 0)


def read_blob(blob: bytes):
    """Parse a blob written by :func:`write_blob` (for tests)."""
    crc, _ = struct.unpack_from("<2I", blob, len(blob) - 8)
    assert zlib.crc32(blob[:-8]) & 0xFFFFFFFF == crc, "checksum"
    assert blob[:4] == BLOB_MAGIC
    ver, n, group, bmax, sink, window, budget = struct.unpack_from(
        "<7I", blob, 4)
    assert ver == BLOB_VERSION
    off = 4 + 28
    streams = []
    for _ in range(n):
        layer, kv, D, k = struct.unpack_from("<4I", blob, off)
        off += 16
        G = D // group
        gp = -(-G // 8) * 8
        widths = np.frombuffer(blob, np.uint8, G, off).astype(np.int64)
        off += gp
        mu = np.frombuffer(blob, "<f8", D, off).copy()
        off += 8 * D
        Vk = np.frombuffer(blob, "<f8", k * D, off).reshape(k, D).copy()
        off += 8 * k * D
        evals = np.frombuffer(blob, "<f8", D, off).copy()
        off += 8 * D
        streams.append(dict(layer=layer, kv=kv, D=D, k=k, widths=widths,
                            mu=mu, basis=Vk.T.copy(), evals=evals))
    return dict(group=group, bmax=bmax, sink=sink, window=window,
                budget_bits=budget, streams=streams)


def stream_calib(entry: dict, sink: int, window: int, budget_bits: int,
                 basis: str = "f64") -> codec.StreamCalib:
    """StreamCalib from a parsed blob entry.  ``basis`` selects the basis
    values the codec multiplies: the calibrated fp64 ('f64'), or the values a
    bf16 ('bf16') or fp16 ('fp16') copy of it holds."""
    B = entry["basis"]
    if basis == "bf16":
        B = fp.bf16_rne_value(B)
    elif basis == "fp16":
        B = fp.fp16_rne(B).astype(np.float64)
    return codec.StreamCalib(entry["mu"], B, entry["widths"], sink, window,
                             budget_bits)
