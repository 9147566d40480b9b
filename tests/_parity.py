"""Shared helpers of the parity tests: oracle calibration of workloads, and
the comparison rules between the CUDA path and the oracle.

Parity rule (compress bitstreams): raw rows bit-exact; per token and group
the GPU's fp16 shift / scale equal the oracle's, except where the oracle's
fp64 pre-rounding value lies within min(1e-3, E) of an fp16 rounding
boundary, E the accumulation bound below (any value the directed rounding
gives for a group minimum or maximum within that distance is then accepted,
and the codes are re-derived in fp64 from the GPU's fields); codes equal
the fp64 rule, except that a code may differ by one where the fp64
coefficient lies within w(c) of a rounding boundary.  Any other difference
is a failure.  The tests report, per configuration, how many codes and
fields differed and the largest field difference in fp16 steps.

The window of coefficient c (absolute, coefficient units) is

    w(c) = min(1e-3, max(1e-3 * step, E(c))),
    E(c) = (D/16 + 16) * 2^-23 * sum_d |V_da x_d| + 2^-23 * (|m_a| + |c|),

where E bounds the error of one fp32 tensor-core accumulation of V^T x
(one rounding of at most one fp32 ulp per 16-term MMA step, plus the
rounding of m = V^T mu and of the final subtraction).  So a difference is
excused only where the fp32 arithmetic itself cannot decide the boundary,
and never farther than 1e-3 from it.

Parity rule (decompress of the oracle's bitstream): relative L2 error at
most 2e-3 and max abs error at most 1 bf16 ulp of the oracle's value plus
1e-3; raw rows bit-exact.
"""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os
from typing import List, Sequence, Tuple

import numpy as np

import synth
from oracle import calibrate, codec, fp

CODE_WINDOW = 1e-3
FIELD_WINDOW = 1e-3

# Per-configuration parity statistics gathered by the GPU tests and printed
# at the end of the session (tests/conftest.py): {config: counts}.
REPORT: dict = {}


def record(config: str, st: dict = None, dst: dict = None) -> None:
    """Add one stream's record statistics (check_records) and/or restore
    statistics (check_decompress) to the session report of `config`."""
    r = REPORT.setdefault(config, dict(
        streams=0, codes=0, code_flips=0, code_flips_outside_1e3_step=0,
        fields=0, field_flips=0, field_dev_steps_max=0, restores=0,
        rel_l2_max=0.0, max_abs=0.0))
    if st is not None:
        r["streams"] += 1
        for k in ("codes", "code_flips", "code_flips_outside_1e3_step",
                  "fields", "field_flips"):
            r[k] += int(st.get(k, 0))
        r["field_dev_steps_max"] = max(r["field_dev_steps_max"],
                                       int(st.get("field_dev_steps_max", 0)))
    if dst is not None:
        r["restores"] += 1
        r["rel_l2_max"] = max(r["rel_l2_max"], float(dst["rel_l2"]))
        r["max_abs"] = max(r["max_abs"], float(dst["max_abs"]))


def fp16_order(h: np.ndarray) -> np.ndarray:
    """Monotone integer position of each fp16 value among all fp16 values
    (adjacent values differ by 1), for counting steps between fields."""
    b = np.asarray(h, dtype=np.float16).view(np.uint16).astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


# ------------------------------------------------------------ calibration
def _calib_one(args):
    name, layer, kv = args
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    w = synth.WORKLOADS[name]
    cb = synth.calib_tokens(w, layer, kv)
    mu, V, evals, widths, _ = calibrate.calibrate_stream(cb, w.budget_bits,
                                                         w.bmax, w.group)
    cols = codec.active_columns(widths)
    # return only the kept columns (the blob stores nothing else)
    Vk = np.zeros_like(V)
    Vk[:, cols] = V[:, cols]
    return layer, kv, mu, Vk, evals, widths


def calibrate_workload(name: str, streams: Sequence[Tuple[int, int]],
                       workers: int = 0) -> List[tuple]:
    """Oracle calibration of the given (layer, kv) streams, in a spawn pool
    when there are several."""
    jobs = [(name, l, kv) for l, kv in streams]
    if len(jobs) <= 2:
        return [_calib_one(j) for j in jobs]
    n = workers or min(len(jobs), os.cpu_count() or 4)
    env = {"OPENBLAS_NUM_THREADS": "1", "OMP_NUM_THREADS": "1",
           "MKL_NUM_THREADS": "1"}
    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        with cf.ProcessPoolExecutor(
                n, mp_context=mp.get_context("spawn")) as ex:
            return list(ex.map(_calib_one, jobs))
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _pca_one(args):
    name, layer, kv = args
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    w = synth.WORKLOADS[name]
    mu, evals, V = calibrate.pca(synth.calib_tokens(w, layer, kv))
    return layer, kv, mu, V, evals


def calibrate_forced(name: str, streams: Sequence[Tuple[int, int]],
                     widths: np.ndarray) -> List[tuple]:
    """Oracle PCA of the given streams with the group widths set by hand
    instead of by the DP (a valid calibration the DP would not pick: it
    reaches kept-component counts the budget allows but the allocation
    never chooses)."""
    jobs = [(name, l, kv) for l, kv in streams]
    if len(jobs) <= 2:
        out = [_pca_one(j) for j in jobs]
    else:
        n = min(len(jobs), os.cpu_count() or 4)
        with cf.ProcessPoolExecutor(
                n, mp_context=mp.get_context("spawn")) as ex:
            out = list(ex.map(_pca_one, jobs))
    wd = np.asarray(widths, dtype=np.int64)
    return [(l, kv, mu, V, ev, wd) for l, kv, mu, V, ev in out]


def blob_for(name: str, entries: Sequence[tuple],
             budget_bits: int = None) -> bytes:
    w = synth.WORKLOADS[name]
    return calibrate.write_blob(entries, w.sink, w.window,
                                budget_bits or w.budget_bits, w.bmax, w.group)


def stream_calibs(blob: bytes):
    """{(layer, kv): (sc_bf16 for compress, sc_fp16 for decompress)}."""
    b = calibrate.read_blob(blob)
    out = {}
    for e in b["streams"]:
        out[(e["layer"], e["kv"])] = (
            calibrate.stream_calib(e, b["sink"], b["window"],
                                   b["budget_bits"], basis="bf16"),
            calibrate.stream_calib(e, b["sink"], b["window"],
                                   b["budget_bits"], basis="fp16"))
    return out


# ----------------------------------------------------------- comparisons
def accumulation_bound(x_rows: np.ndarray, sc: codec.StreamCalib,
                       c: np.ndarray) -> np.ndarray:
    """E(c) of the module docstring, per token and kept component."""
    x = fp.bf16_bits_to_f64(x_rows)
    absprod = np.abs(x) @ np.abs(sc.basis)
    m = sc.mu @ sc.basis
    n_mma = sc.D // 16
    return (n_mma + 16) * 2.0 ** -23 * absprod + \
        2.0 ** -23 * (np.abs(m)[None, :] + np.abs(c))


def coefficient_window(x_rows: np.ndarray, sc: codec.StreamCalib,
                       c: np.ndarray, step: np.ndarray) -> np.ndarray:
    """w(c) of the module docstring, per token and kept component."""
    E = accumulation_bound(x_rows, sc, c)
    return np.minimum(1e-3, np.maximum(1e-3 * step, E))


def check_records(gpu_rec: np.ndarray, x_rows: np.ndarray,
                  sc: codec.StreamCalib) -> dict:
    """Compare GPU records of the compressed rows x_rows (bf16 bits) with
    the fp64 rule.  Returns counts; 'bad' must be 0."""
    n = x_rows.shape[0]
    bits = sc.bits
    if n == 0:
        return dict(bad=0, field_bad=0, code_bad=0, field_flips=0, fields=0,
                    field_dev_steps_max=0, code_flips=0,
                    code_flips_outside_1e3_step=0, codes=0)
    c = codec.coefficients(x_rows, sc)
    ga = bits.shape[0]
    cg = c.reshape(n, ga, 16)
    lo, hi = cg.min(2), cg.max(2)
    lev = (2.0 ** bits - 1.0)[None, :]
    qz = codec.quantise(c, bits)
    so, do = qz.shift.astype(np.float64), qz.scale.astype(np.float64)
    sg, dg, qg = codec.unpack(gpu_rec, bits)
    sg, dg = sg.astype(np.float64), dg.astype(np.float64)
    step = np.repeat(np.where(do > 0, do, 2.0 ** -24), 16, axis=1)
    win = coefficient_window(x_rows, sc, c, step).reshape(n, ga, 16)
    # Fields: the GPU's group minimum and maximum are fp32 coefficients, off
    # by at most the accumulation bound E(c); every fp16 value the directed
    # rounding can give for a value within E of the fp64 minimum (shift), or
    # for a quotient built from a maximum within E (scale), is accepted, and
    # nothing else.
    ebound = np.minimum(1e-3, accumulation_bound(x_rows, sc, c))
    gE = ebound.reshape(n, ga, 16).max(axis=2)     # per group
    with np.errstate(over="ignore", invalid="ignore"):
        shift_ok = (sg == so) | ((sg >= fp.fp16_rd(lo - gE)) &
                                 (sg <= fp.fp16_rd(lo + gE)))
        pre = (hi - sg) / lev
        ptol = gE / lev + 2.0 ** -22 * np.abs(pre)
        ref_scale = fp.fp16_ru(pre).astype(np.float64)
        scale_ok = (dg == ref_scale) | ((dg >= fp.fp16_ru(pre - ptol)) &
                                        (dg <= fp.fp16_ru(pre + ptol)))
    field_bad = ~(shift_ok & scale_ok)
    field_flip = (sg != so) | (dg != do)
    dev = np.maximum(np.abs(fp16_order(sg) - fp16_order(so)),
                     np.abs(fp16_order(dg) - fp16_order(do)))
    # codes from the GPU's fields, in fp64
    with np.errstate(divide="ignore", invalid="ignore"):
        u = (cg - sg[:, :, None]) / dg[:, :, None]
        uwin = win / dg[:, :, None] + 2.0 ** -21 * np.abs(u)
    ref = np.clip(np.floor(u + 0.5), 0, lev[:, :, None])
    ref = np.where(dg[:, :, None] > 0, ref, 0.0)
    ref = np.nan_to_num(ref)
    qg3 = qg.reshape(n, ga, 16).astype(np.float64)
    diff = np.abs(qg3 - ref)
    frac = (u + 0.5) - np.floor(u + 0.5)
    dist = np.minimum(frac, 1 - frac)              # to a boundary, in steps
    near = dist <= uwin
    near_strict = dist <= 1e-3
    code_bad = (diff > 1) | ((diff == 1) & ~near)
    code_bad &= ~field_bad[:, :, None]
    flips = diff == 1
    return dict(bad=int(field_bad.sum() + code_bad.sum()),
                field_bad=int(field_bad.sum()),
                code_bad=int(code_bad.sum()),
                field_flips=int(field_flip.sum()),
                fields=int(2 * field_flip.size),
                field_dev_steps_max=int(dev.max()) if dev.size else 0,
                code_flips=int(flips.sum()),
                code_flips_outside_1e3_step=int((flips & ~near_strict).sum()),
                codes=int(diff.size))


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(e, -125)
    return np.ldexp(1.0, e - 8)


def check_decompress(gpu_bits: np.ndarray, oracle_bits: np.ndarray) -> dict:
    g = fp.bf16_bits_to_f64(gpu_bits)
    o = fp.bf16_bits_to_f64(oracle_bits)
    if o.size == 0:
        return dict(rel_l2=0.0, max_abs=0.0, ok=True)
    err = np.abs(g - o)
    rel = float(np.linalg.norm(g - o) / max(np.linalg.norm(o), 1e-300))
    lim = bf16_ulp(o) + 1e-3
    return dict(rel_l2=rel, max_abs=float(err.max()),
                worst_excess=float((err - lim).max()),
                ok=bool(rel <= 2e-3 and np.all(err <= lim)))
