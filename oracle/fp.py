"""Floating-point formats used by the codec, computed from fp64.

binary16 (fp16): 1 sign, 5 exponent, 10 fraction bits; largest finite 65504.
The microscaling fields (per-group shift and scale, kvtc page, section 2A
"microscaling": a group of components shares a scale factor and a shift) are
stored as fp16.  The shift is rounded DOWN and the scale UP so that every
coefficient of the group maps into [0, 2^b - 1] code units; these directions
are this build's reading (the page does not say how the fields are rounded).

NumPy's float64 -> float16 cast is a single correctly rounded
round-to-nearest-even conversion; directed rounding is obtained from it by
stepping one unit in the last place with ``nextafter`` when the nearest value
lies on the wrong side.  Results that leave the finite range become +-inf and
are reported by the callers as range errors.

bfloat16: 1 sign, 8 exponent, 7 fraction bits (the KV cache's storage type).
"""
from __future__ import annotations

import numpy as np

FP16_MAX = 65504.0


def fp16_rne(v) -> np.ndarray:
    """Nearest fp16 (ties to even) of fp64 values."""
    return np.asarray(v, dtype=np.float64).astype(np.float16)


def fp16_rd(v) -> np.ndarray:
    """Largest fp16 <= v (round toward -inf).  -inf below -65504."""
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):
        h = v.astype(np.float16)
    above = h.astype(np.float64) > v
    with np.errstate(over="ignore"):
        return np.where(above, np.nextafter(h, np.float16(-np.inf)), h)


def fp16_ru(v) -> np.ndarray:
    """Smallest fp16 >= v (round toward +inf).  +inf above 65504."""
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):
        h = v.astype(np.float16)
    below = h.astype(np.float64) < v
    with np.errstate(over="ignore"):
        return np.where(below, np.nextafter(h, np.float16(np.inf)), h)


def fp16_bits(h) -> np.ndarray:
    return np.asarray(h, dtype=np.float16).view(np.uint16)


def fp16_from_bits(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16)


def bf16_rne_value(v) -> np.ndarray:
    """fp64 value of the nearest bf16 (ties to even) of fp64 values.

    A finite v = m * 2^e with 0.5 <= |m| < 1.  bf16 keeps 8 significant bits
    for normal numbers (e >= -125) and a fixed quantum of 2^-133 below that,
    so the result is rint(v * 2^(8-e')) * 2^(e'-8) with e' = max(e, -125);
    ``np.rint`` rounds halves to even.  Single rounding straight from fp64
    (no detour through fp32)."""
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)
    e = np.maximum(e, -125)
    return np.ldexp(np.rint(np.ldexp(v, 8 - e)), e - 8)


def bf16_rne_bits(v) -> np.ndarray:
    """bf16 bit patterns of the nearest bf16 of fp64 values."""
    r = bf16_rne_value(v).astype(np.float32)  # exact: 8 significant bits
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)
