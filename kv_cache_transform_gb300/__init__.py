"""kvtc on GB300: Python binding of ``libkvtc.so`` (argument marshalling only).

Every computation happens in the library's sm_103a kernels; this module only
turns tensors into pointers and status codes into exceptions.  The names
mirror the C ABI in ``include/kvtc.h``:

    kvtc_calib_load, kvtc_calib_free, kvtc_calib_query, kvtc_stream_bytes,
    kvtc_compress, kvtc_decompress, kvtc_decompress_paged,
    kvtc_fields_bound, kvtc_fields_workspace_bytes, kvtc_fields_pack,
    kvtc_fields_unpack, kvtc_decompress_packed, kvtc_device_status,
    kvtc_launch_count, kvtc_strerror

Tensor arguments are torch CUDA tensors (or raw integer device addresses);
``stream`` defaults to torch's current stream.  There is no CPU fallback: if
the library is missing every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvtc.so")

KVTC_OK = 0
KVTC_EINVAL = -1
KVTC_EFORMAT = -2
KVTC_ESIZE = -3
KVTC_ENOMEM = -4
KVTC_ECUDA = -5
KVTC_ERANGE = -6
KVTC_EDEVICE = -7
KVTC_EALIGN = -8
KVTC_ENOTSUP = -9

KVTC_FLAG_RANGE = 1
KVTC_FLAG_TIMEOUT = 2
KVTC_FLAG_BLOCK = 4
KVTC_FLAG_FORMAT = 8

_lib_handle = None


class KvtcError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {kvtc_strerror(code)} ({code})")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib_handle
    if _lib_handle is not None:
        return _lib_handle
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "kv_cache_transform_gb300._build.build() (nvcc, sm_103a)")
    L = ctypes.CDLL(LIB_PATH)
    c_vp, c_i, c_i64, c_sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                              ctypes.c_size_t)
    c_pp = ctypes.POINTER(ctypes.c_void_p)
    c_ip = ctypes.POINTER(ctypes.c_int)
    sig = {
        "kvtc_calib_load": (c_i, [c_vp, c_sz, c_i, c_pp]),
        "kvtc_calib_free": (None, [c_vp]),
        "kvtc_calib_query": (c_i, [c_vp, c_i, c_i, c_ip, c_ip, c_ip, c_ip,
                                   c_ip]),
        "kvtc_stream_bytes": (c_i64, [c_vp, c_i, c_i, c_i64]),
        "kvtc_compress": (c_i, [c_vp, c_i, c_i, c_i, c_pp, c_i64, c_i64, c_vp,
                                c_i64, c_vp]),
        "kvtc_decompress": (c_i, [c_vp, c_i, c_i, c_i, c_vp, c_i64, c_i64,
                                  c_pp, c_i64, c_vp, c_pp]),
        "kvtc_decompress_paged": (c_i, [c_vp, c_i, c_i, c_i, c_pp,
                                        ctypes.POINTER(ctypes.c_int64), c_i,
                                        c_vp, c_i, c_i, c_pp, c_i64, c_vp]),
        "kvtc_device_status": (c_i, [c_vp, c_vp,
                                     ctypes.POINTER(ctypes.c_uint)]),
        "kvtc_strerror": (ctypes.c_char_p, [c_i]),
        "kvtc_calibrate": (c_i, [c_i, c_i, c_ip, c_ip, c_pp, c_i64, c_i64,
                                 c_i, c_i, c_i, c_i, c_vp, c_sz,
                                 ctypes.POINTER(ctypes.c_size_t), c_vp]),
        "kvtc_blob_max_bytes": (c_i64, [c_i, c_i]),
        "kvtc_launch_count": (ctypes.c_uint64, []),
        "kvtc_calib_mean_static": (c_i, [c_i, c_vp, c_i64, c_i64, c_i, c_vp,
                                         c_vp]),
        "kvtc_wait_selftest": (c_i, [c_vp, ctypes.c_uint32, c_vp]),
        "kvtc_fields_bound": (c_i64, [c_vp, c_i, c_i, c_i, c_i64]),
        "kvtc_fields_workspace_bytes": (c_i64, [c_vp, c_i, c_i, c_i]),
        "kvtc_fields_pack": (c_i, [c_vp, c_i, c_i, c_i, c_vp, c_i64, c_i64,
                                   c_vp, c_i64, c_vp, c_vp, c_i64, c_vp]),
        "kvtc_fields_unpack": (c_i, [c_vp, c_i, c_i, c_i, c_vp, c_i64, c_vp,
                                     c_i64, c_vp, c_i64, c_vp]),
        "kvtc_decompress_packed": (c_i, [c_vp, c_i, c_i, c_i, c_vp, c_i64,
                                         c_vp, c_i64, c_pp, c_i64, c_vp,
                                         c_pp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib_handle = L
    return L


def kvtc_launch_count() -> int:
    return int(lib().kvtc_launch_count())


def kvtc_strerror(code: int) -> str:
    return lib().kvtc_strerror(code).decode()


def _check(code: int, what: str) -> int:
    if code < 0:
        raise KvtcError(code, what)
    return code


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _ptr_array(xs: Sequence) -> ctypes.Array:
    arr = (ctypes.c_void_p * max(1, len(xs)))()
    for i, x in enumerate(xs):
        arr[i] = _ptr(x) or None
    return arr


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


class Calib:
    """Handle of a loaded calibration (owns device operands)."""

    def __init__(self, handle: int, device: int):
        self.handle = ctypes.c_void_p(handle)
        self.device = device

    def query(self, layer: int, kv: int) -> dict:
        v = [ctypes.c_int() for _ in range(5)]
        _check(lib().kvtc_calib_query(self.handle, layer, kv,
                                      *[ctypes.byref(x) for x in v]),
               "kvtc_calib_query")
        return dict(zip(("D", "k", "sink", "window", "record_bytes"),
                        (x.value for x in v)))

    def stream_bytes(self, layer: int, kv: int, T: int) -> int:
        return _check(lib().kvtc_stream_bytes(self.handle, layer, kv, T),
                      "kvtc_stream_bytes")

    def free(self) -> None:
        if self.handle:
            lib().kvtc_calib_free(self.handle)
            self.handle = ctypes.c_void_p(0)

    def __del__(self):  # pragma: no cover - best effort
        try:
            self.free()
        except Exception:
            pass


def kvtc_calib_load(blob: bytes, device: int = 0) -> Calib:
    out = ctypes.c_void_p()
    buf = ctypes.create_string_buffer(bytes(blob), len(blob))
    _check(lib().kvtc_calib_load(buf, len(blob), device, ctypes.byref(out)),
           "kvtc_calib_load")
    return Calib(out.value, device)


def kvtc_calibrate(tokens: Sequence, layers: Sequence[int],
                   kvs: Sequence[int], N: int, ld: int, D: int, sink: int,
                   window: int, budget_bits: int, device: int = 0,
                   stream=None) -> bytes:
    """Calibrate streams from device bf16 rows [N][ld]; returns the blob."""
    n = len(tokens)
    cap = _check(lib().kvtc_blob_max_bytes(n, D), "kvtc_blob_max_bytes")
    buf = ctypes.create_string_buffer(cap)
    size = ctypes.c_size_t()
    L = (ctypes.c_int * n)(*layers)
    K = (ctypes.c_int * n)(*kvs)
    _check(lib().kvtc_calibrate(device, n, L, K, _ptr_array(tokens), N, ld,
                                D, sink, window, budget_bits, buf, cap,
                                ctypes.byref(size), _stream(stream) or None),
           "kvtc_calibrate")
    return buf.raw[:size.value]


def kvtc_blob_max_bytes(n: int, D: int) -> int:
    return _check(lib().kvtc_blob_max_bytes(n, D), "kvtc_blob_max_bytes")


def kvtc_calib_mean_static(tokens, N: int, ld: int, D: int, mu_out,
                           device: int = 0, stream=None) -> None:
    """Per-channel mean of device bf16 rows [N][ld] into device fp64 mu_out,
    with no device allocation (for callers that own all device memory)."""
    _check(lib().kvtc_calib_mean_static(device, _ptr(tokens) or None, N, ld,
                                         D, _ptr(mu_out) or None,
                                         _stream(stream) or None),
           "kvtc_calib_mean_static")


def kvtc_calib_free(calib: Calib) -> None:
    calib.free()


def kvtc_calib_query(calib: Calib, layer: int, kv: int) -> dict:
    return calib.query(layer, kv)


def kvtc_stream_bytes(calib: Calib, layer: int, kv: int, T: int) -> int:
    return calib.stream_bytes(layer, kv, T)


def kvtc_compress(calib: Calib, layer0: int, nlayers: int, kv_mask: int,
                  src: Sequence, ld: int, T: int, dst, dst_bytes: int,
                  stream=None) -> None:
    """src: 2*nlayers bf16 [T][ld] tensors (None where kv_mask excludes)."""
    _check(lib().kvtc_compress(calib.handle, layer0, nlayers, kv_mask,
                               _ptr_array(src), ld, T, _ptr(dst) or None,
                               dst_bytes, _stream(stream) or None),
           "kvtc_compress")


def kvtc_decompress(calib: Calib, layer0: int, nlayers: int, kv_mask: int,
                    src, src_bytes: int, T: int, dst: Sequence, ld: int,
                    stream=None, layer_events: Optional[Sequence] = None
                    ) -> None:
    _check(lib().kvtc_decompress(calib.handle, layer0, nlayers, kv_mask,
                                 _ptr(src) or None, src_bytes, T,
                                 _ptr_array(dst), ld,
                                 _stream(stream) or None,
                                 _event_array(layer_events)),
           "kvtc_decompress")


def _event_array(layer_events):
    if layer_events is None:
        return None
    ev = (ctypes.c_void_p * max(1, len(layer_events)))()
    for i, e in enumerate(layer_events):
        ev[i] = e if isinstance(e, int) else int(e.cuda_event)
    return ev


def kvtc_decompress_packed(calib: Calib, layer0: int, nlayers: int,
                           kv_mask: int, src, src_bytes: int, offsets,
                           T: int, dst: Sequence, ld: int, stream=None,
                           layer_events: Optional[Sequence] = None) -> None:
    """Restore from packed streams (offsets as kvtc_fields_pack wrote);
    src and offsets device or pinned host tensors."""
    _check(lib().kvtc_decompress_packed(calib.handle, layer0, nlayers,
                                        kv_mask, _ptr(src) or None, src_bytes,
                                        _ptr(offsets) or None, T,
                                        _ptr_array(dst), ld,
                                        _stream(stream) or None,
                                        _event_array(layer_events)),
           "kvtc_decompress_packed")


def kvtc_decompress_paged(calib: Calib, layer0: int, nlayers: int,
                          kv_mask: int, src: Sequence, T: Sequence[int],
                          block_table, max_blocks: int, block_size: int,
                          cache: Sequence, num_blocks: int,
                          stream=None) -> None:
    Ts = (ctypes.c_int64 * max(1, len(T)))(*T)
    _check(lib().kvtc_decompress_paged(
        calib.handle, layer0, nlayers, kv_mask, _ptr_array(src), Ts, len(T),
        _ptr(block_table) or None, max_blocks, block_size, _ptr_array(cache),
        num_blocks, _stream(stream) or None), "kvtc_decompress_paged")


def kvtc_fields_bound(calib: Calib, layer0: int, nlayers: int,
                      kv_mask: int, T: int) -> int:
    return _check(lib().kvtc_fields_bound(calib.handle, layer0, nlayers,
                                          kv_mask, T), "kvtc_fields_bound")


def kvtc_fields_workspace_bytes(calib: Calib, layer0: int, nlayers: int,
                                kv_mask: int) -> int:
    return _check(lib().kvtc_fields_workspace_bytes(
        calib.handle, layer0, nlayers, kv_mask),
        "kvtc_fields_workspace_bytes")


def kvtc_fields_pack(calib: Calib, layer0: int, nlayers: int, kv_mask: int,
                     src, src_bytes: int, T: int, dst, dst_capacity: int,
                     offsets, workspace, workspace_bytes: int,
                     stream=None) -> None:
    """Pack codec streams; offsets: device int64 [n + 1], written."""
    _check(lib().kvtc_fields_pack(calib.handle, layer0, nlayers, kv_mask,
                                  _ptr(src) or None, src_bytes, T,
                                  _ptr(dst) or None, dst_capacity,
                                  _ptr(offsets) or None,
                                  _ptr(workspace) or None, workspace_bytes,
                                  _stream(stream) or None),
           "kvtc_fields_pack")


def kvtc_fields_unpack(calib: Calib, layer0: int, nlayers: int,
                       kv_mask: int, src, src_bytes: int, offsets, T: int,
                       dst, dst_bytes: int, stream=None) -> None:
    """Restore the codec streams of packed input (offsets as pack wrote)."""
    _check(lib().kvtc_fields_unpack(calib.handle, layer0, nlayers, kv_mask,
                                    _ptr(src) or None, src_bytes,
                                    _ptr(offsets) or None, T,
                                    _ptr(dst) or None, dst_bytes,
                                    _stream(stream) or None),
           "kvtc_fields_unpack")


def kvtc_wait_selftest(calib: Calib, limit_us: int, stream=None) -> None:
    _check(lib().kvtc_wait_selftest(calib.handle, limit_us,
                                    _stream(stream) or None),
           "kvtc_wait_selftest")


def kvtc_device_status(calib: Calib, stream=None) -> int:
    flags = ctypes.c_uint()
    _check(lib().kvtc_device_status(calib.handle, _stream(stream) or None,
                                    ctypes.byref(flags)),
           "kvtc_device_status")
    return flags.value
