"""Host-only checks of the C ABI: the library builds, loads and exports every
declared entry point, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re
import struct
import zlib

import numpy as np
import pytest

import synth
from oracle import calibrate

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def kv():
    from kv_cache_transform_gb300 import _build
    _build.build()
    import kv_cache_transform_gb300 as kv
    return kv


def declared_symbols():
    with open(os.path.join(ROOT, "include", "kvtc.h")) as f:
        txt = f.read()
    return sorted(set(re.findall(r"\b(kvtc_\w+)\s*\(", txt)))


def test_every_declared_symbol_is_exported(kv):
    L = kv.lib()
    syms = declared_symbols()
    assert "kvtc_compress" in syms and "kvtc_decompress_paged" in syms
    for s in syms:
        assert hasattr(L, s), s


def test_strerror(kv):
    assert kv.kvtc_strerror(0) == "ok"
    assert "blob" in kv.kvtc_strerror(kv.KVTC_EFORMAT)
    assert kv.kvtc_strerror(-1234) == "unknown status"


def tiny_blob():
    w = synth.WORKLOADS["tiny"]
    cb = synth.calib_tokens(w, 0, 0)
    mu, V, evals, widths, _ = calibrate.calibrate_stream(cb, w.budget_bits)
    return calibrate.write_blob([(0, 0, mu, V, evals, widths)], w.sink,
                                w.window, w.budget_bits)


def load_raw(kv, blob):
    out = ctypes.c_void_p()
    buf = ctypes.create_string_buffer(blob, len(blob))
    return kv.lib().kvtc_calib_load(buf, len(blob), 0, ctypes.byref(out))


def test_blob_rejections_happen_before_any_cuda_call(kv):
    blob = tiny_blob()
    # bad magic
    assert load_raw(kv, b"XXXX" + blob[4:]) == kv.KVTC_EFORMAT
    # flipped payload byte -> checksum
    bad = bytearray(blob)
    bad[100] ^= 0x40
    assert load_raw(kv, bytes(bad)) == kv.KVTC_EFORMAT
    # truncated
    assert load_raw(kv, blob[:-9]) == kv.KVTC_EFORMAT
    # wrong version with a valid checksum
    body = bytearray(blob[:-8])
    body[4:8] = struct.pack("<I", 2)
    body = bytes(body)
    assert load_raw(kv, body + struct.pack("<2I", zlib.crc32(body), 0)) == \
        kv.KVTC_EFORMAT
    # widths inconsistent with k (claims one more kept column group)
    body = bytearray(blob[:-8])
    k_off = 4 + 28 + 12
    k = struct.unpack_from("<I", body, k_off)[0]
    struct.pack_into("<I", body, k_off, k + 16)
    body = bytes(body)
    assert load_raw(kv, body + struct.pack("<2I", zlib.crc32(body), 0)) == \
        kv.KVTC_EFORMAT
    # null arguments
    out = ctypes.c_void_p()
    assert kv.lib().kvtc_calib_load(None, 10, 0, ctypes.byref(out)) == \
        kv.KVTC_EINVAL


def test_null_handles_are_rejected(kv):
    L = kv.lib()
    arr = (ctypes.c_void_p * 2)()
    assert L.kvtc_compress(None, 0, 1, 1, arr, 128, 10, None, 0, None) == \
        kv.KVTC_EINVAL
    assert L.kvtc_decompress(None, 0, 1, 1, None, 0, 10, arr, 128, None,
                             None) == kv.KVTC_EINVAL
    T = (ctypes.c_int64 * 1)(10)
    assert L.kvtc_decompress_paged(None, 0, 1, 1, arr, T, 1, None, 1, 16,
                                   arr, 1, None) == kv.KVTC_EINVAL
    assert L.kvtc_stream_bytes(None, 0, 0, 10) == kv.KVTC_EINVAL
    flags = ctypes.c_uint()
    assert L.kvtc_device_status(None, None, ctypes.byref(flags)) == \
        kv.KVTC_EINVAL
    assert L.kvtc_fields_bound(None, 0, 1, 1, 10) == kv.KVTC_EINVAL
    assert L.kvtc_fields_workspace_bytes(None, 0, 1, 1) == kv.KVTC_EINVAL
    assert L.kvtc_fields_pack(None, 0, 1, 1, None, 0, 10, None, 0, None,
                              None, 0, None) == kv.KVTC_EINVAL
    assert L.kvtc_fields_unpack(None, 0, 1, 1, None, 0, None, 10, None, 0,
                                None) == kv.KVTC_EINVAL
    assert L.kvtc_decompress_packed(None, 0, 1, 1, None, 0, None, 10, arr,
                                    128, None, None) == kv.KVTC_EINVAL
    L.kvtc_calib_free(None)  # no-op


def test_python_binding_raises_on_error(kv):
    with pytest.raises(kv.KvtcError) as e:
        kv.kvtc_calib_load(b"not a blob at all, definitely not" * 2)
    assert e.value.code == kv.KVTC_EFORMAT


def test_kept_components_beyond_the_kernel_limits_are_refused(kv):
    """Valid blobs the kernels cannot run are refused (ENOTSUP) while
    parsing, before any CUDA call:
    - k = 512 (every group of a D = 512 stream at width 1): the
      reconstruction holds k plus one mean step of 16 fp16 columns in 256
      TMEM columns, so k <= 496;
    - records over 256 bytes (a budget of 2064 bits: R = 272), longer than
      the kernels' record staging takes."""
    D = 512
    widths = np.ones(D // 16, dtype=np.uint8)
    blob = calibrate.write_blob(
        [(0, 0, np.zeros(D), np.eye(D), np.ones(D), widths)], 4, 16,
        int(widths.size * calibrate.width_cost_units(1) * 16))
    assert load_raw(kv, blob) == kv.KVTC_ENOTSUP
    widths = np.zeros(D // 16, dtype=np.uint8)
    widths[:25] = 2
    blob = calibrate.write_blob(
        [(0, 0, np.zeros(D), np.eye(D), np.ones(D), widths)], 4, 16, 2064)
    assert load_raw(kv, blob) == kv.KVTC_ENOTSUP
