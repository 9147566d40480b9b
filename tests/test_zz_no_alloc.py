"""The allocation-free mean entry point, for callers that own all device
memory themselves (a serving engine's preallocated KV pool) or cannot afford
the device-wide synchronisation that cudaMalloc / cudaFree bring.

kvtc_calib_mean_static must give the same per-channel mean as the one
kvtc_calibrate stores in its blob, call after call, while allocating
nothing: its scratch is a fixed array inside the library.  This file is
collected last so that a failure here never hides the other tests."""
import ctypes

import numpy as np
import pytest

import synth
from oracle import calibrate

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kv():
    from kv_cache_transform_gb300 import _build
    _build.build()
    import kv_cache_transform_gb300 as kv
    return kv


def test_static_mean_matches_calibrate_on_consecutive_calls(kv):
    import torch
    cases = [("tiny", 0, 0), ("llama31_8b_8k", 5, 1)]
    rows, refs = [], []
    for name, layer, k in cases:
        w = synth.WORKLOADS[name]
        r = synth.calib_tokens(w, layer, k)
        d = torch.from_numpy(r.view(np.int16).copy()).cuda()
        blob = kv.kvtc_calibrate([d], [layer], [k], w.n_calib, w.D, w.D,
                                 w.sink, w.window, w.budget_bits)
        refs.append(calibrate.read_blob(blob)["streams"][0]["mu"])
        rows.append((d, w))
    # two calls in a row on different inputs, then the first one again: the
    # shared scratch must not carry anything from one call to the next
    for i in (0, 1, 0):
        d, w = rows[i]
        out = torch.full((w.D,), float("nan"), dtype=torch.float64,
                         device="cuda")
        kv.kvtc_calib_mean_static(d, w.n_calib, w.D, w.D, out)
        np.testing.assert_allclose(out.cpu().numpy(), refs[i], rtol=0,
                                   atol=1e-12)


def test_static_mean_rejects_rows_wider_than_its_scratch(kv):
    import torch
    x = torch.zeros((2, 8192), dtype=torch.int16, device="cuda")
    out = torch.zeros(8192, dtype=torch.float64, device="cuda")
    code = kv.lib().kvtc_calib_mean_static(0, ctypes.c_void_p(x.data_ptr()),
                                           2, 8192, 8192,
                                           ctypes.c_void_p(out.data_ptr()),
                                           None)
    assert code == kv.KVTC_ESIZE
