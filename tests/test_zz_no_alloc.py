"""The allocation-free mean entry point, for callers that own all device
memory themselves (a serving engine's preallocated KV pool) or cannot afford
the device-wide synchronisation that cudaMalloc / cudaFree bring.

kvtc_calib_mean_static must give the oracle's per-channel calibration mean
(the mu of the kvtc page's calibration, technical summary 2A), call after
call, while allocating nothing: its scratch is a fixed array inside the
library.  This file is collected last so that a failure here never hides
the other tests."""
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


def test_static_mean_matches_oracle_on_consecutive_calls(kv):
    import torch
    cases = [("tiny", 0, 0), ("llama31_8b_8k", 5, 1)]
    rows, refs, outs = [], [], []
    for name, layer, k in cases:
        w = synth.WORKLOADS[name]
        r = synth.calib_tokens(w, layer, k)
        refs.append(calibrate.pca(r)[0])       # the oracle's mean
        rows.append((torch.from_numpy(r.view(np.int16).copy()).cuda(), w))
        outs.append(torch.empty(w.D, dtype=torch.float64, device="cuda"))
    # two calls in a row on different inputs, then the first one again: the
    # shared scratch must not carry anything from one call to the next
    for i in (0, 1, 0):
        d, w = rows[i]
        outs[i].fill_(float("nan"))
        kv.kvtc_calib_mean_static(d, w.n_calib, w.D, w.D, outs[i])
        np.testing.assert_allclose(outs[i].cpu().numpy(), refs[i], rtol=0,
                                   atol=1e-12)


def test_static_mean_allocates_no_device_memory(kv):
    """After the first call on the device (its one-time set-up), further
    calls leave the driver's free device memory unchanged."""
    import torch
    w = synth.WORKLOADS["llama31_8b_8k"]
    r = synth.calib_tokens(w, 3, 0)
    d = torch.from_numpy(r.view(np.int16).copy()).cuda()
    out = torch.empty(w.D, dtype=torch.float64, device="cuda")
    kv.kvtc_calib_mean_static(d, w.n_calib, w.D, w.D, out)   # set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        kv.kvtc_calib_mean_static(d, w.n_calib, w.D, w.D, out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    np.testing.assert_allclose(out.cpu().numpy(), calibrate.pca(r)[0],
                               rtol=0, atol=1e-12)


def test_static_mean_rejects_rows_wider_than_its_scratch(kv):
    import torch
    x = torch.zeros((2, 8192), dtype=torch.int16, device="cuda")
    out = torch.zeros(8192, dtype=torch.float64, device="cuda")
    code = kv.lib().kvtc_calib_mean_static(0, ctypes.c_void_p(x.data_ptr()),
                                           2, 8192, 8192,
                                           ctypes.c_void_p(out.data_ptr()),
                                           None)
    assert code == kv.KVTC_ESIZE
