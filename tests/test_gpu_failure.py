"""Failure detection on the GPU without a fault: a bounded wait that runs
out reports KVTC_FLAG_TIMEOUT through the sticky flag word, and the context
stays usable (needs a GB300)."""
import numpy as np
import pytest

import synth
from oracle import codec

from _parity import blob_for, calibrate_workload, check_decompress, \
    stream_calibs

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_sets_the_timeout_flag():
    from kv_cache_transform_gb300 import _build
    _build.build()
    import kv_cache_transform_gb300 as kv
    import torch
    name = "tiny"
    w = synth.WORKLOADS[name]
    blob = blob_for(name, calibrate_workload(name, [(0, 0)]))
    calib = kv.kvtc_calib_load(blob, 0)
    assert kv.kvtc_device_status(calib) == 0
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    kv.kvtc_wait_selftest(calib, 50000)  # 50 ms, nothing ever arrives
    b.record()
    assert kv.kvtc_device_status(calib) == kv.KVTC_FLAG_TIMEOUT
    assert a.elapsed_time(b) >= 45.0
    assert kv.kvtc_device_status(calib) == 0  # read and cleared
    # the context is still usable: the GPU restores the oracle's bitstream
    sc_enc, sc_dec = stream_calibs(blob)[(0, 0)]
    T = 300
    x = synth.eval_tokens(w, 0, 0, T=T)
    o = codec.compress_stream(x, sc_enc)
    comp = torch.from_numpy(np.frombuffer(o, np.uint8).copy()).cuda()
    out = torch.zeros((T, w.D), dtype=torch.int16, device="cuda")
    kv.kvtc_decompress(calib, 0, 1, 1, comp, len(o), T, [out], w.D)
    assert kv.kvtc_device_status(calib) == 0
    ref = codec.decompress_stream(o, T, sc_dec)
    got = out.cpu().numpy().view(np.uint16)
    s_, w_, tc = codec.split_tokens(T, w.sink, w.window)
    np.testing.assert_array_equal(got[:s_], ref[:s_])
    np.testing.assert_array_equal(got[T - w_:], ref[T - w_:])
    assert check_decompress(got[s_:T - w_], ref[s_:T - w_])["ok"]
    with pytest.raises(kv.KvtcError):
        kv.kvtc_wait_selftest(calib, 0)
    calib.free()
