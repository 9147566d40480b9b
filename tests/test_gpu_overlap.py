"""Restore/consume overlap (needs a GB300).

Layer-wise decompression exists so that a model can start on layer l while
later layers are still being restored (kvtc page, technical summary 2C;
the TTFT results of section 4).  The bench measures it with a stand-in
consumer (one query per KV head attending over a restored layer) on a
second stream that waits only for layer l's event.  This test checks the
schedule itself: with every output row pre-filled with NaN, the consumer's
per-layer results under the overlapped schedule must be finite and equal
the same consumer run after the whole cache is restored, so no layer was
read before its event."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

pytestmark = pytest.mark.gpu


def test_overlapped_consumer_sees_only_restored_layers():
    import dataclasses
    import torch
    import bench
    from kv_cache_transform_gb300 import _build
    _build.build()
    import kv_cache_transform_gb300 as kv

    w = dataclasses.replace(synth.WORKLOADS["llama31_8b_8k"], layers=6,
                            tokens=3000)
    streams = w.streams()
    T, D = w.tokens, w.D
    cal = [synth.calib_tokens_torch(w, l, k) for l, k in streams]
    blob = kv.kvtc_calibrate(cal, [l for l, _ in streams],
                             [k for _, k in streams], w.n_calib, D, D,
                             w.sink, w.window, w.budget_bits)
    calib = kv.kvtc_calib_load(blob, 0)
    x = [synth.eval_tokens_torch(w, l, k, T=T) for l, k in streams]
    total = sum(calib.stream_bytes(l, k, T) for l, k in streams)
    comp = torch.empty(total, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    kv.kvtc_compress(calib, 0, w.layers, 3, x, D, T, comp, total, stream)
    out = [torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
           for _ in streams]
    q = torch.randn((w.heads, w.head_dim), device="cuda").to(torch.bfloat16)

    def nan_fill():
        for o in out:
            o.view(torch.int16).fill_(0x7FC0)
        torch.cuda.synchronize()

    nan_fill()
    res_o, first_o, all_o = bench.overlap_schedule(
        kv, torch, calib, w, 0, w.layers, comp, out, total, stream, q, True)
    nan_fill()
    res_s, first_s, all_s = bench.overlap_schedule(
        kv, torch, calib, w, 0, w.layers, comp, out, total, stream, q, False)
    assert kv.kvtc_device_status(calib) == 0
    for a, b in zip(res_o, res_s):
        a, b = a.cpu().numpy(), b.cpu().numpy()
        assert np.all(np.isfinite(a)), "a layer was consumed before restore"
        np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-6)
    # the first layer is consumed before the whole cache is back
    assert first_o < all_s
    calib.free()
