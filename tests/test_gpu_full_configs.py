"""Full-size parity of the other workloads, in the launch shapes a user
runs them (needs a GB300).

Each test calibrates every stream with the oracle, runs the whole workload
through the C ABI in one call per direction (the streamed 70B case restores
layer by layer with an event per layer; the paged case restores 64 requests
into 16-token blocks through a seeded random block table), and checks
sampled streams against the oracle:
- compress: the GPU's records of a sampled stream obey the parity rule
  against the oracle's fp64 coefficients of the same input;
- decompress: the sampled streams' bytes in the decompress input are the
  oracle's own bitstreams, so the GPU's restored rows are compared with the
  oracle's restoration of its own bitstream (raw rows bit-exact, the rest
  within the tolerance of the parity rule).
Streams that are not sampled carry the GPU's own bitstreams and exercise the
full-size launch.
"""
import numpy as np
import pytest

import synth
from oracle import codec

from _parity import (blob_for, calibrate_forced, calibrate_workload,
                     check_decompress, check_records, record, stream_calibs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kv():
    from kv_cache_transform_gb300 import _build
    _build.build()
    import kv_cache_transform_gb300 as kv
    return kv


@pytest.fixture(scope="module")
def torch():
    import torch
    assert torch.cuda.is_available()
    return torch


def from_dev(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def check_stream_records(g: bytes, x: np.ndarray, sc_enc, T, w, tag=None):
    """Raw rows bit-exact and every record within the parity rule."""
    s_, w_, tc = codec.split_tokens(T, w.sink, w.window)
    raw = (s_ + w_) * w.D * 2
    o_raw = np.concatenate([x[:s_], x[T - w_:]]).tobytes()
    assert g[:raw] == o_raw, "raw rows differ"
    grec = np.frombuffer(g, np.uint8, tc * sc_enc.R, raw).reshape(tc, sc_enc.R)
    st = check_records(grec, x[s_:T - w_], sc_enc)
    record(tag or w.name, st=st)
    assert st["bad"] == 0, st


def check_stream_restore(got: np.ndarray, oracle_bytes: bytes, T, sc_dec, w,
                         tag=None):
    s_, w_, tc = codec.split_tokens(T, w.sink, w.window)
    ref = codec.decompress_stream(oracle_bytes, T, sc_dec)
    np.testing.assert_array_equal(got[:s_], ref[:s_])
    np.testing.assert_array_equal(got[T - w_:], ref[T - w_:])
    st = check_decompress(got[s_:T - w_], ref[s_:T - w_])
    record(tag or w.name, dst=st)
    assert st["ok"], st


def run_contiguous(kv, torch, name, sample, streamed=False, blob=None,
                   tag=None):
    w = synth.WORKLOADS[name]
    streams = w.streams()
    if blob is None:
        blob = blob_for(name, calibrate_workload(name, streams))
    scs = stream_calibs(blob)
    calib = kv.kvtc_calib_load(blob, 0)
    T, D = w.tokens, w.D
    src = [synth.eval_tokens_torch(w, l, k, T=T).view(torch.int16)
           for l, k in streams]
    total = sum(calib.stream_bytes(l, k, T) for l, k in streams)
    sb = calib.stream_bytes(0, 0, T)
    comp = torch.zeros(total, dtype=torch.uint8, device="cuda")
    kv.kvtc_compress(calib, 0, w.layers, 3, src, D, T, comp, total)
    assert kv.kvtc_device_status(calib) == 0
    gbytes = comp.cpu().numpy()
    dec_in = gbytes.copy()
    oracle_bytes = {}
    for idx in sample:
        l, k = streams[idx]
        sc_enc, _ = scs[(l, k)]
        x = from_dev(src[idx])
        check_stream_records(gbytes[idx * sb:(idx + 1) * sb].tobytes(), x,
                             sc_enc, T, w, tag)
        o = codec.compress_stream(x, sc_enc)
        assert len(o) == sb
        dec_in[idx * sb:(idx + 1) * sb] = np.frombuffer(o, np.uint8)
        oracle_bytes[idx] = o
    del src
    comp.copy_(torch.from_numpy(dec_in))
    outs = [torch.zeros((T, D), dtype=torch.int16, device="cuda")
            for _ in streams]
    if streamed:
        evs = [torch.cuda.Event() for _ in range(w.layers)]
        for e in evs:  # torch creates the CUDA event on its first record
            e.record()
        kv.kvtc_decompress(calib, 0, w.layers, 3, comp, total, T, outs, D,
                           layer_events=evs)
        evs[-1].synchronize()
    else:
        kv.kvtc_decompress(calib, 0, w.layers, 3, comp, total, T, outs, D)
    torch.cuda.synchronize()
    assert kv.kvtc_device_status(calib) == 0
    for idx in sample:
        l, k = streams[idx]
        check_stream_restore(from_dev(outs[idx]), oracle_bytes[idx], T,
                             scs[(l, k)][1], w, tag)
    calib.free()


def test_full_llama31_8b_8k_flat_k256_sampled(kv, torch):
    """Config-2 shape with a flat spectrum: 64 streams x 8192 tokens, the DP
    keeps k = 256 on every stream (single-A-buffer reconstruction)."""
    run_contiguous(kv, torch, "llama31_8b_8k_flat", (0, 1, 33, 62, 63))


def test_full_llama31_8b_8k_k336_sampled(kv, torch):
    """Config-2 workload with 21 one-bit groups set by hand on every stream
    (k = 336, the most its 1024-bit budget holds): the wide projection (two
    MMAs per K step) and reconstruction at full size."""
    name = "llama31_8b_8k"
    w = synth.WORKLOADS[name]
    widths = np.zeros(w.D // 16, dtype=np.int64)
    widths[:21] = 1
    blob = blob_for(name, calibrate_forced(name, w.streams(), widths))
    run_contiguous(kv, torch, name, (0, 1, 30, 63), blob=blob,
                   tag=f"{name}, 21 one-bit groups (k = 336)")


def test_full_cross_layer_pairs_sampled(kv, torch):
    """Cross-layer basis over layer pairs: 32 streams x 8192 tokens of
    D = 2048 (1.07 GB raw), k = 480, 256-byte records."""
    run_contiguous(kv, torch, "llama31_8b_8k_xlayer2", (0, 1, 17, 30, 31))


def test_full_mistral_nemo_12b_32k_sampled(kv, torch):
    """80 streams x 32768 tokens (5.4 GB raw), k = 112, 64-byte records."""
    run_contiguous(kv, torch, "mistral_nemo_12b_32k", (0, 1, 37, 78, 79))


def test_full_llama33_70b_16k_layer_streamed_sampled(kv, torch):
    """160 streams x 16384 tokens (5.4 GB raw), restored layer by layer on
    one stream with an event recorded after each layer."""
    run_contiguous(kv, torch, "llama33_70b_16k", (0, 1, 80, 158, 159),
                   streamed=True)


def test_full_qwen25_7b_paged_sampled(kv, torch):
    """64 requests x 56 streams x 4096 tokens (15 GB of paged cache) restored
    in one call into 16-token blocks through the seeded block table."""
    name = "qwen25_7b_paged"
    w = synth.WORKLOADS[name]
    streams = w.streams()
    entries = calibrate_workload(name, streams)
    blob = blob_for(name, entries)
    scs = stream_calibs(blob)
    calib = kv.kvtc_calib_load(blob, 0)
    T, D, bs = w.tokens, w.D, w.block_size
    table = synth.block_table(w)
    maxb = table.shape[1]
    nblocks = table.size
    sample_req = (0, 17, 63)
    sample_idx = (0, 27, 55)
    sb = calib.stream_bytes(0, 0, T)
    total = sum(calib.stream_bytes(l, k, T) for l, k in streams)
    srcs, oracle_bytes = [], {}
    for r in range(w.requests):
        x = [synth.eval_tokens_torch(w, l, k, request=r, T=T).view(torch.int16)
             for l, k in streams]
        comp = torch.zeros(total, dtype=torch.uint8, device="cuda")
        kv.kvtc_compress(calib, 0, w.layers, 3, x, D, T, comp, total)
        if r in sample_req:
            gbytes = comp.cpu().numpy()
            dec_in = gbytes.copy()
            for idx in sample_idx:
                l, k = streams[idx]
                sc_enc, _ = scs[(l, k)]
                xh = from_dev(x[idx])
                check_stream_records(
                    gbytes[idx * sb:(idx + 1) * sb].tobytes(), xh, sc_enc, T,
                    w)
                o = codec.compress_stream(xh, sc_enc)
                dec_in[idx * sb:(idx + 1) * sb] = np.frombuffer(o, np.uint8)
                oracle_bytes[(r, idx)] = o
            comp.copy_(torch.from_numpy(dec_in))
        srcs.append(comp)
        del x
    assert kv.kvtc_device_status(calib) == 0
    caches = [torch.full((nblocks, bs, D), 0x7FC0, dtype=torch.int16,
                         device="cuda") for _ in streams]
    bt = torch.from_numpy(table).cuda()
    kv.kvtc_decompress_paged(calib, 0, w.layers, 3, srcs, [T] * w.requests,
                             bt, maxb, bs, caches, nblocks)
    torch.cuda.synchronize()
    assert kv.kvtc_device_status(calib) == 0
    t = np.arange(T)
    for idx in sample_idx:
        l, k = streams[idx]
        host = from_dev(caches[idx])
        for r in sample_req:
            got = host[table[r, t // bs], t % bs]
            check_stream_restore(got, oracle_bytes[(r, idx)], T,
                                 scs[(l, k)][1], w)
    calib.free()
