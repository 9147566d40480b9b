"""Field packing on the GPU against the oracle (needs a GB300).

Inputs to the packer are the oracle's own codec streams of seeded synthetic
tokens; the GPU's packed bytes must equal the oracle's packed bytes byte for
byte (integer work), its offsets the oracle's stream sizes, and unpacking
the oracle's packed bytes on the GPU must give back the oracle's codec
streams exactly.  At full size (Llama-3.1-8B shape, 64 streams x 8192
tokens) the pack -> unpack round trip must be the identity on the GPU's
own codec output, with sampled streams replaced by oracle streams and
checked byte for byte.
"""
import numpy as np
import pytest

import synth
from oracle import codec, fieldpack

from _parity import blob_for, calibrate_workload, stream_calibs

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


_CALIBS = {}


def workload_calib(name, streams):
    key = (name, tuple(streams))
    if key not in _CALIBS:
        entries = calibrate_workload(name, streams)
        blob = blob_for(name, entries)
        _CALIBS[key] = (blob, stream_calibs(blob))
    return _CALIBS[key]


def dev_bytes(torch, b: bytes, extra: int = 0):
    t = torch.zeros(max(len(b) + extra, 16), dtype=torch.uint8, device="cuda")
    if b:
        t[:len(b)] = torch.from_numpy(np.frombuffer(b, np.uint8).copy()).cuda()
    return t


def run_pack_parity(kv, torch, name, streams, T):
    w = synth.WORKLOADS[name]
    blob, scs = workload_calib(name, streams)
    calib = kv.kvtc_calib_load(blob, 0)
    layers = sorted({l for l, _ in streams})
    layer0, nl = layers[0], layers[-1] - layers[0] + 1
    kinds = sorted({k for _, k in streams})
    mask = sum(1 << k for k in kinds)
    order = [(l, k) for l in range(layer0, layer0 + nl) for k in kinds]
    codec_streams = [codec.compress_stream(synth.eval_tokens(w, l, k, T=T),
                                           scs[(l, k)][0]) for l, k in order]
    packed_streams = [fieldpack.pack_stream(b, T, scs[s][0])
                      for b, s in zip(codec_streams, order)]
    cb = b"".join(codec_streams)
    pb = b"".join(packed_streams)
    n = len(order)
    bound = kv.kvtc_fields_bound(calib, layer0, nl, mask, T)
    assert bound >= len(pb)
    ws = kv.kvtc_fields_workspace_bytes(calib, layer0, nl, mask)
    src = dev_bytes(torch, cb)
    dst = torch.full((bound,), 0xA5, dtype=torch.uint8, device="cuda")
    offs = torch.full((n + 1,), -7, dtype=torch.int64, device="cuda")
    work = torch.full((ws,), 0x5A, dtype=torch.uint8, device="cuda")
    kv.kvtc_fields_pack(calib, layer0, nl, mask, src, len(cb), T, dst, bound,
                        offs, work, ws)
    assert kv.kvtc_device_status(calib) == 0
    want_offs = np.concatenate([[0], np.cumsum([len(p) for p in
                                                packed_streams])])
    got_offs = offs.cpu().numpy()
    np.testing.assert_array_equal(got_offs, want_offs)
    got = dst.cpu().numpy()[:len(pb)].tobytes()
    for i, s in enumerate(order):
        a, b = want_offs[i], want_offs[i + 1]
        assert got[a:b] == packed_streams[i], f"packed stream {s} differs"
    # unpack the oracle's packed bytes
    psrc = dev_bytes(torch, pb)
    poffs = torch.from_numpy(want_offs.astype(np.int64)).cuda()
    out = torch.full((max(len(cb), 16),), 0xA5, dtype=torch.uint8,
                     device="cuda")
    kv.kvtc_fields_unpack(calib, layer0, nl, mask, psrc, len(pb), poffs, T,
                          out, len(cb))
    assert kv.kvtc_device_status(calib) == 0
    assert out.cpu().numpy()[:len(cb)].tobytes() == cb
    calib.free()
    return len(cb), len(pb)


@pytest.mark.parametrize("T", [0, 1, 4, 20, 21, 147, 148, 276, 1000])
def test_tiny_pack_parity(kv, torch, T):
    """One stream, 32-byte records; T = 20 leaves no coded token (sink 4,
    window 16), 147 and 276 give ragged last tiles."""
    run_pack_parity(kv, torch, "tiny", [(0, 0)], T)


def test_d192_pack_parity(kv, torch):
    run_pack_parity(kv, torch, "edge_d192", [(0, 0), (0, 1)], 700)


def test_d192_256_byte_records_pack_parity(kv, torch):
    run_pack_parity(kv, torch, "edge_d192_r256", [(0, 0), (0, 1)], 600)


def test_d384_fifteen_groups_pack_parity(kv, torch):
    """k = 240: 15 active groups, 30 field slots per record."""
    run_pack_parity(kv, torch, "edge_d384",
                    [(0, 0), (0, 1), (1, 0), (1, 1)], 900)


def test_d384_v_only_pack_parity(kv, torch):
    run_pack_parity(kv, torch, "edge_d384", [(0, 1), (1, 1)], 517)


def test_corrupt_header_is_flagged_and_skipped(kv, torch):
    """A packed stream whose header disagrees with T is skipped with
    KVTC_FLAG_FORMAT; the other streams still restore."""
    name, streams, T = "edge_d192", [(0, 0), (0, 1)], 300
    w = synth.WORKLOADS[name]
    blob, scs = workload_calib(name, streams)
    calib = kv.kvtc_calib_load(blob, 0)
    cbs = [codec.compress_stream(synth.eval_tokens(w, l, k, T=T), scs[(l, k)][0])
           for l, k in streams]
    pbs = [bytearray(fieldpack.pack_stream(b, T, scs[s][0]))
           for b, s in zip(cbs, streams)]
    pbs[0][4] ^= 1                      # T_c of stream 0
    pb = b"".join(bytes(p) for p in pbs)
    offs = np.array([0, len(pbs[0]), len(pb)], dtype=np.int64)
    out = torch.full((len(cbs[0]) + len(cbs[1]),), 0xA5, dtype=torch.uint8,
                     device="cuda")
    kv.kvtc_fields_unpack(calib, 0, 1, 3, dev_bytes(torch, pb), len(pb),
                          torch.from_numpy(offs).cuda(), T, out, out.numel())
    assert kv.kvtc_device_status(calib) == kv.KVTC_FLAG_FORMAT
    host = out.cpu().numpy().tobytes()
    assert host[len(cbs[0]):] == cbs[1]
    assert host[:len(cbs[0])] == b"\xa5" * len(cbs[0])
    # offsets past the end of the input: skipped the same way
    bad = np.array([0, len(pbs[0]), len(pb) + 256], dtype=np.int64)
    kv.kvtc_fields_unpack(calib, 0, 1, 3, dev_bytes(torch, pb), len(pb),
                          torch.from_numpy(bad).cuda(), T, out, out.numel())
    assert kv.kvtc_device_status(calib) == kv.KVTC_FLAG_FORMAT
    calib.free()


def test_full_llama31_8b_8k_round_trip(kv, torch):
    """64 streams x 8192 tokens: GPU compress, pack, unpack is the identity;
    sampled streams carry oracle codec bytes and pack to the oracle's
    packed bytes."""
    name = "llama31_8b_8k"
    w = synth.WORKLOADS[name]
    streams = w.streams()
    blob, scs = workload_calib(name, streams)
    calib = kv.kvtc_calib_load(blob, 0)
    T, D = w.tokens, w.D
    src = [synth.eval_tokens_torch(w, l, k, T=T).view(torch.int16)
           for l, k in streams]
    sb = calib.stream_bytes(0, 0, T)
    total = sb * len(streams)
    comp = torch.zeros(total, dtype=torch.uint8, device="cuda")
    kv.kvtc_compress(calib, 0, w.layers, 3, src, D, T, comp, total)
    del src
    sample = (0, 1, 33, 63)
    host = comp.cpu().numpy()
    oracle_packed = {}
    for idx in sample:
        l, k = streams[idx]
        sc = scs[(l, k)][0]
        o = codec.compress_stream(synth.eval_tokens(w, l, k, T=T), sc)
        host[idx * sb:(idx + 1) * sb] = np.frombuffer(o, np.uint8)
        oracle_packed[idx] = fieldpack.pack_stream(o, T, sc)
    comp.copy_(torch.from_numpy(host))
    bound = kv.kvtc_fields_bound(calib, 0, w.layers, 3, T)
    ws = kv.kvtc_fields_workspace_bytes(calib, 0, w.layers, 3)
    packed = torch.empty(bound, dtype=torch.uint8, device="cuda")
    offs = torch.empty(len(streams) + 1, dtype=torch.int64, device="cuda")
    work = torch.empty(ws, dtype=torch.uint8, device="cuda")
    kv.kvtc_fields_pack(calib, 0, w.layers, 3, comp, total, T, packed, bound,
                        offs, work, ws)
    back = torch.full((total,), 0xA5, dtype=torch.uint8, device="cuda")
    kv.kvtc_fields_unpack(calib, 0, w.layers, 3, packed, bound, offs, T,
                          back, total)
    assert kv.kvtc_device_status(calib) == 0
    assert torch.equal(back, comp)
    o = offs.cpu().numpy()
    pk = packed.cpu().numpy()
    for idx in sample:
        assert pk[o[idx]:o[idx + 1]].tobytes() == oracle_packed[idx]
    # the stage saves bytes on this workload
    assert o[-1] < 0.95 * total
    calib.free()


def test_more_streams_than_one_launch_group(kv, torch):
    """300 streams (150 layers x K, V) in one call: the packer runs two
    launch groups, the second starting from the offset the first wrote."""
    from oracle import calibrate
    w = synth.WORKLOADS["tiny"]
    mu, V, evals, widths, _ = calibrate.calibrate_stream(
        synth.calib_tokens(w, 0, 0), w.budget_bits)
    entries = [(l, k, mu, V, evals, widths)
               for l in range(150) for k in (0, 1)]
    blob = calibrate.write_blob(entries, w.sink, w.window, w.budget_bits)
    sc = stream_calibs(blob)[(0, 0)][0]
    calib = kv.kvtc_calib_load(blob, 0)
    T = 300
    order = [(l, k) for l in range(150) for k in (0, 1)]
    cbs = [codec.compress_stream(synth.eval_tokens(w, l, k, T=T), sc)
           for l, k in order]
    pbs = [fieldpack.pack_stream(b, T, sc) for b in cbs]
    cb, pb = b"".join(cbs), b"".join(pbs)
    bound = kv.kvtc_fields_bound(calib, 0, 150, 3, T)
    ws = kv.kvtc_fields_workspace_bytes(calib, 0, 150, 3)
    dst = torch.full((bound,), 0xA5, dtype=torch.uint8, device="cuda")
    offs = torch.full((301,), -7, dtype=torch.int64, device="cuda")
    work = torch.empty(ws, dtype=torch.uint8, device="cuda")
    kv.kvtc_fields_pack(calib, 0, 150, 3, dev_bytes(torch, cb), len(cb), T,
                        dst, bound, offs, work, ws)
    assert kv.kvtc_device_status(calib) == 0
    want = np.concatenate([[0], np.cumsum([len(p) for p in pbs])])
    np.testing.assert_array_equal(offs.cpu().numpy(), want)
    assert dst.cpu().numpy()[:len(pb)].tobytes() == pb
    out = torch.zeros(len(cb), dtype=torch.uint8, device="cuda")
    kv.kvtc_fields_unpack(calib, 0, 150, 3, dst, bound, offs, T, out, len(cb))
    assert kv.kvtc_device_status(calib) == 0
    assert out.cpu().numpy().tobytes() == cb
    calib.free()


def test_fields_host_refusals(kv, torch):
    """What kvtc_fields_pack and kvtc_fields_unpack refuse on the host,
    before any launch: buffers too small, misaligned pointers, a negative T
    and an invalid K|V mask.  Nothing is written and no device flag is
    raised; the same arguments unchanged then pack and unpack byte for
    byte."""
    name, T = "tiny", 300
    w = synth.WORKLOADS[name]
    blob, scs = workload_calib(name, [(0, 0)])
    calib = kv.kvtc_calib_load(blob, 0)
    comp = dev_bytes(torch, codec.compress_stream(
        synth.eval_tokens(w, 0, 0, T=T), scs[(0, 0)][0]))
    need = calib.stream_bytes(0, 0, T)
    bound = kv.kvtc_fields_bound(calib, 0, 1, 1, T)
    ws = kv.kvtc_fields_workspace_bytes(calib, 0, 1, 1)
    assert ws >= 32
    pk = torch.full((bound + 64,), 0xA5, dtype=torch.uint8, device="cuda")
    offs = torch.full((4,), -7, dtype=torch.int64, device="cuda")
    work = torch.zeros(ws + 64, dtype=torch.uint8, device="cuda")
    back = torch.full((need + 64,), 0x5A, dtype=torch.uint8, device="cuda")
    good = dict(src=comp, src_bytes=need, T=T, dst=pk, cap=bound,
                offsets=offs, work=work, ws=ws, mask=1)

    def pack_refused(**change):
        a = dict(good, **change)
        with pytest.raises(kv.KvtcError) as e:
            kv.kvtc_fields_pack(calib, 0, 1, a["mask"], a["src"],
                                a["src_bytes"], a["T"], a["dst"], a["cap"],
                                a["offsets"], a["work"], a["ws"])
        return e.value.code

    assert pack_refused(src_bytes=need - 16) == kv.KVTC_ESIZE
    assert pack_refused(cap=bound - 16) == kv.KVTC_ESIZE
    assert pack_refused(ws=ws - 16) == kv.KVTC_ESIZE
    assert pack_refused(src=comp.data_ptr() + 8) == kv.KVTC_EALIGN
    assert pack_refused(dst=pk.data_ptr() + 8) == kv.KVTC_EALIGN
    assert pack_refused(work=work.data_ptr() + 8) == kv.KVTC_EALIGN
    assert pack_refused(offsets=offs.data_ptr() + 4) == kv.KVTC_EALIGN
    assert pack_refused(T=-1) == kv.KVTC_EINVAL
    assert pack_refused(mask=0) == kv.KVTC_EINVAL
    torch.cuda.synchronize()
    assert torch.all(pk == 0xA5) and torch.all(offs == -7)
    assert kv.kvtc_device_status(calib) == 0
    kv.kvtc_fields_pack(calib, 0, 1, 1, comp, need, T, pk, bound, offs, work,
                        ws)
    torch.cuda.synchronize()
    size = int(offs[1].item())
    assert int(offs[0].item()) == 0 and 256 <= size <= bound

    def unpack_refused(src=pk, src_bytes=size, offsets=offs, T=T, dst=back,
                       dst_bytes=need):
        with pytest.raises(kv.KvtcError) as e:
            kv.kvtc_fields_unpack(calib, 0, 1, 1, src, src_bytes, offsets, T,
                                  dst, dst_bytes)
        return e.value.code

    assert unpack_refused(dst_bytes=need - 16) == kv.KVTC_ESIZE
    assert unpack_refused(src_bytes=128) == kv.KVTC_ESIZE
    assert unpack_refused(src=pk.data_ptr() + 8) == kv.KVTC_EALIGN
    assert unpack_refused(dst=back.data_ptr() + 8) == kv.KVTC_EALIGN
    assert unpack_refused(offsets=offs.data_ptr() + 4) == kv.KVTC_EALIGN
    assert unpack_refused(T=-1) == kv.KVTC_EINVAL
    torch.cuda.synchronize()
    assert torch.all(back == 0x5A)
    assert kv.kvtc_device_status(calib) == 0
    kv.kvtc_fields_unpack(calib, 0, 1, 1, pk, size, offs, T, back, need)
    torch.cuda.synchronize()
    assert kv.kvtc_device_status(calib) == 0
    assert torch.equal(back[:need], comp[:need])
    assert torch.all(back[need:] == 0x5A)
    calib.free()
