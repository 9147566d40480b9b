"""Restore straight from packed streams on the GPU (needs a GB300).

kvtc_decompress_packed reads the packed streams of the field-packing stage
and unpacks each record's fields inside the restore kernel.  Its output must
be bit-identical to kvtc_decompress of the codec streams the packed bytes
came from (the same kernel arithmetic on the same fields, codes and planes),
and, through that, within the restore tolerance of the oracle: raw rows
exact, coded rows rel L2 <= 2e-3 and every element within 1 bf16 ulp + 1e-3
of the oracle's restore.  Inputs are the oracle's codec and packed streams of
seeded synthetic tokens; at full size (Llama-3.1-8B shape, 64 streams x 8192
tokens) the GPU's own compress and pack feed both restores.
"""
import numpy as np
import pytest

import synth
from oracle import codec, fieldpack

from _parity import (blob_for, calibrate_workload, check_decompress, record,
                     stream_calibs)

pytestmark = pytest.mark.gpu

NAN_BF16 = 0x7FC0


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


def dev_bytes(torch, b: bytes, pinned: bool = False):
    t = torch.zeros(max(len(b), 16), dtype=torch.uint8,
                    pin_memory=pinned)
    if b:
        t[:len(b)] = torch.from_numpy(np.frombuffer(b, np.uint8).copy())
    return t if pinned else t.cuda()


def outputs(torch, n, T, ld):
    return [torch.full((max(T, 1), ld), NAN_BF16, dtype=torch.int16,
                       device="cuda") for _ in range(n)]


def restore_pair(kv, torch, calib, layer0, nl, mask, cb, pb, offs, T, D, ld,
                 n_out, pinned=False, events=False):
    """kvtc_decompress of the codec bytes and kvtc_decompress_packed of the
    packed bytes into NaN-filled outputs; returns both output lists."""
    a = outputs(torch, n_out, T, ld)
    kv.kvtc_decompress(calib, layer0, nl, mask, dev_bytes(torch, cb), len(cb),
                       T, a, ld)
    assert kv.kvtc_device_status(calib) == 0
    b = outputs(torch, n_out, T, ld)
    src = dev_bytes(torch, pb, pinned)
    o = torch.from_numpy(offs.astype(np.int64))
    o = o.pin_memory() if pinned else o.cuda()
    ev = None
    if events:
        ev = [torch.cuda.Event() for _ in range(nl)]
        for e in ev:  # torch creates the CUDA event on its first record
            e.record()
    kv.kvtc_decompress_packed(calib, layer0, nl, mask, src, len(pb), o, T,
                              b, ld, layer_events=ev)
    if ev:
        for e in ev:
            e.synchronize()
    assert kv.kvtc_device_status(calib) == 0
    return a, b


def run_packed_restore(kv, torch, name, streams, T, ld_pad=0, pinned=False,
                       events=False):
    w = synth.WORKLOADS[name]
    blob, scs = workload_calib(name, streams)
    calib = kv.kvtc_calib_load(blob, 0)
    layers = sorted({l for l, _ in streams})
    layer0, nl = layers[0], layers[-1] - layers[0] + 1
    kinds = sorted({k for _, k in streams})
    mask = sum(1 << k for k in kinds)
    order = [(l, k) for l in range(layer0, layer0 + nl) for k in kinds]
    D = w.D
    ld = D + ld_pad
    xs = {s: synth.eval_tokens(w, s[0], s[1], T=T) for s in order}
    cbs = [codec.compress_stream(xs[s], scs[s][0]) for s in order]
    pbs = [fieldpack.pack_stream(b, T, scs[s][0]) for b, s in zip(cbs, order)]
    cb, pb = b"".join(cbs), b"".join(pbs)
    offs = np.concatenate([[0], np.cumsum([len(p) for p in pbs])])
    a, b = restore_pair(kv, torch, calib, layer0, nl, mask, cb, pb, offs, T,
                        D, ld, 2 * nl, pinned, events)
    s_, w_, tc = codec.split_tokens(T, w.sink, w.window)
    for (l, k), cbytes in zip(order, cbs):
        j = 2 * (l - layer0) + k
        assert torch.equal(a[j], b[j]), f"stream {(l, k)} differs"
        if T == 0:
            continue
        got = b[j].cpu().numpy().view(np.uint16)[:T]
        assert np.all(got[:, D:] == NAN_BF16)  # padding columns untouched
        # the decoder's calibration: V_kept held as fp16
        ref = codec.decompress_stream(cbytes, T, scs[(l, k)][1])
        np.testing.assert_array_equal(got[:s_, :D], ref[:s_])
        np.testing.assert_array_equal(got[T - w_:, :D], ref[T - w_:])
        st = check_decompress(got[s_:T - w_, :D], ref[s_:T - w_])
        record(name + " (restore from packed)", dst=st)
        assert st["ok"], st
    calib.free()


@pytest.mark.parametrize("T", [0, 1, 4, 20, 21, 147, 148, 276, 1000])
def test_tiny_packed_restore(kv, torch, T):
    """One stream, 32-byte records: T <= 20 leaves no coded token (sink 4,
    window 16: the raw rows alone, through the copy launch), 21 one coded
    token, 147 and 276 ragged last warps and tiles."""
    run_packed_restore(kv, torch, "tiny", [(0, 0)], T)


def test_d192_packed_restore_padded_rows(kv, torch):
    run_packed_restore(kv, torch, "edge_d192", [(0, 0), (0, 1)], 700,
                       ld_pad=64)


def test_d192_256_byte_records_packed_restore(kv, torch):
    """Every group at width 8: the longest record, packed records of 248
    bytes spread over 16-byte loads that straddle tokens."""
    run_packed_restore(kv, torch, "edge_d192_r256", [(0, 0), (0, 1)], 600)


def test_d384_fifteen_groups_packed_restore(kv, torch):
    """k = 240: 15 active groups, 30 field slots per record (the most field
    packing holds)."""
    run_packed_restore(kv, torch, "edge_d384",
                       [(0, 0), (0, 1), (1, 0), (1, 1)], 900)


def test_d384_v_only_from_pinned_host_with_layer_events(kv, torch):
    """Packed bytes and offsets in pinned host memory, read by the kernels
    over the host link; one completion event per layer."""
    run_packed_restore(kv, torch, "edge_d384", [(0, 1), (1, 1)], 517,
                       pinned=True, events=True)


def test_packed_restore_refusals(kv, torch):
    name = "edge_d192"
    blob, _ = workload_calib(name, [(0, 0), (0, 1)])
    calib = kv.kvtc_calib_load(blob, 0)
    out = outputs(torch, 2, 300, 192)
    src = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    offs = torch.zeros(3, dtype=torch.int64, device="cuda")
    with pytest.raises(kv.KvtcError) as e:      # shorter than 256 a stream
        kv.kvtc_decompress_packed(calib, 0, 1, 3, src, 256, offs, 300, out,
                                  192)
    assert e.value.code == kv.KVTC_ESIZE
    with pytest.raises(kv.KvtcError) as e:      # offsets not 8-byte aligned
        kv.kvtc_decompress_packed(calib, 0, 1, 3, src, 4096,
                                  src[4:].data_ptr(), 300, out, 192)
    assert e.value.code == kv.KVTC_EALIGN
    with pytest.raises(kv.KvtcError) as e:      # pageable host input
        kv.kvtc_decompress_packed(calib, 0, 1, 3, src.cpu(), 4096, offs, 300,
                                  out, 192)
    assert e.value.code == kv.KVTC_EINVAL
    assert kv.kvtc_device_status(calib) == 0
    calib.free()


def zero_records(cb: bytes, T: int, sc) -> bytes:
    """The codec stream with every record set to zeros."""
    s_, w_, tc = codec.split_tokens(T, sc.sink, sc.window)
    b = bytearray(cb)
    at = (s_ + w_) * sc.D * 2
    R = codec.record_bytes(sc.budget_bits)
    b[at:at + tc * R] = bytes(tc * R)
    return bytes(b)


def test_corrupt_packed_streams_are_flagged(kv, torch):
    """A packed stream whose header, slot table or extent does not match is
    flagged KVTC_FLAG_FORMAT without a fault: its coded tokens restore as
    from all-zero records; its raw rows are copied whenever its extent
    frames them; the other stream restores as from intact input."""
    name, streams, T = "edge_d192", [(0, 0), (0, 1)], 300
    w = synth.WORKLOADS[name]
    blob, scs = workload_calib(name, streams)
    calib = kv.kvtc_calib_load(blob, 0)
    D = w.D
    s_, w_, tc = codec.split_tokens(T, w.sink, w.window)
    cbs = [codec.compress_stream(synth.eval_tokens(w, l, k, T=T),
                                 scs[(l, k)][0]) for l, k in streams]
    pbs = [bytearray(fieldpack.pack_stream(b, T, scs[s][0]))
           for b, s in zip(cbs, streams)]
    n0, n1 = len(pbs[0]), len(pbs[1])

    def codec_restore(bufs):
        out = outputs(torch, 2, T, D)
        cb = b"".join(bufs)
        kv.kvtc_decompress(calib, 0, 1, 3, dev_bytes(torch, cb), len(cb), T,
                           out, D)
        assert kv.kvtc_device_status(calib) == 0
        return [o.cpu().numpy().view(np.uint16).copy() for o in out]

    intact = codec_restore(cbs)
    zeroed = codec_restore([zero_records(b, T, scs[s][0])
                            for b, s in zip(cbs, streams)])

    def check(pb_list, offs, bad, raw_kept, nbytes=None):
        # bad: the flagged stream, or a tuple of them
        pb = b"".join(bytes(p) for p in pb_list)
        out = outputs(torch, 2, T, D)
        kv.kvtc_decompress_packed(calib, 0, 1, 3, dev_bytes(torch, pb),
                                  len(pb) if nbytes is None else nbytes,
                                  torch.from_numpy(offs).cuda(), T, out, D)
        assert kv.kvtc_device_status(calib) == kv.KVTC_FLAG_FORMAT
        for j in range(2):
            got = out[j].cpu().numpy().view(np.uint16)
            if j not in (bad if isinstance(bad, tuple) else (bad,)):
                np.testing.assert_array_equal(got, intact[j])
                continue
            want = zeroed[j].copy()
            if raw_kept:
                want[:s_] = intact[j][:s_]
                want[T - w_:] = intact[j][T - w_:]
            else:
                want[:s_] = NAN_BF16
                want[T - w_:] = NAN_BF16
            np.testing.assert_array_equal(got, want)

    good = np.array([0, n0, n0 + n1], dtype=np.int64)
    for at in (0, 4, 8, 10):                # magic, T_c, Rp, slot count
        bad = [bytearray(p) for p in pbs]
        bad[0][at] ^= 1
        check(bad, good, 0, True)
    bad = [bytearray(p) for p in pbs]
    bad[1][16 + 1] = 7                      # a slot's dbits above 6
    check(bad, good, 1, True)
    # stream 1's range shorter than its records, or past the input's end
    check(pbs, np.array([0, n0, n0 + 256], dtype=np.int64), 1, False)
    check(pbs, good, 1, False, nbytes=n0 + n1 - 256)
    # an offset off the 16-byte grid: the end of stream 0 and the start of
    # stream 1, both flagged
    check(pbs, np.array([0, n0 + 8, n0 + n1], dtype=np.int64), (0, 1), False)
    calib.free()


def test_no_coded_token_checks_the_header(kv, torch):
    """T = 12 (sink 4 + 8 window rows, no record): the raw rows come back
    through the copy launch, which also checks magic and T_c; a stream whose
    T_c is wrong is flagged and left untouched, the other restored."""
    name, streams, T = "edge_d192", [(0, 0), (0, 1)], 12
    w = synth.WORKLOADS[name]
    blob, scs = workload_calib(name, streams)
    calib = kv.kvtc_calib_load(blob, 0)
    D = w.D
    cbs = [codec.compress_stream(synth.eval_tokens(w, l, k, T=T),
                                 scs[(l, k)][0]) for l, k in streams]
    pbs = [bytearray(fieldpack.pack_stream(b, T, scs[s][0]))
           for b, s in zip(cbs, streams)]
    pbs[1][4] ^= 1
    pb = b"".join(bytes(p) for p in pbs)
    offs = np.array([0, len(pbs[0]), len(pb)], dtype=np.int64)
    out = outputs(torch, 2, T, D)
    kv.kvtc_decompress_packed(calib, 0, 1, 3, dev_bytes(torch, pb), len(pb),
                              torch.from_numpy(offs).cuda(), T, out, D)
    assert kv.kvtc_device_status(calib) == kv.KVTC_FLAG_FORMAT
    x0 = synth.eval_tokens(w, 0, 0, T=T)
    np.testing.assert_array_equal(out[0].cpu().numpy().view(np.uint16), x0)
    assert np.all(out[1].cpu().numpy().view(np.uint16) == NAN_BF16)
    calib.free()


def test_more_streams_than_one_launch_group(kv, torch):
    """300 streams (150 layers x K, V) in one call: four restore launches of
    up to 96 streams, each finding its streams through the offsets."""
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
    offs = np.concatenate([[0], np.cumsum([len(p) for p in pbs])])
    a, b = restore_pair(kv, torch, calib, 0, 150, 3, b"".join(cbs),
                        b"".join(pbs), offs, T, w.D, w.D, 300)
    for j in range(300):
        assert torch.equal(a[j], b[j]), j
    calib.free()


def test_full_llama31_8b_8k_restore_from_packed(kv, torch):
    """64 streams x 8192 tokens: GPU compress and pack, then the restore from
    the packed bytes (in HBM, and in pinned host memory) equals the restore
    of the codec streams bit for bit."""
    name = "llama31_8b_8k"
    w = synth.WORKLOADS[name]
    streams = w.streams()
    blob, _ = workload_calib(name, streams)
    calib = kv.kvtc_calib_load(blob, 0)
    T, D = w.tokens, w.D
    src = [synth.eval_tokens_torch(w, l, k, T=T).view(torch.int16)
           for l, k in streams]
    total = calib.stream_bytes(0, 0, T) * len(streams)
    comp = torch.zeros(total, dtype=torch.uint8, device="cuda")
    kv.kvtc_compress(calib, 0, w.layers, 3, src, D, T, comp, total)
    del src
    bound = kv.kvtc_fields_bound(calib, 0, w.layers, 3, T)
    ws = kv.kvtc_fields_workspace_bytes(calib, 0, w.layers, 3)
    packed = torch.empty(bound, dtype=torch.uint8, device="cuda")
    offs = torch.empty(len(streams) + 1, dtype=torch.int64, device="cuda")
    work = torch.empty(ws, dtype=torch.uint8, device="cuda")
    kv.kvtc_fields_pack(calib, 0, w.layers, 3, comp, total, T, packed, bound,
                        offs, work, ws)
    assert kv.kvtc_device_status(calib) == 0
    ref = outputs(torch, len(streams), T, D)
    kv.kvtc_decompress(calib, 0, w.layers, 3, comp, total, T, ref, D)
    got = outputs(torch, len(streams), T, D)
    kv.kvtc_decompress_packed(calib, 0, w.layers, 3, packed, bound, offs, T,
                              got, D)
    assert kv.kvtc_device_status(calib) == 0
    for j in range(len(streams)):
        assert torch.equal(ref[j], got[j]), j
    n = int(offs[-1].item())
    host = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    host.copy_(packed[:n])
    hoffs = offs.cpu().pin_memory()
    got = outputs(torch, len(streams), T, D)
    kv.kvtc_decompress_packed(calib, 0, w.layers, 3, host, n, hoffs, T, got,
                              D)
    assert kv.kvtc_device_status(calib) == 0
    for j in range(len(streams)):
        assert torch.equal(ref[j], got[j]), j
    calib.free()
