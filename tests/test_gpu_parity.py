"""CUDA path vs the fp64 oracle, through the C ABI (needs a GB300)."""
import numpy as np
import pytest

import synth
from oracle import codec, fp

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


def to_dev(torch, bits: np.ndarray, ld: int = None):
    T, D = bits.shape
    ld = ld or D
    t = torch.zeros((T, ld), dtype=torch.int16, device="cuda")
    if T:
        t[:, :D] = torch.from_numpy(bits.view(np.int16).copy()).cuda()
    return t


def from_dev(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def run_roundtrip(kv, torch, name, streams, T, ld_pad=0, sample=None,
                  blob=None, tag=None):
    """Compress x of each stream on the GPU and with the oracle, compare;
    decompress the oracle's bitstream on the GPU, compare.  `blob`: a
    calibration to use instead of the oracle's DP calibration of `name`."""
    w = synth.WORKLOADS[name]
    if blob is None:
        blob = blob_for(name, calibrate_workload(name, streams))
    tag = tag or name
    scs = stream_calibs(blob)
    calib = kv.kvtc_calib_load(blob, 0)
    layers = sorted({l for l, _ in streams})
    layer0, nl = layers[0], layers[-1] - layers[0] + 1
    kinds = sorted({k for _, k in streams})
    mask = sum(1 << k for k in kinds)
    D = w.D
    ld = D + ld_pad
    xs, src = {}, [None] * (2 * nl)
    for l, k in streams:
        xs[(l, k)] = synth.eval_tokens(w, l, k, T=T)
        src[2 * (l - layer0) + k] = to_dev(torch, xs[(l, k)], ld)
    order = [(l, k) for l in range(layer0, layer0 + nl) for k in kinds]
    sizes = [calib.stream_bytes(l, k, T) for l, k in order]
    total = sum(sizes)
    dst = torch.full((max(total, 16),), -1, dtype=torch.uint8, device="cuda")
    kv.kvtc_compress(calib, layer0, nl, mask, src, ld, T, dst, total)
    assert kv.kvtc_device_status(calib) == 0
    gpu = dst.cpu().numpy()[:total]
    s_, w_, tc = codec.split_tokens(T, w.sink, w.window)
    off = 0
    oracle_stream = {}
    stats = []
    for (l, k), sz in zip(order, sizes):
        sc_enc, sc_dec = scs[(l, k)]
        g = gpu[off:off + sz].tobytes()
        o = codec.compress_stream(xs[(l, k)], sc_enc)
        assert len(o) == sz
        raw = (s_ + w_) * D * 2
        assert g[:raw] == o[:raw], "raw rows differ"
        R = sc_enc.R
        assert g[raw + tc * R:] == o[raw + tc * R:], "padding differs"
        rows = np.arange(tc) if sample is None else sample(tc)
        grec = np.frombuffer(g, np.uint8, tc * R, raw).reshape(tc, R)[rows]
        st = check_records(grec, xs[(l, k)][s_ + rows], sc_enc)
        record(tag, st=st)
        assert st["bad"] == 0, st
        stats.append(st)
        oracle_stream[(l, k)] = o
        off += sz
    # decompress the oracle's bitstream
    ob = b"".join(oracle_stream[s] for s in order)
    srcd = torch.from_numpy(np.frombuffer(ob, np.uint8).copy()).cuda() \
        if ob else torch.zeros(16, dtype=torch.uint8, device="cuda")
    outs = [None] * (2 * nl)
    for l, k in streams:
        outs[2 * (l - layer0) + k] = torch.full((max(T, 1), ld), 0x7FC0,
                                                dtype=torch.int16,
                                                device="cuda")
    kv.kvtc_decompress(calib, layer0, nl, mask, srcd, len(ob), T, outs, ld)
    assert kv.kvtc_device_status(calib) == 0
    dstats = []
    for l, k in streams:
        sc_enc, sc_dec = scs[(l, k)]
        got = from_dev(outs[2 * (l - layer0) + k])[:T, :D]
        ref = codec.decompress_stream(oracle_stream[(l, k)], T, sc_dec)
        np.testing.assert_array_equal(got[:s_], ref[:s_])
        np.testing.assert_array_equal(got[T - w_:], ref[T - w_:])
        st = check_decompress(got[s_:T - w_], ref[s_:T - w_])
        record(tag, dst=st)
        assert st["ok"], st
        dstats.append(st)
        if ld_pad:  # padding columns untouched
            pad = from_dev(outs[2 * (l - layer0) + k])[:T, D:]
            assert np.all(pad == 0x7FC0)
    calib.free()
    return stats, dstats


@pytest.mark.parametrize("T", [0, 1, 4, 20, 21, 147, 256, 1000, 2049])
def test_tiny_parity(kv, torch, T):
    run_roundtrip(kv, torch, "tiny", [(0, 0)], T)


def test_tiny_row_stride(kv, torch):
    run_roundtrip(kv, torch, "tiny", [(0, 0)], 700, ld_pad=24)


def test_d192_64_column_chunks_odd_k_blocks(kv, torch):
    """D = 192: 64-column output chunks (four accumulators in the ring) and
    three 64-wide K blocks for the projection (the last stage half
    empty)."""
    run_roundtrip(kv, torch, "edge_d192", [(0, 0), (0, 1)], 700)


def test_d192_256_byte_records(kv, torch):
    """Every group at width 8: 256-byte records, the longest the format has
    (the decompress B ring drops to one stage to make room for them)."""
    run_roundtrip(kv, torch, "edge_d192_r256", [(0, 0), (0, 1)], 600)


def test_d384_128_column_chunks(kv, torch):
    """D = 384: three 128-column output chunks (two accumulators), k = 240
    (sixteen MMA K steps with the mean step, every predicated step on)."""
    run_roundtrip(kv, torch, "edge_d384", [(0, 0), (0, 1), (1, 0), (1, 1)],
                  900, ld_pad=64)


def subspace_blob(name, streams, ngroups, width):
    """Calibration built by hand for a row too wide for the oracle's PCA in
    a test (D = 8192): the mean is the generator's, the basis an orthonormal
    basis of the generator's signal subspace (QR of its mixing matrix), and
    the first `ngroups` groups are kept at `width` bits."""
    w = synth.WORKLOADS[name]
    entries = []
    for l, k in streams:
        p = synth.stream_params(w, l, k)
        q, _ = np.linalg.qr(p.A)
        kk = 16 * ngroups
        assert q.shape[1] >= kk
        widths = np.zeros(w.D // 16, dtype=np.int64)
        widths[:ngroups] = width
        entries.append((l, k, p.mu, q[:, :kk], np.zeros(w.D), widths))
    return blob_for(name, entries)


def test_max_d8192(kv, torch):
    """D = 8192, the widest row the kernels take: 128 K blocks per
    projection tile and 32 output chunks per restore tile, contiguous and
    paged (16-token blocks of 256 KB)."""
    name, streams = "edge_d8192", [(0, 0), (0, 1)]
    blob = subspace_blob(name, streams, 14, 2)
    assert {sc.basis.shape for sc, _ in stream_calibs(blob).values()} == \
        {(8192, 224)}
    run_roundtrip(kv, torch, name, streams, 600, blob=blob)
    run_paged(kv, torch, name, streams, [600, 37, 300], blob=blob)


def test_flat_spectrum_k256_takes_the_single_a_buffer(kv, torch):
    """Flat spectrum at 1 bit per coefficient: the DP keeps 16 two-bit
    groups, k = 256.  The projection runs one N = 256 MMA per K step into
    double-buffered accumulators; the reconstruction's A operand (k + 16 =
    272 fp16 columns) takes the single-buffer layout and its B operand two
    ring stages per chunk."""
    run_roundtrip(kv, torch, "llama31_8b_8k_flat",
                  [(0, 0), (0, 1), (1, 0), (1, 1)], 1000)


def test_cross_layer_pairs_k480_one_stage_projection(kv, torch):
    """Cross-layer basis: two layers' rows side by side (D = 2048) under one
    basis, 1 bit per coefficient.  The oracle's DP keeps k = 480 (30
    groups) with 256-byte records: the projection runs two MMAs per K step
    (N = 256 and 224) from a one-stage ring, the reconstruction contracts
    k + 16 = 496 columns, the most its tensor memory holds."""
    name, streams = "llama31_8b_8k_xlayer2", [(0, 0), (0, 1)]
    blob = blob_for(name, calibrate_workload(name, streams))
    assert {sc.basis.shape[1] for sc, _ in stream_calibs(blob).values()} \
        == {480}
    run_roundtrip(kv, torch, name, streams, 1000, ld_pad=64, blob=blob)


def forced_blob(name, streams, ngroups, budget_bits):
    """Oracle basis of `name`'s streams with the first `ngroups` groups at
    width 1 and the rest dropped."""
    w = synth.WORKLOADS[name]
    widths = np.zeros(w.D // 16, dtype=np.int64)
    widths[:ngroups] = 1
    return blob_for(name, calibrate_forced(name, streams, widths),
                    budget_bits)


@pytest.mark.parametrize("ngroups,budget", [(21, 1024), (28, 1408)])
def test_hand_set_widths_k336_and_k448(kv, torch, ngroups, budget):
    """k = 336 (21 one-bit groups, the most a 1024-bit budget holds) and
    k = 448 (28 groups, 176-byte records): the projection issues two MMAs per
    K step (N = 256 and N = k - 256) into one k-column accumulator, and the
    reconstruction contracts k + 16 = 352 or 464 columns from the single A
    buffer, its B operand in two ring stages per chunk."""
    name = "llama31_8b_8k"
    streams = [(2, 0), (2, 1), (3, 0), (3, 1)]
    blob = forced_blob(name, streams, ngroups, budget)
    run_roundtrip(kv, torch, name, streams, 2049, ld_pad=64, blob=blob,
                  tag=f"{name}, {ngroups} one-bit groups (k = "
                      f"{16 * ngroups})")


def mixed_blob(name, specs, budget_bits):
    """Oracle bases of the streams in `specs` {(layer, kv): (groups, width)}
    with that many leading groups at that width each (hand-set widths)."""
    w = synth.WORKLOADS[name]
    entries = []
    for s, (ng, b) in specs.items():
        widths = np.zeros(w.D // 16, dtype=np.int64)
        widths[:ng] = b
        entries += calibrate_forced(name, [s], widths)
    return blob_for(name, entries, budget_bits)


def test_mixed_k_in_one_launch(kv, torch):
    """Six streams of one call keep k = 224, 336, 448, 496, 272 and 256
    (hand-set widths, 256-byte records), 8192 tokens each: 192 super-tiles
    over the CTA pairs, so a pair runs tiles of different streams one after
    another.  The restore launch is wide: its cyclic A slots take tiles of
    15 to 32 K steps back to back (a k = 496 tile fills all 32), each tile
    waiting for the slots it shares with the one before.  The projection
    runs one-K-block ring stages (k > 382 at 256-byte records) and two MMAs
    per K step where k > 256."""
    name = "llama31_8b_8k"
    specs = {(2, 0): (14, 2), (2, 1): (21, 1), (3, 0): (28, 1),
             (3, 1): (31, 1), (4, 0): (17, 2), (4, 1): (16, 2)}
    blob = mixed_blob(name, specs, 2048)
    assert sorted(sc.basis.shape[1] for sc, _ in
                  stream_calibs(blob).values()) == [224, 256, 272, 336, 448,
                                                    496]
    run_roundtrip(kv, torch, name, list(specs), 8192, blob=blob,
                  sample=lambda tc: np.arange(0, tc, 13),
                  tag=f"{name}, k = 224 ... 496 in one launch")


def test_paged_mixed_k(kv, torch):
    """Paged restore of streams keeping k = 224 and k = 496 (256-byte
    records) for five requests of different lengths: the wide paged kernel
    with tiles of 15 and 32 K steps alternating through the cyclic A slots,
    through the block table."""
    name = "qwen25_7b_paged"
    blob = mixed_blob(name, {(0, 0): (14, 2), (0, 1): (31, 1)}, 2048)
    run_paged(kv, torch, name, [(0, 0), (0, 1)], [4096, 700, 4096, 300, 2000],
              blob=blob, tag=f"{name}, k = 224 and 496")


def test_paged_restore_k336(kv, torch):
    """Paged restore of the Qwen-shaped streams (D = 512, two output
    chunks) with 21 one-bit groups: k = 336 through the block table."""
    name = "qwen25_7b_paged"
    streams = [(0, 0), (0, 1)]
    blob = forced_blob(name, streams, 21, 1024)
    run_paged(kv, torch, name, streams, [700, 37, 4096, 300], blob=blob,
              tag=f"{name}, 21 one-bit groups (k = 336)")


def test_llama_shape_several_streams_ragged(kv, torch):
    stats, dstats = run_roundtrip(
        kv, torch, "llama31_8b_8k", [(3, 0), (3, 1), (4, 0), (4, 1)], 1000)
    print(stats, dstats)


def test_more_streams_than_one_launch_holds(kv, torch):
    """100 streams in one call: compress splits them over two launches of at
    most 64 streams, decompress over two of at most 96."""
    streams = [(l, k) for l in range(50) for k in (0, 1)]
    run_roundtrip(kv, torch, "llama33_70b_16k", streams, 400)


def test_nemo_shape_k112(kv, torch):
    run_roundtrip(kv, torch, "mistral_nemo_12b_32k", [(0, 0), (0, 1)], 1500)


def test_paged_restore_and_block_flag(kv, torch):
    run_paged(kv, torch, "qwen25_7b_paged", [(0, 0), (0, 1), (1, 0), (1, 1)],
              [700, 37, 4096, 129])


def test_paged_short_and_raw_only_requests(kv, torch):
    """Requests shorter than a block, with no coded token (sink and window
    only), of one token, with one coded token, and ending one token past a
    256-token tile: sink and window rows exact, coded rows within the
    restore tolerance, partial blocks written row by row."""
    run_paged(kv, torch, "qwen25_7b_paged", [(0, 0), (0, 1)],
              [3, 1, 16, 132, 133, 257, 389, 512])


def test_codec_host_refusals(kv, torch):
    """What kvtc_compress and kvtc_decompress refuse on the host, before any
    launch: a row stride below D or off the 8-element grid, misaligned
    pointers, an output or input buffer too small, a negative T, a layer
    the calibration does not hold and an invalid K|V mask.  Nothing is
    written and no device flag is raised; the same arguments unchanged are
    accepted."""
    name = "tiny"
    w = synth.WORKLOADS[name]
    calib = kv.kvtc_calib_load(blob_for(name, calibrate_workload(
        name, [(0, 0)])), 0)
    T, D = 300, w.D
    x = to_dev(torch, synth.eval_tokens(w, 0, 0, T=T), D)
    need = calib.stream_bytes(0, 0, T)
    comp = torch.full((need + 64,), 0xA5, dtype=torch.uint8, device="cuda")
    out = torch.full((T, D + 8), 0x7FC0, dtype=torch.int16, device="cuda")

    def code(fn, *a):
        with pytest.raises(kv.KvtcError) as e:
            fn(calib, *a)
        return e.value.code

    c = kv.kvtc_compress
    assert code(c, 0, 1, 1, [x], D - 8, T, comp, need) == kv.KVTC_ESIZE
    assert code(c, 0, 1, 1, [x], D + 4, T, comp, need) == kv.KVTC_EALIGN
    assert code(c, 0, 1, 1, [x.data_ptr() + 8], D, T, comp, need) == \
        kv.KVTC_EALIGN
    assert code(c, 0, 1, 1, [x], D, T, comp, need - 16) == kv.KVTC_ESIZE
    assert code(c, 0, 1, 1, [x], D, T, comp.data_ptr() + 8, need) == \
        kv.KVTC_EALIGN
    assert code(c, 0, 1, 1, [x], D, -1, comp, need) == kv.KVTC_EINVAL
    assert code(c, 5, 1, 1, [x], D, T, comp, need) == kv.KVTC_EINVAL
    assert code(c, 0, 1, 0, [x], D, T, comp, need) == kv.KVTC_EINVAL
    d = kv.kvtc_decompress
    assert code(d, 0, 1, 1, comp, need, T, [out], D - 8) == kv.KVTC_ESIZE
    assert code(d, 0, 1, 1, comp, need, T, [out], D + 4) == kv.KVTC_EALIGN
    assert code(d, 0, 1, 1, comp, need, T, [out.data_ptr() + 8], D + 8) == \
        kv.KVTC_EALIGN
    assert code(d, 0, 1, 1, comp, need - 16, T, [out], D + 8) == \
        kv.KVTC_ESIZE
    assert code(d, 0, 1, 1, comp.data_ptr() + 8, need, T, [out], D + 8) == \
        kv.KVTC_EALIGN
    assert code(d, 0, 1, 1, comp, need, -1, [out], D + 8) == kv.KVTC_EINVAL
    assert code(d, 0, 1, 4, comp, need, T, [out], D + 8) == kv.KVTC_EINVAL
    torch.cuda.synchronize()
    assert torch.all(comp == 0xA5) and torch.all(out == 0x7FC0)
    assert kv.kvtc_device_status(calib) == 0
    kv.kvtc_compress(calib, 0, 1, 1, [x], D, T, comp, need)
    kv.kvtc_decompress(calib, 0, 1, 1, comp, need, T, [out], D + 8)
    torch.cuda.synchronize()
    assert kv.kvtc_device_status(calib) == 0
    assert torch.all(comp[need:] == 0xA5) and torch.all(out[:, D:] == 0x7FC0)
    calib.free()


def test_paged_host_refusals(kv, torch):
    """What kvtc_decompress_paged refuses on the host, before any launch:
    a block size other than 16, a block table too narrow for T, misaligned
    stream, pool or block-table pointers, a negative T and an empty pool.
    Nothing is written and no device flag is raised."""
    name = "tiny"
    w = synth.WORKLOADS[name]
    calib = kv.kvtc_calib_load(blob_for(name, calibrate_workload(
        name, [(0, 0)])), 0)
    T, bs, maxb = 100, 16, 7
    src = torch.zeros(calib.stream_bytes(0, 0, T), dtype=torch.uint8,
                      device="cuda")
    cache = torch.full((maxb + 1, bs, w.D), 0x7FC0, dtype=torch.int16,
                       device="cuda")
    bt = torch.arange(maxb, dtype=torch.int32, device="cuda").view(1, maxb)
    good = dict(src=[src], T=[T], block_table=bt, max_blocks=maxb,
                block_size=bs, cache=[cache], num_blocks=maxb + 1)

    def refused(**change):
        a = dict(good, **change)
        with pytest.raises(kv.KvtcError) as e:
            kv.kvtc_decompress_paged(calib, 0, 1, 1, a["src"], a["T"],
                                     a["block_table"], a["max_blocks"],
                                     a["block_size"], a["cache"],
                                     a["num_blocks"])
        return e.value.code

    assert refused(block_size=8) == kv.KVTC_ENOTSUP
    assert refused(max_blocks=maxb - 1, block_table=bt[:, :maxb - 1]
                   .contiguous()) == kv.KVTC_ESIZE
    assert refused(src=[src.data_ptr() + 8]) == kv.KVTC_EALIGN
    assert refused(cache=[cache.data_ptr() + 2]) == kv.KVTC_EALIGN
    assert refused(block_table=bt.data_ptr() + 2) == kv.KVTC_EALIGN
    assert refused(T=[-1]) == kv.KVTC_EINVAL
    assert refused(num_blocks=0) == kv.KVTC_EINVAL
    torch.cuda.synchronize()
    assert torch.all(cache == 0x7FC0)
    assert kv.kvtc_device_status(calib) == 0
    # the same arguments unchanged are accepted
    kv.kvtc_decompress_paged(calib, 0, 1, 1, [src], [T], bt, maxb, bs,
                             [cache], maxb + 1)
    torch.cuda.synchronize()
    assert kv.kvtc_device_status(calib) == 0
    calib.free()


def test_paged_restore_256_byte_records(kv, torch):
    """Paged restore with the longest records (one-stage B ring)."""
    run_paged(kv, torch, "edge_d192_r256", [(0, 0), (0, 1)],
              [600, 21, 300])


def run_paged(kv, torch, name, streams, Ts, blob=None, tag=None):
    w = synth.WORKLOADS[name]
    nl = max(l for l, _ in streams) + 1
    if blob is None:
        blob = blob_for(name, calibrate_workload(name, streams))
    tag = tag or name
    scs = stream_calibs(blob)
    calib = kv.kvtc_calib_load(blob, 0)
    bs = 16
    maxb = -(-max(Ts) // bs)
    nblocks = len(Ts) * maxb + 7
    rng = np.random.default_rng(5)
    table = rng.permutation(nblocks)[:len(Ts) * maxb].astype(np.int32)
    table = table.reshape(len(Ts), maxb)
    D = w.D
    srcs, oracle_bytes = [], []
    for r, T in enumerate(Ts):
        parts = []
        for l, k in streams:
            x = synth.eval_tokens(w, l, k, request=r, T=T)
            parts.append(codec.compress_stream(x, scs[(l, k)][0]))
        b = b"".join(parts)
        oracle_bytes.append(parts)
        srcs.append(torch.from_numpy(np.frombuffer(b, np.uint8).copy()).cuda())
    caches = [torch.full((nblocks, bs, D), 0x7FC0, dtype=torch.int16,
                         device="cuda") for _ in range(2 * nl)]
    bt = torch.from_numpy(table).cuda()
    kv.kvtc_decompress_paged(calib, 0, nl, 3, srcs, Ts, bt, maxb, bs, caches,
                             nblocks)
    assert kv.kvtc_device_status(calib) == 0
    host = [from_dev(c) for c in caches]
    for r, T in enumerate(Ts):
        s_, w_, tc = codec.split_tokens(T, w.sink, w.window)
        for j, (l, k) in enumerate(streams):
            ref = codec.decompress_stream(oracle_bytes[r][j], T, scs[(l, k)][1])
            t = np.arange(T)
            got = host[j][table[r, t // bs], t % bs]
            np.testing.assert_array_equal(got[:s_], ref[:s_])
            np.testing.assert_array_equal(got[T - w_:], ref[T - w_:])
            st = check_decompress(got[s_:T - w_], ref[s_:T - w_])
            record(tag + " (paged)", dst=st)
            assert st["ok"], st
    # untouched blocks keep their contents
    used = set(table[r, t] for r, T in enumerate(Ts)
               for t in range(-(-T // bs)))
    free = [b for b in range(nblocks) if b not in used]
    for c in host:
        assert np.all(c[free] == 0x7FC0)
    # an out-of-range block id is skipped and flagged, not a fault
    bad = table.copy()
    bad[-1, 1] = nblocks + 3
    bad[0, 0] = -1
    kv.kvtc_decompress_paged(calib, 0, nl, 3, srcs, Ts,
                             torch.from_numpy(bad).cuda(), maxb, bs, caches,
                             nblocks)
    assert kv.kvtc_device_status(calib) & kv.KVTC_FLAG_BLOCK
    assert kv.kvtc_device_status(calib) == 0  # cleared after reading
    calib.free()


def test_layer_events_match_single_launch(kv, torch):
    name = "llama31_8b_8k"
    w = synth.WORKLOADS[name]
    streams = [(l, k) for l in range(3) for k in (0, 1)]
    entries = calibrate_workload(name, streams)
    blob = blob_for(name, entries)
    calib = kv.kvtc_calib_load(blob, 0)
    T = 600
    src = [to_dev(torch, synth.eval_tokens(w, l, k, T=T)) for l, k in streams]
    total = sum(calib.stream_bytes(l, k, T) for l, k in streams)
    comp = torch.zeros(total, dtype=torch.uint8, device="cuda")
    kv.kvtc_compress(calib, 0, 3, 3, src, w.D, T, comp, total)
    a = [torch.zeros((T, w.D), dtype=torch.int16, device="cuda")
         for _ in streams]
    b = [torch.zeros((T, w.D), dtype=torch.int16, device="cuda")
         for _ in streams]
    kv.kvtc_decompress(calib, 0, 3, 3, comp, total, T, a, w.D)
    evs = [torch.cuda.Event() for _ in range(3)]
    for e in evs:  # torch creates the CUDA event on its first record
        e.record()
    kv.kvtc_decompress(calib, 0, 3, 3, comp, total, T, b, w.D,
                       layer_events=evs)
    evs[0].synchronize()
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert kv.kvtc_device_status(calib) == 0
    calib.free()


def test_restore_from_pinned_host_memory(kv, torch):
    """kvtc_decompress and kvtc_decompress_paged given pinned host memory
    read it over the host link and restore exactly what they restore from
    device memory; pageable host memory is refused before any launch."""
    name = "llama31_8b_8k"
    w = synth.WORKLOADS[name]
    streams = [(l, k) for l in range(2) for k in (0, 1)]
    entries = calibrate_workload(name, streams)
    blob = blob_for(name, entries)
    calib = kv.kvtc_calib_load(blob, 0)
    T = 700
    src = [to_dev(torch, synth.eval_tokens(w, l, k, T=T)) for l, k in streams]
    total = sum(calib.stream_bytes(l, k, T) for l, k in streams)
    comp = torch.zeros(total, dtype=torch.uint8, device="cuda")
    kv.kvtc_compress(calib, 0, 2, 3, src, w.D, T, comp, total)
    pinned = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    pinned.copy_(comp)
    torch.cuda.synchronize()

    def restore(inp):
        out = [torch.full((T, w.D), 0x7FC0, dtype=torch.int16, device="cuda")
               for _ in streams]
        kv.kvtc_decompress(calib, 0, 2, 3, inp, total, T, out, w.D)
        torch.cuda.synchronize()
        return out

    for x, y in zip(restore(comp), restore(pinned)):
        assert torch.equal(x, y)
    assert kv.kvtc_device_status(calib) == 0
    # paged, one request, from pinned memory
    bs, maxb = 16, -(-T // 16)
    bt = torch.arange(maxb, dtype=torch.int32, device="cuda").view(1, maxb)
    caches = [torch.zeros((maxb, bs, w.D), dtype=torch.int16, device="cuda")
              for _ in streams]
    kv.kvtc_decompress_paged(calib, 0, 2, 3, [pinned], [T], bt, maxb, bs,
                             caches, maxb)
    torch.cuda.synchronize()
    ref = restore(comp)
    for c, r in zip(caches, ref):
        assert torch.equal(c.view(-1, w.D)[:T], r)
    assert kv.kvtc_device_status(calib) == 0
    # pageable host memory: refused on the host
    pageable = np.zeros(total + 16, dtype=np.uint8)
    addr = (pageable.ctypes.data + 15) // 16 * 16
    with pytest.raises(kv.KvtcError) as e:
        kv.kvtc_decompress(calib, 0, 2, 3, addr, total, T, ref, w.D)
    assert e.value.code == kv.KVTC_EINVAL
    with pytest.raises(kv.KvtcError) as e:
        kv.kvtc_decompress_paged(calib, 0, 2, 3, [addr], [T], bt, maxb, bs,
                                 caches, maxb)
    assert e.value.code == kv.KVTC_EINVAL
    calib.free()


def test_full_llama31_8b_8k_sampled(kv, torch):
    """Full workload as the bench launches it (64 streams x 8192 tokens, one
    call each way); eight streams are checked against the oracle in full."""
    name = "llama31_8b_8k"
    w = synth.WORKLOADS[name]
    streams = w.streams()
    entries = calibrate_workload(name, streams)
    blob = blob_for(name, entries)
    scs = stream_calibs(blob)
    calib = kv.kvtc_calib_load(blob, 0)
    T, D = w.tokens, w.D
    src = [synth.eval_tokens_torch(w, l, k, T=T).view(torch.int16)
           for l, k in streams]
    total = sum(calib.stream_bytes(l, k, T) for l, k in streams)
    comp = torch.zeros(total, dtype=torch.uint8, device="cuda")
    kv.kvtc_compress(calib, 0, w.layers, 3, src, D, T, comp, total)
    outs = [torch.zeros((T, D), dtype=torch.int16, device="cuda")
            for _ in streams]
    kv.kvtc_decompress(calib, 0, w.layers, 3, comp, total, T, outs, D)
    assert kv.kvtc_device_status(calib) == 0
    sb = calib.stream_bytes(0, 0, T)
    s_, w_, tc = codec.split_tokens(T, w.sink, w.window)
    raw = (s_ + w_) * D * 2
    gbytes = comp.cpu().numpy()
    worst = 0.0
    for idx in (0, 1, 14, 27, 40, 51, 62, 63):
        l, k = streams[idx]
        sc_enc, sc_dec = scs[(l, k)]
        x = from_dev(src[idx])
        g = gbytes[idx * sb:(idx + 1) * sb].tobytes()
        o = codec.compress_stream(x, sc_enc)
        assert g[:raw] == o[:raw]
        grec = np.frombuffer(g, np.uint8, tc * sc_enc.R, raw).reshape(
            tc, sc_enc.R)
        st = check_records(grec, x[s_:T - w_], sc_enc)
        record(name, st=st)
        assert st["bad"] == 0, (idx, st)
        # GPU decompress of the GPU bitstream vs the oracle decompressing
        # the same bitstream
        ref = codec.decompress_stream(g, T, sc_dec)
        got = from_dev(outs[idx])
        np.testing.assert_array_equal(got[:s_], x[:s_])
        np.testing.assert_array_equal(got[T - w_:], x[T - w_:])
        dst = check_decompress(got[s_:T - w_], ref[s_:T - w_])
        record(name, dst=dst)
        assert dst["ok"], (idx, dst)
        worst = max(worst, dst["rel_l2"])
    calib.free()
