"""Pins for the oracle's calibration: PCA, DP allocation, blob format."""
import itertools

import numpy as np
import pytest

import synth
from oracle import calibrate, codec, fp


@pytest.fixture(scope="module")
def tiny():
    w = synth.WORKLOADS["tiny"]
    cb = synth.calib_tokens(w, 0, 0)
    return w, cb, calibrate.pca(cb)


def test_basis_orthonormal_and_sorted(tiny):
    w, cb, (mu, evals, V) = tiny
    assert np.abs(V.T @ V - np.eye(w.D)).max() <= 1e-9
    assert np.all(np.diff(evals) <= 0)
    idx = np.argmax(np.abs(V), axis=0)
    assert np.all(V[idx, np.arange(w.D)] > 0)  # sign rule


def test_pca_matches_svd_of_centred_data(tiny):
    w, cb, (mu, evals, V) = tiny
    x = fp.bf16_bits_to_f64(cb)
    np.testing.assert_allclose(mu, x.mean(0), rtol=0, atol=1e-15)
    _, s, vt = np.linalg.svd(x - mu, full_matrices=False)
    np.testing.assert_allclose(evals, s ** 2 / x.shape[0], rtol=1e-9,
                               atol=1e-15)
    # well separated leading components agree up to sign
    for i in range(16):
        d = abs(abs(vt[i] @ V[:, i]) - 1)
        assert d < 1e-8


def test_spectrum_matches_generator(tiny):
    """Eigenvalues of x = mu + A z + 0.01 eps are sigma_i^2 + 1e-4 (plus the
    bf16 storage noise) up to sampling error."""
    w, cb, (mu, evals, V) = tiny
    sigma2 = np.arange(1, w.rank + 1, dtype=float) ** (-2 * w.spectrum_p)
    rel = evals[:8] / (sigma2[:8] + 1e-4) - 1
    assert np.all(np.abs(rel) < 0.15)
    noise = evals[w.rank:]
    assert np.all(noise > 0) and np.all(noise < 3e-4)


def brute_force(E, budget_bits):
    G, nb = E.shape
    U = budget_bits // 16
    best, arg, count = np.inf, None, 0
    for combo in itertools.product(range(nb), repeat=G):
        cost = sum(calibrate.width_cost_units(b) for b in combo)
        if cost > U:
            continue
        v = sum(E[g, b] for g, b in enumerate(combo))
        if v < best - 1e-12:
            best, arg, count = v, combo, 1
        elif abs(v - best) <= 1e-12:
            count += 1
    return best, arg, count


@pytest.mark.parametrize("G", [1, 2, 3, 4])
def test_dp_matches_brute_force(G):
    rng = np.random.default_rng(100 + G)
    for trial in range(6):
        if trial % 2 == 0:   # realistic: decreasing in b
            E = np.sort(rng.exponential(1.0, (G, 9)), axis=1)[:, ::-1].copy()
        else:                # arbitrary tables
            E = rng.uniform(0, 1, (G, 9))
        for u in range(0, G * 10 + 2):
            budget = 16 * u + int(rng.integers(0, 16))
            widths = calibrate.allocate_bits(E, budget)
            cost = sum(calibrate.width_cost_units(int(b)) for b in widths)
            assert cost * 16 <= budget
            val = sum(E[g, b] for g, b in enumerate(widths))
            best, arg, count = brute_force(E, budget)
            assert abs(val - best) <= 1e-12 * max(1.0, best)
            if count == 1:
                assert tuple(int(b) for b in widths) == arg


def test_dp_special_cases():
    rng = np.random.default_rng(7)
    E = np.sort(rng.exponential(1.0, (6, 9)), axis=1)[:, ::-1].copy()
    E += np.arange(9)[::-1][None, :] * 1e-3  # strictly decreasing in b
    assert np.all(calibrate.allocate_bits(E, 0) == 0)
    assert np.all(calibrate.allocate_bits(E, 47) == 0)  # 1-bit group costs 48
    assert np.all(calibrate.allocate_bits(E, 6 * (32 + 128)) == 8)


def test_dp_prefers_high_variance_groups(tiny):
    """Widths never increase along the descending spectrum for the tiny
    workload, and dropped groups carry the least energy."""
    w, cb, _ = tiny
    mu, V, evals, widths, E = calibrate.calibrate_stream(cb, w.budget_bits)
    assert widths[0] > 0
    assert np.all(np.diff(widths) <= 0)
    used = sum(calibrate.width_cost_units(int(b)) for b in widths) * 16
    assert used <= w.budget_bits


def test_distortion_table_definition(tiny):
    w, cb, (mu, evals, V) = tiny
    c = (fp.bf16_bits_to_f64(cb) - mu) @ V
    E = calibrate.distortion_table(c)
    np.testing.assert_allclose(E[:, 0], (c.reshape(len(c), -1, 16) ** 2)
                               .sum((0, 2)), rtol=1e-12)
    # group energies sum to the total variance times N (trace)
    np.testing.assert_allclose(E[:, 0].sum(), evals.sum() * len(c),
                               rtol=1e-9)
    assert np.all(np.diff(E[0, 1:]) < 0)


def test_blob_round_trip(tiny):
    w, cb, _ = tiny
    mu, V, evals, widths, E = calibrate.calibrate_stream(cb, w.budget_bits)
    blob = calibrate.write_blob([(0, 0, mu, V, evals, widths)], w.sink,
                                w.window, w.budget_bits)
    b = calibrate.read_blob(blob)
    assert b["sink"] == w.sink and b["window"] == w.window
    s = b["streams"][0]
    cols = codec.active_columns(widths)
    np.testing.assert_array_equal(s["basis"], V[:, cols])
    np.testing.assert_array_equal(s["widths"], widths)
    np.testing.assert_array_equal(s["mu"], mu)
    bad = bytearray(blob)
    bad[40] ^= 1
    with pytest.raises(AssertionError):
        calibrate.read_blob(bytes(bad))


@pytest.mark.parametrize("b", range(1, 9))
def test_distortion_table_equals_codec_error_at_every_width(tiny, b):
    """Column b of the distortion table is the squared error the codec
    itself makes at uniform width b (kvtc page, technical summary 2A: the
    DP minimises reconstruction error measured on calibration data).

    The codec path is independent of the table's own loop: every group is
    given width b through the stream's widths, the rows are compressed into
    records (fields and bit-planes), unpacked and reconstructed as
    x_hat = mu + V c_hat in fp64.  With the full orthonormal basis,
    Parseval makes ||x - x_hat||^2 equal to ||c - c_hat||^2, so the summed
    column must match the reconstruction error in x space, and each group's
    entry the error of its 16 coefficients."""
    w, cb, (mu, evals, V) = tiny
    G = w.D // 16
    x = fp.bf16_bits_to_f64(cb)
    c = (x - mu) @ V
    E = calibrate.distortion_table(c)
    widths = np.full(G, b)
    budget = G * (32 + 16 * 8)
    sc = codec.StreamCalib(mu, V, widths, 0, 0, budget)
    buf = codec.compress_stream(cb, sc)
    xh = codec.decompress_stream(buf, cb.shape[0], sc, exact=True)
    err_x = ((x - xh) ** 2).sum()
    np.testing.assert_allclose(E[:, b].sum(), err_x, rtol=1e-9)
    shift, scale, q = codec.unpack(codec.stream_records(buf, cb.shape[0], sc),
                                   sc.bits)
    chat = codec.dequantise(shift, scale, q)
    per_group = ((c - chat) ** 2).reshape(len(c), G, 16).sum(axis=(0, 2))
    np.testing.assert_allclose(E[:, b], per_group, rtol=1e-9, atol=0)
    # a wider code never does worse on the same group
    if b > 1:
        assert np.all(E[:, b] <= E[:, b - 1] * (1 + 1e-12))


def test_dp_units_beyond_ten_per_group_change_nothing():
    """No group costs more than 10 units (two fp16 fields plus 8 planes of
    16 bits), so the widths the DP picks with U units equal those with
    min(U, 10 G) units, ties included: the library's device DP caps its
    table there."""
    rng = np.random.default_rng(0)
    for trial in range(200):
        G = int(rng.integers(1, 9))
        if trial % 2:
            E = rng.uniform(0, 1, (G, 9))
        else:
            E = np.sort(rng.exponential(1, (G, 9)), axis=1)[:, ::-1].copy()
        if trial % 5 == 0:
            E[:, 3:] = E[:, 3:4]     # equal errors above width 3: ties
        for budget in (int(rng.integers(0, 16 * 12 * G)), 16 * 10 * G + 7,
                       16 * 40 * G, 1 << 16):
            full = calibrate.allocate_bits(E, budget)
            capped = calibrate.allocate_bits(E, 16 * min(budget // 16,
                                                         10 * G))
            assert np.array_equal(full, capped)
