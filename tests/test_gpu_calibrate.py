"""Library calibration (kvtc_calibrate, GPU) vs the oracle's calibration on
the same calibration rows."""
import numpy as np
import pytest

import synth
from oracle import calibrate, codec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kv():
    from kv_cache_transform_gb300 import _build
    _build.build()
    import kv_cache_transform_gb300 as kv
    return kv


@pytest.mark.parametrize("name,streams", [
    ("tiny", [(0, 0)]),
    ("llama31_8b_8k", [(0, 0), (7, 1)]),
    ("mistral_nemo_12b_32k", [(3, 0)]),
])
def test_calibrate_matches_oracle(kv, name, streams):
    import torch
    w = synth.WORKLOADS[name]
    rows = [synth.calib_tokens(w, l, k) for l, k in streams]
    dev = [torch.from_numpy(r.view(np.int16).copy()).cuda() for r in rows]
    blob = kv.kvtc_calibrate(dev, [l for l, _ in streams],
                             [k for _, k in streams], w.n_calib, w.D, w.D,
                             w.sink, w.window, w.budget_bits)
    got = calibrate.read_blob(blob)          # parses and checks the CRC
    assert got["sink"] == w.sink and got["window"] == w.window
    assert got["budget_bits"] == w.budget_bits
    for (l, k), r, e in zip(streams, rows, got["streams"]):
        assert (e["layer"], e["kv"]) == (l, k)
        mu, V, evals, widths, E = calibrate.calibrate_stream(r, w.budget_bits)
        np.testing.assert_allclose(e["mu"], mu, rtol=0, atol=1e-12)
        np.testing.assert_allclose(e["evals"], evals, rtol=0,
                                   atol=1e-9 * evals[0])
        # objective of the library's widths on the oracle's table equals the
        # oracle's optimum (ties may pick other widths)
        obj = lambda wd: sum(E[g, b] for g, b in enumerate(wd))
        assert abs(obj(e["widths"]) - obj(widths)) <= 1e-6 * obj(widths)
        cost = sum(calibrate.width_cost_units(int(b)) for b in e["widths"])
        assert cost * 16 <= w.budget_bits
        # kept vectors: orthonormal, and the well-separated leading ones
        # equal the oracle's (same sign rule)
        B = e["basis"]
        assert np.abs(B.T @ B - np.eye(B.shape[1])).max() < 1e-9
        cols = codec.active_columns(e["widths"])
        lead = [i for i, c in enumerate(cols) if c < 8]
        for i in lead:
            np.testing.assert_allclose(B[:, i], V[:, cols[i]], atol=1e-7)
