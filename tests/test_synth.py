"""The seeded input generators: reproducible and of the stated recipe."""
import numpy as np

from verify_matvec_gb300 import synth


def test_weights_reproducible_and_in_range():
    a = synth.weight_blocks(64, 256, stream=5)
    b = synth.weight_blocks(64, 256, stream=5)
    np.testing.assert_array_equal(a, b)
    assert not np.array_equal(a, synth.weight_blocks(64, 256, stream=6))
    s = a[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    assert s.min() >= np.float16(1e-3) and s.max() <= np.float16(1e-2)
    qs = a[:, :, 2:]
    lo, hi = np.bincount((qs & 15).ravel(), minlength=16), np.bincount((qs >> 4).ravel(), minlength=16)
    assert lo.min() > 0.8 * lo.mean() and hi.min() > 0.8 * hi.mean()


def test_activations_outliers():
    x = synth.activations(3, 4096, stream=9, outliers=True)
    assert x.dtype == np.float32 and x.shape == (3, 4096)
    for c in range(3):
        assert np.sum(np.abs(x[c]) > 6.0) >= 30  # ~41 outliers of magnitude ~20


def test_router_distinct_and_softmax():
    ids, wts = synth.router(5, 8, 256)
    assert ids.dtype == np.int32 and wts.dtype == np.float32
    for t in range(5):
        assert len(set(ids[t].tolist())) == 8
        assert abs(float(wts[t].astype(np.float64).sum()) - 1.0) < 1e-6
    d = synth.distinct_experts(ids, 256)
    assert len(d) == len(set(ids.ravel().tolist()))
