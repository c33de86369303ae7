"""The hyper-connection Sinkhorn normalisation (cbq_hc_sinkhorn) on the GPU
against the oracle's fp64 evaluation of the same rounds, entry by entry,
within (8 + 16 * iters) * 2^-24: batch sizes from one matrix to more than a
grid of 128-thread blocks with a ragged last block, round counts from 0 to
the limit, wide and narrow logits, the degenerate cases (equal logits, a
rank-one matrix, a doubly stochastic input), in place, and the output buffer
guarded on both sides."""
import numpy as np
import pytest

from oracle import oracle as O
from tests.gpu_util import Guarded, cuda
from verify_matvec_gb300 import cbq, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return cuda()


def _tol(iters):
    return (8 + 16 * iters) * 2.0 ** -24


def _run(torch, c, iters):
    d = torch.from_numpy(np.ascontiguousarray(c, dtype=np.float32)).cuda()
    g = Guarded(torch, d.shape, torch.float32)
    cbq.cbq_hc_sinkhorn(d, iters, out=g.view)
    torch.cuda.synchronize()
    g.check()
    return g.view.cpu().numpy()


@pytest.mark.parametrize("n", [1, 5, 127, 128, 129, 1000, 40_003])
@pytest.mark.parametrize("iters", [0, 1, 3, 20])
def test_matches_oracle(torch, n, iters):
    c = synth.hc_logits(n, stream=synth.S_HC * 100 + n % 97)
    got = _run(torch, c, iters)
    want = O.hc_sinkhorn(c, iters)
    np.testing.assert_allclose(got, want, rtol=0, atol=_tol(iters))


@pytest.mark.parametrize("scale", [0.01, 3.0, 10.0])
def test_logit_scales(torch, scale):
    """Narrow logits (nearly uniform), wide ones (spread up to ~80: entries
    down to e^-80, still normal fp32), many rounds."""
    c = synth.hc_logits(3000, scale=scale, stream=synth.S_HC * 100 + 1)
    if scale == 10.0:  # keep every matrix within the contract's spread of 80
        spread = c.reshape(3000, -1).max(1) - c.reshape(3000, -1).min(1)
        c = c[spread <= 80.0]
    for iters in (5, 100):
        np.testing.assert_allclose(_run(torch, c, iters), O.hc_sinkhorn(c, iters), rtol=0, atol=_tol(iters))


def test_degenerate_matrices(torch):
    """Equal logits give 1/4 everywhere; a rank-one exp(c) is uniform after one
    round; a doubly stochastic input stays where it is; the largest round
    count the ABI accepts."""
    eq = np.full((3, 4, 4), 2.5, np.float32)
    for iters in (1, 7):
        np.testing.assert_array_equal(_run(torch, eq, iters), np.full((3, 4, 4), 0.25))
    rng = np.random.default_rng(3)
    a = np.round(rng.uniform(-3, 3, (4, 4, 1)) * 16) / 16
    b = np.round(rng.uniform(-3, 3, (4, 1, 4)) * 16) / 16
    r1 = (a + b).astype(np.float32)
    np.testing.assert_allclose(_run(torch, r1, 1), np.full((4, 4, 4), 0.25), rtol=0, atol=_tol(1))
    vals = np.array([0.5, 0.25, 0.125, 0.125])
    P = np.array([[vals[(i + j) % 4] for j in range(4)] for i in range(4)])
    c = np.log(P).astype(np.float32)[None]
    np.testing.assert_allclose(_run(torch, c, 50)[0], P, rtol=0, atol=1e-6)
    big = synth.hc_logits(33, stream=synth.S_HC * 100 + 2)
    it = cbq.CBQ_HC_MAX_ITERS
    np.testing.assert_allclose(_run(torch, big, it), O.hc_sinkhorn(big, it), rtol=0, atol=_tol(it))


def test_in_place_and_offset(torch):
    """out may be the logits buffer itself; a view starting at a later matrix
    (16-byte aligned) normalises only that range."""
    c = synth.hc_logits(300, stream=synth.S_HC * 100 + 3)
    d = torch.from_numpy(c).cuda()
    want = O.hc_sinkhorn(c, 20)
    sub = d[100:200]
    cbq.cbq_hc_sinkhorn(sub, 20, out=sub)
    got = d.cpu().numpy()
    np.testing.assert_array_equal(got[:100], c[:100])
    np.testing.assert_array_equal(got[200:], c[200:])
    np.testing.assert_allclose(got[100:200], want[100:200], rtol=0, atol=_tol(20))
