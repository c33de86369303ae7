"""The bounded waits of the layer kernel and of the tensor-core path, run out
on purpose through their give-up test modes (cbq_moe_debug_stall,
cbq_debug_mmq_stall): a wait for a dependency count that is never reached, or
for a weight stage that never arrives.  Every wait in the
kernels has a 1 s limit; when it runs out the kernel records a timeout bit in
the handle's error word and the CTA winds down without leaving a copy in
flight.  The tests check the bits the host reads, and that the handle keeps
working: the next calls give the same bits as a call before the stall, with a
clean error word.  No GPU fault is involved: the waits end by their limit."""
import numpy as np
import pytest

from tests.gpu_util import cuda
from verify_matvec_gb300 import cbq, synth

pytestmark = pytest.mark.gpu

E, H, F = 8, 256, 128
TIMEOUT_BITS = cbq.CBQ_DEVERR_PIPE_TIMEOUT | cbq.CBQ_DEVERR_DEPENDENCY_TIMEOUT


@pytest.fixture(scope="module")
def torch():
    return cuda()


@pytest.fixture(scope="module")
def layer(torch):
    gu = synth.expert_blocks(E, 2 * F, H, stream=801)
    dn = synth.expert_blocks(E, H, F, stream=802)
    return cbq.Moe(gu, dn, E, H, F)


@pytest.mark.parametrize("mode,must", [(1, TIMEOUT_BITS), (2, cbq.CBQ_DEVERR_PIPE_TIMEOUT)])
@pytest.mark.parametrize("n_tok,k", [(1, 4), (3, 2)])
def test_wait_gives_up_and_handle_recovers(torch, layer, mode, must, n_tok, k):
    L = layer
    h = synth.activations(n_tok, H, stream=810 + n_tok)
    ids, wts = synth.router(n_tok, k, E, stream=811 + n_tok)
    hd, idd, wd = (torch.from_numpy(a).cuda() for a in (h, ids, wts))
    y_ok = cbq.cbq_moe_matvec(L, hd, idd, wd).cpu().numpy()
    assert cbq.cbq_moe_get_error(L) == 0
    cbq.cbq_moe_debug_stall(L, mode)
    try:
        cbq.cbq_moe_matvec(L, hd, idd, wd)
        torch.cuda.synchronize()
        err = cbq.cbq_moe_get_error(L)
    finally:
        cbq.cbq_moe_debug_stall(L, 0)
    assert err & must, f"error word {err:#x}"
    assert err & ~TIMEOUT_BITS == 0, f"error word {err:#x}"
    for _ in range(2):
        y = cbq.cbq_moe_matvec(L, hd, idd, wd).cpu().numpy()
        np.testing.assert_array_equal(y, y_ok)
        assert cbq.cbq_moe_get_error(L) == 0


@pytest.mark.parametrize("n", [8, 16])
def test_tensor_core_wait_gives_up_and_handle_recovers(torch, n):
    """The first CTA of the tensor-core kernel fills no stage: every role's
    wait for it runs out, the CTA frees its tensor memory and exits, the
    error word holds the pipe timeout bit only, and the next calls give the
    bits of a call before the stall."""
    M, K = 384, 512  # three 128-row tiles: CTA 0 gives up, the others finish
    W = cbq.Weights(synth.weight_blocks(M, K, stream=820), M, K)
    x = torch.from_numpy(synth.activations(n, K, stream=821)).cuda()
    y_ok = cbq.cbq_matmat(W, x).cpu().numpy()
    assert cbq.cbq_weights_get_error(W) == 0
    cbq.cbq_debug_mmq_stall(W, 1)
    try:
        cbq.cbq_matmat(W, x)
        torch.cuda.synchronize()
        err = cbq.cbq_weights_get_error(W)
    finally:
        cbq.cbq_debug_mmq_stall(W, 0)
    assert err == cbq.CBQ_DEVERR_PIPE_TIMEOUT, f"error word {err:#x}"
    for _ in range(2):
        y = cbq.cbq_matmat(W, x).cpu().numpy()
        np.testing.assert_array_equal(y, y_ok)
        assert cbq.cbq_weights_get_error(W) == 0
