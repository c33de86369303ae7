"""The allocation-free dense entry point, cbq_matvec_static.

Some callers cannot allocate device memory while they run (hosts that fix
their device memory at start-up); cbq_matvec_static serves them by keeping its
quantized activations in a scratch array the library declares statically on
each device (one aligned column needs none: it is quantized inside the matvec
kernel).  This file is named to be collected last.  It checks, through the C
ABI, that two calls in a row give the same bits as cbq_matvec on the same
inputs and stay within the parity bound of the oracle, and that a K beyond the
scratch's limit is refused before anything runs.
"""
import numpy as np
import pytest

from oracle import oracle as O
from tests.gpu_util import assert_within_bound, cuda
from verify_matvec_gb300 import cbq, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return cuda()


@pytest.mark.parametrize("M,K,n,offset", [(4096, 4096, 1, 0), (4096, 4096, 1, 1), (1000, 2080, 5, 0)])
def test_static_scratch_matches_matvec_on_two_calls(torch, M, K, n, offset):
    """offset 1 puts x 4 bytes past a 16-byte boundary (the scratch path for
    one column)."""
    W = synth.weight_blocks(M, K, stream=901 + n)
    Wh = cbq.Weights(W, M, K)
    for call in range(2):  # the second call must not depend on the first's scratch
        x = synth.activations(n, K, stream=910 + 10 * n + call, outliers=(call == 0))
        buf = torch.zeros(n * K + offset, dtype=torch.float32, device="cuda")
        buf[offset:] = torch.from_numpy(x).cuda().reshape(-1)
        xd = buf[offset:].view(n, K)
        assert (xd.data_ptr() % 16 == 0) == (offset == 0)
        y_static = cbq.cbq_matvec_static(Wh, xd).cpu().numpy()
        y_ref = cbq.cbq_matvec(Wh, xd).cpu().numpy()
        np.testing.assert_array_equal(y_static, y_ref)
        qx, dx = O.quantize_act(x)
        bound = O.matvec_bound(W, M, K, qx, dx)
        assert_within_bound(y_static, O.matvec_q(W, M, K, qx, dx), bound, what=f"call {call} vs oracle")


def test_static_scratch_refuses_large_k(torch):
    K = cbq.CBQ_STATIC_SCRATCH_MAX_K + 32
    W = synth.weight_blocks(32, K, stream=920)
    Wh = cbq.Weights(W, 32, K)
    x = torch.zeros((1, K), dtype=torch.float32, device="cuda")
    with pytest.raises(cbq.CbqError) as err:
        cbq.cbq_matvec_static(Wh, x)
    assert err.value.status == cbq.CBQ_EINVAL
