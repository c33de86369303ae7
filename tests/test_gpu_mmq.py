"""The tensor-core (tcgen05) path for up to 16 columns (cbq_matmat) against
the oracle: the per-block integer dots bit for bit with the oracle's block
dots (every level and activation exact in the fp16 operands, every block sum
exact in the fp32 accumulator), and y within the same per-output bound as the
dp4a path, on ragged and full-size shapes and partial tiles (a pair count
that is odd, a block count that is not a multiple of the four-block batch)."""
import numpy as np
import pytest

from oracle import oracle as O
from tests.gpu_util import assert_within_bound, cuda
from verify_matvec_gb300 import cbq, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return cuda()


def _dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("M,K,n", [(256, 1024, 16), (256, 1024, 1), (70, 160, 8), (33, 96, 16), (1000, 2080, 11),
                                   (128, 4096, 16)])
def test_block_dots_bit_exact(torch, M, K, n):
    W = synth.weight_blocks(M, K, stream=701 + M + n)
    qx = np.random.default_rng(M + K + n).integers(-127, 128, size=(n, K)).astype(np.int8)
    qx[0, :32] = 127                      # extreme block: every product at its largest
    Wh = cbq.Weights(W, M, K)
    s = cbq.cbq_debug_mmq_block_dots(Wh, _dev(torch, qx)).cpu().numpy()
    np.testing.assert_array_equal(s, O.block_dots(W, M, K, qx))
    assert cbq.cbq_weights_get_error(Wh) == 0


def test_block_dots_every_codebook_entry(torch):
    """Blocks of one index each (0..15) against all-ones and alternating columns."""
    M, K = 128, 512
    blk = np.zeros((M, K // 32, 18), dtype=np.uint8)
    blk[:, :, 0:2] = np.frombuffer(np.float16(0.01).tobytes(), np.uint8)
    for r in range(M):
        for b in range(K // 32):
            i = (r + b) % 16
            blk[r, b, 2:] = i | (i << 4)
    qx = np.ones((3, K), dtype=np.int8)
    qx[1, ::2] = -1
    qx[2] = np.arange(K) % 255 - 127
    s = cbq.cbq_debug_mmq_block_dots(cbq.Weights(blk, M, K), _dev(torch, qx)).cpu().numpy()
    np.testing.assert_array_equal(s, O.block_dots(blk, M, K, qx))


def _check(torch, W, M, K, x, rows=None):
    Wh = cbq.Weights(W, M, K)
    y = cbq.cbq_matmat(Wh, _dev(torch, x)).cpu().numpy()
    qx, dx = O.quantize_act(x)
    yr = O.matvec_q(W, M, K, qx, dx, rows=rows)
    b = O.matvec_bound(W, M, K, qx, dx, rows=rows)
    assert_within_bound(y if rows is None else y[:, rows], yr, b)
    assert cbq.cbq_weights_get_error(Wh) == 0
    return Wh, y


@pytest.mark.parametrize("M,K,n", [(70, 160, 6), (33, 32, 16), (300, 1056, 8), (4096, 4096, 16), (4096, 4096, 9),
                                   (1000, 2080, 1)])
def test_matmat_vs_oracle(torch, M, K, n):
    W = synth.weight_blocks(M, K, stream=720 + M + n)
    x = synth.activations(n, K, stream=721 + n, outliers=True)
    _check(torch, W, M, K, x)


@pytest.mark.parametrize("n", [8, 16])
def test_matmat_16384_all_rows_and_repeatable(torch, n):
    """Every row of a 16384 x 4096 call at n = 8 (the N = 8 MMAs) and 16,
    and the same bits on a second call."""
    M, K = 16384, 4096
    W = synth.weight_blocks(M, K, stream=730)
    x = synth.activations(n, K, stream=731)
    Wh, y = _check(torch, W, M, K, x)
    y2 = cbq.cbq_matmat(Wh, _dev(torch, x)).cpu().numpy()
    np.testing.assert_array_equal(y, y2)
