"""The weight converter (cbq_quantize_weights) on the GPU against the oracle's
converter, byte for byte: random matrices of several shapes (a block count
that is not a multiple of the eight blocks a warp takes per step included),
blocks built to hit every decision edge (weights on the codebook grid,
weights exactly between two levels, equal largest magnitudes of either
sign, all-zero blocks, scales that round to zero or to a binary16
subnormal), a full-size 16384 x 4096 matrix, and the converted blocks fed
to the matvec."""
import numpy as np
import pytest

from oracle import oracle as O
from tests.gpu_util import cuda
from verify_matvec_gb300 import cbq, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return cuda()


def _convert(torch, w):
    return cbq.cbq_quantize_weights(torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).cuda()).cpu().numpy()


@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (5, 32), (70, 160), (257, 4096), (1000, 2080)])
def test_random_matrices_bit_exact(torch, M, K):
    rng = np.random.default_rng(M + K)
    w = (rng.standard_normal((M, K)) * rng.uniform(1e-3, 4.0, (M, 1))).astype(np.float32)
    np.testing.assert_array_equal(_convert(torch, w), O.quantize_weights(w, M, K))


def _edge_blocks():
    rng = np.random.default_rng(7)
    rows = []
    levels = O.CODEBOOK.astype(np.float32)
    half = (levels[:-1] + levels[1:]) / 2
    for sign in (1, -1):
        for dwv in (2.0 ** -6, 0.00787353515625, 3.0517578125e-05):  # plain, rounded, binary16 subnormal
            dw = np.float32(sign * dwv)
            idx = rng.integers(0, 16, 32)
            idx[5] = 0
            rows.append(dw * levels[idx])                                 # on the grid
            t = dw * half[rng.integers(0, 15, 32)]                        # on the cell boundaries
            t[0] = -127 * dw
            rows.append(t)
    r = rng.standard_normal(32).astype(np.float32)
    r[3], r[17] = 2.5, -2.5                                               # equal magnitudes, either sign
    rows.append(r)
    rows.append(-r)
    rows.append(np.zeros(32, np.float32))                                 # zero block
    z = np.zeros(32, np.float32)
    z[9] = 1e-7                                                           # scale rounds to zero
    z[20] = -4e-8
    rows.append(z)
    rows.append(np.full(32, -0.0, np.float32))
    rows.append(np.full(32, 3.0, np.float32))                             # constant block
    return np.stack(rows).astype(np.float32)


def test_decision_edges_bit_exact(torch):
    w = _edge_blocks()
    M = w.shape[0]
    np.testing.assert_array_equal(_convert(torch, w), O.quantize_weights(w, M, 32))
    # the same blocks laid along K, in every position of a warp's eight-block step
    for shift in range(8):
        wk = np.concatenate([np.zeros((1, 32 * shift), np.float32), w.reshape(1, -1)], axis=1)
        np.testing.assert_array_equal(_convert(torch, wk), O.quantize_weights(wk, 1, wk.shape[1]))


def test_full_size_matrix_and_matvec(torch):
    """A 16384 x 4096 matrix: the blocks equal the oracle's, and a handle built
    from the device blocks gives the matvec of those blocks."""
    M, K = 16384, 4096
    rng = np.random.default_rng(21)
    w = (rng.standard_normal((M, K)) * 0.02).astype(np.float32)
    wd = torch.from_numpy(w).cuda()
    blocks = cbq.cbq_quantize_weights(wd)
    torch.cuda.synchronize()
    ref = O.quantize_weights(w, M, K)
    np.testing.assert_array_equal(blocks.cpu().numpy(), ref)
    Wh = cbq.Weights(blocks, M, K)
    x = synth.activations(1, K, stream=22)
    y = cbq.cbq_matvec(Wh, torch.from_numpy(x).cuda()).cpu().numpy()
    qx, dx = O.quantize_act(x)
    rows = np.arange(0, M, 97)
    yr = O.matvec_q(ref, M, K, qx, dx, rows=rows)
    b = O.matvec_bound(ref, M, K, qx, dx, rows=rows)
    assert np.all(np.abs(y[:, rows] - yr) <= 1e-4 * b)
    assert cbq.cbq_weights_get_error(Wh) == 0


def test_output_offset_and_stream_order(torch):
    """Blocks written at a 2-byte (not 4-byte) aligned offset, into a buffer
    whose other bytes stay untouched; two conversions in a row on one stream."""
    M, K = 9, 224
    rng = np.random.default_rng(23)
    w1 = rng.standard_normal((M, K)).astype(np.float32)
    w2 = rng.standard_normal((M, K)).astype(np.float32)
    n = M * (K // 32) * 18
    buf = torch.full((n + 4,), 0xAB, dtype=torch.uint8, device="cuda")
    out = buf[2:2 + n]
    assert out.data_ptr() % 4 == 2
    cbq.cbq_quantize_weights(torch.from_numpy(w1).cuda(), out=out)
    cbq.cbq_quantize_weights(torch.from_numpy(w2).cuda(), out=out)
    got = buf.cpu().numpy()
    assert got[0] == got[1] == got[-2] == got[-1] == 0xAB
    np.testing.assert_array_equal(got[2:2 + n].reshape(M, K // 32, 18), O.quantize_weights(w2, M, K))
