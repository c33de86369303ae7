"""Dense path on the GPU (through the C ABI) against the CPU oracle.

Bit-exact: activation quantization and every per-block int32 dot.  Within
1e-4 * sum_i |w_i * xhat_i| per output: the fp32 matvec.  Exact on the GPU
too: doubling every scale doubles y, negating x negates y, a zero scale gives
a zero row.
"""
import numpy as np
import pytest

from oracle import oracle as O
from tests.gpu_util import Guarded, assert_within_bound, cuda
from verify_matvec_gb300 import cbq, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return cuda()


def _dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# --------------------------------------------------------- quantization ---

@pytest.mark.parametrize("n,K,outliers", [(1, 1024, False), (1, 4096, True), (5, 4096, False),
                                          (3, 2048, True), (2, 32, False), (5, 96, True)])
def test_quantize_bit_exact(torch, n, K, outliers):
    x = synth.activations(n, K, stream=101 + K + n, outliers=outliers)
    x[0, :32] = 0.0                         # an all-zero block
    x[-1, 32 * (K // 64):32 * (K // 64) + 32] = 3.0  # a constant block
    gq, gd = Guarded(torch, (n, K), torch.int8), Guarded(torch, (n, K // 32), torch.float32)
    qx, dx = cbq.cbq_quantize_act(_dev(torch, x), qx=gq.view, dx=gd.view)
    gq.check()
    gd.check()
    qr, dr = O.quantize_act(x)
    np.testing.assert_array_equal(qx.cpu().numpy(), qr)
    np.testing.assert_array_equal(dx.cpu().numpy().view(np.uint32), dr.view(np.uint32))


def test_quantize_golden_ties(torch, golden_dir):
    from tests.test_oracle import _read_quant_cases
    cases = _read_quant_cases(golden_dir)
    X = np.array([[float(v) for v in c["x"]] for c in cases], dtype=np.float32)
    qx, _ = cbq.cbq_quantize_act(_dev(torch, X))
    np.testing.assert_array_equal(qx.cpu().numpy(), np.array([[int(v) for v in c["q"]] for c in cases]))


# ------------------------------------------------------------ block dots ---

@pytest.mark.parametrize("M,K", [(256, 1024), (70, 160), (33, 32), (1, 96), (130, 4096)])
@pytest.mark.parametrize("n", [1, 2, 3, 5])
def test_block_dots_bit_exact(torch, M, K, n):
    W = synth.weight_blocks(M, K, stream=201 + M)
    Wh = cbq.Weights(W, M, K)
    qx = np.random.default_rng(M * 7 + n).integers(-127, 128, size=(n, K)).astype(np.int8)
    qx[0, :32] = 127
    s = cbq.cbq_debug_block_dots(Wh, _dev(torch, qx)).cpu().numpy()
    np.testing.assert_array_equal(s, O.block_dots(W, M, K, qx))


def test_block_dots_every_codebook_entry(torch):
    M, K = 32, 512
    W = np.zeros((M, K // 32, 18), dtype=np.uint8)
    for r in range(M):
        W[r, :, 2:] = (r % 16) | ((15 - r % 16) << 4)
    Wh = cbq.Weights(W, M, K)
    qx = np.ones((4, K), dtype=np.int8)
    qx[1] = -1
    qx[2, ::2] = 127
    qx[3] = np.random.default_rng(5).integers(-127, 128, size=K)
    s = cbq.cbq_debug_block_dots(Wh, _dev(torch, qx)).cpu().numpy()
    np.testing.assert_array_equal(s, O.block_dots(W, M, K, qx))


# ---------------------------------------------------------------- matvec ---

def _check_matvec(torch, W, M, K, x, rows=None):
    Wh = cbq.Weights(W, M, K)
    g = Guarded(torch, (x.shape[0], M), torch.float32)
    y = cbq.cbq_matvec(Wh, _dev(torch, x), y=g.view).cpu().numpy()
    g.check()
    qx, dx = O.quantize_act(x)
    yr = O.matvec_q(W, M, K, qx, dx, rows=rows)
    b = O.matvec_bound(W, M, K, qx, dx, rows=rows)
    assert_within_bound(y if rows is None else y[:, rows], yr, b)
    assert cbq.cbq_weights_get_error(Wh) == 0
    return Wh, y


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_matvec_tiny_config(torch, n):
    M, K = 256, 1024
    W = synth.weight_blocks(M, K, stream=synth.S_W)
    _check_matvec(torch, W, M, K, synth.activations(n, K, stream=synth.S_X))


@pytest.mark.parametrize("M,K", [(70, 160), (33, 32), (1, 4096), (100, 2080)])
@pytest.mark.parametrize("n", [1, 3, 5])
def test_matvec_ragged(torch, M, K, n):
    W = synth.weight_blocks(M, K, stream=301 + M + K)
    _check_matvec(torch, W, M, K, synth.activations(n, K, stream=302, outliers=True))


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_matvec_4096_full(torch, n):
    M = K = 4096
    W = synth.weight_blocks(M, K, stream=synth.S_W)
    _check_matvec(torch, W, M, K, synth.activations(n, K, stream=synth.S_X + n, outliers=(n == 1)))


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_matvec_16384_all_rows(torch, n):
    M, K = 16384, 4096
    W = synth.weight_blocks(M, K, stream=synth.S_W + 50)
    _check_matvec(torch, W, M, K, synth.activations(n, K, stream=synth.S_X + 50, outliers=True))


@pytest.mark.parametrize("n", [1, 5])
def test_matvec_single_group_items_all_rows(torch, n):
    """32,800 x 2080: 513 pairs of row groups, more than the resident CTAs, so
    the launcher takes single-group work items (1,026 of them, several per
    CTA), with a ragged last pair (one real group) and an odd chunk count
    (65 blocks, padded to 68: the last stage holds one chunk of four blocks,
    three of them padding).  Every row against the oracle."""
    M, K = 32800, 2080
    W = synth.weight_blocks(M, K, stream=synth.S_W + 60)
    _check_matvec(torch, W, M, K, synth.activations(n, K, stream=synth.S_X + 60, outliers=True))


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("K", [1024, 1056])
def test_matvec_q_equals_matvec_and_host_entry(torch, n, K):
    """cbq_matvec quantizes inside the matvec kernel for one 16-byte aligned
    column and through the quantization kernel otherwise; both, the
    pre-quantized entry and the host entry give the same bits."""
    M = 300
    W = synth.weight_blocks(M, K, stream=401)
    x = synth.activations(n, K, stream=402 + n, outliers=True)
    Wh = cbq.Weights(W, M, K)
    y = cbq.cbq_matvec(Wh, _dev(torch, x)).cpu().numpy()
    qx, dx = cbq.cbq_quantize_act(_dev(torch, x))
    yq = cbq.cbq_matvec_q(Wh, qx, dx).cpu().numpy()
    np.testing.assert_array_equal(yq, y)
    yh = cbq.cbq_matvec_host(Wh, x)
    np.testing.assert_array_equal(yh, y)
    buf = torch.zeros(n * K + 1, dtype=torch.float32, device="cuda")
    buf[1:] = _dev(torch, x).reshape(-1)
    xm = buf[1:].view(n, K)  # 4 bytes past a 16-byte boundary
    assert xm.data_ptr() % 16 == 4
    np.testing.assert_array_equal(cbq.cbq_matvec(Wh, xm).cpu().numpy(), y)


def test_matvec_exact_invariants(torch):
    M, K, n = 200, 2048, 5
    W = synth.weight_blocks(M, K, stream=501)
    W[7, :, 0:2] = 0
    x = synth.activations(n, K, stream=502)
    Wh = cbq.Weights(W, M, K)
    y = cbq.cbq_matvec(Wh, _dev(torch, x)).cpu().numpy()
    assert np.all(y[:, 7] == 0)
    yn = cbq.cbq_matvec(Wh, _dev(torch, -x)).cpu().numpy()
    np.testing.assert_array_equal(yn, -y)
    W2 = W.copy()
    bits = W2[:, :, 0:2].copy().view(np.uint16)
    nz = bits != 0
    bits[nz] += np.uint16(0x0400)
    W2[:, :, 0:2] = bits.view(np.uint8)
    y2 = cbq.cbq_matvec(cbq.Weights(W2, M, K), _dev(torch, x)).cpu().numpy()
    np.testing.assert_array_equal(y2, 2 * y)


def test_output_head_all_rows_bench_shape(torch):
    """The 129280 x 4096 head at n = 5, launched as the benchmark launches it,
    every row against the oracle."""
    M, K, n = 129280, 4096, 5
    W = synth.weight_blocks(M, K, stream=synth.S_HEAD)
    x = synth.activations(n, K, stream=synth.S_HEAD_X)
    _check_matvec(torch, W, M, K, x)


def test_largest_k_accepted_and_correct(torch):
    """K = 27,136 (848 blocks: the most the 5-column staging fits beside a
    four-stage weight ring and the 5-column partial-sum set in 227 KB), ragged
    M, a partial last stage."""
    M, K = 70, 27136
    W = synth.weight_blocks(M, K, stream=450)
    for n in (1, 5):
        _check_matvec(torch, W, M, K, synth.activations(n, K, stream=451 + n, outliers=True))


def test_k_beyond_staging_limit_refused(torch):
    M, K = 32, 27168
    with pytest.raises(cbq.CbqError) as info:
        cbq.Weights(synth.weight_blocks(M, K, stream=452), M, K)
    assert info.value.status == cbq.CBQ_EINVAL


@pytest.mark.parametrize("n", [1, 2, 5])
def test_back_to_back_calls_on_one_handle(torch, n):
    """Many calls on one handle, enqueued without a synchronization between
    them (each call's first kernel may become resident while the previous call
    still runs), give the bits of calls made one at a time; so do the
    pre-quantized entry and the static-scratch entry."""
    M, K = 1000, 2048
    Wh = cbq.Weights(synth.weight_blocks(M, K, stream=460), M, K)
    xs = [_dev(torch, synth.activations(n, K, stream=461 + i)) for i in range(4)]
    ref = []
    for x in xs:
        ref.append(cbq.cbq_matvec(Wh, x).cpu().numpy())
        torch.cuda.synchronize()
    ys = [torch.empty((n, M), dtype=torch.float32, device="cuda") for _ in range(40)]
    for i, y in enumerate(ys):
        cbq.cbq_matvec(Wh, xs[i % 4], y=y)
    torch.cuda.synchronize()
    for i, y in enumerate(ys):
        np.testing.assert_array_equal(y.cpu().numpy(), ref[i % 4])
    qd = [cbq.cbq_quantize_act(x) for x in xs]
    for i, y in enumerate(ys):  # the three entry points interleaved, still unsynchronized
        if i % 3 == 0:
            cbq.cbq_matvec_q(Wh, qd[i % 4][0], qd[i % 4][1], y=y)
        elif i % 3 == 1:
            cbq.cbq_matvec_static(Wh, xs[i % 4], y=y)
        else:
            cbq.cbq_matvec(Wh, xs[i % 4], y=y)
    torch.cuda.synchronize()
    for i, y in enumerate(ys):
        np.testing.assert_array_equal(y.cpu().numpy(), ref[i % 4])
    assert cbq.cbq_weights_get_error(Wh) == 0
