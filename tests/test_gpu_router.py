"""Routed-expert selection on the GPU (cbq_router_topk) against the CPU
oracle, and the routed layer fed by router logits (cbq_moe_matvec_logits).

Ids are integer decisions taken on the same fp32 logits: bit-exact.  The
weights are an fp64 softmax rounded to fp32 on both sides: equal up to one
fp32 ulp (the two exp implementations differ by a few fp64 ulps).
"""
import numpy as np
import pytest

from oracle import oracle as O
from tests.gpu_util import Guarded, cuda
from tests.test_gpu_moe import _check_layer
from verify_matvec_gb300 import cbq, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return cuda()


def _dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _logits(n_tok, E, seed, ties=False):
    g = np.random.default_rng(seed)
    lg = g.standard_normal((n_tok, E)).astype(np.float32)
    if ties:
        lg = np.round(lg * 4).astype(np.float32) / 4  # many equal logits
    return lg


def _check_router(torch, lg, k):
    gi, gw = Guarded(torch, (lg.shape[0], k), torch.int32), Guarded(torch, (lg.shape[0], k), torch.float32)
    ids, wts = cbq.cbq_router_topk(_dev(torch, lg), k, ids=gi.view, wts=gw.view)
    gi.check()
    gw.check()
    ids, wts = ids.cpu().numpy(), wts.cpu().numpy()
    ids_r, wts_r = O.router_topk(lg, k)
    np.testing.assert_array_equal(ids, ids_r)
    ref32 = wts_r.astype(np.float32)
    assert np.all(np.abs(wts - ref32) <= np.spacing(ref32)), "weights beyond one fp32 ulp"
    return ids, wts


@pytest.mark.parametrize("n_tok,E,k", [(1, 1, 1), (1, 8, 4), (5, 256, 8), (5, 20, 16), (3, 33, 7),
                                       (200, 256, 8), (2, 16384, 16)])
@pytest.mark.parametrize("ties", [False, True])
def test_router_topk_matches_oracle(torch, n_tok, E, k, ties):
    _check_router(torch, _logits(n_tok, E, 700 + E + k, ties), k)


def test_router_all_equal_logits_pick_lowest_indices(torch):
    lg = np.full((2, 40), 1.5, dtype=np.float32)
    ids, wts = _check_router(torch, lg, 6)
    np.testing.assert_array_equal(ids, np.tile(np.arange(6), (2, 1)))
    np.testing.assert_array_equal(wts, np.full((2, 6), np.float32(1 / 6)))


def test_router_rejects_bad_arguments(torch):
    lg = _dev(torch, _logits(2, 8, 1))
    for k in (0, 9, 17):
        with pytest.raises(cbq.CbqError) as info:
            cbq.cbq_router_topk(lg, k)
        assert info.value.status == cbq.CBQ_EINVAL
    big = torch.zeros((1, cbq.CBQ_ROUTER_MAX_E + 1), dtype=torch.float32, device="cuda")
    with pytest.raises(cbq.CbqError) as info:
        cbq.cbq_router_topk(big, 4)
    assert info.value.status == cbq.CBQ_EINVAL


E_W, H_W, F_W = 20, 256, 128


@pytest.fixture(scope="module")
def layer(torch):
    gu = synth.expert_blocks(E_W, 2 * F_W, H_W, stream=710)
    dn = synth.expert_blocks(E_W, H_W, F_W, stream=711)
    return gu, dn, cbq.Moe(gu, dn, E_W, H_W, F_W)


@pytest.mark.parametrize("n_tok,k", [(1, 4), (5, 8), (5, 16), (3, 2)])
def test_layer_from_logits(torch, layer, n_tok, k):
    """The logits entry equals the ids entry fed by the GPU router (same
    bits), picks the oracle's experts, and matches the oracle's layer."""
    gu, dn, L = layer
    lg = _logits(n_tok, E_W, 720 + n_tok + k, ties=(k == 8))
    h = synth.activations(n_tok, H_W, stream=721 + n_tok)
    y = cbq.cbq_moe_matvec_logits(L, _dev(torch, h), _dev(torch, lg), k).cpu().numpy()
    ids, wts = cbq.cbq_router_topk(_dev(torch, lg), k)
    y2 = cbq.cbq_moe_matvec(L, _dev(torch, h), ids, wts).cpu().numpy()
    np.testing.assert_array_equal(y, y2)
    ids_np, wts_np = ids.cpu().numpy(), wts.cpu().numpy()
    np.testing.assert_array_equal(ids_np, O.router_topk(lg, k)[0])
    _check_layer(torch, L, gu, dn, E_W, H_W, F_W, h, ids_np, wts_np, 1)


def test_full_layer_from_logits_batch5_top8(torch):
    """The 256-expert layer (4096 x 2048) from router logits of 5 tokens: the
    GPU picks the oracle's experts and the layer matches the oracle's."""
    from tests.test_gpu_moe import E, F, H
    g = np.random.default_rng(730)
    lg = g.standard_normal((5, E)).astype(np.float32)
    ids_r, _ = O.router_topk(lg, 8)
    used = synth.distinct_experts(ids_r, E)
    gu = np.zeros((E, 2 * F, H // 32, 18), dtype=np.uint8)
    dn = np.zeros((E, H, F // 32, 18), dtype=np.uint8)
    for e in used:
        gu[e] = synth.weight_blocks(2 * F, H, stream=synth.S_GATE_UP * 1000 + int(e))
        dn[e] = synth.weight_blocks(H, F, stream=synth.S_DOWN * 1000 + int(e))
    L = cbq.Moe(gu, dn, E, H, F)
    h = synth.activations(5, H, stream=731)
    y = cbq.cbq_moe_matvec_logits(L, _dev(torch, h), _dev(torch, lg), 8).cpu().numpy()
    ids, wts = cbq.cbq_router_topk(_dev(torch, lg), 8)
    ids_np, wts_np = ids.cpu().numpy(), wts.cpu().numpy()
    np.testing.assert_array_equal(ids_np, ids_r)
    y2 = _check_layer(torch, L, gu, dn, E, H, F, h, ids_np, wts_np, 1)
    np.testing.assert_array_equal(y, y2)
