"""Routed-expert path (gate_up + SwiGLU + requant, down + combine) on the GPU
against the CPU oracle, stage by stage and end to end.

Stage 1: the fp32 intermediate a of every (token, slot) within the bound
propagated from the gate/up tolerance.  Requantization: (qa, da) bit-exact
with the oracle's quantization of the GPU's own a.  Stage 2: y within
1e-4 * sum_j |r_j| * sum_i |wd_i * ahat_i| of the oracle's down+combine fed
the GPU's own (qa, da).  End to end: y against the oracle's own a, with the
extra term sum_j |r_j| sum_i |wd_i| |ahat_gpu - ahat_ref| for requantization
flips near rounding ties.
"""
import numpy as np
import pytest

from oracle import oracle as O
from tests.gpu_util import TOL, Guarded, assert_within_bound, cuda
from tests.test_oracle import _np_dequant
from verify_matvec_gb300 import cbq, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return cuda()


def _dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _check_layer(torch, L, gu, dn, E, H, F, h, ids, wts, swiglu, expect_bad=0, shared=None):
    """shared = (gate_up, down) blocks of the shared expert L holds, or None."""
    n_tok, k = ids.shape
    N = n_tok * k
    cbq.cbq_moe_set_debug(L, True)
    g = Guarded(torch, (n_tok, H), torch.float32)
    y = cbq.cbq_moe_matvec(L, _dev(torch, h), _dev(torch, ids), _dev(torch, wts), swiglu=swiglu,
                           y=g.view).cpu().numpy()
    g.check()
    a_g, qa_g, da_g = (t.cpu().numpy() for t in
                       cbq.cbq_moe_debug_intermediate(L, N + (n_tok if shared is not None else 0)))
    err = cbq.cbq_moe_get_error(L)
    assert err == (cbq.CBQ_DEVERR_BAD_EXPERT_ID if expect_bad else 0)
    if shared is not None:
        sgu, sdn = shared
        y_sh, nbad_sh = O.moe_shared(gu, dn, E, H, F, sgu, sdn, h, ids, wts, swiglu=swiglu)
        assert nbad_sh == expect_bad
        # The checks below then run on an equivalent routed layer: the experts
        # the tokens use, then the shared one, in a compact table; every token
        # gets one more slot (last, weight 1) on the shared expert.  The GPU
        # keeps the shared slots after the routed ones (N + t).
        used = np.unique(ids[(ids >= 0) & (ids < E)])
        remap = {int(e): i for i, e in enumerate(used)}
        ids_c = np.array([[remap.get(int(e), -1) for e in row] for row in ids], dtype=np.int32)
        gu = np.concatenate([gu[used], sgu[None]])
        dn = np.concatenate([dn[used], sdn[None]])
        E = len(used) + 1
        ids = np.concatenate([ids_c, np.full((n_tok, 1), E - 1, np.int32)], axis=1)
        wts = np.concatenate([wts, np.ones((n_tok, 1), np.float32)], axis=1)
        gpu_slot = [t * k + j if j < k else N + t for t in range(n_tok) for j in range(k + 1)]
        a_g, qa_g, da_g = a_g[gpu_slot], qa_g[gpu_slot], da_g[gpu_slot]
        k += 1
    valid = ((ids >= 0) & (ids < E)).ravel()

    # stage 1: a per slot against the oracle's g, u and their bounds
    qh, dh = O.quantize_act(h)
    for p in np.flatnonzero(valid):
        t, e = p // k, int(ids.ravel()[p])
        G = gu[e].reshape(2 * F, -1)
        g = O.matvec_q(G[:F].ravel(), F, H, qh[t], dh[t])[0]
        u = O.matvec_q(G[F:].ravel(), F, H, qh[t], dh[t])[0]
        bg = TOL * O.matvec_bound(G[:F].ravel(), F, H, qh[t], dh[t])[0]
        bu = TOL * O.matvec_bound(G[F:].ravel(), F, H, qh[t], dh[t])[0]
        if swiglu:
            sg = np.array([O.silu(v) for v in g])
            a_ref = sg * u
            lim = 1.1 * np.abs(u) * bg + np.abs(sg) * bu + 1.1 * bg * bu
        else:
            a_ref = g * u
            lim = np.abs(u) * bg + np.abs(g) * bu + bg * bu
        lim = lim + 4 * 2.0 ** -24 * np.abs(a_ref) + 1e-30
        assert np.all(np.abs(a_g[p] - a_ref) <= lim), f"slot {p}: a outside bound"
        # requantization: bit-exact on the GPU's own a
        qa_r, da_r = O.quantize_act(a_g[p])
        np.testing.assert_array_equal(qa_g[p], qa_r)
        np.testing.assert_array_equal(da_g[p].view(np.uint32), da_r.view(np.uint32))

    # stage 2: down + combine from the GPU's own quantized intermediate
    qa_use = np.where(valid[:, None], qa_g, 0).astype(np.int8)
    da_use = np.where(valid[:, None], da_g, 0).astype(np.float32)
    y2, yb, nbad = O.moe_down_combine(dn, E, H, F, ids, wts, qa_use, da_use)
    assert nbad == expect_bad
    assert_within_bound(y, y2, yb, what="y (stage 2)")

    # end to end against the oracle's own intermediate
    y_ref, _, qa_r, da_r, nbad = O.moe(gu, dn, E, H, F, h, ids, wts, swiglu=swiglu, want_intermediate=True)
    extra = np.zeros_like(y_ref)
    for p in np.flatnonzero(valid):
        t, e = p // k, int(ids.ravel()[p])
        dah = np.abs(qa_use[p].astype(np.float64) * np.repeat(da_use[p].astype(np.float64), 32)
                     - qa_r[p].astype(np.float64) * np.repeat(da_r[p].astype(np.float64), 32))
        if np.any(dah):
            extra[t] += abs(float(wts.ravel()[p])) * (np.abs(_np_dequant(dn[e], H, F)) @ dah)
    assert_within_bound(y, y_ref, yb + extra / TOL, what="y (end to end)")
    if shared is not None:
        assert_within_bound(y, y_sh, yb + extra / TOL, what="y (end to end, shared-expert oracle)")
    return y


# ------------------------------------------------------------- small layer -

E_S, H_S, F_S = 8, 256, 128


@pytest.fixture(scope="module")
def small(torch):
    gu = synth.expert_blocks(E_S, 2 * F_S, H_S, stream=601)
    dn = synth.expert_blocks(E_S, H_S, F_S, stream=602)
    return gu, dn, cbq.Moe(gu, dn, E_S, H_S, F_S)


@pytest.mark.parametrize("n_tok,k", [(1, 1), (1, 4), (3, 2), (5, 3), (5, 8), (2, 8)])
@pytest.mark.parametrize("swiglu", [1, 0])
def test_small_layer(torch, small, n_tok, k, swiglu):
    gu, dn, L = small
    h = synth.activations(n_tok, H_S, stream=603 + n_tok)
    ids, wts = synth.router(n_tok, k, E_S, stream=604 + k)
    _check_layer(torch, L, gu, dn, E_S, H_S, F_S, h, ids, wts, swiglu)


def test_duplicates_and_bad_ids(torch, small):
    gu, dn, L = small
    h = synth.activations(5, H_S, stream=610)
    ids = np.array([[3, 3, 1], [9, 2, -4], [2, 2, 2], [0, 7, 3], [3, 3, 3]], dtype=np.int32)
    wts = np.random.default_rng(3).random((5, 3)).astype(np.float32)
    _check_layer(torch, L, gu, dn, E_S, H_S, F_S, h, ids, wts, 1, expect_bad=2)


def test_nothing_routed_gives_zero(torch, small):
    gu, dn, L = small
    h = synth.activations(2, H_S, stream=611)
    ids = np.array([[-1, 8], [100, -7]], dtype=np.int32)
    wts = np.ones((2, 2), dtype=np.float32)
    y = cbq.cbq_moe_matvec(L, _dev(torch, h), _dev(torch, ids), _dev(torch, wts)).cpu().numpy()
    assert np.all(y == 0)
    assert cbq.cbq_moe_get_error(L) == cbq.CBQ_DEVERR_BAD_EXPERT_ID
    assert cbq.cbq_moe_get_error(L) == 0  # read clears


def test_nothing_routed_gives_zero_one_token(torch, small):
    """One token (the layer kernel forms y itself): no valid id still writes y."""
    gu, dn, L = small
    h = synth.activations(1, H_S, stream=614)
    ids = np.array([[-3, 8, 11]], dtype=np.int32)
    wts = np.ones((1, 3), dtype=np.float32)
    y = cbq.cbq_moe_matvec(L, _dev(torch, h), _dev(torch, ids), _dev(torch, wts),
                           y=torch.full((1, H_S), 7.0, device="cuda")).cpu().numpy()
    assert np.all(y == 0)
    assert cbq.cbq_moe_get_error(L) == cbq.CBQ_DEVERR_BAD_EXPERT_ID


def test_error_word_is_per_handle(torch, small):
    """A bad id on one handle shows in that handle's error word only."""
    gu, dn, L = small
    L2 = cbq.Moe(gu, dn, E_S, H_S, F_S)
    h = synth.activations(2, H_S, stream=615)
    bad = np.array([[1, 99], [2, 3]], dtype=np.int32)
    ids, wts = synth.router(2, 2, E_S, stream=616)
    cbq.cbq_moe_matvec(L, _dev(torch, h), _dev(torch, bad), _dev(torch, wts))
    cbq.cbq_moe_matvec(L2, _dev(torch, h), _dev(torch, ids), _dev(torch, wts))
    torch.cuda.synchronize()
    assert cbq.cbq_moe_get_error(L2) == 0
    assert cbq.cbq_moe_get_error(L) == cbq.CBQ_DEVERR_BAD_EXPERT_ID


def test_host_entry_matches(torch, small):
    gu, dn, L = small
    h = synth.activations(4, H_S, stream=612)
    ids, wts = synth.router(4, 3, E_S, stream=613)
    y = cbq.cbq_moe_matvec(L, _dev(torch, h), _dev(torch, ids), _dev(torch, wts)).cpu().numpy()
    np.testing.assert_array_equal(cbq.cbq_moe_matvec_host(L, h, ids, wts), y)


def test_expert_block_dots(torch, small):
    gu, dn, L = small
    qx = np.random.default_rng(9).integers(-127, 128, size=(3, H_S)).astype(np.int8)
    s = cbq.cbq_moe_debug_block_dots(L, 5, 0, _dev(torch, qx)).cpu().numpy()
    np.testing.assert_array_equal(s, O.block_dots(gu[5], 2 * F_S, H_S, qx))
    qx = np.random.default_rng(10).integers(-127, 128, size=(2, F_S)).astype(np.int8)
    s = cbq.cbq_moe_debug_block_dots(L, 7, 1, _dev(torch, qx)).cpu().numpy()
    np.testing.assert_array_equal(s, O.block_dots(dn[7], H_S, F_S, qx))


def test_repeated_calls_are_deterministic(torch, small):
    gu, dn, L = small
    h = _dev(torch, synth.activations(5, H_S, stream=614))
    ids, wts = synth.router(5, 8, E_S, stream=615)
    ids, wts = _dev(torch, ids), _dev(torch, wts)
    ys = [cbq.cbq_moe_matvec(L, h, ids, wts).cpu().numpy() for _ in range(3)]
    np.testing.assert_array_equal(ys[0], ys[1])
    np.testing.assert_array_equal(ys[0], ys[2])


# --------------------------------------------------------- full-size layer -

E, H, F = 256, 4096, 2048


@pytest.fixture(scope="module")
def full(torch):
    """The 256-expert layer; only the experts the two routing tables use are
    drawn, the rest stay zero (their bytes are never read)."""
    ids1, wts1 = synth.router(1, 4, E, stream=synth.S_IDS)
    ids5, wts5 = synth.router(5, 8, E, stream=synth.S_IDS + 1)
    used = np.union1d(synth.distinct_experts(ids1, E), synth.distinct_experts(ids5, E))
    gu = np.zeros((E, 2 * F, H // 32, 18), dtype=np.uint8)
    dn = np.zeros((E, H, F // 32, 18), dtype=np.uint8)
    for e in used:
        gu[e] = synth.weight_blocks(2 * F, H, stream=synth.S_GATE_UP * 1000 + int(e))
        dn[e] = synth.weight_blocks(H, F, stream=synth.S_DOWN * 1000 + int(e))
    L = cbq.Moe(gu, dn, E, H, F)
    return gu, dn, L, (ids1, wts1), (ids5, wts5)


def test_full_layer_batch1_top4(torch, full):
    gu, dn, L, (ids, wts), _ = full
    h = synth.activations(1, H, stream=synth.S_H)
    _check_layer(torch, L, gu, dn, E, H, F, h, ids, wts, 1)


def test_full_layer_batch5_top8(torch, full):
    gu, dn, L, _, (ids, wts) = full
    h = synth.activations(5, H, stream=synth.S_H + 1)
    _check_layer(torch, L, gu, dn, E, H, F, h, ids, wts, 1)


# ------------------------------------------------------------- edge shapes -

@pytest.fixture(scope="module")
def wide(torch):
    """20 experts, so 5 tokens can each route top-16 (80 slots, the maximum)."""
    E_, H_, F_ = 20, 256, 128
    gu = synth.expert_blocks(E_, 2 * F_, H_, stream=620)
    dn = synth.expert_blocks(E_, H_, F_, stream=621)
    return gu, dn, cbq.Moe(gu, dn, E_, H_, F_), (E_, H_, F_)


def test_maximum_slots_5x16(torch, wide):
    gu, dn, L, (E_, H_, F_) = wide
    h = synth.activations(5, H_, stream=622)
    ids, wts = synth.router(5, 16, E_, stream=623)
    _check_layer(torch, L, gu, dn, E_, H_, F_, h, ids, wts, 1)


def test_expert_serving_more_than_five_slots(torch, wide):
    """Expert 3 takes 8 slots (repeated ids are served as extra columns), so
    its items run as two column chunks (5 + 3)."""
    gu, dn, L, (E_, H_, F_) = wide
    h = synth.activations(5, H_, stream=624)
    ids = np.array([[3, 3, 3], [3, 3, 1], [3, 0, 2], [3, 5, 6], [7, 3, 19]], dtype=np.int32)
    wts = np.random.default_rng(5).random((5, 3)).astype(np.float32)
    _check_layer(torch, L, gu, dn, E_, H_, F_, h, ids, wts, 1)


@pytest.mark.parametrize("H_,F_", [(160, 96), (1120, 352)])
def test_ragged_layer_dims(torch, H_, F_):
    """Block counts that are not multiples of 4 (padded blocks) or of 32
    (a partial last stage), in both the gate_up and the down passes."""
    E_ = 6
    gu = synth.expert_blocks(E_, 2 * F_, H_, stream=630 + H_)
    dn = synth.expert_blocks(E_, H_, F_, stream=631 + F_)
    L = cbq.Moe(gu, dn, E_, H_, F_)
    for n_tok, k in ((1, 2), (5, 4)):
        h = synth.activations(n_tok, H_, stream=632 + n_tok)
        ids, wts = synth.router(n_tok, k, E_, stream=633 + k)
        _check_layer(torch, L, gu, dn, E_, H_, F_, h, ids, wts, 1)


@pytest.mark.parametrize("H_,n_tok", [(27648, 5), (32768, 1), (33792, 1)])
def test_large_hidden(torch, H_, n_tok):
    """Large hidden sizes: five tokens through the quantization kernel; one
    token quantized in the layer kernel (32,768 = 1,024 staged blocks, the
    most it stages) and, one block group beyond that, through the
    quantization kernel."""
    E_, F_ = 3, 64
    gu = synth.expert_blocks(E_, 2 * F_, H_, stream=640)
    dn = synth.expert_blocks(E_, H_, F_, stream=641)
    L = cbq.Moe(gu, dn, E_, H_, F_)
    h = synth.activations(n_tok, H_, stream=642)
    ids, wts = synth.router(n_tok, 2, E_, stream=643)
    _check_layer(torch, L, gu, dn, E_, H_, F_, h, ids, wts, 1)


def test_one_token_quantized_in_kernel_matches_kernel_path(torch, small):
    """One token with h 16-byte aligned is quantized inside the layer kernel;
    shifted by 4 bytes it goes through the quantization kernel: same bits."""
    gu, dn, L = small
    h = synth.activations(1, H_S, stream=650, outliers=True)
    ids, wts = synth.router(1, 4, E_S, stream=651)
    y = cbq.cbq_moe_matvec(L, _dev(torch, h), _dev(torch, ids), _dev(torch, wts)).cpu().numpy()
    buf = torch.zeros(H_S + 1, dtype=torch.float32, device="cuda")
    buf[1:] = _dev(torch, h).reshape(-1)
    hm = buf[1:].view(1, H_S)
    assert hm.data_ptr() % 16 == 4
    ym = cbq.cbq_moe_matvec(L, hm, _dev(torch, ids), _dev(torch, wts)).cpu().numpy()
    np.testing.assert_array_equal(ym, y)


@pytest.mark.parametrize("n_tok,k", [(1, 4), (5, 8)])
def test_back_to_back_layer_calls(torch, small, n_tok, k):
    """Layer calls on one handle enqueued without a synchronization between
    them, alternating routing tables and the ids and logits entries, give the
    bits of calls made one at a time."""
    gu, dn, L = small
    tabs = []
    for i in range(3):
        h = _dev(torch, synth.activations(n_tok, H_S, stream=660 + i))
        ids, wts = synth.router(n_tok, k, E_S, stream=663 + i)
        tabs.append((h, _dev(torch, ids), _dev(torch, wts)))
    ref = []
    for h, ids, wts in tabs:
        ref.append(cbq.cbq_moe_matvec(L, h, ids, wts).cpu().numpy())
        torch.cuda.synchronize()
    lg = _dev(torch, np.random.default_rng(666).standard_normal((n_tok, E_S)).astype(np.float32))
    y_lg = cbq.cbq_moe_matvec_logits(L, tabs[0][0], lg, k).cpu().numpy()
    ys = [torch.empty((n_tok, H_S), dtype=torch.float32, device="cuda") for _ in range(30)]
    for i, y in enumerate(ys):
        if i % 4 == 3:
            cbq.cbq_moe_matvec_logits(L, tabs[0][0], lg, k, y=y)
        else:
            h, ids, wts = tabs[i % 3]
            cbq.cbq_moe_matvec(L, h, ids, wts, y=y)
    torch.cuda.synchronize()
    for i, y in enumerate(ys):
        np.testing.assert_array_equal(y.cpu().numpy(), y_lg if i % 4 == 3 else ref[i % 3])
    assert cbq.cbq_moe_get_error(L) == 0


# ----------------------------------------------------------- shared expert -

@pytest.fixture(scope="module")
def small_shared(torch):
    """The small layer on its own handle, with a shared expert drawn apart
    from the routed ones."""
    gu = synth.expert_blocks(E_S, 2 * F_S, H_S, stream=601)
    dn = synth.expert_blocks(E_S, H_S, F_S, stream=602)
    sgu = synth.expert_blocks(1, 2 * F_S, H_S, stream=670)[0]
    sdn = synth.expert_blocks(1, H_S, F_S, stream=671)[0]
    L = cbq.Moe(gu, dn, E_S, H_S, F_S)
    cbq.cbq_moe_set_shared(L, sgu, sdn)
    return gu, dn, (sgu, sdn), L


@pytest.mark.parametrize("n_tok,k", [(1, 1), (1, 4), (3, 2), (5, 8)])
@pytest.mark.parametrize("swiglu", [1, 0])
def test_shared_expert_small(torch, small_shared, n_tok, k, swiglu):
    gu, dn, sh, L = small_shared
    h = synth.activations(n_tok, H_S, stream=672 + n_tok)
    ids, wts = synth.router(n_tok, k, E_S, stream=673 + k)
    _check_layer(torch, L, gu, dn, E_S, H_S, F_S, h, ids, wts, swiglu, shared=sh)


def test_shared_expert_bad_ids_are_not_the_shared_one(torch, small_shared):
    """A routed id equal to E (the shared expert's place in the kernels) or
    any other out-of-range id skips its slot; the shared slot still runs."""
    gu, dn, sh, L = small_shared
    h = synth.activations(3, H_S, stream=680)
    ids = np.array([[E_S, 1], [-1, E_S], [2, 2]], dtype=np.int32)
    wts = np.random.default_rng(11).random((3, 2)).astype(np.float32)
    _check_layer(torch, L, gu, dn, E_S, H_S, F_S, h, ids, wts, 1, expect_bad=3, shared=sh)


def test_shared_expert_alone(torch, small_shared):
    """Every routed id out of range: y is the shared expert's FFN."""
    gu, dn, sh, L = small_shared
    h = synth.activations(2, H_S, stream=681)
    ids = np.array([[-3, E_S + 1], [E_S, -1]], dtype=np.int32)
    y = _check_layer(torch, L, gu, dn, E_S, H_S, F_S, h, ids, np.ones((2, 2), np.float32), 1, expect_bad=4,
                     shared=sh)
    assert np.any(y != 0)


def test_shared_expert_block_dots(torch, small_shared):
    gu, dn, (sgu, sdn), L = small_shared
    qx = np.random.default_rng(12).integers(-127, 128, size=(2, H_S)).astype(np.int8)
    s = cbq.cbq_moe_debug_block_dots(L, E_S, 0, _dev(torch, qx)).cpu().numpy()
    np.testing.assert_array_equal(s, O.block_dots(sgu, 2 * F_S, H_S, qx))
    qx = np.random.default_rng(13).integers(-127, 128, size=(4, F_S)).astype(np.int8)
    s = cbq.cbq_moe_debug_block_dots(L, E_S, 1, _dev(torch, qx)).cpu().numpy()
    np.testing.assert_array_equal(s, O.block_dots(sdn, H_S, F_S, qx))


def test_shared_expert_set_replace_remove(torch, small):
    """Setting a shared expert, replacing it (from device memory) and removing
    it: each state computes its own layer, and removal gives back the routed
    layer's bits and the handle's byte count."""
    gu, dn, L = small
    h_np = synth.activations(5, H_S, stream=682)
    ids_np, wts_np = synth.router(5, 3, E_S, stream=683)
    h, ids, wts = _dev(torch, h_np), _dev(torch, ids_np), _dev(torch, wts_np)
    y0 = cbq.cbq_moe_matvec(L, h, ids, wts).cpu().numpy()
    b0 = L.device_bytes()
    with pytest.raises(cbq.CbqError):  # no shared expert: id E names nothing
        cbq.cbq_moe_debug_block_dots(L, E_S, 0, _dev(torch, np.zeros((1, H_S), np.int8)))
    try:
        cbq.cbq_moe_set_shared(L, gu[1], dn[1])  # a copy of routed expert 1
        assert L.device_bytes() > b0
        _check_layer(torch, L, gu, dn, E_S, H_S, F_S, h_np, ids_np, wts_np, 1, shared=(gu[1], dn[1]))
        cbq.cbq_moe_set_shared(L, _dev(torch, gu[4]), _dev(torch, dn[4]))
        _check_layer(torch, L, gu, dn, E_S, H_S, F_S, h_np, ids_np, wts_np, 1, shared=(gu[4], dn[4]))
        # every router weight 0: the shared expert's output alone, whatever the ids
        z = np.zeros_like(wts_np)
        o4 = _check_layer(torch, L, gu, dn, E_S, H_S, F_S, h_np, ids_np, z, 1, shared=(gu[4], dn[4]))
        o4b = cbq.cbq_moe_matvec(L, h, _dev(torch, np.full((5, 1), 1, np.int32)), _dev(torch, z[:, :1]))
        np.testing.assert_array_equal(o4b.cpu().numpy(), o4)
    finally:
        cbq.cbq_moe_set_shared(L, None, None)
    assert L.device_bytes() == b0
    np.testing.assert_array_equal(cbq.cbq_moe_matvec(L, h, ids, wts).cpu().numpy(), y0)
    with pytest.raises(ValueError):
        cbq.cbq_moe_set_shared(L, gu[1][:-1], dn[1])


def test_shared_expert_with_maximum_slots(torch, wide):
    """5 tokens x top-16 plus 5 shared slots: 85 columns, the most a call
    has."""
    gu, dn, L, (E_, H_, F_) = wide
    sgu = synth.expert_blocks(1, 2 * F_, H_, stream=684)[0]
    sdn = synth.expert_blocks(1, H_, F_, stream=685)[0]
    h = synth.activations(5, H_, stream=686)
    ids, wts = synth.router(5, 16, E_, stream=687)
    cbq.cbq_moe_set_shared(L, sgu, sdn)
    try:
        _check_layer(torch, L, gu, dn, E_, H_, F_, h, ids, wts, 1, shared=(sgu, sdn))
    finally:
        cbq.cbq_moe_set_shared(L, None, None)


@pytest.mark.parametrize("n_tok,k", [(1, 4), (5, 8)])
def test_shared_expert_full_size(torch, full, n_tok, k):
    gu, dn, L, t1, t5 = full
    ids, wts = t1 if n_tok == 1 else t5
    sgu = synth.weight_blocks(2 * F, H, stream=synth.S_GATE_UP * 1000 + 999)
    sdn = synth.weight_blocks(H, F, stream=synth.S_DOWN * 1000 + 999)
    h = synth.activations(n_tok, H, stream=synth.S_H + 7 + n_tok)
    cbq.cbq_moe_set_shared(L, sgu, sdn)
    try:
        _check_layer(torch, L, gu, dn, E, H, F, h, ids, wts, 1, shared=(sgu, sdn))
    finally:
        cbq.cbq_moe_set_shared(L, None, None)


@pytest.mark.parametrize("n_tok,k", [(1, 4), (5, 8)])
def test_inputs_written_just_before_the_call(torch, small, n_tok, k):
    """Each call's token and routing table are written by a device copy on the
    same stream right before it (no synchronization in between), so the
    call's first kernel must wait for that copy before it reads them."""
    gu, dn, L = small
    tabs = []
    for i in range(4):
        h = _dev(torch, synth.activations(n_tok, H_S, stream=690 + i))
        ids, wts = synth.router(n_tok, k, E_S, stream=694 + i)
        tabs.append((h, _dev(torch, ids), _dev(torch, wts)))
    ref = []
    for h, ids, wts in tabs:
        ref.append(cbq.cbq_moe_matvec(L, h, ids, wts).cpu().numpy())
        torch.cuda.synchronize()
    hb, ib, wb = (torch.empty_like(t) for t in tabs[0])
    ys = [torch.empty((n_tok, H_S), dtype=torch.float32, device="cuda") for _ in range(16)]
    for i, y in enumerate(ys):
        h, ids, wts = tabs[i % 4]
        hb.copy_(h)
        ib.copy_(ids)
        wb.copy_(wts)
        cbq.cbq_moe_matvec(L, hb, ib, wb, y=y)
    torch.cuda.synchronize()
    for i, y in enumerate(ys):
        np.testing.assert_array_equal(y.cpu().numpy(), ref[i % 4])
    assert cbq.cbq_moe_get_error(L) == 0
