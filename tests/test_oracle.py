"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Every test here runs on the CPU.  The pins are hand-worked fixtures
(tests/golden), exact-rational properties, numpy library routines (fp16
decoding, fp64 matmul) and invariants of the mathematics (linearity, sign
symmetry, zero scales, closed forms, the silu odd-part identity, the k=1
reduction of the routed-expert FFN).  Each one is chosen so that a plausible
slip in the oracle (a dropped factor, a swapped nibble, a wrong tie rule, a
gate/up swap, a misindexed router weight) fails at least one of them.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import oracle as O
from verify_matvec_gb300 import synth

QK = 32


# ---------------------------------------------------------------- fixtures --

def _read_codebook(golden_dir):
    with open(os.path.join(golden_dir, "codebook.txt")) as f:
        vals = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    return np.array([int(v) for v in vals[0].split()], dtype=np.int8)


def _read_quant_cases(golden_dir):
    cases, cur = [], {}
    with open(os.path.join(golden_dir, "quantize_blocks.txt")) as f:
        for ln in f:
            if ln.startswith("#") or not ln.strip():
                continue
            key, val = ln.split(":", 1)
            cur[key] = val.split()
            if key == "q":
                cases.append(cur)
                cur = {}
    return cases


def _read_block_cases(golden_dir):
    blocks = []
    with open(os.path.join(golden_dir, "block_dots.txt")) as f:
        for ln in f:
            if ln.startswith("#") or not ln.strip():
                continue
            parts = ln.split()
            if parts[0] == "block":
                bits = int(parts[2], 16)
                qs = [int(b, 16) for b in parts[3:]]
                assert len(qs) == 16
                blk = np.array([bits & 0xFF, bits >> 8] + qs, dtype=np.uint8)
                blocks.append({"name": parts[1], "blk": blk, "dots": []})
            elif parts[0] == "w":
                blocks[-1]["w"] = np.array([float(v) for v in parts[1:]])
            elif parts[0] == "dot":
                eq = parts.index("=")
                qx = np.array([int(v) for v in parts[1:eq]], dtype=np.int8)
                blocks[-1]["dots"].append((qx, int(parts[eq + 1])))
    return blocks


def _np_dequant(W, M, K):
    """Independent fp64 dequantization with numpy bit operations."""
    cb = O.CODEBOOK.astype(np.float64)
    Wb = np.asarray(W, dtype=np.uint8).reshape(M, K // QK, 18)
    scale = Wb[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    qs = Wb[:, :, 2:]
    idx = np.concatenate([qs & 0x0F, qs >> 4], axis=2)
    return (scale[:, :, None] * cb[idx]).reshape(M, K)


# ------------------------------------------------------------- codebook ----

def test_codebook_matches_fixture(golden_dir):
    cb = _read_codebook(golden_dir)
    assert cb.tolist() == O.CODEBOOK.tolist()
    assert int(cb.astype(np.int64).sum()) == -94
    for i in range(16):
        blk = np.zeros(18, dtype=np.uint8)
        blk[0:2] = [0x00, 0x3C]  # scale 1.0
        blk[2:] = i | (i << 4)
        np.testing.assert_array_equal(O.dequantize_block(blk), np.full(32, float(cb[i])))


def test_half_to_float_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([O.half_to_float(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# --------------------------------------------------------- quantization ----

def test_quantize_golden_blocks(golden_dir):
    for case in _read_quant_cases(golden_dir):
        x = np.array([float(v) for v in case["x"]], dtype=np.float32)
        q, d = O.quantize_act(x)
        assert q.tolist() == [int(v) for v in case["q"]]
        if case["d"][0] != "None":
            assert float(d[0]) == float(case["d"][0])


def test_quantize_golden_blocks_as_columns_and_rows(golden_dir):
    cases = _read_quant_cases(golden_dir)
    X = np.array([[float(v) for v in c["x"]] for c in cases], dtype=np.float32)
    Q = np.array([[int(v) for v in c["q"]] for c in cases], dtype=np.int8)
    q_cols, _ = O.quantize_act(X)                   # n columns of one block
    np.testing.assert_array_equal(q_cols, Q)
    q_row, d_row = O.quantize_act(X.reshape(1, -1))  # one column of n blocks
    np.testing.assert_array_equal(q_row.reshape(Q.shape), Q)
    assert d_row.shape == (1, len(cases))


def _exact_checks(x, q, d):
    """q is the nearest integer to x/d up to the fp32 rounding of the quotient,
    d is fl32(amax/127), and exact half-integer quotients round to even."""
    amax = Fraction(float(np.max(np.abs(x))))
    d_exact = amax / 127
    df = Fraction(float(d))
    if amax == 0:
        assert df == 0 and not np.any(q)
        return
    ulp = Fraction(float(np.spacing(np.float32(d))))
    assert abs(df - d_exact) <= ulp / 2
    for xi, qi in zip(x.tolist(), q.tolist()):
        r = Fraction(xi) / df
        assert abs(r - qi) <= Fraction(1, 2) + abs(r) * Fraction(1, 2 ** 23)
        if r.denominator == 2:
            assert qi % 2 == 0
        assert -127 <= qi <= 127


def test_quantize_exact_rational_properties():
    g = np.random.default_rng(7)
    for trial in range(200):
        x = g.standard_normal(32).astype(np.float32) * np.float32(10.0 ** g.integers(-3, 4))
        if trial % 3 == 0:  # force exact ties: amax = 127 * 2^e so d = 2^e
            e = int(g.integers(-6, 6))
            x = (g.integers(-254, 255, 32) / 2.0 * 2.0 ** e).astype(np.float32)
            x[g.integers(0, 32)] = np.float32(127 * 2.0 ** e)
        q, d = O.quantize_act(x)
        _exact_checks(x, q, d[0])


def test_quantize_sign_symmetry_and_power_of_two_scaling():
    x = synth.activations(3, 256, stream=77, outliers=True)
    q, d = O.quantize_act(x)
    qn, dn = O.quantize_act(-x)
    np.testing.assert_array_equal(qn, -q)
    np.testing.assert_array_equal(dn, d)
    q4, d4 = O.quantize_act(x * np.float32(4.0))
    np.testing.assert_array_equal(q4, q)
    np.testing.assert_array_equal(d4, d * np.float32(4.0))


def test_quantize_extreme_element_maps_to_127():
    x = synth.activations(4, 512, stream=78)
    q, _ = O.quantize_act(x)
    xb = x.reshape(4, 16, 32)
    qb = q.reshape(4, 16, 32)
    am = np.argmax(np.abs(xb), axis=2)
    top = np.take_along_axis(qb, am[:, :, None], axis=2)[:, :, 0]
    sign = np.sign(np.take_along_axis(xb, am[:, :, None], axis=2)[:, :, 0])
    np.testing.assert_array_equal(top, (127 * sign).astype(np.int8))


# ---------------------------------------------------- block format / dots --

def test_nibble_layout_one_hot():
    for p in range(32):
        for i in (1, 7, 8, 15):
            blk = np.zeros(18, dtype=np.uint8)
            blk[0:2] = [0x00, 0x3C]
            if p < 16:
                blk[2 + p] = i
            else:
                blk[2 + p - 16] = i << 4
            got = [O.block_index(blk, j) for j in range(32)]
            want = [i if j == p else 0 for j in range(32)]
            assert got == want
            qx = np.zeros(32, dtype=np.int8)
            qx[p] = 3
            s = O.block_dots(blk, 1, 32, qx)
            # every other element has index 0 but meets qx == 0
            assert int(s[0, 0, 0]) == 3 * int(O.CODEBOOK[i])


def test_block_dots_golden(golden_dir):
    for case in _read_block_cases(golden_dir):
        np.testing.assert_array_equal(O.dequantize_block(case["blk"]), case["w"])
        for qx, s in case["dots"]:
            assert int(O.block_dots(case["blk"], 1, 32, qx)[0, 0, 0]) == s, case["name"]


def test_codebook_table_dots():
    for i in range(16):
        blk = np.zeros(18, dtype=np.uint8)
        blk[2:] = i | (i << 4)
        s = O.block_dots(blk, 1, 32, np.ones(32, dtype=np.int8))
        assert int(s[0, 0, 0]) == 32 * int(O.CODEBOOK[i])


def test_block_dots_brute_force_small():
    M, K = 3, 96
    W = synth.weight_blocks(M, K, stream=90)
    qx = np.random.default_rng(3).integers(-127, 128, size=(2, K)).astype(np.int8)
    s = O.block_dots(W, M, K, qx)
    Wd = _np_dequant(W, M, K)
    scale = W[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    for c in range(2):
        for r in range(M):
            for b in range(K // QK):
                ints = Wd[r, 32 * b:32 * b + 32] / scale[r, b]
                assert np.all(ints == np.round(ints))
                assert int(s[c, r, b]) == int(np.dot(ints.astype(np.int64), qx[c, 32 * b:32 * b + 32]))


# --------------------------------------------------------------- matvec ----

@pytest.mark.parametrize("M,K,n", [(7, 64, 1), (33, 320, 3), (64, 1024, 5)])
def test_matvec_equals_dequantize_then_dot(M, K, n):
    W = synth.weight_blocks(M, K, stream=11)
    x = synth.activations(n, K, stream=12, outliers=True)
    qx, dx = O.quantize_act(x)
    xhat = qx.astype(np.float64) * np.repeat(dx.astype(np.float64), QK, axis=1)
    ref = xhat @ _np_dequant(W, M, K).T
    y = O.matvec(W, M, K, x)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-15)
    np.testing.assert_array_equal(O.matvec_q(W, M, K, qx, dx), y)


def test_matvec_scale_linearity_exact():
    M, K = 40, 256
    W = synth.weight_blocks(M, K, stream=13)
    x = synth.activations(2, K, stream=14)
    y = O.matvec(W, M, K, x)
    W2 = W.copy()
    bits = W2[:, :, 0:2].copy().view(np.uint16)
    W2[:, :, 0:2] = (bits + np.uint16(0x0400)).view(np.uint8)  # exponent + 1: dw * 2
    np.testing.assert_array_equal(O.matvec(W2, M, K, x), 2.0 * y)


def test_matvec_sign_symmetry_exact():
    M, K = 40, 256
    W = synth.weight_blocks(M, K, stream=15)
    x = synth.activations(3, K, stream=16)
    np.testing.assert_array_equal(O.matvec(W, M, K, -x), -O.matvec(W, M, K, x))


def test_matvec_zero_scale_rows():
    M, K = 16, 128
    W = synth.weight_blocks(M, K, stream=17)
    W[5, :, 0:2] = 0        # +0 scale
    W[9, :, 0:2] = [0, 0x80]  # -0 scale
    y = O.matvec(W, M, K, synth.activations(2, K, stream=18))
    assert np.all(y[:, 5] == 0) and np.all(y[:, 9] == 0)
    assert np.all(y[:, [0, 1, 2, 3]] != 0)


def test_matvec_constant_index_closed_form():
    M, K, i = 4, 192, 13
    W = synth.weight_blocks(M, K, stream=19)
    W[:, :, 2:] = i | (i << 4)
    x = synth.activations(1, K, stream=20)
    qx, dx = O.quantize_act(x)
    dw = W[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    qsum = qx.reshape(K // QK, QK).astype(np.int64).sum(axis=1).astype(np.float64)
    want = float(O.CODEBOOK[i]) * (dw * dx[0].astype(np.float64) * qsum).sum(axis=1)
    np.testing.assert_allclose(O.matvec(W, M, K, x)[0], want, rtol=1e-13)


def test_matvec_rows_subset_and_bound():
    M, K = 50, 256
    W = synth.weight_blocks(M, K, stream=21)
    x = synth.activations(2, K, stream=22, outliers=True)
    qx, dx = O.quantize_act(x)
    y = O.matvec_q(W, M, K, qx, dx)
    rows = np.array([49, 0, 17, 17, 3])
    np.testing.assert_array_equal(O.matvec_q(W, M, K, qx, dx, rows=rows), y[:, rows])
    b = O.matvec_bound(W, M, K, qx, dx)
    assert np.all(b >= np.abs(y))
    xhat = qx.astype(np.float64) * np.repeat(dx.astype(np.float64), QK, axis=1)
    np.testing.assert_allclose(b, np.abs(xhat) @ np.abs(_np_dequant(W, M, K)).T, rtol=1e-12)
    np.testing.assert_array_equal(O.matvec_bound(W, M, K, qx, dx, rows=rows), b[:, rows])


# ------------------------------------------------------------------ silu ---

def test_silu_identities():
    assert O.silu(0.0) == 0.0
    for z in (0.1, 0.5, 1.0, 3.0, 7.5, 20.0):
        assert abs((O.silu(z) - O.silu(-z)) - z) <= 1e-15 * max(1.0, z)
    assert abs(O.silu(40.0) - 40.0) <= 40.0 * 1e-15
    assert abs(O.silu(-40.0)) <= 1e-15
    assert abs(O.silu(1.0) - 1.0 / (1.0 + np.exp(-1.0))) <= 1e-16


# ------------------------------------------------------------------- MoE ---

E_, H_, F_ = 6, 64, 32


@pytest.fixture(scope="module")
def tiny_layer():
    gu = synth.expert_blocks(E_, 2 * F_, H_, stream=31)
    dn = synth.expert_blocks(E_, H_, F_, stream=32)
    return gu, dn


def _expert_slot(gu, dn, e, h, swiglu):
    """One (token, slot) through the pinned matvec pieces, gate rows first."""
    qh, dh = O.quantize_act(h)
    g_rows = gu[e].reshape(2 * F_, -1)
    g = O.matvec_q(g_rows[:F_].ravel(), F_, H_, qh, dh)[0]
    u = O.matvec_q(g_rows[F_:].ravel(), F_, H_, qh, dh)[0]
    if swiglu:
        a = np.array([O.silu(v) * w for v, w in zip(g, u)]).astype(np.float32)
    else:
        a = (g * u).astype(np.float32)
    qa, da = O.quantize_act(a)
    return O.matvec_q(dn[e].ravel(), H_, F_, qa, da)[0], a


@pytest.mark.parametrize("swiglu", [1, 0])
def test_moe_k1_reduces_to_matvecs(tiny_layer, swiglu):
    gu, dn = tiny_layer
    h = synth.activations(1, H_, stream=33)
    for e in range(E_):
        y, a, qa, da, nbad = O.moe(gu, dn, E_, H_, F_, h, np.array([[e]]), np.array([[1.0]]),
                                   swiglu=swiglu, want_intermediate=True)
        want, a_want = _expert_slot(gu, dn, e, h[0], swiglu)
        assert nbad == 0
        np.testing.assert_array_equal(a[0], a_want)
        np.testing.assert_array_equal(y[0], want)


def test_moe_gate_and_up_are_not_interchangeable(tiny_layer):
    gu, dn = tiny_layer
    h = synth.activations(1, H_, stream=34)
    ids, wts = np.array([[2]]), np.array([[1.0]])
    y = O.moe(gu, dn, E_, H_, F_, h, ids, wts)
    sw = gu.copy()
    rows = sw[2].reshape(2 * F_, -1).copy()
    sw[2] = np.concatenate([rows[F_:], rows[:F_]]).reshape(sw[2].shape)
    assert not np.allclose(O.moe(sw, dn, E_, H_, F_, h, ids, wts), y)
    z = gu.copy()
    zr = z[2].reshape(2 * F_, H_ // QK, 18)
    zr[F_:, :, 0:2] = 0  # up half scaled to zero -> a == 0 -> y == 0
    z[2] = zr.reshape(z[2].shape)
    assert np.all(O.moe(z, dn, E_, H_, F_, h, ids, wts) == 0)


def test_moe_router_weights_and_slots(tiny_layer):
    gu, dn = tiny_layer
    h = synth.activations(1, H_, stream=35)
    ids = np.array([[4, 1]])
    wts = np.array([[0.75, 0.25]], dtype=np.float32)
    y = O.moe(gu, dn, E_, H_, F_, h, ids, wts)
    y4 = O.moe(gu, dn, E_, H_, F_, h, np.array([[4]]), np.array([[1.0]]))
    y1 = O.moe(gu, dn, E_, H_, F_, h, np.array([[1]]), np.array([[1.0]]))
    np.testing.assert_allclose(y, 0.75 * y4 + 0.25 * y1, rtol=1e-12, atol=1e-14)
    # doubling every router weight doubles y exactly
    np.testing.assert_array_equal(O.moe(gu, dn, E_, H_, F_, h, ids, 2 * wts), 2 * y)
    # slot order only changes the fp64 summation order
    np.testing.assert_allclose(O.moe(gu, dn, E_, H_, F_, h, ids[:, ::-1], wts[:, ::-1]), y,
                               rtol=1e-12, atol=1e-14)


def test_moe_tokens_are_independent(tiny_layer):
    gu, dn = tiny_layer
    h = synth.activations(5, H_, stream=36)
    ids, wts = synth.router(5, 3, E_, stream=37)
    y = O.moe(gu, dn, E_, H_, F_, h, ids, wts)
    for t in range(5):
        np.testing.assert_array_equal(O.moe(gu, dn, E_, H_, F_, h[t:t + 1], ids[t:t + 1], wts[t:t + 1])[0], y[t])


def test_moe_bad_ids_and_duplicates(tiny_layer):
    gu, dn = tiny_layer
    h = synth.activations(1, H_, stream=38)
    y_ok = O.moe(gu, dn, E_, H_, F_, h, np.array([[3]]), np.array([[0.5]]))
    y, _, _, _, nbad = O.moe(gu, dn, E_, H_, F_, h, np.array([[3, E_, -1]]),
                             np.array([[0.5, 0.3, 0.2]]), want_intermediate=True)
    assert nbad == 2
    np.testing.assert_array_equal(y, y_ok)
    y_dup = O.moe(gu, dn, E_, H_, F_, h, np.array([[3, 3]]), np.array([[0.25, 0.25]]))
    np.testing.assert_allclose(y_dup, y_ok, rtol=1e-12, atol=1e-14)


def test_moe_down_combine_matches_full(tiny_layer):
    gu, dn = tiny_layer
    h = synth.activations(4, H_, stream=39)
    ids, wts = synth.router(4, 2, E_, stream=40)
    y, a, qa, da, _ = O.moe(gu, dn, E_, H_, F_, h, ids, wts, want_intermediate=True)
    y2, yb, nbad = O.moe_down_combine(dn, E_, H_, F_, ids, wts, qa, da)
    assert nbad == 0
    np.testing.assert_array_equal(y2, y)
    assert np.all(yb >= np.abs(y))
    qa2, da2 = O.quantize_act(a)
    np.testing.assert_array_equal(qa2, qa)
    np.testing.assert_array_equal(da2, da)


def test_moe_large_gate_makes_silu_identity(tiny_layer):
    """Gate rows pushed far positive: silu(g) = g to fp32, so a = g*u."""
    gu, dn = tiny_layer
    big = gu.copy()
    r = big[0].reshape(2 * F_, H_ // QK, 18)
    r[:F_, :, 2:] = 0xFF                       # every gate index -> codebook max 113
    r[:F_, :, 0:2] = np.frombuffer(np.float16(0.5).tobytes(), dtype=np.uint8)
    big[0] = r.reshape(big[0].shape)
    h = np.abs(synth.activations(1, H_, stream=41))  # positive input -> g >> 0
    _, a1, _, _, _ = O.moe(big, dn, E_, H_, F_, h, np.array([[0]]), np.array([[1.0]]),
                           swiglu=1, want_intermediate=True)
    _, a0, _, _, _ = O.moe(big, dn, E_, H_, F_, h, np.array([[0]]), np.array([[1.0]]),
                           swiglu=0, want_intermediate=True)
    np.testing.assert_allclose(a1, a0, rtol=1e-6)


# ------------------------------------------------------ shared expert ------

def _shared(tiny_layer, e):
    """Expert e of the tiny table as a stand-alone shared expert."""
    gu, dn = tiny_layer
    return gu[e].copy(), dn[e].copy()


def test_moe_shared_zero_scales_give_the_routed_layer(tiny_layer):
    gu, dn = tiny_layer
    sgu, sdn = _shared(tiny_layer, 5)
    sdn.reshape(H_, F_ // QK, 18)[:, :, 0:2] = 0  # every down scale zero: o_sh == 0
    h = synth.activations(3, H_, stream=42)
    ids, wts = synth.router(3, 2, E_, stream=43)
    y, nbad = O.moe_shared(gu, dn, E_, H_, F_, sgu, sdn, h, ids, wts)
    assert nbad == 0
    np.testing.assert_array_equal(y, O.moe(gu, dn, E_, H_, F_, h, ids, wts))


@pytest.mark.parametrize("swiglu", [1, 0])
def test_moe_shared_alone_is_one_dense_ffn(tiny_layer, swiglu):
    """Every routed id out of range: each token gets exactly the shared
    expert's FFN, built here from the pinned matvec pieces."""
    gu, dn = tiny_layer
    sgu, sdn = _shared(tiny_layer, 2)
    h = synth.activations(2, H_, stream=44)
    ids = np.array([[-1, E_], [E_ + 3, -9]], dtype=np.int32)
    y, nbad = O.moe_shared(gu, dn, E_, H_, F_, sgu, sdn, h, ids, np.ones((2, 2), np.float32), swiglu=swiglu)
    assert nbad == 4
    for t in range(2):
        want, _ = _expert_slot(sgu[None], sdn[None], 0, h[t], swiglu)
        np.testing.assert_array_equal(y[t], want)


def test_moe_shared_is_one_more_slot_of_weight_one(tiny_layer):
    """The shared expert appended to the table as expert E and to every
    token's slots (last, weight 1) gives the same layer."""
    gu, dn = tiny_layer
    sgu, sdn = _shared(tiny_layer, 1)
    sgu[0, 0] ^= 0x5A  # differ from every routed expert
    h = synth.activations(4, H_, stream=45)
    ids, wts = synth.router(4, 3, E_, stream=46)
    y, _ = O.moe_shared(gu, dn, E_, H_, F_, sgu, sdn, h, ids, wts)
    ids_a = np.concatenate([ids, np.full((4, 1), E_, np.int32)], axis=1)
    wts_a = np.concatenate([wts, np.ones((4, 1), np.float32)], axis=1)
    y_a = O.moe(np.concatenate([gu, sgu[None]]), np.concatenate([dn, sdn[None]]), E_ + 1, H_, F_, h, ids_a, wts_a)
    np.testing.assert_allclose(y, y_a, rtol=1e-12, atol=1e-14)


def test_moe_shared_equal_to_a_routed_expert(tiny_layer):
    """Shared expert == routed expert e, top-1 to e with weight w:
    y = (w + 1) * o_e, token by token."""
    gu, dn = tiny_layer
    sgu, sdn = _shared(tiny_layer, 4)
    h = synth.activations(3, H_, stream=47)
    ids = np.full((3, 1), 4, np.int32)
    wts = np.array([[0.25], [0.5], [2.0]], np.float32)
    y, _ = O.moe_shared(gu, dn, E_, H_, F_, sgu, sdn, h, ids, wts)
    y1 = O.moe(gu, dn, E_, H_, F_, h, ids, np.ones_like(wts))
    np.testing.assert_allclose(y, (wts.astype(np.float64) + 1.0) * y1, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------- router top-k --

def _read_router_cases(golden_dir):
    cases, cur = [], {}
    with open(os.path.join(golden_dir, "router_topk.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            cur[key] = val.split()
            if key == "terms":
                cases.append(cur)
                cur = {}
    return cases


def test_router_topk_golden(golden_dir):
    cases = _read_router_cases(golden_dir)
    assert len(cases) == 4
    for c in cases:
        k = int(c["k"][0])
        logits = np.array([[float(v) for v in c["logits"]]], dtype=np.float32)
        ids, wts = O.router_topk(logits, k)
        np.testing.assert_array_equal(ids[0], [int(v) for v in c["ids"]])
        terms = np.exp(np.array([float(v) for v in c["terms"]]))
        np.testing.assert_allclose(wts[0], terms / terms.sum(), rtol=1e-15)


def test_router_topk_matches_stable_sort_and_library_softmax():
    """Ids against a stable descending argsort (lower index first among
    equal logits); weights against scipy's softmax of the selected logits."""
    special = pytest.importorskip("scipy.special")
    g = np.random.default_rng(21)
    for E, k in ((8, 1), (16, 4), (64, 8), (256, 8), (20, 16), (7, 7)):
        logits = g.standard_normal((5, E)).astype(np.float32)
        logits[1, 3] = logits[1, 5] = logits[1].max() + 1  # a tie at the top
        logits[2] = np.round(logits[2])  # many ties
        ids, wts = O.router_topk(logits, k)
        for t in range(5):
            ref = np.argsort(-logits[t].astype(np.float64), kind="stable")[:k]
            np.testing.assert_array_equal(ids[t], ref)
            np.testing.assert_allclose(wts[t], special.softmax(logits[t][ref].astype(np.float64)), rtol=1e-13)


def test_router_topk_invariants():
    g = np.random.default_rng(22)
    logits = np.round(g.standard_normal((5, 64)) * 64).astype(np.float32) / 64  # exact after +8
    ids, wts = O.router_topk(logits, 8)
    np.testing.assert_allclose(wts.sum(axis=1), 1.0, rtol=1e-15)
    assert np.all(np.diff(wts, axis=1) <= 0)  # descending logits give descending weights
    ids2, wts2 = O.router_topk(logits + np.float32(8.0), 8)  # a common shift changes nothing
    np.testing.assert_array_equal(ids2, ids)
    np.testing.assert_allclose(wts2, wts, rtol=1e-14)
    distinct = (g.permutation(5 * 64).reshape(5, 64) / 64.0).astype(np.float32)
    ids_d, wts_d = O.router_topk(distinct, 8)
    perm = g.permutation(64)  # relabelled experts: the same choices under the new labels
    ids3, wts3 = O.router_topk(distinct[:, perm], 8)
    np.testing.assert_array_equal(perm[ids3], ids_d)
    np.testing.assert_array_equal(wts3, wts_d)


# ------------------------------------------------------ weight converter ---

def _read_convert_cases(golden_dir):
    cases = []
    with open(os.path.join(golden_dir, "convert_blocks.txt")) as f:
        for line in f:
            if not line.startswith("convert "):
                continue
            head, tail = line.split("=")
            parts = head.split()
            w = np.array([float(v) for v in parts[2:]], dtype=np.float32)
            blk = np.array([int(b, 16) for b in tail.split()], dtype=np.uint8)
            assert w.size == 32 and blk.size == 18
            cases.append((parts[1], w, blk))
    return cases


def test_float_to_half_matches_numpy():
    """binary16 rounding against numpy's float32 -> float16 conversion: every
    finite binary16 value, the midpoints between neighbours (ties to even),
    and random float32 across the subnormal, normal and overflow ranges."""
    bits = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    h = bits.view(np.float16)
    finite = np.isfinite(h)
    vals = [h[finite].astype(np.float32)]
    hs = np.sort(np.unique(np.abs(h[finite].astype(np.float64))))
    mids = (hs[:-1] + hs[1:]) / 2  # exact in fp32 (12 significant bits)
    vals += [mids.astype(np.float32), -mids.astype(np.float32)]
    rng = np.random.default_rng(11)
    for lo, hi in ((-30, -24), (-24, -14), (-14, 16), (15, 17)):
        e = rng.uniform(lo, hi, 4000)
        vals.append((np.sign(rng.standard_normal(4000)) * 2.0 ** e).astype(np.float32))
    vals.append(np.array([65504, 65519.99, 65520, 1e30, np.inf, -np.inf, 0.0, -0.0], dtype=np.float32))
    for v in np.concatenate(vals):
        want = int(np.float32(v).astype(np.float16).view(np.uint16))
        assert O.float_to_half(v) == want, (float(v), hex(want))


def test_convert_golden_blocks(golden_dir):
    for name, w, blk in _read_convert_cases(golden_dir):
        np.testing.assert_array_equal(O.quantize_weights(w, 1, 32).ravel(), blk, err_msg=name)


def test_convert_grid_round_trip():
    """Weights that are exactly dw * codebook[index] with a level -127 present
    (the unique largest magnitude) come back as exactly those bytes: the
    scale rule, the index search, the nibble packing and the byte order."""
    rng = np.random.default_rng(12)
    M, K = 7, 96
    nb = K // 32
    blocks = np.zeros((M, nb, 18), dtype=np.uint8)
    w = np.zeros((M, K), dtype=np.float32)
    for r in range(M):
        for b in range(nb):
            dw = np.float16(rng.uniform(1e-3, 1e-2) * rng.choice([-1, 1]))
            idx = rng.integers(1, 16, 32)
            idx[rng.integers(0, 32)] = 0
            hb = int(np.array(dw).view(np.uint16))
            blocks[r, b, 0], blocks[r, b, 1] = hb & 0xFF, hb >> 8
            blocks[r, b, 2:] = (idx[:16] | (idx[16:] << 4)).astype(np.uint8)
            w[r, 32 * b:32 * b + 32] = (np.float32(dw) * O.CODEBOOK[idx].astype(np.float32))
    np.testing.assert_array_equal(O.quantize_weights(w, M, K), blocks)


def test_convert_brute_force_exact():
    """Random blocks: the scale by numpy (fp32 division, float16 rounding) and
    every index by an exact-rational search over the 16 levels (lowest index
    among equal distances)."""
    rng = np.random.default_rng(13)
    w = (rng.standard_normal((5, 64)) * rng.uniform(0.01, 3.0, (5, 1))).astype(np.float32)
    w[2, 40] = w[2, 33] = -np.abs(w[2]).max() * 1.5  # equal largest magnitudes: the first one counts
    got = O.quantize_weights(w, 5, 64)
    for r in range(5):
        for b in range(2):
            x = w[r, 32 * b:32 * b + 32]
            m = x[int(np.argmax(np.abs(x)))]  # argmax takes the first of equal values
            dw = np.float16(np.float32(m) / np.float32(-127.0))
            blk = got[r, b]
            assert int(blk[0]) | (int(blk[1]) << 8) == int(np.array(dw).view(np.uint16))
            D = Fraction(float(dw))
            for i in range(32):
                dist = [abs(Fraction(float(x[i])) - D * int(O.CODEBOOK[j])) for j in range(16)]
                want = dist.index(min(dist))
                have = int(blk[2 + i] & 0xF) if i < 16 else int(blk[2 + i - 16] >> 4)
                assert have == want, (r, b, i)


def test_convert_error_bound_and_zero_blocks():
    """Every weight comes back within 14 scale units of itself (half the widest
    gap between levels is 12; a weight of the other sign than the largest one
    can sit 127 - 113 = 14 units past the last level), plus the scale's own
    rounding; an all-zero block converts to zero bytes."""
    rng = np.random.default_rng(14)
    M, K = 6, 128
    w = rng.standard_normal((M, K)).astype(np.float32)
    w[3, 32:64] = 0.0
    blocks = O.quantize_weights(w, M, K)
    assert not blocks[3, 1].any()
    for r in range(M):
        for b in range(K // 32):
            dq = O.dequantize_block(blocks[r, b])
            x = w[r, 32 * b:32 * b + 32].astype(np.float64)
            dw = abs(O.half_to_float(int(blocks[r, b, 0]) | (int(blocks[r, b, 1]) << 8)))
            assert np.all(np.abs(dq - x) <= 14 * dw + 127 * dw * 2.0 ** -10)


# ---- sinkhorn normalisation of the hyper-connection matrices ----------------

def _logits(rng, n, nhc, scale=1.0, step=1.0 / 64):
    """Logits on a grid of 1/64 in [-4*scale, 4*scale]: exact in fp32, so a
    shifted copy stays exact too."""
    return (np.round(rng.uniform(-4 * scale, 4 * scale, (n, nhc, nhc)) / step) * step).astype(np.float32)


def test_sinkhorn_zero_rounds_is_the_shifted_exponential():
    """With no round the output is exp(c - max c): numpy's exp, 1 at the
    largest logit."""
    rng = np.random.default_rng(40)
    c = _logits(rng, 7, 4)
    got = O.hc_sinkhorn(c, 0)
    want = np.exp(c.astype(np.float64) - c.reshape(7, -1).max(axis=1)[:, None, None])
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=0)
    assert np.all(got.reshape(7, -1).max(axis=1) == 1.0)


@pytest.mark.parametrize("nhc", [2, 3, 4])
def test_sinkhorn_rank_one_is_uniform_after_one_round(nhc):
    """c_ij = a_i + b_j makes exp(c) rank one: one row step gives identical
    rows, the column step then gives every entry 1/nhc."""
    rng = np.random.default_rng(41 + nhc)
    a = np.round(rng.uniform(-3, 3, (5, nhc, 1)) * 16) / 16
    b = np.round(rng.uniform(-3, 3, (5, 1, nhc)) * 16) / 16
    c = (a + b).astype(np.float32)
    np.testing.assert_allclose(O.hc_sinkhorn(c, 1), np.full((5, nhc, nhc), 1.0 / nhc), rtol=0, atol=1e-14)


def test_sinkhorn_two_by_two_limit_closed_form():
    """A positive 2 x 2 matrix [[a, b], [c, d]] converges to [[p, 1-p], [1-p,
    p]] with p = sqrt(ad) / (sqrt(ad) + sqrt(bc)) (the only doubly stochastic
    matrix of the form diag(x) P diag(y))."""
    rng = np.random.default_rng(44)
    c = _logits(rng, 9, 2, scale=0.5)
    e = np.exp(c.astype(np.float64))
    ad = np.sqrt(e[:, 0, 0] * e[:, 1, 1])
    bc = np.sqrt(e[:, 0, 1] * e[:, 1, 0])
    p = ad / (ad + bc)
    want = np.stack([np.stack([p, 1 - p], -1), np.stack([1 - p, p], -1)], -2)
    np.testing.assert_allclose(O.hc_sinkhorn(c, 400), want, rtol=0, atol=1e-12)


def test_sinkhorn_doubly_stochastic_input_is_a_fixed_point():
    """A Latin square of 1/2, 1/4, 1/8, 1/8 is doubly stochastic: given its
    logarithms (rounded to fp32) the rounds leave it where it is, within the
    rounding of the logits."""
    vals = np.array([0.5, 0.25, 0.125, 0.125])
    P = np.array([[vals[(i + j) % 4] for j in range(4)] for i in range(4)])
    c = np.log(P).astype(np.float32)[None]
    for iters in (1, 5, 50):
        np.testing.assert_allclose(O.hc_sinkhorn(c, iters)[0], P, rtol=0, atol=1e-6)


def test_sinkhorn_sums_row_shift_and_permutations():
    """After every round the columns sum to 1; with many rounds the rows do
    too; a constant added to one row of logits changes nothing (the row step
    removes it); permuting rows and columns of the logits permutes the
    result."""
    rng = np.random.default_rng(45)
    c = _logits(rng, 6, 4)
    for iters in (1, 2, 7):
        out = O.hc_sinkhorn(c, iters)
        np.testing.assert_allclose(out.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    out = O.hc_sinkhorn(c, 300)
    np.testing.assert_allclose(out.sum(axis=2), 1.0, rtol=0, atol=1e-12)
    shifted = c.copy()
    shifted[:, 2, :] += np.float32(1.25)
    np.testing.assert_allclose(O.hc_sinkhorn(shifted, 3), O.hc_sinkhorn(c, 3), rtol=0, atol=1e-14)
    pr, pc = np.array([2, 0, 3, 1]), np.array([1, 3, 0, 2])
    got = O.hc_sinkhorn(c[:, pr][:, :, pc], 4)
    np.testing.assert_allclose(got, O.hc_sinkhorn(c, 4)[:, pr][:, :, pc], rtol=0, atol=1e-14)
