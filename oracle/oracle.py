"""numpy front end of the C oracle (cbq_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check in the
package entry module and by the benchmark's CPU-baseline leg.  The product
path (the CUDA library and its binding) never imports this module.

Every function takes and returns numpy arrays; the arithmetic all happens in
the C file, which this module compiles with gcc on first use (or which the
package build compiles ahead of time).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cbq_oracle.c")
_HDR = os.path.join(_HERE, "cbq_oracle.h")
_LIB = os.path.join(_HERE, "libcbq_oracle.so")
_lock = threading.Lock()
_lib = None

QK = 32
BLOCK_BYTES = 18
# The same 16 levels as the C table; kept here only to let tests index it.
CODEBOOK = np.array([-127, -104, -83, -65, -49, -35, -22, -10,
                     1, 13, 25, 38, 53, 69, 89, 113], dtype=np.int8)

_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile libcbq_oracle.so next to its source (gcc, no GPU needed)."""
    stale = (not os.path.exists(_LIB) or
             os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    """Declare the argument and result types of the oracle's C functions."""
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I = ctypes.c_int
    lib.oracle_half_to_float.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_float.restype = ctypes.c_float
    lib.oracle_block_index.argtypes = [P, I]
    lib.oracle_block_index.restype = I
    lib.oracle_dequantize_block.argtypes = [P, P]
    lib.oracle_quantize_act.argtypes = [P, I64, I, P, P]
    lib.oracle_block_dots.argtypes = [P, I64, I64, P, I, P]
    lib.oracle_matvec_q.argtypes = [P, I64, I64, P, P, I, P]
    lib.oracle_matvec_q_rows.argtypes = [P, I64, I64, P, P, I, P, I64, P]
    lib.oracle_matvec.argtypes = [P, I64, I64, P, I, P]
    lib.oracle_matvec_bound.argtypes = [P, I64, I64, P, P, I, P]
    lib.oracle_matvec_bound_rows.argtypes = [P, I64, I64, P, P, I, P, I64, P]
    lib.oracle_silu.argtypes = [ctypes.c_double]
    lib.oracle_silu.restype = ctypes.c_double
    lib.oracle_moe.argtypes = [P, P, I, I64, I64, P, I, P, P, I, I, P, P, P, P]
    lib.oracle_moe.restype = I
    lib.oracle_moe_shared.argtypes = [P, P, I, I64, I64, P, P, P, I, P, P, I, I, P]
    lib.oracle_moe_shared.restype = I
    lib.oracle_moe_down_combine.argtypes = [P, I, I64, I64, I, P, P, I, P, P, P, P]
    lib.oracle_moe_down_combine.restype = I
    lib.oracle_router_topk.argtypes = [P, I, I, I, P, P]
    lib.oracle_router_topk.restype = None
    lib.oracle_float_to_half.argtypes = [ctypes.c_float]
    lib.oracle_float_to_half.restype = ctypes.c_uint16
    lib.oracle_quantize_weights_block.argtypes = [P, P]
    lib.oracle_quantize_weights.argtypes = [P, I64, I64, P]
    lib.oracle_hc_sinkhorn.argtypes = [P, I64, I, I, P]
    lib.oracle_hc_sinkhorn.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        _lib = _bind(ctypes.CDLL(build()))
        return _lib


@contextlib.contextmanager
def using_library(path):
    """Run the wrappers of this module against another build of the oracle's
    C source (the mutation tests plant one mistake per build) for the
    duration of the block."""
    global _lib
    other = _bind(ctypes.CDLL(path))
    with _lock:
        saved = _lib
        _lib = other
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _blocks(W: np.ndarray, M: int, K: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    if K % QK or W.size != M * (K // QK) * BLOCK_BYTES:
        raise ValueError("weight blocks do not match M x K")
    return W


def half_to_float(bits: int) -> float:
    return float(_load().oracle_half_to_float(int(bits)))


def block_index(blk: np.ndarray, i: int) -> int:
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    return int(_load().oracle_block_index(_p(blk), int(i)))


def dequantize_block(blk: np.ndarray) -> np.ndarray:
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    out = np.empty(QK, dtype=np.float64)
    _load().oracle_dequantize_block(_p(blk), _p(out))
    return out


def quantize_act(x: np.ndarray):
    """x: (n, K) or (K,) fp32 -> (qx int8 same shape, dx fp32 (n, K/32))."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    x2 = x.reshape(-1, x.shape[-1])
    n, K = x2.shape
    if K % QK:
        raise ValueError("K must be a multiple of 32")
    qx = np.empty((n, K), dtype=np.int8)
    dx = np.empty((n, K // QK), dtype=np.float32)
    if n and K:
        _load().oracle_quantize_act(_p(x2), K, n, _p(qx), _p(dx))
    return qx.reshape(x.shape), dx.reshape(x.shape[:-1] + (K // QK,))


def block_dots(W, M, K, qx):
    qx = np.ascontiguousarray(qx, dtype=np.int8).reshape(-1, K)
    n = qx.shape[0]
    s = np.empty((n, M, K // QK), dtype=np.int32)
    _load().oracle_block_dots(_p(_blocks(W, M, K)), M, K, _p(qx), n, _p(s))
    return s


def matvec_q(W, M, K, qx, dx, rows=None):
    """fp64 y (n, M) from quantized activations; rows=None for all rows."""
    qx = np.ascontiguousarray(qx, dtype=np.int8).reshape(-1, K)
    dx = np.ascontiguousarray(dx, dtype=np.float32).reshape(-1, K // QK)
    n = qx.shape[0]
    W = _blocks(W, M, K)
    if rows is None:
        y = np.empty((n, M), dtype=np.float64)
        _load().oracle_matvec_q(_p(W), M, K, _p(qx), _p(dx), n, _p(y))
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        y = np.empty((n, rows.size), dtype=np.float64)
        _load().oracle_matvec_q_rows(_p(W), M, K, _p(qx), _p(dx), n, _p(rows), rows.size, _p(y))
    return y


def matvec(W, M, K, x):
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, K)
    n = x.shape[0]
    y = np.empty((n, M), dtype=np.float64)
    _load().oracle_matvec(_p(_blocks(W, M, K)), M, K, _p(x), n, _p(y))
    return y


def matvec_bound(W, M, K, qx, dx, rows=None):
    qx = np.ascontiguousarray(qx, dtype=np.int8).reshape(-1, K)
    dx = np.ascontiguousarray(dx, dtype=np.float32).reshape(-1, K // QK)
    n = qx.shape[0]
    W = _blocks(W, M, K)
    if rows is None:
        b = np.empty((n, M), dtype=np.float64)
        _load().oracle_matvec_bound(_p(W), M, K, _p(qx), _p(dx), n, _p(b))
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        b = np.empty((n, rows.size), dtype=np.float64)
        _load().oracle_matvec_bound_rows(_p(W), M, K, _p(qx), _p(dx), n, _p(rows), rows.size, _p(b))
    return b


def silu(z: float) -> float:
    return float(_load().oracle_silu(float(z)))


def moe(gate_up, down, E, H, F, h, ids, wts, swiglu=1, want_intermediate=False):
    """Routed-expert FFN.  Returns y (n_tok, H) fp64 [, a, qa, da, n_bad]."""
    h = np.ascontiguousarray(h, dtype=np.float32).reshape(-1, H)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    n_tok, k = ids.shape
    wts = np.ascontiguousarray(wts, dtype=np.float32).reshape(n_tok, k)
    gate_up = np.ascontiguousarray(gate_up, dtype=np.uint8)
    down = np.ascontiguousarray(down, dtype=np.uint8)
    if gate_up.size != E * 2 * F * (H // QK) * BLOCK_BYTES or down.size != E * H * (F // QK) * BLOCK_BYTES:
        raise ValueError("expert weights do not match E, H, F")
    y = np.empty((n_tok, H), dtype=np.float64)
    a = np.empty((n_tok * k, F), dtype=np.float32)
    qa = np.empty((n_tok * k, F), dtype=np.int8)
    da = np.empty((n_tok * k, F // QK), dtype=np.float32)
    nbad = _load().oracle_moe(_p(gate_up), _p(down), E, H, F, _p(h), n_tok, _p(ids), _p(wts), k,
                              int(swiglu), _p(y), _p(a), _p(qa), _p(da))
    if want_intermediate:
        return y, a, qa, da, nbad
    return y


def moe_shared(gate_up, down, E, H, F, sh_gate_up, sh_down, h, ids, wts, swiglu=1):
    """Routed layer plus the shared expert (weight 1 for every token).
    Returns y (n_tok, H) fp64 and the number of out-of-range routed ids."""
    h = np.ascontiguousarray(h, dtype=np.float32).reshape(-1, H)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    n_tok, k = ids.shape
    wts = np.ascontiguousarray(wts, dtype=np.float32).reshape(n_tok, k)
    gate_up = np.ascontiguousarray(gate_up, dtype=np.uint8)
    down = np.ascontiguousarray(down, dtype=np.uint8)
    sh_gate_up = np.ascontiguousarray(sh_gate_up, dtype=np.uint8)
    sh_down = np.ascontiguousarray(sh_down, dtype=np.uint8)
    gu1, dn1 = 2 * F * (H // QK) * BLOCK_BYTES, H * (F // QK) * BLOCK_BYTES
    if gate_up.size != E * gu1 or down.size != E * dn1 or sh_gate_up.size != gu1 or sh_down.size != dn1:
        raise ValueError("expert weights do not match E, H, F")
    y = np.empty((n_tok, H), dtype=np.float64)
    nbad = _load().oracle_moe_shared(_p(gate_up), _p(down), E, H, F, _p(sh_gate_up), _p(sh_down), _p(h), n_tok,
                                     _p(ids), _p(wts), k, int(swiglu), _p(y))
    return y, nbad


def moe_down_combine(down, E, H, F, ids, wts, qa, da):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    n_tok, k = ids.shape
    wts = np.ascontiguousarray(wts, dtype=np.float32).reshape(n_tok, k)
    qa = np.ascontiguousarray(qa, dtype=np.int8).reshape(n_tok * k, F)
    da = np.ascontiguousarray(da, dtype=np.float32).reshape(n_tok * k, F // QK)
    down = np.ascontiguousarray(down, dtype=np.uint8)
    y = np.empty((n_tok, H), dtype=np.float64)
    yb = np.empty((n_tok, H), dtype=np.float64)
    nbad = _load().oracle_moe_down_combine(_p(down), E, H, F, n_tok, _p(ids), _p(wts), k,
                                           _p(qa), _p(da), _p(y), _p(yb))
    return y, yb, nbad


def router_topk(logits, k):
    """ids (n_tok, k) int32 and fp64 softmax weights of the k largest logits."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    n_tok, E = logits.shape
    ids = np.empty((n_tok, k), dtype=np.int32)
    wts = np.empty((n_tok, k), dtype=np.float64)
    _load().oracle_router_topk(_p(logits), n_tok, E, k, _p(ids), _p(wts))
    return ids, wts


def float_to_half(x: float) -> int:
    """binary16 bits of fp32 x, rounded to nearest even."""
    return int(_load().oracle_float_to_half(float(np.float32(x))))


def quantize_weights(w: np.ndarray, M: int, K: int) -> np.ndarray:
    """The weight converter: fp32 w (M, K) -> blocks (M, K/32, 18) uint8."""
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(M, K)
    out = np.empty((M, K // QK, BLOCK_BYTES), dtype=np.uint8)
    _load().oracle_quantize_weights(_p(w), M, K, _p(out))
    return out


def hc_sinkhorn(logits, iters: int) -> np.ndarray:
    """Sinkhorn normalisation of fp32 logits (..., nhc, nhc): exp(c - max c),
    then `iters` rounds of row then column normalisation, fp64 out."""
    c = np.ascontiguousarray(logits, dtype=np.float32)
    nhc = c.shape[-1]
    assert c.shape[-2] == nhc
    n = c.size // (nhc * nhc)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_hc_sinkhorn(_p(c), n, nhc, int(iters), _p(out))
    return out
