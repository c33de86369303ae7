"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module only draws random numbers and lays them out in the canonical
block format; it holds none of the quantized-matvec arithmetic.  Each tensor
gets its own counter-keyed numpy stream (``default_rng([seed, stream])``), so
any tensor can be regenerated alone.

Canonical block (18 bytes per 32 weights along K): bytes 0-1 the fp16 scale
(little-endian), bytes 2-17 the index bytes, byte j holding element j in its
low nibble and element j+16 in its high nibble.  Drawing every index byte
uniformly in 0..255 draws both nibbles uniformly in 0..15.

Workload recipe (the five shapes of the codebook-4bit decode and verify
workloads; see the design notes for the sizes):
  weights      indices uniform 0..15; scales fp16(U[1e-3, 1e-2]);
  activations  N(0,1) fp32, optionally with exactly round(0.01*K) entries per
               column multiplied by 20 (outliers);
  router       per token k distinct expert ids drawn uniformly without
               replacement, weights = softmax of k N(0,1) logits (fp32).
"""
from __future__ import annotations

import numpy as np

SEED = 0x5EED
QK = 32
BLOCK_BYTES = 18

# stream ids, one per tensor role
S_W, S_X, S_GATE_UP, S_DOWN, S_H, S_IDS, S_HEAD, S_HEAD_X, S_MISC, S_HC = range(1, 11)


def rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(stream)])


def weight_blocks(M: int, K: int, seed: int = SEED, stream: int = S_W,
                  scale_lo: float = 1e-3, scale_hi: float = 1e-2) -> np.ndarray:
    """Canonical blocks of an M x K matrix: uint8 array (M, K/32, 18)."""
    if K % QK:
        raise ValueError("K must be a multiple of 32")
    nb = K // QK
    g = rng(seed, stream)
    out = np.empty((M, nb, BLOCK_BYTES), dtype=np.uint8)
    scales = g.uniform(scale_lo, scale_hi, size=(M, nb)).astype(np.float16)
    out[:, :, 0:2] = scales.view(np.uint8).reshape(M, nb, 2)
    out[:, :, 2:] = g.integers(0, 256, size=(M, nb, 16), dtype=np.uint8)
    return out


def expert_blocks(E: int, M: int, K: int, seed: int = SEED, stream: int = S_GATE_UP,
                  out: np.ndarray | None = None) -> np.ndarray:
    """E experts of M x K each, expert e drawn from stream (stream, e)."""
    nb = K // QK
    if out is None:
        out = np.empty((E, M, nb, BLOCK_BYTES), dtype=np.uint8)
    for e in range(E):
        out[e] = weight_blocks(M, K, seed, stream * 1000 + e)
    return out


def activations(n: int, K: int, seed: int = SEED, stream: int = S_X,
                outliers: bool = False) -> np.ndarray:
    """n columns of K fp32 values from N(0,1); optional 1% x20 outliers."""
    g = rng(seed, stream)
    x = g.standard_normal((n, K)).astype(np.float32)
    if outliers:
        m = int(round(0.01 * K))
        for c in range(n):
            pos = g.choice(K, size=m, replace=False)
            x[c, pos] *= np.float32(20.0)
    return x


def router(n_tok: int, k: int, E: int, seed: int = SEED, stream: int = S_IDS):
    """ids (n_tok, k) int32 distinct per token; wts (n_tok, k) fp32 softmax."""
    g = rng(seed, stream)
    ids = np.empty((n_tok, k), dtype=np.int32)
    wts = np.empty((n_tok, k), dtype=np.float32)
    for t in range(n_tok):
        ids[t] = g.choice(E, size=k, replace=False)
        logits = g.standard_normal(k)
        ex = np.exp(logits - logits.max())
        wts[t] = (ex / ex.sum()).astype(np.float32)
    return ids, wts


def hc_logits(n: int, nhc: int = 4, scale: float = 1.0, seed: int = SEED, stream: int = S_HC) -> np.ndarray:
    """Hyper-connection mixing logits (n, nhc, nhc) fp32 ~ N(0, scale^2)."""
    return (rng(seed, stream).standard_normal((n, nhc, nhc)) * scale).astype(np.float32)


def distinct_experts(ids: np.ndarray, E: int) -> np.ndarray:
    """Sorted distinct in-range expert ids of a routing table (for byte counts)."""
    v = np.asarray(ids).ravel()
    v = v[(v >= 0) & (v < E)]
    return np.unique(v)
