"""CPU oracle for ring decode -- TEST INFRASTRUCTURE ONLY (same rules as
``oracle.attention``: only tests, smoke() and bench.py's CPU legs use it).

What is computed, and the readings taken:

  * Decoding generates one token at a time, so the query has length 1
    ([CH] §5.6 "推理适用性"; [FT] "局限与未来", the inference point).  The new
    token's query q attends to every entry of the KV cache, whose last row is
    the new token's own key/value: the causal rule t_k <= t_q then admits every
    cached key, so no mask is applied.
  * The cache is spread over the ring: each host keeps one segment and the
    partial results travel the ring ([CH] §5.6; [AQ] "超长序列推理与 KV Cache
    分发": every card holds one segment of the cache).  The pages do not say
    how a cache whose length is not a multiple of N is cut; the reading here
    is c = ceil(S / N) rows per block, block j = rows [j*c, min((j+1)*c, S)),
    so trailing blocks may be short or empty (a growing cache fills the ring
    front to back).  An empty block contributes the empty partial (O = 0,
    lse = -inf).
  * The partials are folded with the LogSumExp merge ([FT] "Online Softmax")
    in the ring order of the host that holds the newest token, i.e. the last
    block's host (N - 1): blocks N-1, N-2, ..., 0.

Pins: tests/test_oracle.py (the test_decode_* functions).
"""
from __future__ import annotations

import numpy as np

from .attention import lse_merge, ring_order


def decode_attention(q, k, v):
    """Plain definition for ONE query vector of ONE head.

    q: float64 [D]; k, v: float64 [L, D] with L >= 0.
    Returns (o [D], lse): o = sum_t e^{s_t - lse} v_t with s_t = q.k_t / sqrt(D)
    and lse = ln sum_t e^{s_t} (max-subtracted); L = 0 gives (0, -inf).
    """
    L, D = k.shape
    if L == 0:
        return np.zeros(D), -np.inf
    s = (k @ q) / np.sqrt(D)
    m = s.max()
    e = np.exp(s - m)
    l = e.sum()
    return (e @ v) / l, m + np.log(l)


def decode_blocks(S: int, N: int):
    """Row ranges [(start, end)] of the N ring blocks of an S-row cache."""
    if S < 1 or N < 1:
        raise ValueError("S and N must be >= 1")
    c = -(-S // N)
    return [(min(j * c, S), min((j + 1) * c, S)) for j in range(N)]


def ring_decode(q, k, v, N: int, holder: int | None = None):
    """Ring decode of ONE head: per-block partials merged along the ring.

    q: float64 [D]; k, v: float64 [S, D].  ``holder`` is the host that holds
    the query (default: the last block's host).  Returns (o [D], lse).
    """
    S, D = k.shape
    blocks = decode_blocks(S, N)
    holder = N - 1 if holder is None else holder
    o, lse = np.zeros(D), -np.inf
    for j in ring_order(holder, N):
        a, b = blocks[j]
        oj, lj = decode_attention(q, k[a:b], v[a:b])
        mo, ml = lse_merge(o[None], np.array([lse]), oj[None], np.array([lj]))
        o, lse = mo[0], float(ml[0])
    return o, lse


def decode_batch(q, k, v, N: int):
    """``ring_decode`` over every (b, h): q [B, H, D], k/v [B, H, S, D].

    Returns (o [B, H, D], lse [B, H])."""
    B, H, S, D = k.shape
    o = np.zeros((B, H, D))
    lse = np.zeros((B, H))
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = ring_decode(q[b, h], k[b, h], v[b, h], N)
    return o, lse
