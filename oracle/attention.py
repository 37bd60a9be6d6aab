"""CPU oracle for ring-order blockwise attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline
leg and its ``--impl reference`` arm) may import or run anything in this
package.  The product path (``ring_attention_fwd_gb300`` and its CUDA library)
never imports it and shares no code with it.

Everything is float64 NumPy, written for a reader to check against the pages
by eye.  Pages cited (title and section only):

  [FT]  "Ring Attention如何让大模型突破百万Token上下文：从环形通信到计算重叠的技术突围"
        (answer.freetools.me)
  [CH]  "Ring Attention with Blockwise Transformers for Near Infinite Context",
        reading notes on arXiv 2310.01889 (papers.chlience.com)
  [AQ]  "Ring Attention" explainer, sushi-conveyor analogy (aiqz.cc)

What the method computes, and the readings taken where the pages are silent:

  * Exact scaled dot-product attention softmax(Q K^T / sqrt(D)) V, per batch
    b and head h ([CH] §5.1; [FT] "一个100M Token的序列需要多少内存").  D is
    the per-head key dimension d_k ([AQ] §分块注意力, S_b = Q_i K_b^T / sqrt(d_k)).
  * The sequence is cut into N equal blocks of c = S/N rows ([CH] §5.2;
    [FT] "Ring Attention的核心洞察", steps 1-2).  Tensors arrive in *storage
    order*.  Contiguous layout: storage row p holds token p.  Striped layout:
    token t lives on virtual device t mod N ([FT] "因果掩码的负载均衡挑战",
    the Token [0,4,8,12,...] list), at row t div N of that device's block, so
    storage row p = i*c + r holds token r*N + i.
  * Causal masking is token level: token t_q sees key token t_k iff
    t_k <= t_q ([AQ] §工程实现, third point).  For contiguous blocks this makes
    whole blocks j > i invisible, which the ring loop skips ([AQ] §工程实现,
    the S_ij -> -inf (j > i) equation).
  * LSE is the natural log of sum_k exp(s_qk) over visible keys, in scaled
    score units ([FT] "Online Softmax" LogSumExp form).  A row with no visible
    key has O = 0 and LSE = -inf (cannot occur under the causal rule, since
    every token sees itself; it can occur for a partial state).
  * Backward: the pages only say the backward re-sweeps the ring to
    accumulate dQ, dK, dV from the saved softmax state ([CH] §5.2, last
    paragraph).  The oracle uses the gradient of the definition above, with
    D_vec = rowsum(dO * O) taken from the *given* O (the saved output).

Parity pins live in ``tests/test_oracle.py``; nothing here is "parity
unpinned".
"""
from __future__ import annotations

import numpy as np

CONTIGUOUS = "contiguous"
STRIPED = "striped"
_LAYOUTS = (CONTIGUOUS, STRIPED)


# ----------------------------------------------------------------------------
# Layout: storage row <-> token position
# ----------------------------------------------------------------------------
def token_positions(S: int, N: int, layout: str) -> np.ndarray:
    """Token position held by each storage row p (int64 array of length S).

    Contiguous: block i holds tokens i*c .. i*c+c-1 ([FT] "Ring Attention的核心
    洞察", step 1).  Striped: device i holds tokens i, i+N, i+2N, ... ([FT]
    "因果掩码的负载均衡挑战"), so row r of block i is token r*N + i.
    """
    if layout not in _LAYOUTS:
        raise ValueError(layout)
    if N <= 0 or S % N:
        raise ValueError("S must be a positive multiple of N")
    p = np.arange(S, dtype=np.int64)
    if layout == CONTIGUOUS:
        return p
    c = S // N
    i, r = np.divmod(p, c)
    return r * N + i


def visible(tq: np.ndarray, tk: np.ndarray, causal: bool) -> np.ndarray:
    """Boolean [len(tq), len(tk)]: may query token tq see key token tk."""
    if not causal:
        return np.ones((tq.size, tk.size), dtype=bool)
    return tk[None, :] <= tq[:, None]


# ----------------------------------------------------------------------------
# Form 1: the plain definition, full-row softmax per query row
# ----------------------------------------------------------------------------
def attention_rows(q, k, v, rows, n_blocks: int, causal: bool, layout: str):
    """O and LSE of the given storage rows of ONE head.

    q, k, v: float64 [S, D].  rows: int array of storage rows.
    Returns (o [len(rows), D], lse [len(rows)]).  Softmax over each full row of
    scores, max-subtracted (the naive reference of [AQ] §Python 演示).
    """
    S, D = k.shape
    rows = np.asarray(rows, dtype=np.int64)
    s = (q[rows] @ k.T) / np.sqrt(D)
    if causal:      # (non-causal: every key visible; q and k may differ in length)
        pos = token_positions(S, n_blocks, layout)
        s = np.where(visible(pos[rows], pos, causal), s, -np.inf)
    m = s.max(axis=1)
    any_vis = np.isfinite(m)
    m_safe = np.where(any_vis, m, 0.0)
    e = np.exp(s - m_safe[:, None])           # exp(-inf) = 0 on masked entries
    l = e.sum(axis=1)
    o = np.zeros((rows.size, D))
    o[any_vis] = (e[any_vis] @ v) / l[any_vis, None]
    lse = np.full(rows.size, -np.inf)
    lse[any_vis] = m[any_vis] + np.log(l[any_vis])
    return o, lse


def naive_attention(q, k, v, n_blocks: int, causal: bool, layout: str, row_chunk: int = 512):
    """Plain definition over all rows.  q, k, v: float64 [B, H, S, D].

    Returns (o [B,H,S,D], lse [B,H,S]).  Rows are processed in chunks so that
    long sequences fit in memory; each chunk is ``attention_rows``.
    """
    B, H, S, D = q.shape
    o = np.zeros((B, H, S, D))
    lse = np.zeros((B, H, S))
    for b in range(B):
        for h in range(H):
            for r0 in range(0, S, row_chunk):
                rows = np.arange(r0, min(S, r0 + row_chunk))
                o[b, h, rows], lse[b, h, rows] = attention_rows(
                    q[b, h], k[b, h], v[b, h], rows, n_blocks, causal, layout)
    return o, lse


# ----------------------------------------------------------------------------
# Form 2: the literal ring loop with the online-softmax update
# ----------------------------------------------------------------------------
def ring_order(i: int, N: int) -> list:
    """KV blocks in the order query block i meets them on the ring.

    At step s, host i holds the block of host (i - s) mod N: it sends to i+1
    and receives from i-1 ([FT] "Ring Attention的核心洞察", step 3; [AQ]
    §环状拓扑 and the demo's ``src = (device - step) % num_devices``).
    """
    return [(i - s) % N for s in range(N)]


def ring_block_attention(q, k, v, i: int, n_blocks: int, causal: bool, layout: str,
                         order=None):
    """Online-softmax sweep of query block i over KV blocks, ONE head.

    Follows [AQ] §分块注意力, in the page's normalised-output form:
        S_b  = Q_i K_b^T / sqrt(d_k)
        m    <- max(m_old, rowmax(S_b))
        l    <- l_old * exp(m_old - m) + rowsum(exp(S_b - m))
        O    <- (l_old * exp(m_old - m) / l) * O + (exp(S_b - m) / l) * V_b
    starting from m = -inf, l = 0, O = 0 ([AQ] §Python 演示).  Contiguous
    causal blocks j > i are skipped whole ([AQ] §工程实现); all other masking is
    per token (entries set to -inf).  ``order`` overrides the ring order (any
    permutation gives the same result: [FT] "Ring Attention的核心洞察", [CH] §4).

    Returns (o_i [c, D], lse_i [c]).
    """
    S, D = k.shape
    N = n_blocks
    c = S // N
    pos = token_positions(S, N, layout)
    qi = q[i * c:(i + 1) * c]
    tq = pos[i * c:(i + 1) * c]
    m = np.full(c, -np.inf)
    l = np.zeros(c)
    o = np.zeros((c, D))
    for j in (ring_order(i, N) if order is None else order):
        if causal and layout == CONTIGUOUS and j > i:
            continue                                  # whole block invisible
        kj = k[j * c:(j + 1) * c]
        vj = v[j * c:(j + 1) * c]
        sb = (qi @ kj.T) / np.sqrt(D)
        sb = np.where(visible(tq, pos[j * c:(j + 1) * c], causal), sb, -np.inf)
        m_new = np.maximum(m, sb.max(axis=1))
        seen = np.isfinite(m_new)                     # rows that saw any key so far
        m_ref = np.where(seen, m_new, 0.0)            # exp(-inf - (-inf)) := 0
        scale_old = np.where(np.isfinite(m), np.exp(m - m_ref), 0.0)
        e = np.exp(sb - m_ref[:, None])
        l_new = l * scale_old + e.sum(axis=1)
        o_new = np.zeros_like(o)
        o_new[seen] = ((l[seen] * scale_old[seen] / l_new[seen])[:, None] * o[seen]
                       + (e[seen] @ vj) / l_new[seen, None])
        m, l, o = m_new, l_new, o_new
    lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return o, lse


def ring_attention(q, k, v, n_blocks: int, causal: bool, layout: str, order_fn=None):
    """Every query block's ring sweep.  q, k, v: float64 [B, H, S, D].

    ``order_fn(i, N)`` may replace ``ring_order`` (to test order invariance).
    Returns (o [B,H,S,D], lse [B,H,S]).
    """
    B, H, S, D = q.shape
    N = n_blocks
    c = S // N
    o = np.zeros((B, H, S, D))
    lse = np.zeros((B, H, S))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                order = None if order_fn is None else order_fn(i, N)
                o[b, h, i * c:(i + 1) * c], lse[b, h, i * c:(i + 1) * c] = ring_block_attention(
                    q[b, h], k[b, h], v[b, h], i, N, causal, layout, order)
    return o, lse


def block_pair_attention(q, k, v, i: int, j: int, n_blocks: int, causal: bool, layout: str):
    """Partial state of query block i over the keys of block j only, ONE head.

    What host i holds after attending its queries to the one KV block j it
    has in a ring round ([CH] §5.2): softmax over block j's visible keys.
    q, k, v: float64 [S, D] of the whole sequence (storage order), so that the
    token positions of both blocks are those of `layout`.  Rows that see none
    of block j's keys get O = 0, LSE = -inf.  Returns (o [c, D], lse [c]).
    """
    S, D = k.shape
    c = S // n_blocks
    pos = token_positions(S, n_blocks, layout)
    qi = q[i * c:(i + 1) * c]
    kj, vj = k[j * c:(j + 1) * c], v[j * c:(j + 1) * c]
    s = (qi @ kj.T) / np.sqrt(D)
    s = np.where(visible(pos[i * c:(i + 1) * c], pos[j * c:(j + 1) * c], causal), s, -np.inf)
    m = s.max(axis=1)
    seen = np.isfinite(m)
    e = np.exp(s - np.where(seen, m, 0.0)[:, None])
    l = e.sum(axis=1)
    o = np.zeros((c, D))
    o[seen] = (e[seen] @ vj) / l[seen, None]
    lse = np.full(c, -np.inf)
    lse[seen] = m[seen] + np.log(l[seen])
    return o, lse


# ----------------------------------------------------------------------------
# LogSumExp merge of two partial states
# ----------------------------------------------------------------------------
def lse_merge(o_a, lse_a, o_b, lse_b):
    """Merge two partial (O, lse) states over disjoint key sets.

    [FT] "Online Softmax": l = l1 e^{m1-m} + l2 e^{m2-m}, and in log space
    log l = log(e^{log l1 + m1 - m} + e^{log l2 + m2 - m}).  With lse = m + log l
    for each part, the merged lse is M + log(e^{lse_a - M} + e^{lse_b - M}),
    M = max(lse_a, lse_b), and each normalised output is re-weighted by its
    share of the total mass: O = e^{lse_a - lse} O_a + e^{lse_b - lse} O_b.
    Both -inf (no key seen on either side): lse = -inf, O = 0.
    o_*: [..., D]; lse_*: [...].
    """
    lse_a = np.asarray(lse_a, dtype=np.float64)
    lse_b = np.asarray(lse_b, dtype=np.float64)
    M = np.maximum(lse_a, lse_b)
    none = ~np.isfinite(M)
    M_safe = np.where(none, 0.0, M)
    wa_un = np.exp(lse_a - M_safe)
    wb_un = np.exp(lse_b - M_safe)
    tot = wa_un + wb_un
    lse = np.where(none, -np.inf, M_safe + np.log(np.where(none, 1.0, tot)))
    wa = np.where(none, 0.0, wa_un / np.where(none, 1.0, tot))
    wb = np.where(none, 0.0, wb_un / np.where(none, 1.0, tot))
    o = wa[..., None] * o_a + wb[..., None] * o_b
    return o, lse


# ----------------------------------------------------------------------------
# Backward: gradient of the definition, given the saved O and LSE
# ----------------------------------------------------------------------------
def _probabilities(q, k, lse, n_blocks, causal, layout, rows=None):
    """P = exp(S - LSE) on visible entries, 0 elsewhere, for ONE head."""
    S, D = k.shape
    pos = token_positions(S, n_blocks, layout)
    rows = np.arange(S) if rows is None else np.asarray(rows, dtype=np.int64)
    s = (q[rows] @ k.T) / np.sqrt(D)
    vis = visible(pos[rows], pos, causal)
    lse_r = lse[rows]
    ok = vis & np.isfinite(lse_r)[:, None]
    return np.where(ok, np.exp(np.where(ok, s - lse_r[:, None], -np.inf)), 0.0)


def attention_bwd_head(q, k, v, o, lse, do, n_blocks: int, causal: bool, layout: str):
    """dQ, dK, dV of ONE head (all float64 [S, D]; lse [S]).

    With P = exp(S - LSE), S = Q K^T / sqrt(D):
        dV = P^T dO,  dP = dO V^T,  D_vec = rowsum(dO * O),
        dS = P * (dP - D_vec),  dQ = dS K / sqrt(D),  dK = dS^T Q / sqrt(D).
    """
    S, D = q.shape
    P = _probabilities(q, k, lse, n_blocks, causal, layout)
    dV = P.T @ do
    dP = do @ v.T
    Dvec = (do * o).sum(axis=1)
    dS = P * (dP - Dvec[:, None])
    dQ = (dS @ k) / np.sqrt(D)
    dK = (dS.T @ q) / np.sqrt(D)
    return dQ, dK, dV


def attention_bwd_head_chunked(q, k, v, o, lse, do, n_blocks: int, causal: bool, layout: str,
                               row_chunk: int = 256):
    """``attention_bwd_head`` for sequences whose S x S matrix of
    probabilities does not fit in memory (ONE head; float64 [S, D], lse [S]).

    The query rows are taken ``row_chunk`` at a time.  A chunk's rows of dQ
    depend on that chunk alone; its contributions to dK and dV are added up
    over the chunks, as dK_j and dV_j accumulate one query block per ring
    round ([CH] §5.2).  Same formulas as ``attention_bwd_head``:
        dV += P_c^T dO_c,  dS_c = P_c * (dO_c V^T - rowsum(dO_c * O_c)),
        dQ_c = dS_c K / sqrt(D),  dK += dS_c^T Q_c / sqrt(D).
    """
    S, D = q.shape
    dQ = np.zeros((S, D))
    dK = np.zeros((S, D))
    dV = np.zeros((S, D))
    for r0 in range(0, S, row_chunk):
        rows = np.arange(r0, min(S, r0 + row_chunk))
        P = _probabilities(q, k, lse, n_blocks, causal, layout, rows=rows)
        dV += P.T @ do[rows]
        dP = do[rows] @ v.T
        Dvec = (do[rows] * o[rows]).sum(axis=1)
        dS = P * (dP - Dvec[:, None])
        dQ[rows] = (dS @ k) / np.sqrt(D)
        dK += (dS.T @ q[rows]) / np.sqrt(D)
    return dQ, dK, dV


def block_pair_bwd(q, k, v, o, lse, do, i: int, j: int, n_blocks: int, causal: bool, layout: str):
    """One ring round of the backward, ONE head: the contributions of query
    block i against KV block j alone.

    The pages only say the backward, like the forward, sweeps the KV blocks
    around the ring to accumulate dQ, dK, dV ([CH] §5.2).  Restricting the
    gradient of ``attention_bwd_head`` to the keys of block j gives, with
    P_ij = exp(Q_i K_j^T / sqrt(D) - LSE_i) on visible entries (LSE_i the
    block's FINAL log-sum-exp):
        dV_j += P_ij^T dO_i,  dS_ij = P_ij * (dO_i V_j^T - rowsum(dO_i * O_i)),
        dQ_i += dS_ij K_j / sqrt(D),  dK_j += dS_ij^T Q_i / sqrt(D).
    q, k, v, o, do: float64 [S, D] of the whole head; lse [S].  Returns the
    three contributions (dq_i, dk_j, dv_j), each [c, D].
    """
    S, D = q.shape
    c = S // n_blocks
    rq = np.arange(i * c, (i + 1) * c)
    rk = np.arange(j * c, (j + 1) * c)
    pos = token_positions(S, n_blocks, layout)
    s = (q[rq] @ k[rk].T) / np.sqrt(D)
    ok = visible(pos[rq], pos[rk], causal) & np.isfinite(lse[rq])[:, None]
    P = np.where(ok, np.exp(np.where(ok, s - lse[rq][:, None], -np.inf)), 0.0)
    dv = P.T @ do[rq]
    Dvec = (do[rq] * o[rq]).sum(axis=1)
    dS = P * (do[rq] @ v[rk].T - Dvec[:, None])
    return (dS @ k[rk]) / np.sqrt(D), (dS.T @ q[rq]) / np.sqrt(D), dv


def attention_bwd(q, k, v, o, lse, do, n_blocks: int, causal: bool, layout: str):
    """Batched ``attention_bwd_head``: all float64 [B, H, S, D] (lse [B, H, S])."""
    B, H = q.shape[:2]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = attention_bwd_head(
                q[b, h], k[b, h], v[b, h], o[b, h], lse[b, h], do[b, h], n_blocks, causal, layout)
    return dq, dk, dv


def attention_bwd_dq_rows(q, k, v, do, rows, n_blocks: int, causal: bool, layout: str):
    """dQ of selected storage rows of ONE head, from Q, K, V, dO alone.

    Each row's gradient needs only that row's own O and LSE, which are
    recomputed here from the definition (``attention_rows``).
    """
    S, D = q.shape
    rows = np.asarray(rows, dtype=np.int64)
    o_r, lse_r = attention_rows(q, k, v, rows, n_blocks, causal, layout)
    full_lse = np.full(S, -np.inf)
    full_lse[rows] = lse_r
    P = _probabilities(q, k, full_lse, n_blocks, causal, layout, rows=rows)
    dP = do[rows] @ v.T
    Dvec = (do[rows] * o_r).sum(axis=1)
    dS = P * (dP - Dvec[:, None])
    return (dS @ k) / np.sqrt(D)


def attention_bwd_kv_rows(q, k, v, do, key_rows, n_blocks: int, causal: bool, layout: str,
                          row_chunk: int = 512, query_rows=None):
    """dK and dV of selected key rows of ONE head, from Q, K, V, dO alone.

    Every query row that can see one of the keys (all rows, or under the causal
    rule the rows whose token is not earlier than the earliest selected key) has
    its O and LSE recomputed from the definition (``attention_rows``); then
        dV(k) = sum_q P(q,k) dO(q),   dS(q,k) = P(q,k) (dO(q).v_k - D_vec(q)),
        dK(k) = sum_q dS(q,k) q / sqrt(D),   D_vec(q) = dO(q).O(q).
    ``query_rows`` (storage rows) restricts both sums to those queries: the
    parts over a partition of the rows add up to the whole, as dK_j and dV_j
    accumulate one query block per ring round ([CH] §5.2).
    Returns (dK [len(key_rows), D], dV [len(key_rows), D]).
    """
    S, D = q.shape
    key_rows = np.asarray(key_rows, dtype=np.int64)
    pos = token_positions(S, n_blocks, layout)
    if causal:
        q_rows = np.nonzero(pos >= pos[key_rows].min())[0]
    else:
        q_rows = np.arange(S)
    if query_rows is not None:
        q_rows = np.intersect1d(q_rows, np.asarray(query_rows, dtype=np.int64))
    dK = np.zeros((key_rows.size, D))
    dV = np.zeros((key_rows.size, D))
    kk, vk = k[key_rows], v[key_rows]
    for c0 in range(0, q_rows.size, row_chunk):
        rows = q_rows[c0:c0 + row_chunk]
        o_r, lse_r = attention_rows(q, k, v, rows, n_blocks, causal, layout)
        s = (q[rows] @ kk.T) / np.sqrt(D)
        vis = visible(pos[rows], pos[key_rows], causal) & np.isfinite(lse_r)[:, None]
        P = np.where(vis, np.exp(np.where(vis, s - lse_r[:, None], -np.inf)), 0.0)
        dP = do[rows] @ vk.T
        Dvec = (do[rows] * o_r).sum(axis=1)
        dS = P * (dP - Dvec[:, None])
        dV += P.T @ do[rows]
        dK += (dS.T @ q[rows]) / np.sqrt(D)
    return dK, dV


# ----------------------------------------------------------------------------
# Work per virtual device (load balance)
# ----------------------------------------------------------------------------
def visible_pairs_per_device(S: int, N: int, layout: str, causal: bool) -> np.ndarray:
    """Number of visible (query, key) pairs whose query block is device i.

    Counted from the mask definition, row by row: a causal query at token t
    sees t + 1 keys; a non-causal one sees S.
    """
    pos = token_positions(S, N, layout)
    per_row = (pos + 1) if causal else np.full(S, S, dtype=np.int64)
    return per_row.reshape(N, S // N).sum(axis=1)


def block_rectangle_work(S: int, N: int, layout: str, causal: bool) -> np.ndarray:
    """Per device, sum of c*c over the block pairs its ring sweep does not skip.

    This is the block-level count of [FT] "因果掩码的负载均衡挑战" (device i of 4
    computes 25 x 25(i+1) when 100 tokens are split contiguously).
    """
    c = S // N
    out = np.zeros(N, dtype=np.int64)
    for i in range(N):
        for j in ring_order(i, N):
            if causal and layout == CONTIGUOUS and j > i:
                continue
            out[i] += c * c
    return out
