"""Ring forward across processes: one query block per rank, K/V blocks rotate.

The multi-device form of the method ("Ring Attention with Blockwise
Transformers for Near Infinite Context" notes, §5.2; "Ring Attention如何让大模型
突破百万Token上下文…", "Ring Attention的核心洞察" steps 1-5): rank i of an N-rank
group holds query block i and KV block i.  In round s it attends its queries
to the KV block it holds -- block (i - s) mod N -- while sending that block to
rank i+1 and receiving the next one from rank i-1, so the transfer overlaps
the compute.  After N rounds every rank has seen every KV block; the partial
states are folded with the LogSumExp merge.  Contiguous causal rounds whose
block lies entirely in the future (j > i) are skipped (the block is still
forwarded).

The block compute and the merge default to the library's ``fwd_step_fold``
(bf16: each round's partial is merged into the float32 running state inside
the forward kernel's epilogue, one launch per round) or ``fwd_step`` and
``merge`` (CUDA tensors, NCCL process group).  Both are parameters, so the
exchange protocol can be exercised elsewhere with other implementations.

``ring_backward`` is the training backward: dQ_i stays at host i while the
float32 accumulators of dK_j, dV_j travel with K_j, V_j; after the N rounds
one more hop returns each to its owner.

``ring_decode`` is the inference form (reading notes §5.6; "Ring Attention"
explainer, "超长序列推理与 KV Cache 分发"): every rank keeps one segment of the
KV cache and decodes the new token's query against it; the small partial
states, not the cache, then travel the ring.
"""
from __future__ import annotations

import datetime

import torch
import torch.distributed as dist


def ring_order(i: int, n: int):
    """KV block held by rank i in rounds 0..n-1: i, i-1, ... (mod n)."""
    return [(i - s) % n for s in range(n)]


def ring_forward(q, k, v, *, causal: bool = True, layout: str = "contiguous", group=None, step=None,
                 merge=None, timeout_s: float | None = None):
    """Ring attention forward for this rank's block.

    q, k, v: this rank's blocks [B, H, c, D] (block index = rank in `group`).
    step(q, k_j, v_j, n, i, j) -> (o, lse): partial state of block i over
    block j; merge(o, lse, o_j, lse_j) folds a partial into (o, lse) in place.
    timeout_s: give up (RuntimeError) if a round's exchange has not completed
    within this many seconds, instead of waiting for a peer that is gone.
    The running state starts empty (O = 0, lse = -inf) and stays in float32
    (float64 if q is float64) across the rounds; each round's partial, bf16
    from the library's step, is folded into it, so the output is rounded once
    rather than once per round.
    Returns (o, lse) of this rank's query rows, o in the state's dtype.
    """
    n = dist.get_world_size(group)
    i = dist.get_rank(group)
    fold = None
    if step is None and merge is None and q.dtype == torch.bfloat16:
        from . import binding

        def fold(qq, kk, vv, nn, ii, jj, oo, ll):
            binding.fwd_step_fold(qq, kk, vv, nn, ii, jj, causal, layout, o_acc=oo, lse_acc=ll)
    elif step is None or merge is None:
        from . import binding
        step = step or (lambda qq, kk, vv, nn, ii, jj: binding.fwd_step(qq, kk, vv, nn, ii, jj, causal, layout))
        merge = merge or (lambda o, l, oj, lj: binding.merge(o, l, oj, lj))
    send_to, recv_from = (i + 1) % n, (i - 1) % n
    bufs = [(torch.empty_like(k), torch.empty_like(v)) for _ in range(2 if n > 1 else 0)]
    cur_k, cur_v = k, v
    B, H, c, D = q.shape
    state = torch.float64 if q.dtype == torch.float64 else torch.float32
    o = torch.zeros((B, H, c, D), dtype=state, device=q.device)
    lse = torch.full((B, H, c), float("-inf"), dtype=state if state == torch.float64 else torch.float32,
                     device=q.device)
    for s, j in enumerate(ring_order(i, n)):
        reqs = []
        if s < n - 1:   # forward the block we hold, receive the next one
            nk, nv = bufs[s % 2]
            ops = [dist.P2POp(dist.isend, cur_k, send_to, group), dist.P2POp(dist.irecv, nk, recv_from, group),
                   dist.P2POp(dist.isend, cur_v, send_to, group), dist.P2POp(dist.irecv, nv, recv_from, group)]
            reqs = dist.batch_isend_irecv(ops)
        if not (causal and layout == "contiguous" and j > i):
            if fold is not None:
                fold(q, cur_k, cur_v, n, i, j, o, lse)
            else:
                oj, lj = step(q, cur_k, cur_v, n, i, j)
                merge(o, lse, oj, lj)
        for r in reqs:
            ok = r.wait(datetime.timedelta(seconds=timeout_s)) if timeout_s is not None else r.wait()
            if ok is False:
                raise RuntimeError(f"ring round {s}: exchange with ranks {recv_from}/{send_to} timed out")
        if s < n - 1:
            cur_k, cur_v = bufs[s % 2]
    return o, lse


def ring_decode(q, k, v, *, group=None, step=None, merge=None, timeout_s: float | None = None,
                lse_dtype=torch.float32):
    """Ring decode for this rank.

    q: the new token's query [B, H, D], the same on every rank; k, v: this
    rank's cache segment [B, H, c_i, D] (c_i may be 0).  The rank computes its
    segment's partial state, then for N-1 rounds forwards the partial it last
    received (first its own) to rank i+1 and merges the one arriving from
    rank i-1, so every rank ends with the full (o, lse), merged in its ring
    order i, i-1, ..., i+1.
    step(q, k, v) -> (o, lse) partial over one segment (default: the library's
    ``decode`` with one block); merge as for ring_forward.  lse_dtype: the
    dtype of the LSE that ``step`` returns (used for an empty segment).
    Returns (o [B, H, D], lse [B, H])."""
    n = dist.get_world_size(group)
    i = dist.get_rank(group)
    if step is None or merge is None:
        from . import binding
        step = step or (lambda qq, kk, vv: binding.decode(qq, kk, vv, 1))
        merge = merge or (lambda o, l, oj, lj: binding.merge(o, l, oj, lj))
    B, H, D = q.shape
    if k.shape[2] > 0:
        own_o, own_l = step(q, k, v)
    else:   # empty segment: the empty partial
        own_o = torch.zeros_like(q)
        own_l = torch.full((B, H), float("-inf"), dtype=lse_dtype, device=q.device)
    o, lse = own_o.clone(), own_l.clone()
    send_to, recv_from = (i + 1) % n, (i - 1) % n
    cur_o, cur_l = own_o, own_l
    for s in range(1, n):
        new_o, new_l = torch.empty_like(own_o), torch.empty_like(own_l)
        ops = [dist.P2POp(dist.isend, cur_o, send_to, group), dist.P2POp(dist.irecv, new_o, recv_from, group),
               dist.P2POp(dist.isend, cur_l, send_to, group), dist.P2POp(dist.irecv, new_l, recv_from, group)]
        for r in dist.batch_isend_irecv(ops):
            ok = r.wait(datetime.timedelta(seconds=timeout_s)) if timeout_s is not None else r.wait()
            if ok is False:
                raise RuntimeError(f"decode round {s}: exchange with ranks {recv_from}/{send_to} timed out")
        merge(o, lse, new_o, new_l)
        cur_o, cur_l = new_o, new_l
    return o, lse


def _wait_all(reqs, timeout_s, what):
    for r in reqs:
        ok = r.wait(datetime.timedelta(seconds=timeout_s)) if timeout_s is not None else r.wait()
        if ok is False:
            raise RuntimeError(f"{what}: exchange timed out")


def ring_backward(q, k, v, o, lse, do, *, causal: bool = True, layout: str = "contiguous", group=None, step=None,
                  timeout_s: float | None = None):
    """Ring backward for this rank's blocks.

    q, k, v, o, do: this rank's blocks [B, H, c, D]; lse: its final [B, H, c]
    LSE from the forward.  In round s the rank holds KV block j = (i - s) mod N;
    the float32 accumulators dK_j, dV_j travel the ring with it, one rank
    behind: the rank adds query block i's contributions (``step``) to its own
    dQ_i and to a zeroed partial of dK_j, dV_j, and only then waits for the
    accumulators of block j from rank i-1, adds the partial into them and
    passes them on to rank i+1.  K_j, V_j and the accumulators therefore both
    move while the rounds compute.  After the last round the accumulators hop
    once more, which brings each rank's own dK_i, dV_i home.  Contiguous causal
    rounds j > i add nothing and are skipped (the data is still forwarded).
    Per pair of ranks the transfers are posted in the same order on both sides
    (K_j, V_j of round s, then the accumulators of round s), as point-to-point
    backends match them by order.
    step(q, k_j, v_j, o, lse, do, dq, dk_j, dv_j, n, i, j) adds in place
    (default: the library's ``bwd_step``).  Returns float32 (dq, dk, dv)."""
    n = dist.get_world_size(group)
    i = dist.get_rank(group)
    if step is None:
        from . import binding

        def step(qq, kk, vv, oo, ll, dd, gq, gk, gv, nn, ii, jj):
            binding.bwd_step(qq, kk, vv, oo, ll, dd, gq, gk, gv, nn, ii, jj, causal, layout)
    send_to, recv_from = (i + 1) % n, (i - 1) % n
    f32 = dict(dtype=torch.float32, device=q.device)
    dq = torch.zeros(q.shape, **f32)
    kv = [k, v]
    sent = []                     # (requests, tensors) of the accumulators last passed on
    for s, j in enumerate(ring_order(i, n)):
        acc, acc_reqs = None, []
        if s > 0:                 # block j's accumulators from rank i-1, needed after this round's compute
            acc = [torch.empty(k.shape, **f32), torch.empty(v.shape, **f32)]
            acc_reqs = dist.batch_isend_irecv([dist.P2POp(dist.irecv, acc[0], recv_from, group),
                                               dist.P2POp(dist.irecv, acc[1], recv_from, group)])
        kv_reqs, nxt = [], None
        if s < n - 1:             # K_j, V_j move on while this round computes
            nxt = [torch.empty_like(kv[0]), torch.empty_like(kv[1])]
            kv_reqs = dist.batch_isend_irecv([
                dist.P2POp(dist.isend, kv[0], send_to, group), dist.P2POp(dist.irecv, nxt[0], recv_from, group),
                dist.P2POp(dist.isend, kv[1], send_to, group), dist.P2POp(dist.irecv, nxt[1], recv_from, group)])
        part = [torch.zeros(k.shape, **f32), torch.zeros(v.shape, **f32)]
        if not (causal and layout == "contiguous" and j > i):
            step(q, kv[0], kv[1], o, lse, do, dq, part[0], part[1], n, i, j)
        if acc is None:
            acc = part
        else:
            _wait_all(acc_reqs, timeout_s, f"backward round {s}: accumulators from rank {recv_from}")
            acc[0] += part[0]
            acc[1] += part[1]
        for reqs, _ in sent:
            _wait_all(reqs, timeout_s, f"backward round {s}: accumulators to rank {send_to}")
        sent = [(dist.batch_isend_irecv([dist.P2POp(dist.isend, acc[0], send_to, group),
                                         dist.P2POp(dist.isend, acc[1], send_to, group)]), acc)]
        _wait_all(kv_reqs, timeout_s, f"backward round {s} with ranks {recv_from}/{send_to}")
        kv = nxt
    home = [torch.empty(k.shape, **f32), torch.empty(v.shape, **f32)]
    reqs = dist.batch_isend_irecv([dist.P2POp(dist.irecv, home[0], recv_from, group),
                                   dist.P2POp(dist.irecv, home[1], recv_from, group)])
    _wait_all(reqs + sent[0][0], timeout_s, f"backward: own accumulators from rank {recv_from}")
    return dq, home[0], home[1]
