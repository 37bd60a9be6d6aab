"""Helpers shared by the GPU parity tests (inputs, sampling, comparison).

Expected values always come from ``oracle`` on the CPU; GPU outputs are only
ever compared, never fed back into the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as orc
from ring_attention_fwd_gb300.inputs import as_float64, make_inputs

# Tolerances (max absolute error) for the forward: bf16 inputs with float32
# accumulation -> O <= 2e-2, LSE <= 1e-3; float32 workload <= 1e-4.
TOL = {"bf16": dict(o=2e-2, lse=1e-3), "f32": dict(o=1e-4, lse=1e-4)}

# Limits of the backward's whole-sequence identities, per head and column:
# |sum_k dK| <= SUM_DK_LIMIT * ||dK||_2 and
# |sum_k dV - sum_q dO| <= SUM_DV_LIMIT * sqrt(||dV||_2^2 + ||dO||_2^2).
# tests/test_tolerance_derivation.py derives them from the bf16 rounding points
# of the kernels (CPU only).
SUM_DK_LIMIT = 5e-2
SUM_DV_LIMIT = 1e-2


def to_cuda(inp: dict) -> dict:
    return {k: v.cuda() for k, v in inp.items()}


def sample_rows(S: int, N: int, n_random: int, seed: int) -> np.ndarray:
    """First/last rows, every block boundary, and random rows (sorted, unique)."""
    c = S // N
    rows = set(range(min(S, 32))) | set(range(max(0, S - 32), S))
    for i in range(N):
        rows |= {i * c, i * c + c - 1, min(S - 1, i * c + 127), min(S - 1, i * c + 128)}
    rng = np.random.default_rng(seed)
    rows |= set(rng.integers(0, S, size=n_random).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def max_err(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_inf = np.isneginf(a) & np.isneginf(b)
    d = np.abs(np.where(both_inf, 0.0, a) - np.where(both_inf, 0.0, b))
    return float(np.nanmax(np.where(np.isnan(d), np.inf, d))) if d.size else 0.0


def grad_errors(g, ref):
    """(max |g - ref| / max(1, max |ref|), relative Frobenius error): the
    backward's two figures, bounded by 2e-2 and 1e-2 for bf16."""
    g = np.asarray(g, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = max(1.0, float(np.abs(ref).max()))
    fro = float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30))
    return max_err(g, ref) / scale, fro


def fwd_full_check(ra, inp: dict, N: int, causal: bool, layout: str, dtype: str):
    """Run the CUDA forward and compare every output with the oracle."""
    dev = to_cuda(inp)
    o, lse = ra.fwd(dev["q"], dev["k"], dev["v"], N, causal, layout)
    torch.cuda.synchronize()
    ra.check_device_status()
    q, k, v = (as_float64(inp[x]) for x in ("q", "k", "v"))
    ro, rl = orc.naive_attention(q, k, v, N, causal, layout)
    eo = max_err(o.float().cpu().numpy(), ro)
    el = max_err(lse.cpu().numpy(), rl)
    return eo, el


def attention_rows_chunked(q, k, v, rows, N: int, causal: bool, layout: str, chunk: int = 64):
    """``oracle.attention_rows`` over ``rows``, ``chunk`` rows per call, so that
    the rows-by-S score matrix of a million-token sequence stays small."""
    rows = np.asarray(rows, dtype=np.int64)
    o = np.zeros((rows.size, q.shape[1]))
    lse = np.zeros(rows.size)
    for c0 in range(0, rows.size, chunk):
        o[c0:c0 + chunk], lse[c0:c0 + chunk] = orc.attention_rows(q, k, v, rows[c0:c0 + chunk], N, causal, layout)
    return o, lse


def fwd_sampled_check(ra, inp: dict, N: int, causal: bool, layout: str, heads, n_random: int, seed: int):
    """Run the CUDA forward on the full workload; compare sampled rows of the
    given heads with the oracle's row-by-row definition.  Also checks that
    every output is finite."""
    dev = to_cuda(inp)
    o, lse = ra.fwd(dev["q"], dev["k"], dev["v"], N, causal, layout)
    torch.cuda.synchronize()
    ra.check_device_status()
    assert bool(torch.isfinite(lse).all()), "non-finite LSE"
    assert bool(torch.isfinite(o.float()).all()), "non-finite O"
    B, H, S, D = inp["q"].shape
    eo = el = 0.0
    for (b, h) in heads:
        rows = sample_rows(S, N, n_random, seed + 31 * h)
        q = inp["q"][b, h].to(torch.float64).numpy()
        k = inp["k"][b, h].to(torch.float64).numpy()
        v = inp["v"][b, h].to(torch.float64).numpy()
        ro, rl = attention_rows_chunked(q, k, v, rows, N, causal, layout)
        go = o[b, h, torch.from_numpy(rows).cuda()].float().cpu().numpy()
        gl = lse[b, h, torch.from_numpy(rows).cuda()].cpu().numpy()
        eo = max(eo, max_err(go, ro))
        el = max(el, max_err(gl, rl))
    return eo, el, o, lse


def workload_inputs(w: dict, with_grad: bool = False) -> dict:
    """The workload's seeded inputs; dO is drawn after Q, K, V, so asking for it
    leaves Q, K, V unchanged."""
    return make_inputs(w["B"], w["H"], w["S"], w["D"], w["seed"], dtype=w["dtype"], scale=w["scale"],
                       with_grad=w["grad"] or with_grad)


def head_arrays(inp: dict, b: int, h: int, names=("q", "k", "v", "do")) -> dict:
    """float64 NumPy copies of one (b, h) slab of the given inputs (exact)."""
    return {x: inp[x][b, h].to(torch.float64).numpy() for x in names if x in inp}


def keys_in_every_block(S: int, N: int, per_block: int, seed: int) -> np.ndarray:
    """Storage rows of ``per_block`` keys in each of the N blocks: the block's
    first row, its last row, and random rows between (sorted, unique)."""
    c = S // N
    rng = np.random.default_rng(seed)
    keys = set()
    for i in range(N):
        keys |= {i * c, i * c + c - 1}
        keys |= set((i * c + rng.integers(0, c, size=max(0, per_block - 2))).tolist())
    return np.array(sorted(keys), dtype=np.int64)


def pooled_fwd_check(inp: dict, o, lse, N: int, causal: bool, layout: str, heads, n_random: int, seed: int):
    """Sampled rows of every listed head against ``oracle.attention_rows``,
    computed on all host cores; returns the max errors (O, LSE)."""
    import oracle_pool as op
    S = inp["q"].shape[2]
    eo = el = 0.0
    for (b, h) in heads:
        rows = sample_rows(S, N, n_random, seed + 31 * h)
        paths = op.share(f"fwd{b}_{h}", **head_arrays(inp, b, h, ("q", "k", "v")))
        ro, rl = op.fwd_rows(paths, rows, N, causal, layout)
        op.release(paths)
        idx = torch.from_numpy(rows).to(o.device)
        eo = max(eo, max_err(o[b, h, idx].float().cpu().numpy(), ro))
        el = max(el, max_err(lse[b, h, idx].cpu().numpy(), rl))
    return eo, el
