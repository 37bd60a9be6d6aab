"""Backward parity: CUDA ra_bwd (through the C ABI) vs the CPU oracle.

Tolerance for dQ, dK, dV (bf16 inputs, float32 accumulation, bf16 outputs):
max |g - ref| <= 2e-2 * max(1, max |ref|), and relative Frobenius error
<= 1e-2.  Derivation: P and dS enter the tensor cores rounded to bf16
(relative 2^-9); the outputs are rounded to bf16 (relative 2^-9); float32
accumulation adds ~1e-6 relative; so ~4e-3 of the largest gradient entry,
with a 5x margin for sums of correlated rounding errors.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from gpu_helpers import (SUM_DK_LIMIT, SUM_DV_LIMIT, TOL, fwd_sampled_check, head_arrays, keys_in_every_block,
                         max_err, sample_rows, workload_inputs)
from ring_attention_fwd_gb300.inputs import LONG_WORKLOADS, WORKLOADS, as_float64, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import ring_attention_fwd_gb300 as ra
    assert torch.cuda.is_available()
    return ra


def _close(g, ref, name):
    g = np.asarray(g, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = max(1.0, float(np.abs(ref).max()))
    e = max_err(g, ref)
    assert e <= 2e-2 * scale, f"{name}: max err {e:.3e} (scale {scale:.3e})"
    fro = float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30))
    assert fro <= 1e-2, f"{name}: relative Frobenius {fro:.3e}"


BWD_CASES = [
    (1, 1, 256, 1, True, "contiguous"),
    (1, 2, 512, 2, True, "contiguous"),
    (1, 2, 512, 2, True, "striped"),
    (2, 1, 1024, 4, False, "contiguous"),
    (1, 1, 384, 3, True, "striped"),
    (1, 2, 600, 3, True, "contiguous"),     # c = 200: ragged KV and query tiles
    (1, 1, 1000, 5, True, "striped"),       # c = 200, striped
    (1, 1, 128, 8, True, "striped"),        # c = 16
    (1, 3, 2048, 4, True, "striped"),
    (1, 2, 2048, 8, False, "striped"),
    (3, 2, 768, 3, True, "striped"),        # B > 1, causal
    (1, 2, 8, 8, True, "contiguous"),       # c = 1: one token per block
]


@pytest.mark.parametrize("B,H,S,N,causal,layout", BWD_CASES)
def test_bwd_shapes_from_oracle_state(ra, B, H, S, N, causal, layout):
    """The kernel alone: it is given the oracle's O (rounded to bf16) and LSE
    (rounded to float32); the expected gradient uses those same rounded values."""
    inp = make_inputs(B, H, S, 128, seed=300 + S + N, with_grad=True)
    q, k, v, do = (as_float64(inp[x]) for x in ("q", "k", "v", "do"))
    o_ref, lse_ref = orc.naive_attention(q, k, v, N, causal, layout)
    o_bf = torch.from_numpy(o_ref).to(torch.bfloat16)
    lse_f = torch.from_numpy(lse_ref).float()
    rq, rk, rv = orc.attention_bwd(q, k, v, o_bf.double().numpy(), lse_f.double().numpy(), do, N, causal, layout)
    dev = {x: inp[x].cuda() for x in ("q", "k", "v", "do")}
    dq, dk, dv = ra.bwd(dev["q"], dev["k"], dev["v"], o_bf.cuda(), lse_f.cuda(), dev["do"], N, causal, layout)
    torch.cuda.synchronize()
    ra.check_device_status()
    _close(dq.double().cpu().numpy(), rq, "dQ")
    _close(dk.double().cpu().numpy(), rk, "dK")
    _close(dv.double().cpu().numpy(), rv, "dV")


@pytest.mark.parametrize("layout", ["striped", "contiguous"])
def test_fwd_then_bwd_against_exact_gradient(ra, layout):
    """The composition: the GPU forward's (O, LSE) feed the GPU backward; the
    oracle computes the gradient from Q, K, V, dO alone."""
    B, H, S, N = 1, 2, 1536, 6
    inp = make_inputs(B, H, S, 128, seed=401, with_grad=True)
    q, k, v, do = (as_float64(inp[x]) for x in ("q", "k", "v", "do"))
    o_ref, lse_ref = orc.naive_attention(q, k, v, N, True, layout)
    rq, rk, rv = orc.attention_bwd(q, k, v, o_ref, lse_ref, do, N, True, layout)
    dev = {x: inp[x].cuda() for x in ("q", "k", "v", "do")}
    o, lse = ra.fwd(dev["q"], dev["k"], dev["v"], N, True, layout)
    dq, dk, dv = ra.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], N, True, layout)
    torch.cuda.synchronize()
    _close(dq.double().cpu().numpy(), rq, "dQ")
    _close(dk.double().cpu().numpy(), rk, "dK")
    _close(dv.double().cpu().numpy(), rv, "dV")


def test_bwd_deterministic_and_workspace_reuse(ra):
    """dQ, dK and dV are each written once per row by one CTA, with no
    atomics, so two runs are bit-identical.  A workspace reused without
    clearing gives the same result."""
    inp = {k: v.cuda() for k, v in make_inputs(1, 2, 1024, 128, seed=5, with_grad=True).items()}
    o, lse = ra.fwd(inp["q"], inp["k"], inp["v"], 4, True, "striped")
    ws = torch.full((ra.bwd_workspace_bytes(1, 2, 1024, 128, 4),), 0x7f, dtype=torch.uint8, device="cuda")
    a = ra.bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], 4, True, "striped", workspace=ws)
    b = ra.bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], 4, True, "striped", workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def check_sum_identities(dk, dv, do, heads):
    """Every row of P sums to 1 and every row of dS to 0, so for every head and
    column  sum_k dK = 0  and  sum_k dV = sum_q dO  (each query sees at least
    its own key).  Checked over all S keys, so every key block of the full-size
    output takes part; the sums run in float64 on the device."""
    for h in heads:
        gk = dk[0, h].double()
        gv = dv[0, h].double()
        gd = do[0, h].double()
        rk = gk.sum(0).abs() / gk.norm(dim=0).clamp_min(1e-30)
        rv = (gv.sum(0) - gd.sum(0)).abs() / (gv.norm(dim=0) ** 2 + gd.norm(dim=0) ** 2).sqrt()
        assert float(rk.max()) <= SUM_DK_LIMIT, f"sum_k dK head {h}: {float(rk.max()):.3e} of ||dK||"
        assert float(rv.max()) <= SUM_DV_LIMIT, f"sum_k dV - sum_q dO head {h}: {float(rv.max()):.3e}"


def _sampled_bwd_check(ra, w, dq_heads, kv_head, n_keys, late_only, late_window=2048, n_random=96):
    inp = workload_inputs(w, with_grad=True)
    N, causal, layout = w["N"], w["causal"], w["layout"]
    B, H, S, D = inp["q"].shape
    dev = {x: inp[x].cuda() for x in ("q", "k", "v", "do")}
    o, lse = ra.fwd(dev["q"], dev["k"], dev["v"], N, causal, layout)
    dq, dk, dv = ra.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], N, causal, layout)
    torch.cuda.synchronize()
    ra.check_device_status()
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t.float()).all())
    check_sum_identities(dk, dv, dev["do"], range(H))
    del o, lse, dev
    for h in dq_heads:
        rows = sample_rows(S, N, n_random, 7 + h)
        q, k, v, do = (inp[x][0, h].to(torch.float64).numpy() for x in ("q", "k", "v", "do"))
        ref = np.concatenate([orc.attention_bwd_dq_rows(q, k, v, do, rows[c0:c0 + 64], N, causal, layout)
                              for c0 in range(0, rows.size, 64)])
        _close(dq[0, h, torch.from_numpy(rows).cuda()].double().cpu().numpy(), ref, f"dQ rows head {h}")
    q, k, v, do = (inp[x][0, kv_head].to(torch.float64).numpy() for x in ("q", "k", "v", "do"))
    pos = orc.token_positions(S, N, layout)
    rng = np.random.default_rng(11)
    if late_only:   # keys among the last tokens: only that many queries see them
        cand = np.nonzero(pos >= S - late_window)[0]
    else:
        cand = np.arange(S)
    keys = np.sort(rng.choice(cand, size=n_keys, replace=False))
    rk, rv = orc.attention_bwd_kv_rows(q, k, v, do, keys, N, causal, layout, row_chunk=128)
    kidx = torch.from_numpy(keys).cuda()
    _close(dk[0, kv_head, kidx].double().cpu().numpy(), rk, "dK rows")
    _close(dv[0, kv_head, kidx].double().cpu().numpy(), rv, "dV rows")


def _wide_bwd_check(ra, w, kv_heads, keys_per_block, n_random):
    """Full-size forward+backward on the GPU, then, with the oracle on all host
    cores: dQ on sampled rows (every block boundary, random rows) of EVERY
    head, and dK/dV on keys in EVERY ring block of ``kv_heads`` -- keys of
    the first blocks are seen by (nearly) every query, so the oracle recomputes
    the whole head for them.  The sum identities cover every key of every head."""
    import oracle_pool as op
    inp = workload_inputs(w, with_grad=True)
    N, causal, layout = w["N"], w["causal"], w["layout"]
    B, H, S, D = inp["q"].shape
    dev = {x: inp[x].cuda() for x in ("q", "k", "v", "do")}
    o, lse = ra.fwd(dev["q"], dev["k"], dev["v"], N, causal, layout)
    dq, dk, dv = ra.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], N, causal, layout)
    torch.cuda.synchronize()
    ra.check_device_status()
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t.float()).all())
    check_sum_identities(dk, dv, dev["do"], range(H))
    del o, lse, dev
    for h in range(H):
        paths = op.share(f"h{h}", **head_arrays(inp, 0, h))
        rows = sample_rows(S, N, n_random, 7 + h)
        ref = op.dq_rows(paths, rows, N, causal, layout)
        _close(dq[0, h, torch.from_numpy(rows).cuda()].double().cpu().numpy(), ref, f"dQ rows head {h}")
        if h in kv_heads:
            keys = keys_in_every_block(S, N, keys_per_block, 11 + h)
            rk, rv = op.kv_rows(paths, keys, N, causal, layout, S)
            kidx = torch.from_numpy(keys).cuda()
            _close(dk[0, h, kidx].double().cpu().numpy(), rk, f"dK rows head {h}")
            _close(dv[0, h, kidx].double().cpu().numpy(), rv, f"dV rows head {h}")
        op.release(paths)


def test_fwdbwd_64k_workload_backward_wide(ra):
    """The 65536-token striped forward+backward workload at full size: dQ rows
    of all 32 heads; dK/dV on 3 keys of each of the 16 blocks of two heads."""
    _wide_bwd_check(ra, WORKLOADS["fwdbwd_64k"], kv_heads=(5, 30), keys_per_block=3, n_random=32)


def test_long_128k_workload_backward_wide(ra):
    """The benchmark's workload and launch configuration (131072 tokens, 32
    blocks, causal contiguous): dQ rows of all 32 heads; dK/dV on 2 keys of
    each of the 32 blocks of two heads, the early blocks' keys included (the
    longest ring re-sweeps of the backward)."""
    _wide_bwd_check(ra, WORKLOADS["long_128k"], kv_heads=(9, 26), keys_per_block=2, n_random=32)


def test_million_token_forward_backward_sampled(ra):
    """A 1,048,576-token causal sequence (2 heads of 128, 64 blocks of 16384
    tokens): the lengths the method exists for.  Forward rows and dQ rows
    sampled over the whole sequence and every block boundary, dK/dV on keys
    among the last 1024 tokens, and the whole-sequence sum identities over all
    keys of both heads."""
    w = dict(LONG_WORKLOADS["long_1m"], H=2)
    inp = workload_inputs(w)
    eo, el, _, _ = fwd_sampled_check(ra, {x: inp[x] for x in ("q", "k", "v")}, w["N"], True, "contiguous",
                                     [(0, 0), (0, 1)], 32, 8)
    assert eo <= TOL["bf16"]["o"] and el <= TOL["bf16"]["lse"], (eo, el)
    del inp
    torch.cuda.empty_cache()
    _sampled_bwd_check(ra, w, dq_heads=(1,), kv_head=0, n_keys=32, late_only=True, late_window=1024,
                       n_random=16)

