"""ra_fwd_step (one ring host, one KV block) and its chaining with ra_merge,
on the GPU, against the oracle and against the fused ra_fwd."""
import numpy as np
import pytest
import torch

import oracle as orc
from gpu_helpers import TOL, max_err
from ring_attention_fwd_gb300.inputs import as_float64, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import ring_attention_fwd_gb300 as ra
    assert torch.cuda.is_available()
    return ra


def _blocks(t, N):
    B, H, S, D = t.shape
    c = S // N
    return [t[:, :, b * c:(b + 1) * c].contiguous() for b in range(N)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_single_pairs_match_oracle(ra, fwd_kernel, layout, dtype):
    N, c = 4, 200 if dtype == "bf16" else 48
    D = 128 if dtype == "bf16" else 64
    inp = make_inputs(1, 2, N * c, D, seed=31, dtype=dtype)
    q, k, v = (as_float64(inp[x]) for x in ("q", "k", "v"))
    qb, kb, vb = (_blocks(inp[x].cuda(), N) for x in ("q", "k", "v"))
    tol = TOL[dtype]
    for i, j in [(2, 2), (2, 0), (0, 3), (3, 1), (1, 2)]:   # diagonal, past, future (contiguous: empty)
        o, lse = ra.fwd_step(qb[i], kb[j], vb[j], N, i, j, True, layout)
        torch.cuda.synchronize()
        for h in range(2):
            ro, rl = orc.block_pair_attention(q[0, h], k[0, h], v[0, h], i, j, N, True, layout)
            assert max_err(o[0, h].double().cpu().numpy(), ro) <= tol["o"], (i, j, h)
            assert max_err(lse[0, h].cpu().numpy(), rl) <= tol["lse"], (i, j, h)


@pytest.mark.parametrize("layout,causal", [("contiguous", True), ("striped", True), ("striped", False)])
def test_chained_steps_equal_fused_forward(ra, layout, causal):
    """Each virtual host runs its N ring steps and merges them: the result is
    the fused kernel's (and the oracle's) rows of that host."""
    B, H, N, c = 1, 2, 4, 256
    inp = make_inputs(B, H, N * c, 128, seed=32)
    dev = {x: inp[x].cuda() for x in ("q", "k", "v")}
    o_full, lse_full = ra.fwd(dev["q"], dev["k"], dev["v"], N, causal, layout)
    qb, kb, vb = (_blocks(dev[x], N) for x in ("q", "k", "v"))
    q, k, v = (as_float64(inp[x]) for x in ("q", "k", "v"))
    ro, rl = orc.naive_attention(q, k, v, N, causal, layout)
    for i in range(N):
        o = lse = None
        for j in orc.ring_order(i, N):
            oj, lj = ra.fwd_step(qb[i], kb[j], vb[j], N, i, j, causal, layout)
            if o is None:
                o, lse = oj, lj
            else:
                ra.merge(o, lse, oj, lj)
        torch.cuda.synchronize()
        sl = slice(i * c, (i + 1) * c)
        assert max_err(o.double().cpu().numpy(), ro[:, :, sl]) <= TOL["bf16"]["o"]
        assert max_err(lse.cpu().numpy(), rl[:, :, sl]) <= TOL["bf16"]["lse"]
        assert max_err(o.float().cpu().numpy(), o_full[:, :, sl].float().cpu().numpy()) <= TOL["bf16"]["o"]


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_chained_steps_32_blocks_float32_state(ra, layout):
    """32 ring hosts (the block count of the 131072-token workload), each
    chaining its 32 ring steps: with the running output kept in float32 and
    every bf16 partial folded into it (what ring.ring_forward does), the
    result matches the oracle at the forward's tolerance, and rounding the
    state to bf16 after every round is never more accurate."""
    B, H, N, c = 1, 2, 32, 128
    inp = make_inputs(B, H, N * c, 128, seed=33)
    dev = {x: inp[x].cuda() for x in ("q", "k", "v")}
    qb, kb, vb = (_blocks(dev[x], N) for x in ("q", "k", "v"))
    q, k, v = (as_float64(inp[x]) for x in ("q", "k", "v"))
    ro, rl = orc.naive_attention(q, k, v, N, True, layout)
    err32 = err16 = 0.0
    for i in range(N):
        o32 = torch.zeros((B, H, c, 128), dtype=torch.float32, device="cuda")
        l32 = torch.full((B, H, c), float("-inf"), dtype=torch.float32, device="cuda")
        o16 = l16 = None
        for j in orc.ring_order(i, N):
            if layout == "contiguous" and j > i:
                continue
            oj, lj = ra.fwd_step(qb[i], kb[j], vb[j], N, i, j, True, layout)
            ra.merge(o32, l32, oj, lj)
            if o16 is None:
                o16, l16 = oj.clone(), lj.clone()
            else:
                ra.merge(o16, l16, oj, lj)
        torch.cuda.synchronize()
        sl = slice(i * c, (i + 1) * c)
        err32 = max(err32, max_err(o32.double().cpu().numpy(), ro[:, :, sl]))
        err16 = max(err16, max_err(o16.double().cpu().numpy(), ro[:, :, sl]))
        assert max_err(l32.cpu().numpy(), rl[:, :, sl]) <= TOL["bf16"]["lse"]
    assert err32 <= TOL["bf16"]["o"], err32
    assert err32 <= err16, (err32, err16)


@pytest.mark.parametrize("layout,causal", [("contiguous", True), ("striped", True), ("striped", False)])
def test_fold_chain_32_blocks(ra, fwd_kernel, layout, causal):
    """ra_fwd_step_fold: every host folds its 32 rounds, in ring order, into a
    float32 state inside the forward epilogue; the state equals the oracle's
    rows at the forward's tolerance, and agrees with the step + merge chain."""
    B, H, N, c = 1, 2, 32, 128
    inp = make_inputs(B, H, N * c, 128, seed=34)
    dev = {x: inp[x].cuda() for x in ("q", "k", "v")}
    qb, kb, vb = (_blocks(dev[x], N) for x in ("q", "k", "v"))
    q, k, v = (as_float64(inp[x]) for x in ("q", "k", "v"))
    ro, rl = orc.naive_attention(q, k, v, N, causal, layout)
    for i in range(N):
        o = torch.full((B, H, c, 128), float("nan"), dtype=torch.float32, device="cuda")   # never read while empty
        lse = torch.full((B, H, c), float("-inf"), dtype=torch.float32, device="cuda")
        o2 = torch.zeros_like(o)
        l2 = lse.clone()
        for j in orc.ring_order(i, N):
            ra.fwd_step_fold(qb[i], kb[j], vb[j], N, i, j, causal, layout, o_acc=o, lse_acc=lse)
            oj, lj = ra.fwd_step(qb[i], kb[j], vb[j], N, i, j, causal, layout)
            ra.merge(o2, l2, oj, lj)
        torch.cuda.synchronize()
        ra.check_device_status()
        sl = slice(i * c, (i + 1) * c)
        assert max_err(o.double().cpu().numpy(), ro[:, :, sl]) <= TOL["bf16"]["o"], i
        assert max_err(lse.cpu().numpy(), rl[:, :, sl]) <= TOL["bf16"]["lse"], i
        assert max_err(o.cpu().numpy(), o2.cpu().numpy()) <= TOL["bf16"]["o"], i


def test_fold_leaves_unseen_rows_and_empty_rounds_alone(ra):
    """A contiguous causal round j > i folds nothing; a striped round j > i
    hides each query's own row, so row 0 of block i sees no key of block j and
    its state stays bit-identical."""
    B, H, N, c = 1, 1, 4, 128
    inp = make_inputs(B, H, N * c, 128, seed=35)
    qb, kb, vb = (_blocks(inp[x].cuda(), N) for x in ("q", "k", "v"))
    g = torch.Generator().manual_seed(3)
    o = torch.randn((B, H, c, 128), generator=g).cuda()
    lse = torch.randn((B, H, c), generator=g).cuda()
    o0, l0 = o.clone(), lse.clone()
    ra.fwd_step_fold(qb[1], kb[3], vb[3], N, 1, 3, True, "contiguous", o_acc=o, lse_acc=lse)
    torch.cuda.synchronize()
    assert torch.equal(o, o0) and torch.equal(lse, l0)
    ra.fwd_step_fold(qb[1], kb[3], vb[3], N, 1, 3, True, "striped", o_acc=o, lse_acc=lse)
    torch.cuda.synchronize()
    assert torch.equal(o[0, 0, 0], o0[0, 0, 0]) and torch.equal(lse[0, 0, 0], l0[0, 0, 0])
    assert not torch.equal(o[0, 0, 1:], o0[0, 0, 1:])


def _grad_tol(ref):
    return 2e-2 * max(1.0, float(np.abs(ref).max()))


def _bwd_inputs(B, H, N, c, seed):
    inp = make_inputs(B, H, N * c, 128, seed=seed, with_grad=True)
    q, k, v, do = (as_float64(inp[x]) for x in ("q", "k", "v", "do"))
    return inp, q, k, v, do


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_bwd_step_pairs_match_oracle(ra, layout):
    """One round (query block i, KV block j) added into zeroed float32
    accumulators equals the oracle's pair contributions (O, LSE: the oracle's
    final forward state, rounded as the GPU would hold them)."""
    B, H, N, c = 1, 2, 4, 200
    inp, q, k, v, do = _bwd_inputs(B, H, N, c, seed=33)
    ro, rl = orc.naive_attention(q, k, v, N, True, layout)
    o_dev = torch.from_numpy(ro).to(torch.bfloat16)
    o64 = o_dev.double().numpy()
    l_dev = torch.from_numpy(rl).float()
    l64 = l_dev.double().numpy()
    blk = lambda t, b: t[:, :, b * c:(b + 1) * c].contiguous().cuda()
    for i, j in [(2, 2), (2, 0), (0, 3), (3, 1), (1, 2)]:
        dq, dk, dv = (torch.zeros(B, H, c, 128, device="cuda") for _ in range(3))
        ra.bwd_step(blk(inp["q"], i), blk(inp["k"], j), blk(inp["v"], j), blk(o_dev, i),
                    l_dev[:, :, i * c:(i + 1) * c].contiguous().cuda(), blk(inp["do"], i), dq, dk, dv, N, i, j,
                    True, layout)
        torch.cuda.synchronize()
        ra.check_device_status()
        for h in range(H):
            rq, rk, rv = orc.block_pair_bwd(q[0, h], k[0, h], v[0, h], o64[0, h], l64[0, h], do[0, h], i, j, N,
                                            True, layout)
            for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
                assert max_err(g[0, h].cpu().numpy(), r) <= _grad_tol(r), (i, j, h, name)


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_bwd_steps_chained_equal_full_backward(ra, layout):
    """Every host's N rounds, accumulated in float32 as a ring would (dQ_i at
    its host, dK_j/dV_j travelling), give the full gradient of the oracle and
    agree with the fused ra_bwd."""
    B, H, N, c = 1, 2, 4, 256
    inp, q, k, v, do = _bwd_inputs(B, H, N, c, seed=34)
    dev = {x: inp[x].cuda() for x in ("q", "k", "v", "do")}
    o, lse = ra.fwd(dev["q"], dev["k"], dev["v"], N, True, layout)
    fq, fk, fv = ra.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], N, True, layout)
    blk = lambda t, b: t[:, :, b * c:(b + 1) * c].contiguous()
    dq = [torch.zeros(B, H, c, 128, device="cuda") for _ in range(N)]
    dk = [torch.zeros(B, H, c, 128, device="cuda") for _ in range(N)]
    dv = [torch.zeros(B, H, c, 128, device="cuda") for _ in range(N)]
    for i in range(N):
        for j in orc.ring_order(i, N):
            ra.bwd_step(blk(dev["q"], i), blk(dev["k"], j), blk(dev["v"], j), blk(o, i), blk(lse, i),
                        blk(dev["do"], i), dq[i], dk[j], dv[j], N, i, j, True, layout)
    torch.cuda.synchronize()
    ra.check_device_status()
    gq, gk, gv = (torch.cat(x, dim=2).cpu().numpy() for x in (dq, dk, dv))
    o64 = o.double().cpu().numpy()
    l64 = lse.double().cpu().numpy()
    rq, rk, rv = orc.attention_bwd(q, k, v, o64, l64, do, N, True, layout)
    for name, g, r, f in (("dq", gq, rq, fq), ("dk", gk, rk, fk), ("dv", gv, rv, fv)):
        assert max_err(g, r) <= _grad_tol(r), name
        assert max_err(g, f.float().cpu().numpy()) <= _grad_tol(r), name
