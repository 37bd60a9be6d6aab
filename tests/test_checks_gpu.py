"""The bounds-checked build (libringattn_checked.so) on the GPU.

Every global index of the epilogues, merge, preprocess, decode, feedforward
and float32 kernels, and every TMA box start, is checked against its tensor's
extent in that build; an access out of bounds is skipped and recorded.  Small
odd shapes (one token per block, ragged tiles, B > 1, empty decode blocks,
unaligned merge rows) go through every entry point, and each call must leave
zero violations and match the oracle.  The same build counts the forward's
O rescales, which shows the correction branch of the online softmax running
on the peaked inputs at least as often as the inputs force it
(``tests/peaked.py``).
"""
import numpy as np
import pytest
import torch

import oracle as orc
from gpu_helpers import TOL, max_err
from peaked import PEAKED_CASES, rescale_events, tile_maxima
from ring_attention_fwd_gb300.inputs import (as_float64, make_decode_inputs, make_ffn_inputs, make_inputs,
                                             make_peaked_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import ring_attention_fwd_gb300 as ra
    assert torch.cuda.is_available()
    ra.use_checked_build(True)
    assert ra.version().endswith("checked")
    ra.read_checks()            # start from a clear record
    yield ra
    ra.use_checked_build(False)


def _clean(ra, what, need_boxes=False):
    r = ra.read_checks()
    assert r["violations"] == 0, f"{what}: out-of-bounds access {r}"
    assert r["accesses_checked"] > 0, f"{what}: nothing was checked {r}"
    if need_boxes:
        assert r["tma_boxes_checked"] > 0, f"{what}: no TMA box was checked {r}"
    return r


def _grad_close(g, ref, name):
    scale = max(1.0, float(np.abs(ref).max()))
    assert max_err(g, ref) <= 2e-2 * scale, name
    assert np.linalg.norm(g - ref) <= 1e-2 * max(np.linalg.norm(ref), 1e-30), name


@pytest.mark.parametrize("B,H,S,N,causal,layout", [
    (1, 2, 8, 8, True, "contiguous"),       # c = 1
    (1, 1, 128, 8, True, "striped"),        # c = 16: the unit's second query tile starts past S
    (1, 2, 600, 3, True, "contiguous"),     # c = 200: ragged tiles
    (1, 1, 1000, 5, True, "striped"),
    (3, 2, 768, 3, True, "striped"),        # B > 1
    (2, 1, 1024, 4, False, "contiguous"),
])
def test_checked_forward_backward(ra, fwd_kernel, B, H, S, N, causal, layout):
    inp = make_inputs(B, H, S, 128, seed=700 + S + N, with_grad=True)
    q, k, v, do = (as_float64(inp[x]) for x in ("q", "k", "v", "do"))
    dev = {x: inp[x].cuda() for x in ("q", "k", "v", "do")}
    o, lse = ra.fwd(dev["q"], dev["k"], dev["v"], N, causal, layout)
    _clean(ra, "forward", need_boxes=True)
    ro, rl = orc.naive_attention(q, k, v, N, causal, layout)
    assert max_err(o.double().cpu().numpy(), ro) <= TOL["bf16"]["o"]
    assert max_err(lse.double().cpu().numpy(), rl) <= TOL["bf16"]["lse"]
    # the backward on the oracle's saved state (O in bf16, LSE in float32)
    o_bf = torch.from_numpy(ro).to(torch.bfloat16)
    l_f = torch.from_numpy(rl).float()
    dq, dk, dv = ra.bwd(dev["q"], dev["k"], dev["v"], o_bf.cuda(), l_f.cuda(), dev["do"], N, causal, layout)
    _clean(ra, "backward", need_boxes=True)
    rq, rk, rv = orc.attention_bwd(q, k, v, o_bf.double().numpy(), l_f.double().numpy(), do, N, causal, layout)
    for name, g, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        _grad_close(g.double().cpu().numpy(), r, name)


@pytest.mark.parametrize("B,H,S,D,N,causal,layout", [
    (1, 1, 256, 64, 4, False, "contiguous"),
    (1, 2, 300, 32, 3, True, "striped"),
    (1, 1, 130, 8, 5, True, "striped"),
])
def test_checked_forward_f32(ra, B, H, S, D, N, causal, layout):
    inp = make_inputs(B, H, S, D, seed=800 + S, dtype="f32")
    o, lse = ra.fwd(*(inp[x].cuda() for x in ("q", "k", "v")), N, causal, layout)
    _clean(ra, "f32 forward")
    ro, rl = orc.naive_attention(*(as_float64(inp[x]) for x in ("q", "k", "v")), N, causal, layout)
    assert max_err(o.double().cpu().numpy(), ro) <= TOL["f32"]["o"]
    assert max_err(lse.double().cpu().numpy(), rl) <= TOL["f32"]["lse"]


def test_checked_ring_steps_and_merge(ra):
    B, H, S, N, layout = 1, 2, 1024, 4, "striped"
    c = S // N
    inp = make_inputs(B, H, S, 128, seed=901, with_grad=True)
    q, k, v = (as_float64(inp[x]) for x in ("q", "k", "v"))
    blk = lambda t, b: t[:, :, b * c:(b + 1) * c].contiguous().cuda()
    for i, j in ((2, 2), (1, 3), (3, 0)):                 # diagonal, striped j > i, j < i
        o, lse = ra.fwd_step(blk(inp["q"], i), blk(inp["k"], j), blk(inp["v"], j), N, i, j, True, layout)
        _clean(ra, f"fwd_step {i},{j}", need_boxes=True)
        for h in range(H):
            ro, rl = orc.block_pair_attention(q[0, h], k[0, h], v[0, h], i, j, N, True, layout)
            assert max_err(o[0, h].double().cpu().numpy(), ro) <= TOL["bf16"]["o"]
            assert max_err(lse[0, h].double().cpu().numpy(), rl) <= TOL["bf16"]["lse"]
        o_acc = torch.zeros((B, H, c, 128), dtype=torch.float32, device="cuda")
        l_acc = torch.full((B, H, c), float("-inf"), dtype=torch.float32, device="cuda")
        ra.fwd_step_fold(blk(inp["q"], i), blk(inp["k"], j), blk(inp["v"], j), N, i, j, True, layout, o_acc=o_acc,
                         lse_acc=l_acc)
        _clean(ra, f"fwd_step_fold {i},{j}", need_boxes=True)
        for h in range(H):
            ro, rl = orc.block_pair_attention(q[0, h], k[0, h], v[0, h], i, j, N, True, layout)
            assert max_err(o_acc[0, h].double().cpu().numpy(), ro) <= TOL["bf16"]["o"]
            assert max_err(l_acc[0, h].double().cpu().numpy(), rl) <= TOL["bf16"]["lse"]
        acc = [torch.zeros((B, H, c, 128), dtype=torch.float32, device="cuda") for _ in range(3)]
        o_full, lse_full = ra.fwd(*(inp[x].cuda() for x in ("q", "k", "v")), N, True, layout)
        ra.read_checks()
        ra.bwd_step(blk(inp["q"], i), blk(inp["k"], j), blk(inp["v"], j), o_full[:, :, i * c:(i + 1) * c].contiguous(),
                    lse_full[:, :, i * c:(i + 1) * c].contiguous(), blk(inp["do"], i), *acc, N, i, j, True, layout)
        _clean(ra, f"bwd_step {i},{j}", need_boxes=True)
    for dtype, D in ((torch.bfloat16, 128), (torch.bfloat16, 100), (torch.float32, 64), (torch.float32, 6)):
        rows = 257
        g = torch.Generator().manual_seed(D)
        oa, ob = (torch.randn(rows, D, generator=g).to(dtype) for _ in range(2))
        la, lb = (torch.randn(rows, generator=g) * 3 for _ in range(2))
        la[::7] = -float("inf")
        lb[::5] = -float("inf")
        ga, gla = oa.cuda(), la.cuda()
        ra.merge(ga, gla, ob.cuda(), lb.cuda())
        _clean(ra, f"merge {dtype} D={D}")
        ro, rl = orc.lse_merge(oa.double().numpy(), la.double().numpy(), ob.double().numpy(), lb.double().numpy())
        tol = 2e-2 if dtype == torch.bfloat16 else 1e-5
        assert max_err(ga.double().cpu().numpy(), ro) <= tol and max_err(gla.double().cpu().numpy(), rl) <= 1e-5


@pytest.mark.parametrize("B,H,S,N", [(1, 2, 3000, 4), (2, 1, 100, 7), (1, 1, 64, 1)])
def test_checked_decode(ra, B, H, S, N):
    inp = make_decode_inputs(B, H, S, 128, seed=950 + S)
    o, lse = ra.decode(*(inp[x].cuda() for x in ("q", "k", "v")), N)
    _clean(ra, "decode")
    for b in range(B):
        for h in range(H):
            ro, rl = orc.ring_decode(*(as_float64(inp[x][b, h]) for x in ("q", "k", "v")), N)
            assert max_err(o[b, h].double().cpu().numpy(), ro) <= 2e-2
            assert abs(float(lse[b, h]) - rl) <= 1e-3


def test_checked_feedforward(ra):
    inp = make_ffn_inputs(300, 256, 384, seed=13)
    y = ra.ffn(*(inp[x].cuda() for x in ("x", "w1", "w3", "w2")), 128)
    _clean(ra, "feedforward", need_boxes=True)
    ref = orc.blockwise_ffn(*(as_float64(inp[x]) for x in ("x", "w1", "w3", "w2")), 128)
    assert max_err(y.double().cpu().numpy(), ref) <= 2e-2 * max(1.0, float(np.abs(ref).max()))


@pytest.mark.parametrize("B,H,S,N,causal,layout,mode", PEAKED_CASES)
def test_checked_counts_forced_rescales(ra, fwd_kernel, B, H, S, N, causal, layout, mode):
    """Device count of rows whose O was rescaled >= what the inputs force."""
    inp = make_peaked_inputs(B, H, S, N, seed=500 + S + N, mode=mode)
    q, k = as_float64(inp["q"]), as_float64(inp["k"])
    forced = sum(int(rescale_events(tile_maxima(q[b, h], k[b, h], N, causal, layout)).sum())
                 for b in range(B) for h in range(H))
    o, lse = ra.fwd(inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(), N, causal, layout)
    r = _clean(ra, "peaked forward", need_boxes=True)
    assert forced > 0
    assert r["fwd_rescale_rows"] >= forced, (r, forced)
    assert r["fwd_rescale_passes"] > 0, r
    ro, rl = orc.naive_attention(q, k, as_float64(inp["v"]), N, causal, layout)
    assert max_err(o.double().cpu().numpy(), ro) <= TOL["bf16"]["o"]
    assert max_err(lse.double().cpu().numpy(), rl) <= TOL["bf16"]["lse"]


def test_checked_build_full_size_workloads(ra):
    """The largest extents the library meets in the specified workloads, with
    every index and TMA box checked: the 131072-token forward and backward
    (32 heads, 32 blocks), the 262144-token ring decode and the 7B-shaped
    feedforward.  Zero violations, finite outputs (values are checked against
    the oracle by the default build's tests)."""
    from ring_attention_fwd_gb300.inputs import DECODE_WORKLOADS, FFN_WORKLOADS, WORKLOADS
    w = WORKLOADS["long_128k"]
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    B, H, S, N = w["B"], w["H"], w["S"], w["N"]
    q, k, v, do = (torch.randn((B, H, S, 128), device="cuda", generator=g).mul_(0.5).to(torch.bfloat16)
                   for _ in range(4))
    o, lse = ra.fwd(q, k, v, N, True, "contiguous")
    r = _clean(ra, "131072-token forward", need_boxes=True)
    assert bool(torch.isfinite(lse).all()) and bool(torch.isfinite(o.float()).all())
    dq, dk, dv = ra.bwd(q, k, v, o, lse, do, N, True, "contiguous")
    _clean(ra, "131072-token backward", need_boxes=True)
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t.float()).all())
    del q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()
    d = DECODE_WORKLOADS["decode_256k"]
    qd = torch.randn((d["B"], d["H"], 128), device="cuda", generator=g).to(torch.bfloat16)
    kc, vc = (torch.randn((d["B"], d["H"], d["S"], 128), device="cuda", generator=g).to(torch.bfloat16)
              for _ in range(2))
    od, ld = ra.decode(qd, kc, vc, d["N"])
    _clean(ra, "262144-token decode")
    assert bool(torch.isfinite(ld).all()) and bool(torch.isfinite(od.float()).all())
    del kc, vc
    f = FFN_WORKLOADS["ffn_7b"]
    x = torch.randn((f["T"], f["h"]), device="cuda", generator=g).to(torch.bfloat16)
    w1, w3 = (torch.randn((f["f"], f["h"]), device="cuda", generator=g).mul_(f["h"] ** -0.5).to(torch.bfloat16)
              for _ in range(2))
    w2 = torch.randn((f["h"], f["f"]), device="cuda", generator=g).mul_(f["f"] ** -0.5).to(torch.bfloat16)
    y = ra.ffn(x, w1, w3, w2, f["block_rows"])
    _clean(ra, "7B-shaped feedforward", need_boxes=True)
    assert bool(torch.isfinite(y.float()).all())
