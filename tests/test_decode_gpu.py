"""Ring decode on the GPU (ra_decode through the C ABI) against the oracle:
small ragged caches element by element, the per-host step chained with
ra_merge, and the full 256K-token workload on every head."""
import numpy as np
import pytest
import torch

import oracle as orc
from gpu_helpers import TOL, max_err
from ring_attention_fwd_gb300.inputs import DECODE_WORKLOADS, make_decode_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import ring_attention_fwd_gb300 as ra
    assert torch.cuda.is_available()
    return ra


def _f64(t):
    return t.to(torch.float64).numpy()


def _check(ra, inp, N, tol=TOL["bf16"]):
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    o, lse = ra.decode(q, k, v, N)
    torch.cuda.synchronize()
    ra.check_device_status()
    go, gl = o.float().cpu().numpy(), lse.cpu().numpy()
    B, H = inp["q"].shape[:2]
    for b in range(B):          # one head at a time: a 256K-row cache is 0.5 GB in float64
        for h in range(H):
            ro, rl = orc.ring_decode(_f64(inp["q"][b, h]), _f64(inp["k"][b, h]), _f64(inp["v"][b, h]), N)
            assert max_err(go[b, h], ro) <= tol["o"], (b, h)
            assert max_err(gl[b, h], rl) <= tol["lse"], (b, h)
    return o, lse


@pytest.mark.parametrize("B,H,S,N", [(2, 3, 1, 1), (2, 3, 63, 1), (1, 2, 64, 3), (2, 3, 1000, 3),
                                     (1, 2, 4097, 8), (1, 2, 5, 9), (1, 4, 20000, 7), (3, 1, 777, 777)])
def test_decode_matches_oracle(ra, B, H, S, N):
    _check(ra, make_decode_inputs(B, H, S, 128, seed=S + N), N)


def test_decode_peaked_scores(ra):
    """Scaled inputs make a few keys dominate (scores up to ~100): the running
    maximum and the merges must keep the result exact."""
    _check(ra, make_decode_inputs(2, 2, 3000, 128, seed=7, scale=3.0), 5)


def test_decode_step_chain_equals_ring(ra):
    """Each ring block decoded alone (N = 1 on its segment) and merged in the
    ring order of the last block's host equals the whole-cache call."""
    B, H, S, N = 1, 3, 5000, 4
    inp = make_decode_inputs(B, H, S, 128, seed=9)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    o_full, l_full = ra.decode(q, k, v, N)
    blocks = orc.decode_blocks(S, N)
    o = lse = None
    for j in orc.ring_order(N - 1, N):
        a, b = blocks[j]
        oj, lj = ra.decode(q, k[:, :, a:b].contiguous(), v[:, :, a:b].contiguous(), 1)
        if o is None:
            o, lse = oj, lj
        else:
            ra.merge(o, lse, oj, lj)
    torch.cuda.synchronize()
    ro, rl = orc.decode_batch(_f64(inp["q"]), _f64(inp["k"]), _f64(inp["v"]), N)
    assert max_err(o.float().cpu().numpy(), ro) <= TOL["bf16"]["o"]
    assert max_err(lse.cpu().numpy(), rl) <= TOL["bf16"]["lse"]
    assert max_err(o.float().cpu().numpy(), o_full.float().cpu().numpy()) <= TOL["bf16"]["o"]


def test_decode_full_workload_every_head(ra):
    w = DECODE_WORKLOADS["decode_256k"]
    inp = make_decode_inputs(w["B"], w["H"], w["S"], w["D"], w["seed"], scale=w["scale"])
    o, lse = _check(ra, inp, w["N"])
    assert bool(torch.isfinite(o.float()).all()) and bool(torch.isfinite(lse).all())


def test_decode_kernel_timing_records(ra):
    inp = make_decode_inputs(1, 2, 3000, 128, seed=3)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    ra.set_kernel_timing(True)
    try:
        ra.decode(q, k, v, 4)
        names = [n for n, ms in ra.kernel_times() if ms >= 0]
    finally:
        ra.set_kernel_timing(False)
    assert names == ["decode_split", "decode_combine"]
