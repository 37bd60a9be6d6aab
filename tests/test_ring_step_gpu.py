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
def test_single_pairs_match_oracle(ra, layout, dtype):
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
