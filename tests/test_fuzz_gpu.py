"""Seeded random-shape parity sweep on the GPU: forward, backward, decode and
the feedforward against the oracle, over shapes drawn at random (ragged
blocks, several heads and batches, both layouts, causal and not, caches
shorter than the ring, ragged feedforward blocks).  Sizes stay small so the
float64 oracle checks every element."""
import numpy as np
import pytest
import torch

import oracle as orc
from gpu_helpers import TOL, max_err
from ring_attention_fwd_gb300.inputs import as_float64, make_decode_inputs, make_ffn_inputs, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import ring_attention_fwd_gb300 as ra
    assert torch.cuda.is_available()
    return ra


def _attn_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        N = int(rng.integers(1, 9))
        c = int(rng.integers(1, 300))
        cases.append(dict(B=int(rng.integers(1, 3)), H=int(rng.integers(1, 4)), N=N, S=N * c,
                          causal=bool(rng.random() < 0.7), layout=["contiguous", "striped"][int(rng.integers(0, 2))],
                          seed=int(rng.integers(0, 1 << 30))))
    return cases


@pytest.mark.parametrize("case", _attn_cases(12, 2024), ids=lambda c: f"B{c['B']}H{c['H']}S{c['S']}N{c['N']}"
                         f"{'c' if c['causal'] else 'n'}{c['layout'][0]}")
def test_fuzz_forward_backward(ra, fwd_kernel, case):
    B, H, S, N = case["B"], case["H"], case["S"], case["N"]
    inp = make_inputs(B, H, S, 128, seed=case["seed"], with_grad=True)
    dev = {k: v.cuda() for k, v in inp.items()}
    o, lse = ra.fwd(dev["q"], dev["k"], dev["v"], N, case["causal"], case["layout"])
    torch.cuda.synchronize()
    ra.check_device_status()
    q, k, v, do = (as_float64(inp[x]) for x in ("q", "k", "v", "do"))
    ro, rl = orc.naive_attention(q, k, v, N, case["causal"], case["layout"])
    assert max_err(o.float().cpu().numpy(), ro) <= TOL["bf16"]["o"]
    assert max_err(lse.cpu().numpy(), rl) <= TOL["bf16"]["lse"]
    # the backward on the saved state as stored (the oracle's O rounded to
    # bf16, LSE to float32); the expected gradient uses that same state
    o_bf = torch.from_numpy(ro).to(torch.bfloat16)
    l_f = torch.from_numpy(rl).float()
    dq, dk, dv = ra.bwd(dev["q"], dev["k"], dev["v"], o_bf.cuda(), l_f.cuda(), dev["do"], N, case["causal"],
                        case["layout"])
    torch.cuda.synchronize()
    ra.check_device_status()
    rq, rk, rv = orc.attention_bwd(q, k, v, o_bf.double().numpy(), l_f.double().numpy(), do, N,
                                   case["causal"], case["layout"])
    for g, r in ((dq, rq), (dk, rk), (dv, rv)):
        g = g.double().cpu().numpy()
        assert max_err(g, r) <= 2e-2 * max(1.0, float(np.abs(r).max()))
        assert np.linalg.norm(g - r) <= 1e-2 * max(np.linalg.norm(r), 1e-30)


def _decode_cases(n, seed):
    rng = np.random.default_rng(seed)
    return [dict(B=int(rng.integers(1, 3)), H=int(rng.integers(1, 5)), S=int(rng.integers(1, 9000)),
                 N=int(rng.integers(1, 40)), seed=int(rng.integers(0, 1 << 30))) for _ in range(n)]


@pytest.mark.parametrize("case", _decode_cases(10, 2025), ids=lambda c: f"B{c['B']}H{c['H']}S{c['S']}N{c['N']}")
def test_fuzz_decode(ra, case):
    inp = make_decode_inputs(case["B"], case["H"], case["S"], 128, seed=case["seed"])
    o, lse = ra.decode(*(inp[x].cuda() for x in ("q", "k", "v")), case["N"])
    torch.cuda.synchronize()
    ra.check_device_status()
    ro, rl = orc.decode_batch(*(as_float64(inp[x]) for x in ("q", "k", "v")), case["N"])
    assert max_err(o.float().cpu().numpy(), ro) <= TOL["bf16"]["o"]
    assert max_err(lse.cpu().numpy(), rl) <= TOL["bf16"]["lse"]


def _ffn_cases(n, seed):
    rng = np.random.default_rng(seed)
    return [dict(T=int(rng.integers(1, 700)), h=256 * int(rng.integers(1, 3)), f=128 * int(rng.integers(1, 6)),
                 c=int(rng.integers(1, 400)), seed=int(rng.integers(0, 1 << 30))) for _ in range(n)]


@pytest.mark.parametrize("case", _ffn_cases(8, 2026), ids=lambda c: f"T{c['T']}h{c['h']}f{c['f']}c{c['c']}")
def test_fuzz_ffn(ra, case):
    inp = make_ffn_inputs(case["T"], case["h"], case["f"], seed=case["seed"])
    y = ra.ffn(*(inp[x].cuda() for x in ("x", "w1", "w3", "w2")), case["c"])
    torch.cuda.synchronize()
    ra.check_device_status()
    ref = orc.blockwise_ffn(*(as_float64(inp[x]) for x in ("x", "w1", "w3", "w2")), case["c"])
    g = y.double().cpu().numpy()
    assert max_err(g, ref) <= 2e-2 * max(1.0, float(np.abs(ref).max()))
    assert np.linalg.norm(g - ref) <= 1e-2 * max(np.linalg.norm(ref), 1e-30)
