"""Forward parity: CUDA path (through the C ABI) vs the CPU oracle."""
import numpy as np
import pytest
import torch

from gpu_helpers import TOL, fwd_full_check, pooled_fwd_check, to_cuda, workload_inputs
from ring_attention_fwd_gb300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import ring_attention_fwd_gb300 as ra
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return ra


def test_tiny_f32_workload(ra):
    w = WORKLOADS["tiny_f32"]
    eo, el = fwd_full_check(ra, workload_inputs(w), w["N"], w["causal"], w["layout"], "f32")
    assert eo <= TOL["f32"]["o"] and el <= TOL["f32"]["lse"], (eo, el)


@pytest.mark.parametrize("B,H,S,D,N,causal,layout", [
    (1, 1, 256, 64, 4, True, "contiguous"),
    (1, 2, 300, 32, 3, True, "striped"),        # c = 100: ragged tiles
    (2, 1, 192, 128, 1, False, "contiguous"),
    (1, 1, 130, 8, 5, True, "striped"),          # c = 26
])
def test_f32_shapes(ra, B, H, S, D, N, causal, layout):
    inp = make_inputs(B, H, S, D, seed=100 + S, dtype="f32")
    eo, el = fwd_full_check(ra, inp, N, causal, layout, "f32")
    assert eo <= TOL["f32"]["o"] and el <= TOL["f32"]["lse"], (eo, el)


BF16_CASES = [
    (1, 1, 256, 1, True, "contiguous"),     # one block
    (1, 2, 512, 2, True, "contiguous"),
    (1, 2, 512, 2, True, "striped"),
    (2, 1, 1024, 4, False, "contiguous"),
    (1, 1, 384, 3, True, "striped"),        # c = 128: unit taller than a block
    (1, 2, 600, 3, True, "contiguous"),     # c = 200: ragged KV tile and unit
    (1, 1, 1000, 5, True, "striped"),       # c = 200, striped
    (1, 1, 128, 8, True, "striped"),        # c = 16: every tile ragged
    (1, 3, 2048, 4, True, "striped"),
    (1, 2, 4096, 8, False, "striped"),
    (3, 2, 1536, 6, True, "contiguous"),    # c = 256
    (1, 2, 8, 8, True, "contiguous"),       # c = 1: one token per block
    (2, 1, 16, 16, True, "striped"),        # c = 1, striped
]


@pytest.mark.parametrize("B,H,S,N,causal,layout", BF16_CASES)
def test_bf16_shapes(ra, fwd_kernel, B, H, S, N, causal, layout):
    inp = make_inputs(B, H, S, 128, seed=200 + S + N, dtype="bf16")
    eo, el = fwd_full_check(ra, inp, N, causal, layout, "bf16")
    assert eo <= TOL["bf16"]["o"] and el <= TOL["bf16"]["lse"], (eo, el)


def test_bf16_deterministic(ra):
    inp = {k: v.cuda() for k, v in make_inputs(1, 4, 2048, 128, seed=7).items()}
    o1, l1 = ra.fwd(inp["q"], inp["k"], inp["v"], 4, True, "striped")
    o2, l2 = ra.fwd(inp["q"], inp["k"], inp["v"], 4, True, "striped")
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_causal_8k_workload_full(ra):
    w = WORKLOADS["causal_8k"]
    eo, el = fwd_full_check(ra, workload_inputs(w), w["N"], w["causal"], w["layout"], "bf16")
    assert eo <= TOL["bf16"]["o"] and el <= TOL["bf16"]["lse"], (eo, el)


def _run_fwd(ra, inp, N, causal, layout):
    dev = to_cuda({x: inp[x] for x in ("q", "k", "v")})
    o, lse = ra.fwd(dev["q"], dev["k"], dev["v"], N, causal, layout)
    torch.cuda.synchronize()
    ra.check_device_status()
    assert bool(torch.isfinite(lse).all()), "non-finite LSE"
    assert bool(torch.isfinite(o.float()).all()), "non-finite O"
    return o, lse


def _every_head(inp):
    B, H = inp["q"].shape[:2]
    return [(b, h) for b in range(B) for h in range(H)]


@pytest.mark.parametrize("layout", ["striped", "contiguous"])
def test_balance_32k_workload_every_head(ra, layout):
    """The 32768-token workload in both layouts: sampled rows (every block
    boundary and random rows) of all 16 heads against the oracle."""
    w = WORKLOADS["balance_32k"]
    inp = workload_inputs(w)
    o, lse = _run_fwd(ra, inp, w["N"], w["causal"], layout)
    eo, el = pooled_fwd_check(inp, o, lse, w["N"], w["causal"], layout, _every_head(inp), 128, 3)
    assert eo <= TOL["bf16"]["o"] and el <= TOL["bf16"]["lse"], (eo, el)


def test_long_128k_workload_sampled(ra):
    """The 131072-token workload, in the launch configuration the benchmark
    times; sampled rows of every head against the oracle.  The call must not
    allocate device memory beyond its outputs (working set of the method:
    a constant number of blocks per virtual host, here none extra)."""
    w = WORKLOADS["long_128k"]
    inp = workload_inputs(w)
    dev = {k: v.cuda() for k, v in inp.items()}
    B, H, S, D = inp["q"].shape
    o = torch.empty_like(dev["q"])
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    ra.fwd(dev["q"], dev["k"], dev["v"], w["N"], True, "contiguous", o=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.cuda.max_memory_allocated() == base
    del dev, o, lse
    o, lse = _run_fwd(ra, inp, w["N"], w["causal"], w["layout"])
    eo, el = pooled_fwd_check(inp, o, lse, w["N"], w["causal"], w["layout"], _every_head(inp), 64, 4)
    assert eo <= TOL["bf16"]["o"] and el <= TOL["bf16"]["lse"], (eo, el)


def test_fwdbwd_64k_workload_forward_every_head(ra):
    w = WORKLOADS["fwdbwd_64k"]
    inp = workload_inputs(w)
    o, lse = _run_fwd(ra, inp, w["N"], w["causal"], w["layout"])
    eo, el = pooled_fwd_check(inp, o, lse, w["N"], w["causal"], w["layout"], _every_head(inp), 64, 5)
    assert eo <= TOL["bf16"]["o"] and el <= TOL["bf16"]["lse"], (eo, el)


def test_per_device_timing_buffer(ra, fwd_kernel):
    """Timing hooks: every visited (virtual host, ring step) gets time, every
    skipped one (contiguous causal, j > i) none."""
    N = 4
    inp = {k: v.cuda() for k, v in make_inputs(1, 2, 2048, 128, seed=9).items()}
    buf = torch.zeros(N * N, dtype=torch.int64, device="cuda")
    ra.set_timing_buffer(buf)
    try:
        ra.fwd(inp["q"], inp["k"], inp["v"], N, True, "contiguous")
        torch.cuda.synchronize()
    finally:
        ra.set_timing_buffer(None)
    t = buf.view(N, N).cpu().numpy()
    for i in range(N):
        for s in range(N):
            j = (i - s) % N
            assert (t[i, s] > 0) == (j <= i), (i, s, t)


PAIR_EQUAL_CASES = [
    (1, 2, 1024, 2, True, "contiguous", 1.0),
    (1, 3, 4000, 4, True, "striped", 1.0),      # c = 1000: ragged units and KV tiles
    (2, 2, 2000, 2, False, "contiguous", 1.0),
    (1, 2, 200, 4, True, "contiguous", 1.0),     # c = 50: a pair unit holds all of a block
    (1, 4, 32768, 8, True, "contiguous", 4.0),   # peaked scores: O rescaled mid-sweep
    (1, 32, 131072, 32, True, "contiguous", 0.5),  # the 131072-token workload's shape
]


@pytest.mark.parametrize("B,H,S,N,causal,layout,scale", PAIR_EQUAL_CASES)
def test_pair_and_single_kernels_bit_identical(ra, B, H, S, N, causal, layout, scale):
    """The SM-pair forward issues the same MMAs over the same tiles, in the
    same order, and runs the same per-row softmax code as the one-CTA-per-SM
    kernel: O and LSE agree bit for bit, including rows beyond a ragged block
    and rows that rescale."""
    g = torch.Generator(device="cuda")
    g.manual_seed(S + N)
    q, k, v = (torch.randn((B, H, S, 128), device="cuda", generator=g).mul_(scale).to(torch.bfloat16)
               for _ in range(3))
    out = {}
    try:
        for kind in ("single", "pair"):
            ra.set_fwd_kernel(kind)
            out[kind] = ra.fwd(q, k, v, N, causal, layout)
            torch.cuda.synchronize()
            ra.check_device_status()
    finally:
        ra.set_fwd_kernel("single")
    assert torch.equal(out["single"][0], out["pair"][0])
    assert torch.equal(out["single"][1], out["pair"][1])


def test_kernel_selection_and_names(ra):
    """The timing records name the forward kernel that ran."""
    inp = {x: torch.randn((1, 2, 1024, 128), device="cuda").to(torch.bfloat16) for x in "qkv"}
    names = []
    for kind in ("pair", "single"):
        ra.set_fwd_kernel(kind)
        ra.set_kernel_timing(True)
        try:
            ra.fwd(inp["q"], inp["k"], inp["v"], 4, True, "contiguous")
            names.append([n for n, _ in ra.kernel_times()])
        finally:
            ra.set_kernel_timing(False)
            ra.set_fwd_kernel("single")
    assert names == [["fwd_pair"], ["fwd"]]


def test_kernel_timing_records(ra):
    """Opt-in kernel timing: one record per kernel of every timed call, in
    order, with positive durations; nothing is recorded once it is off."""
    inp = {k: v.cuda() for k, v in make_inputs(1, 2, 1024, 128, seed=12, with_grad=True).items()}
    ra.set_kernel_timing(True)
    try:
        o, lse = ra.fwd(inp["q"], inp["k"], inp["v"], 4, True, "striped")
        ra.bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], 4, True, "striped")
        t = ra.kernel_times(with_clock=True)
    finally:
        ra.set_kernel_timing(False)
    assert [n for n, _, _ in t] == ["fwd", "bwd_prep", "bwd_dkv", "bwd_dq"]
    assert all(ms > 0 for _, ms, _ in t)
    mhz = {n: c for n, _, c in t}
    assert mhz["bwd_prep"] == -1                       # no clock record for the preprocess
    for n in ("fwd", "bwd_dkv", "bwd_dq"):             # the tensor-core kernels report their SM clock
        assert 200 < mhz[n] < 2600, (n, mhz[n])
    ra.fwd(inp["q"], inp["k"], inp["v"], 4, True, "striped")
    assert ra.kernel_times() == []
