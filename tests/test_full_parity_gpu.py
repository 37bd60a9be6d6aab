"""Full-mode parity: every element of every head of the large workloads
against the whole oracle (every row and every key, float64), computed on all
host cores.

The 32768-token workload in both layouts, forward and backward, runs by
default.  The 65536-token forward+backward workload and the 131072-token
forward take the oracle tens of minutes of host time; they run when
RA_FULL_PARITY=1.  The 131072-token forward+backward (about 45 minutes of
the oracle on 16 cores) runs when RA_FULL_PARITY=2."""
import os
import time

import numpy as np
import pytest
import torch

from gpu_helpers import TOL, grad_errors, head_arrays, max_err, workload_inputs
from ring_attention_fwd_gb300.inputs import WORKLOADS

pytestmark = pytest.mark.gpu
FULL = os.environ.get("RA_FULL_PARITY") == "1"
FULL_128K_BWD = os.environ.get("RA_FULL_PARITY") == "2"
GRAD_MAX, GRAD_FRO = 2e-2, 1e-2     # the backward's bounds (tests/test_bwd_gpu.py)


@pytest.fixture(scope="module")
def ra():
    import ring_attention_fwd_gb300 as ra
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return ra


def _full_check(ra, w, layout, with_bwd, row_chunk):
    """Runs the CUDA forward (and backward) on the whole workload, then the
    whole oracle head by head, a batch of heads at a time; returns the worst
    errors over all heads and the oracle's wall time."""
    import oracle_pool as op
    inp = workload_inputs(w, with_grad=with_bwd)
    B, H = inp["q"].shape[:2]
    N, causal = w["N"], w["causal"]
    dev = {k: v.cuda() for k, v in inp.items()}
    o, lse = ra.fwd(dev["q"], dev["k"], dev["v"], N, causal, layout)
    grads = None
    if with_bwd:
        grads = dict(zip(("dq", "dk", "dv"), ra.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], N, causal,
                                                    layout)))
    torch.cuda.synchronize()
    ra.check_device_status()
    del dev
    heads = [(b, h) for b in range(B) for h in range(H)]
    names = ("q", "k", "v", "do") if with_bwd else ("q", "k", "v")
    worst = {"o": 0.0, "lse": 0.0}
    if with_bwd:
        worst.update({n: (0.0, 0.0) for n in ("dq", "dk", "dv")})
    t0 = time.time()
    per = op.workers()
    for b0 in range(0, len(heads), per):
        batch = heads[b0:b0 + per]
        shared = [op.share(f"in{b}_{h}", **head_arrays(inp, b, h, names)) for (b, h) in batch]
        try:
            for n, out in op.full_heads(shared, N, causal, layout, with_bwd, row_chunk):
                b, h = batch[n]
                try:
                    worst["o"] = max(worst["o"], max_err(o[b, h].float().cpu().numpy(), np.load(out["o"])))
                    worst["lse"] = max(worst["lse"], max_err(lse[b, h].cpu().numpy(), np.load(out["lse"])))
                    if with_bwd:
                        for name, g in grads.items():
                            e, f = grad_errors(g[b, h].float().cpu().numpy(), np.load(out[name]))
                            worst[name] = (max(worst[name][0], e), max(worst[name][1], f))
                finally:
                    op.release(out)
        finally:
            for p in shared:
                op.release(p)
    return worst, time.time() - t0


def _assert_within(worst, with_bwd):
    assert worst["o"] <= TOL["bf16"]["o"] and worst["lse"] <= TOL["bf16"]["lse"], worst
    if with_bwd:
        for name in ("dq", "dk", "dv"):
            e, f = worst[name]
            assert e <= GRAD_MAX and f <= GRAD_FRO, (name, worst[name])


@pytest.mark.parametrize("layout", ["striped", "contiguous"])
def test_balance_32k_full_forward_backward(ra, layout):
    """32768 tokens, 16 heads, 16 ring blocks: O, LSE, dQ, dK and dV of every
    row of every head."""
    worst, secs = _full_check(ra, WORKLOADS["balance_32k"], layout, True, 256)
    print(f"balance_32k {layout} full: {worst}, oracle {secs:.0f} s")
    _assert_within(worst, True)


def test_batch2_noncausal_16k_full_forward_backward(ra):
    """B = 2, 4 heads, 16384 tokens, 8 ring blocks, every key visible: the
    unmasked path and the batch dimension, every element."""
    w = dict(B=2, H=4, S=16384, D=128, N=8, causal=False, layout="contiguous", dtype="bf16", seed=16, scale=1.0,
             grad=True)
    worst, secs = _full_check(ra, w, w["layout"], True, 256)
    print(f"batch 2 non-causal 16k full: {worst}, oracle {secs:.0f} s")
    _assert_within(worst, True)


@pytest.mark.skipif(not FULL, reason="oracle takes tens of minutes: set RA_FULL_PARITY=1")
def test_fwdbwd_64k_full_forward_backward(ra):
    """65536 tokens, 32 heads, 16 ring blocks, causal striped: every element."""
    w = WORKLOADS["fwdbwd_64k"]
    worst, secs = _full_check(ra, w, w["layout"], True, 256)
    print(f"fwdbwd_64k full: {worst}, oracle {secs:.0f} s")
    _assert_within(worst, True)


@pytest.mark.skipif(not FULL, reason="oracle takes tens of minutes: set RA_FULL_PARITY=1")
def test_long_128k_full_forward(ra):
    """131072 tokens, 32 heads, 32 ring blocks, causal contiguous (the
    benchmark's workload): O and LSE of every row of every head."""
    w = WORKLOADS["long_128k"]
    worst, secs = _full_check(ra, w, w["layout"], False, 128)
    print(f"long_128k full forward: {worst}, oracle {secs:.0f} s")
    _assert_within(worst, False)


@pytest.mark.skipif(not FULL_128K_BWD, reason="oracle takes about 45 minutes: set RA_FULL_PARITY=2")
def test_long_128k_full_forward_backward(ra):
    """131072 tokens, 32 heads, 32 ring blocks, causal contiguous (the
    benchmark's workload): O, LSE, dQ, dK and dV of every row of every head."""
    w = WORKLOADS["long_128k"]
    worst, secs = _full_check(ra, w, w["layout"], True, 128)
    print(f"long_128k full forward+backward: {worst}, oracle {secs:.0f} s")
    _assert_within(worst, True)
