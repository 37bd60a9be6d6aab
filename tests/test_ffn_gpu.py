"""Blockwise gated feedforward on the GPU (ra_ffn through the C ABI) against
the oracle: small ragged shapes element by element, several block sizes, and
sampled rows of the LLaMA-7B-shaped workload."""
import numpy as np
import pytest
import torch

import oracle as orc
from gpu_helpers import max_err
from ring_attention_fwd_gb300.inputs import FFN_WORKLOADS, make_ffn_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import ring_attention_fwd_gb300 as ra
    assert torch.cuda.is_available()
    return ra


def _f64(t):
    return t.to(torch.float64).numpy()


def _tol_ok(g, r):
    """The intermediate is stored in bf16 (relative 2^-9) and so is Y:
    max error <= 2e-2 * max(1, |ref|_inf) and relative Frobenius <= 1e-2."""
    err = max_err(g, r)
    rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    return err <= 2e-2 * max(1.0, float(np.abs(r).max())) and rel <= 1e-2, (err, rel)


@pytest.mark.parametrize("T,h,f,c", [(300, 256, 384, 128), (128, 256, 128, 128), (1, 512, 256, 1),
                                     (1000, 512, 1024, 1000), (1000, 512, 1024, 256), (777, 768, 640, 500)])
def test_ffn_matches_oracle(ra, T, h, f, c):
    inp = make_ffn_inputs(T, h, f, seed=T + h + f)
    dev = {k: v.cuda() for k, v in inp.items()}
    y = ra.ffn(dev["x"], dev["w1"], dev["w3"], dev["w2"], c)
    torch.cuda.synchronize()
    ra.check_device_status()
    ref = orc.blockwise_ffn(_f64(inp["x"]), _f64(inp["w1"]), _f64(inp["w3"]), _f64(inp["w2"]), c)
    ok, why = _tol_ok(y.double().cpu().numpy(), ref)
    assert ok, why


def test_ffn_block_size_does_not_change_the_result(ra):
    """Rows are independent, so every block size gives bit-identical rows."""
    inp = make_ffn_inputs(640, 512, 512, seed=5)
    dev = {k: v.cuda() for k, v in inp.items()}
    ys = [ra.ffn(dev["x"], dev["w1"], dev["w3"], dev["w2"], c) for c in (640, 256, 128)]
    torch.cuda.synchronize()
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])


def test_ffn_full_workload_sampled_rows(ra):
    w = FFN_WORKLOADS["ffn_7b"]
    inp = make_ffn_inputs(w["T"], w["h"], w["f"], w["seed"])
    dev = {k: v.cuda() for k, v in inp.items()}
    y = ra.ffn(dev["x"], dev["w1"], dev["w3"], dev["w2"], w["block_rows"])
    torch.cuda.synchronize()
    ra.check_device_status()
    assert bool(torch.isfinite(y.float()).all())
    c = w["block_rows"]
    rng = np.random.default_rng(0)
    rows = sorted({0, 127, 128, c - 1, c, w["T"] - 1} | set(rng.integers(0, w["T"], 58).tolist()))
    ref = orc.ffn_rows(_f64(inp["x"][rows]), _f64(inp["w1"]), _f64(inp["w3"]), _f64(inp["w2"]))
    ok, why = _tol_ok(y[rows].double().cpu().numpy(), ref)
    assert ok, why


def test_ffn_kernel_timing_records(ra):
    inp = make_ffn_inputs(512, 256, 256, seed=3)
    dev = {k: v.cuda() for k, v in inp.items()}
    ra.set_kernel_timing(True)
    try:
        ra.ffn(dev["x"], dev["w1"], dev["w3"], dev["w2"], 256)
        names = [n for n, ms in ra.kernel_times() if ms >= 0]
    finally:
        ra.set_kernel_timing(False)
    assert names == ["ffn_up", "ffn_down", "ffn_up", "ffn_down"]
