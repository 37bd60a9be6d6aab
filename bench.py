"""Benchmark: ring-order blockwise attention forward + backward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload long_128k|fwdbwd_64k|balance_32k|causal_8k|long_1m|decode_256k|ffn_7b]

A step is one pass of the whole path over one batch of synthetic input: the
forward (O, LSE) followed by the backward (dQ, dK, dV) from the saved state.
Default workload: 131072 tokens, 32 heads of dim 128, 32 ring blocks of
4096, causal, contiguous, inputs N(0,1) x 0.5 in bf16.  The inputs (1 GiB
each) are larger than L2, so no flush is needed between steps.

The `e2e` figure runs the same steps through the public API from pinned host
memory: every step uploads its inputs and downloads every output, on two copy
streams (one per direction) that overlap the neighbouring steps' compute
(device tensors double-buffered), as a training loop would prefetch.
`e2e.link_alone` times one step's copies with nothing else running (each
direction alone and both at once), the bound the host link sets on `e2e`.

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent replicas; the real multi-GPU ring exchange is not built), the
timing is the max over ranks and `value` sums the ranks' work.

`--workload long_1m` runs the same step on 1,048,576 tokens (4 heads, 64 ring
blocks of 16384).

`--workload decode_256k` measures ring decode instead (one new token against
a resident 256K-token KV cache; HBM-bound, reported in GB/s).

`--workload ffn_7b` measures the blockwise gated feedforward of a LLaMA-7B-shaped
layer over 16384 tokens in blocks of 4096 (tensor-bound, TFLOP/s).

`--impl reference` times the CPU oracle (float64 NumPy) on the host cores, on
a bounded sample of the same workload, and prints the same JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ring-order blockwise attn fwd+bwd TFLOP/s, % GB300 BF16 peak (S=128K)"
UNIT = "TFLOP/s"

# DRAM traffic per launch of a kernel, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), valid only for the kernel
# code it was taken on: the hash of csrc/<file> without comments (_src_hash)
# at capture time.
NCU_TRAFFIC = {
    "fwd": {"sha256": "a8b983f4ad109f5ccb021fb5f887f6e32dedae180da1253e95220a5374f1b78f", "workload": "long_128k", "bytes_per_launch": (27.160 + 1.250) * 1e9},
    "bwd_dkv": {"sha256": "2cd114dc083486b62a781ff2c5c5b85003f5c222d07ef62ba0a8939e8e86990d", "workload": "long_128k", "bytes_per_launch": (11.253 + 2.136) * 1e9},
    "bwd_dq": {"sha256": "2cd114dc083486b62a781ff2c5c5b85003f5c222d07ef62ba0a8939e8e86990d", "workload": "long_128k", "bytes_per_launch": (8.710 + 1.069) * 1e9},
    "decode_split": {"sha256": "db519d009c6e14d06bbde7b8df9ec6dab5ec5aeb1dc7cbff5fa4dc7eeea7a5b8", "workload": "decode_256k", "bytes_per_launch": 4295068000 + 6642688},
    "ffn_up": {"sha256": "e3c1fddde6a2bcd126b3ceb1de1f6d6f977d1cc7e45d80e1a639318de4a2afb1", "workload": "ffn_7b", "bytes_per_launch": (218.333 + 79.864) * 1e6},
}


def _src_hash(names) -> str:
    """SHA-256 of csrc/<name> (or of several files, in order) with // comments
    and blank lines removed: the recorded traffic stays valid across comment
    edits, not code changes."""
    import re
    lines = []
    for name in ([names] if isinstance(names, str) else names):
        with open(os.path.join(ROOT, "ring_attention_fwd_gb300", "csrc", name)) as f:
            lines += [re.sub(r"//.*$", "", ln).rstrip() for ln in f]
    return hashlib.sha256("\n".join(ln for ln in lines if ln).encode()).hexdigest()


def _hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured copy bandwidth"
    except Exception:
        return 6800.0, "fallback"


def merge_bandwidth(rows: int, D: int, launches: int = 20) -> dict:
    """ra_merge at one ring round's size: `rows` rows of D, bf16 state and
    partial, and a float32 state folding a bf16 partial (what ring_forward
    does each round).  Every launch is timed alone with CUDA events after a
    write of 512 MB has pushed the operands out of L2; the median is reported
    against the measured HBM copy bandwidth.  Algorithmic bytes per row: read
    both states and both LSEs, write the merged state and LSE."""
    import torch
    import ring_attention_fwd_gb300 as ra
    hbm, hsrc = _hbm_peak()
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    out = {"rows": rows, "D": D, "l2": "flushed before each launch (512 MB write)", "peak": hbm,
           "peak_kind": hsrc, "launches": launches}
    for name, adt, bdt in (("bf16", torch.bfloat16, torch.bfloat16), ("f32_state_bf16_partial", torch.float32,
                                                                       torch.bfloat16)):
        oa = torch.randn((rows, D), device="cuda", generator=g).to(adt)
        ob = torch.randn((rows, D), device="cuda", generator=g).to(bdt)
        la = torch.randn((rows,), device="cuda", generator=g)
        lb = torch.randn((rows,), device="cuda", generator=g)
        nbytes = rows * (2 * D * oa.element_size() + D * ob.element_size() + 12)
        ms = []
        for k in range(launches + 2):
            flush.fill_(k & 0xff)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            ra.merge(oa, la, ob, lb)
            e1.record()
            e1.synchronize()
            if k >= 2:
                ms.append(e0.elapsed_time(e1))
        med = statistics.median(ms)
        out[name] = {"bytes": nbytes, "ms": med, "gbps": nbytes / (med * 1e-3) / 1e9,
                     "frac_of_hbm": nbytes / (med * 1e-3) / 1e9 / hbm}
    ra.check_device_status()
    return out


def ring_round(dev: dict, N: int, causal: bool, layout: str, launches: int = 10) -> dict:
    """One ring round at the workload's block size (host N-1 against block 0,
    every key visible): the step folded into a float32 state in the kernel's
    epilogue (ra_fwd_step_fold) against the step writing its partial and a
    separate merge into the same state.  Median of `launches` each."""
    import torch
    import ring_attention_fwd_gb300 as ra
    B, H, S, D = dev["q"].shape
    c = S // N
    qi = dev["q"][:, :, (N - 1) * c:].contiguous()
    kj, vj = dev["k"][:, :, :c].contiguous(), dev["v"][:, :, :c].contiguous()
    o_acc = torch.zeros((B, H, c, D), dtype=torch.float32, device="cuda")
    l_acc = torch.zeros((B, H, c), dtype=torch.float32, device="cuda")
    oj, lj = torch.empty_like(qi), torch.empty_like(l_acc)

    def timed(fn):
        ms = []
        for k in range(launches + 2):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            if k >= 2:
                ms.append(e0.elapsed_time(e1))
        return statistics.median(ms)

    fold = timed(lambda: ra.fwd_step_fold(qi, kj, vj, N, N - 1, 0, causal, layout, o_acc=o_acc, lse_acc=l_acc))
    step = timed(lambda: ra.fwd_step(qi, kj, vj, N, N - 1, 0, causal, layout, o=oj, lse=lj))
    both = timed(lambda: (ra.fwd_step(qi, kj, vj, N, N - 1, 0, causal, layout, o=oj, lse=lj),
                          ra.merge(o_acc, l_acc, oj, lj)))
    ra.check_device_status()
    return {"rows": B * H * c, "fold_ms": fold, "step_ms": step, "step_then_merge_ms": both,
            "fold_saves": 1.0 - fold / both}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm = [float(r[1]) for r in self.rows if len(r) > 8 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) > 8 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in self.rows if len(r) > 8 for k in range(4)
                          if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def pipelined_e2e(steps: int, stream, h2d_list, compute, d2h_list, warmup: int = 2) -> float:
    """End-to-end loop with the host<->device copies overlapped with compute,
    as a training or serving loop prefetches: one copy stream uploads step
    k+1's inputs and another downloads step k's results (both directions of
    the link at once) while the compute stream runs step k; device inputs and
    outputs are double-buffered (sets 0 and 1).  The first upload and the
    last download are not hidden.

    h2d_list(b) / d2h_list(b): [(dst, src)] copies for buffer set b;
    compute(b): one step on set b, on the current stream.
    Returns ms per step, CUDA events from the first upload to the last download."""
    import torch
    if warmup:
        pipelined_e2e(warmup, stream, h2d_list, compute, d2h_list, warmup=0)   # untimed
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    up.wait_stream(stream)
    down.wait_stream(stream)
    with torch.cuda.stream(up):
        for dst, src in h2d_list(0):
            dst.copy_(src, non_blocking=True)
        ev_in[0].record(up)
    for k in range(steps):
        b = k % 2
        stream.wait_event(ev_in[b])
        if k >= 2:
            stream.wait_event(ev_out[b])          # step k-2's results are out of set b
        with torch.cuda.stream(stream):
            compute(b)
        ev_done[b].record(stream)
        if k + 1 < steps:
            nb = (k + 1) % 2
            with torch.cuda.stream(up):
                if k >= 1:
                    up.wait_event(ev_done[nb])    # step k-1 no longer reads set nb
                for dst, src in h2d_list(nb):
                    dst.copy_(src, non_blocking=True)
                ev_in[nb].record(up)
        with torch.cuda.stream(down):
            down.wait_event(ev_done[b])
            for dst, src in d2h_list(b):
                dst.copy_(src, non_blocking=True)
            ev_out[b].record(down)
    stream.wait_stream(up)
    stream.wait_stream(down)
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def link_times(stream, h2d, d2h) -> dict:
    """One step's host<->device copies with no compute beside them: uploads
    alone, downloads alone, and both directions at once (on two streams), so
    an e2e figure can be read against what the host link allows.
    h2d / d2h: [(dst, src)] copies.  Returns ms and GB/s."""
    import torch
    up, down = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(pairs_up, pairs_down):
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s0.record(stream)
        up.wait_stream(stream)
        down.wait_stream(stream)
        with torch.cuda.stream(up):
            for dst, src in pairs_up:
                dst.copy_(src, non_blocking=True)
        with torch.cuda.stream(down):
            for dst, src in pairs_down:
                dst.copy_(src, non_blocking=True)
        stream.wait_stream(up)
        stream.wait_stream(down)
        s1.record(stream)
        torch.cuda.synchronize()
        return s0.elapsed_time(s1)

    bu = sum(src.numel() * src.element_size() for _, src in h2d)
    bd = sum(src.numel() * src.element_size() for _, src in d2h)
    # three samples each, interleaved; the spread shows a slow outlier (a first
    # touch, another tenant on the host link) instead of hiding it in a minimum
    hs, ds, bs = [], [], []
    for _ in range(3):
        hs.append(timed(h2d, []))
        ds.append(timed([], d2h))
        bs.append(timed(h2d, d2h))
    h_ms, d_ms, b_ms = (statistics.median(x) for x in (hs, ds, bs))
    return {"h2d_ms": h_ms, "d2h_ms": d_ms, "both_ms": b_ms, "h2d_gbs": bu / h_ms / 1e6, "d2h_gbs": bd / d_ms / 1e6,
            "stat": "median of 3", "h2d_ms_all": hs, "d2h_ms_all": ds, "both_ms_all": bs}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ----------------------------------------------------------------- CPU oracle
def oracle_full(inp, w, with_bwd: bool):
    """Time the whole oracle on the whole workload: every head, every row
    (``naive_attention``) and, with the backward, ``attention_bwd_head_chunked``
    on the oracle's own O and LSE.  One process; NumPy's BLAS uses the host
    cores.  Returns (flops by the benchmark's convention, seconds, description)."""
    import oracle as orc
    B, H, S, D = inp["q"].shape
    N, causal, layout = w["N"], w["causal"], w["layout"]
    t0 = time.perf_counter()
    for b in range(B):
        for h in range(H):
            q, k, v = (inp[x][b, h].double().numpy() for x in ("q", "k", "v"))
            o, lse = orc.naive_attention(q[None, None], k[None, None], v[None, None], N, causal, layout,
                                         row_chunk=128)
            if with_bwd:
                orc.attention_bwd_head_chunked(q, k, v, o[0, 0], lse[0, 0], inp["do"][b, h].double().numpy(), N,
                                               causal, layout, row_chunk=128)
    dt = time.perf_counter() - t0
    from ring_attention_fwd_gb300 import flops as fl
    f = fl.fwd_flops(B, H, S, D, causal) * (3.5 if with_bwd else 1.0)
    return f, dt, (f"the whole workload: {B * H} heads, every row, forward" + (" and backward" if with_bwd else "")
                   + ", float64")


def oracle_sample(inp, w, budget_s: float):
    """Time the oracle on sampled query rows of one head (forward LSE/O and
    the dQ rows of the backward), growing the sample until `budget_s` is
    spent.  Returns (flops, seconds, description)."""
    import numpy as np
    import oracle as orc
    q = inp["q"][0, 0].double().numpy()
    k = inp["k"][0, 0].double().numpy()
    v = inp["v"][0, 0].double().numpy()
    do = inp["do"][0, 0].double().numpy() if "do" in inp else v
    S, D, N = w["S"], w["D"], w["N"]
    pos = orc.token_positions(S, N, w["layout"])
    rng = np.random.default_rng(0)
    flops = 0.0
    rows_done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        rows = np.sort(rng.choice(S, size=64, replace=False))
        orc.attention_rows(q, k, v, rows, N, w["causal"], w["layout"])
        orc.attention_bwd_dq_rows(q, k, v, do, rows, N, w["causal"], w["layout"])
        vis = (pos[rows] + 1) if w["causal"] else np.full(rows.size, S)
        # forward 4*D per visible pair; the backward's dQ rows 2.5x that (convention)
        flops += float(vis.sum()) * 4 * D * 3.5
        rows_done += rows.size
    dt = time.perf_counter() - t0
    return flops, dt, f"{rows_done} random query rows of head 0 (forward O/LSE + backward dQ), row by row"


def run_reference(args, w):
    import torch
    from ring_attention_fwd_gb300.inputs import make_inputs
    ws, rank, _ = _dist()
    if rank != 0:
        return
    cores = len(os.sched_getaffinity(0))
    inp = make_inputs(1, 1, w["S"], w["D"], w["seed"], dtype=w["dtype"], scale=w["scale"], with_grad=True)
    per_step = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(inp, w, per_step / 4)
    tot_f = tot_t = 0.0
    desc = ""
    for _ in range(args.steps):
        f, t, desc = oracle_sample(inp, w, per_step)
        tot_f += f
        tot_t += t
    val = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, **{k: w[k] for k in ("B", "H", "S", "D", "N", "causal", "layout")},
                   "input_scale": w["scale"], "step": "fwd+bwd"},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"per step: {desc}; numpy float64, BLAS threads = {cores}"},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU arm
def run_ours(args, w):
    import torch
    import ring_attention_fwd_gb300 as ra
    from ring_attention_fwd_gb300 import flops as fl
    from ring_attention_fwd_gb300.inputs import make_inputs

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    ra.set_fwd_kernel(args.fwd_kernel)
    B, H, S, D, N = w["B"], w["H"], w["S"], w["D"], w["N"]
    causal, layout = w["causal"], w["layout"]
    inp = make_inputs(B, H, S, D, w["seed"], dtype=w["dtype"], scale=w["scale"], with_grad=True)
    host = {k: v.pin_memory() for k, v in inp.items()}
    dev = {k: v.cuda() for k, v in host.items()}
    o = torch.empty_like(dev["q"])
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.empty_like(dev["q"]) for _ in range(3))
    wsb = ra.bwd_workspace_bytes(B, H, S, D, N)
    work = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def has_bwd():
        try:
            ra.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], N, causal, layout, dq=dq, dk=dk, dv=dv,
                   workspace=work)
            return True
        except ra.RingAttnError as e:
            if e.code == ra.binding.RA_ERR_UNSUPPORTED:
                return False
            raise

    ra.fwd(dev["q"], dev["k"], dev["v"], N, causal, layout, o=o, lse=lse)
    with_bwd = has_bwd()
    torch.cuda.synchronize()
    ra.check_device_status()
    f_fwd = fl.fwd_flops(B, H, S, D, causal)
    f_bwd = fl.bwd_flops(B, H, S, D, causal) if with_bwd else 0
    f_step = f_fwd + f_bwd

    ev = []

    def step(record):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ra.fwd(dev["q"], dev["k"], dev["v"], N, causal, layout, o=o, lse=lse)
        e1.record(stream)
        if with_bwd:
            ra.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], N, causal, layout, dq=dq, dk=dk, dv=dv,
                   workspace=work)
        e2.record(stream)
        if record:
            ev.append((e0, e1, e2))

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ra.set_kernel_timing(True)   # the library records CUDA events around each of its kernels
    with ClockSampler(local) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            step(True)
        t1.record(stream)
        torch.cuda.synchronize()
    ktimes = ra.kernel_times(with_clock=True)
    ra.set_kernel_timing(False)
    ra.check_device_status()
    per_kernel, kernel_mhz = {}, {}
    for name, ms, mhz in ktimes:
        per_kernel.setdefault(name, []).append(ms)
        if mhz > 0:
            kernel_mhz.setdefault(name, []).append(mhz)
    total_ms = t0.elapsed_time(t1)
    if ws > 1:
        tt = torch.tensor([total_ms], device="cuda")
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        torch.distributed.barrier()
        total_ms = float(tt.item())
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in ev)
    bwd_ms = statistics.mean(b.elapsed_time(c) for _, b, c in ev) if with_bwd else None
    ms_step = total_ms / args.steps
    value = f_step * ws / (ms_step * 1e-3) / 1e12

    e2e_ms = link = None
    if not args.kernels_only:
        # end to end through the public API with host buffers: every step uploads
        # its inputs from pinned memory and downloads every output, overlapped with
        # the neighbouring steps' compute (double-buffered device tensors)
        outs_host = {"o": torch.empty_like(o, device="cpu").pin_memory(),
                     "lse": torch.empty_like(lse, device="cpu").pin_memory()}
        if with_bwd:
            for n in ("dq", "dk", "dv"):
                outs_host[n] = torch.empty_like(dq, device="cpu").pin_memory()
        in_names = ["q", "k", "v"] + (["do"] if with_bwd else [])
        h2d = sum(host[n].numel() * host[n].element_size() for n in in_names)
        d2h = sum(t.numel() * t.element_size() for t in outs_host.values())
        ins = [dev, {n: torch.empty_like(dev[n]) for n in in_names}]
        outs = [{"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv},
                {"o": torch.empty_like(o), "lse": torch.empty_like(lse), "dq": torch.empty_like(dq),
                 "dk": torch.empty_like(dk), "dv": torch.empty_like(dv)}]

        def e2e_compute(b):
            x, y = ins[b], outs[b]
            ra.fwd(x["q"], x["k"], x["v"], N, causal, layout, o=y["o"], lse=y["lse"])
            if with_bwd:
                ra.bwd(x["q"], x["k"], x["v"], y["o"], y["lse"], x["do"], N, causal, layout, dq=y["dq"], dk=y["dk"],
                       dv=y["dv"], workspace=work)

        e2e_steps = max(8, args.steps)          # amortises the unhidden first upload and last download
        # The host link is shared with the machine's other GPUs and shows one-off stalls of 100-200 ms
        # on a 4.3 GB copy: the pipelined loop runs three times and the median stands (all reported).
        e2e_runs = [pipelined_e2e(e2e_steps, stream, lambda b: [(ins[b][n], host[n]) for n in in_names],
                                  e2e_compute, lambda b: [(outs_host[n], outs[b][n]) for n in outs_host])
                    for _ in range(3)]
        e2e_ms = statistics.median(e2e_runs)
        link = link_times(stream, [(ins[1][n], host[n]) for n in in_names], [(outs_host[n], outs[0][n]) for n in outs_host])
        if ws > 1:
            tt = torch.tensor([e2e_ms], device="cuda")
            torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
            e2e_ms = float(tt.item())

    burst, sustained, src = _peaks()
    # Algorithmic FLOPs per launch of each tensor-core kernel.  The backward's
    # five GEMMs (S, dP, dV, dK, dQ; 2.5x the forward's two) split as four in
    # the dK/dV kernel and one (dQ) in the dQ kernel, which also recomputes S
    # and dP (executed: three GEMMs).
    gemm = f_fwd / 2
    algo = {"fwd": f_fwd, "fwd_pair": f_fwd, "bwd_dkv": 4 * gemm, "bwd_dq": 1 * gemm}
    executed = {"fwd": f_fwd, "fwd_pair": f_fwd, "bwd_dkv": 4 * gemm, "bwd_dq": 3 * gemm}
    kernels = {}
    clocks = clk.summary()
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    for name, lst in per_kernel.items():
        mean_ms = statistics.mean(lst)
        kernels[name] = {"launches": len(lst), "ms": mean_ms}
        if name in algo:
            kernels[name]["tflops_algorithmic"] = algo[name] / (mean_ms * 1e-3) / 1e12
            kernels[name]["tflops_executed"] = executed[name] / (mean_ms * 1e-3) / 1e12
            # per clock, apart from the power cap: executed FLOP over (cycles x SMs x the
            # dense bf16 tensor rate of 8192 FLOP per clock per SM).  The clock is the one
            # the kernel itself measured (its first CTA's cycle counter against the global
            # timer); nvidia-smi's median over the whole step is kept beside it for reference.
            if name in kernel_mhz:
                mhz = statistics.median(kernel_mhz[name])
                cyc = mean_ms * 1e-3 * mhz * 1e6
                kernels[name]["sm_mhz_in_kernel"] = mhz
                kernels[name]["mcycles"] = cyc / 1e6
                kernels[name]["per_clock_frac"] = executed[name] / (cyc * sms * 8192)
            if clocks.get("sm_mhz"):
                cyc = mean_ms * 1e-3 * clocks["sm_mhz"] * 1e6
                kernels[name]["per_clock_frac_at_smi_median"] = executed[name] / (cyc * sms * 8192)
    dom = max((n for n in kernels if n in algo), key=lambda n: kernels[n]["ms"])
    achieved = kernels[dom]["tflops_algorithmic"]
    src_file = {"fwd": ("fwd_bf16.cu", "fwd_softmax.cuh"), "fwd_pair": ("fwd_bf16_pair.cu", "fwd_softmax.cuh"),
                "bwd_dkv": "bwd_bf16.cu", "bwd_dq": "bwd_bf16.cu"}[dom]
    tr = NCU_TRAFFIC.get(dom)
    traffic = tr["bytes_per_launch"] if tr and tr["sha256"] == _src_hash(src_file) and \
        tr["workload"] == args.workload and args.heads == 0 else None
    roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved,
                "peak": sustained, "unit": UNIT, "frac": achieved / sustained, "traffic": traffic,
                "algorithmic_flops_per_launch": algo[dom], "avg_launch_ms": kernels[dom]["ms"],
                "peak_kind": f"{src} sustained bf16 (burst {burst})", "frac_of_burst": achieved / burst}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "H": H, "S": S, "D": D, "N": N, "causal": causal,
                   "layout": layout, "input_scale": w["scale"], "step": "fwd+bwd" if with_bwd else "fwd only",
                   "l2": "inputs larger than L2 (1 GiB per tensor), no flush",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "fwd_kernel": args.fwd_kernel,
        "fwd": {"ms": fwd_ms, "tflops": f_fwd / (fwd_ms * 1e-3) / 1e12,
                "frac_of_peak": f_fwd / (fwd_ms * 1e-3) / 1e12 / sustained},
        "bwd": ({"ms": bwd_ms, "tflops": f_bwd / (bwd_ms * 1e-3) / 1e12,
                 "frac_of_peak": f_bwd / (bwd_ms * 1e-3) / 1e12 / sustained} if with_bwd else None),
        "tokens_per_s": B * S * ws / (ms_step * 1e-3),
        "flops_per_step": {"convention": f_step,
                           "exact_visible_pairs": fl.fwd_flops_exact(B, H, S, D, causal) * (3.5 if with_bwd else 1.0),
                           "value_exact_tflops": fl.fwd_flops_exact(B, H, S, D, causal) * (3.5 if with_bwd else 1.0)
                           * ws / (ms_step * 1e-3) / 1e12},
        "roofline": roofline,
        "e2e": ({"value": f_step * ws / (e2e_ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": e2e_ms,
                 "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                 "stat": "median of 3 runs", "ms_per_step_all": e2e_runs,
                 "copies": "overlapped with the neighbouring steps' compute on two copy streams (up, down); "
                           "double-buffered",
                 "link_alone": link} if e2e_ms is not None else None),
        "kernels": kernels,
        "gpu_launches": len(ktimes),
        "clocks": clocks,
        # one ring round's merge (a host's c query rows of every head), outside the timed region
        "merge": None if args.kernels_only else merge_bandwidth(B * H * (S // N), D),
        "ring_round": None if args.kernels_only else ring_round(dev, N, causal, layout),
    }
    if rank == 0 and not args.no_cpu_baseline:
        cores = len(os.sched_getaffinity(0))
        if args.oracle_full:
            f, t, desc = oracle_full(inp, w, with_bwd)
        else:
            inp1 = {k: v[:1, :1] for k, v in inp.items()}
            f, t, desc = oracle_sample(inp1, w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": f / t / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc + f"; {t:.1f} s of numpy float64"}
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_balance(args):
    """Per-virtual-host work and time of the forward, striped vs contiguous
    (the 32768-token, 16-block workload by default): analytic visible-pair
    FLOPs per block, CTA-time per (block, ring step) from the kernel's
    %globaltimer hooks, and the makespan of N hosts that each ran their block
    alone on a GPU like this one (sum over ring steps of the slowest host;
    no communication).  Prints one JSON line."""
    import torch
    import ring_attention_fwd_gb300 as ra
    from ring_attention_fwd_gb300 import flops as fl
    from ring_attention_fwd_gb300.inputs import WORKLOADS, make_inputs
    w = dict(WORKLOADS[args.workload])
    B, H, S, D, N = w["B"], w["H"], w["S"], w["D"], w["N"]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    inp = {k: v.cuda() for k, v in make_inputs(B, H, S, D, w["seed"], scale=w["scale"]).items()}
    out = {"workload": args.workload, "B": B, "H": H, "S": S, "D": D, "N": N, "causal": True, "layouts": {}}
    buf = torch.zeros(N * N, dtype=torch.int64, device="cuda")
    for layout in ("contiguous", "striped"):
        for _ in range(args.warmup):
            ra.fwd(inp["q"], inp["k"], inp["v"], N, True, layout)
        times, kms = [], []
        for _ in range(args.steps):
            buf.zero_()
            ra.set_timing_buffer(buf)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            ra.fwd(inp["q"], inp["k"], inp["v"], N, True, layout)
            e1.record()
            torch.cuda.synchronize()
            ra.set_timing_buffer(None)
            times.append(buf.view(N, N).double().cpu())
            kms.append(e0.elapsed_time(e1))
        ra.check_device_status()
        t = sum(times) / len(times) / 1e6                  # CTA-ms per (block, ring step)
        pairs = fl.visible_pairs_per_block(S, N, layout, True)
        per_dev_ms = (t.sum(dim=1) / sms).tolist()         # block i alone on all SMs
        makespan = float((t.max(dim=0).values / sms).sum())
        out["layouts"][layout] = {
            "flops_per_block": [4 * D * H * B * p for p in pairs],
            "flops_max_over_min": max(pairs) / min(pairs),
            "time_ms_per_block": per_dev_ms,
            "time_max_over_min": max(per_dev_ms) / min(per_dev_ms),
            "simulated_makespan_ms": makespan,
            "kernel_ms": statistics.mean(kms),
        }
    L = out["layouts"]
    out["striped_speedup_of_simulated_makespan"] = (L["contiguous"]["simulated_makespan_ms"] /
                                                    L["striped"]["simulated_makespan_ms"])
    out["pages_context"] = "striped 1.45x at 256K, 1.65x at 786K tokens, multi-device, hardware not stated"
    print(json.dumps(out), flush=True)


DECODE_METRIC = "ring decode attention KV-cache read GB/s (256K-token context, one new token)"


def _decode_bytes(B, H, S, D):
    """Algorithmic bytes of one decode call: read q, K, V (bf16); write O (bf16), LSE (f32)."""
    return B * H * (2 * S * D * 2 + D * 2 + D * 2 + 4)


def decode_oracle_sample(inp, w, budget_s: float):
    """Time the oracle's ring decode head by head until `budget_s` is spent.
    Returns (bytes, seconds, description)."""
    import oracle as orc
    B, H, S, D, N = w["B"], w["H"], w["S"], w["D"], w["N"]
    done, nbytes = 0, 0.0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s or done == 0:
        b, h = divmod(done % (B * H), H)
        orc.ring_decode(inp["q"][b, h].double().numpy(), inp["k"][b, h].double().numpy(),
                        inp["v"][b, h].double().numpy(), N)
        nbytes += _decode_bytes(1, 1, S, D)
        done += 1
    dt = time.perf_counter() - t0
    return nbytes, dt, f"{done} heads of the workload, ring decode of each head in numpy float64"


def run_decode(args, w):
    """Ring decode: one query token per (b, h) against a resident KV cache."""
    import torch
    from ring_attention_fwd_gb300.inputs import make_decode_inputs
    ws, rank, local = _dist()
    B, H, S, D, N = w["B"], w["H"], w["S"], w["D"], w["N"]
    cfg = {"workload": args.workload, "B": B, "H": H, "S": S, "D": D, "N": N, "query_tokens": 1,
           "l2": "KV cache (4.3 GB) larger than L2, no flush",
           "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"}
    cores = len(os.sched_getaffinity(0))
    if args.impl == "reference":
        if rank != 0:
            return
        inp = make_decode_inputs(1, 2, S, D, w["seed"], scale=w["scale"])
        w1 = dict(w, B=1, H=2)
        per_step = max(1.0, 60.0 / max(1, args.steps + args.warmup))
        for _ in range(args.warmup):
            decode_oracle_sample(inp, w1, per_step / 4)
        tot_b = tot_t = 0.0
        desc = ""
        for _ in range(args.steps):
            nb, t, desc = decode_oracle_sample(inp, w1, per_step)
            tot_b += nb
            tot_t += t
        val = tot_b / tot_t / 1e9
        print(json.dumps({
            "impl": "reference", "metric": DECODE_METRIC, "value": val, "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg,
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"per step: {desc}"},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)
        return

    import ring_attention_fwd_gb300 as ra
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    inp = make_decode_inputs(B, H, S, D, w["seed"], scale=w["scale"])
    dev = {k: v.cuda() for k, v in inp.items()}
    o = torch.empty_like(dev["q"])
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    work = torch.empty(ra.decode_workspace_bytes(B, H, S, D, N), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        ra.decode(dev["q"], dev["k"], dev["v"], N, o=o, lse=lse, workspace=work)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ra.check_device_status()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    steps = args.steps * 20          # a call takes well under a millisecond
    ra.set_kernel_timing(True)
    with ClockSampler(local) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        time.sleep(0.3)              # at least one clock sample
    ktimes = ra.kernel_times()
    ra.set_kernel_timing(False)
    ra.check_device_status()
    total_ms = t0.elapsed_time(t1)
    if ws > 1:
        tt = torch.tensor([total_ms], device="cuda")
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(tt.item())
    ms_step = total_ms / steps
    nbytes = _decode_bytes(B, H, S, D)
    value = nbytes * ws / (ms_step * 1e-3) / 1e9
    per_kernel = {}
    for name, ms in ktimes:
        per_kernel.setdefault(name, []).append(ms)
    kernels = {n: {"launches": len(l), "ms": statistics.mean(l)} for n, l in per_kernel.items()}
    split_ms = kernels["decode_split"]["ms"]
    split_bytes = B * H * (2 * S * D * 2 + D * 2)          # reads q, K, V
    hbm, hsrc = _hbm_peak()
    achieved = split_bytes / (split_ms * 1e-3) / 1e9
    # the combine reads every partial (the workspace: items x (D + 1) floats, padded to 256 B)
    # and writes O (bf16) and LSE (f32) per head
    comb = kernels.get("decode_combine")
    if comb:
        cb = ra.decode_workspace_bytes(B, H, S, D, N) + B * H * (2 * D + 4)
        comb.update(bytes=cb, gbps=cb / (comb["ms"] * 1e-3) / 1e9, frac_of_hbm=cb / (comb["ms"] * 1e-3) / 1e9 / hbm,
                    bound="latency: one CTA per head walks its partials serially")
    tr = NCU_TRAFFIC.get("decode_split")
    traffic = tr["bytes_per_launch"] if tr and tr["sha256"] == _src_hash("decode.cu") and \
        tr["workload"] == args.workload else None

    # end to end: the cache stays resident (it is the server's state); each
    # step copies the new query in from pinned memory and the result out
    qh = inp["q"].pin_memory()
    oh = torch.empty_like(o, device="cpu").pin_memory()
    lh = torch.empty_like(lse, device="cpu").pin_memory()

    def e2e_step():
        dev["q"].copy_(qh, non_blocking=True)
        step()
        oh.copy_(o, non_blocking=True)
        lh.copy_(lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a.elapsed_time(b) / steps
    line = {
        "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
        "tokens_per_s": B * ws / (ms_step * 1e-3),
        "roofline": {"bound": "hbm", "kernel": "decode_split", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic, "algorithmic_bytes_per_launch": split_bytes,
                     "avg_launch_ms": split_ms, "peak_kind": hsrc},
        "e2e": {"value": nbytes * ws / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": qh.numel() * qh.element_size(),
                "d2h_bytes_per_step": oh.numel() * oh.element_size() + lh.numel() * lh.element_size()},
        "kernels": kernels,
        "gpu_launches": len(ktimes),
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        nb, t, desc = decode_oracle_sample({k: v[:1, :2] for k, v in inp.items()}, dict(w, B=1, H=2),
                                           args.cpu_seconds)
        line["cpu_baseline"] = {"value": nb / t / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": desc + f"; {t:.1f} s"}
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


FFN_METRIC = "blockwise gated FFN TFLOP/s (LLaMA-7B-shaped layer, 16384 tokens, blocks of 4096)"


def ffn_oracle_sample(inp, w, budget_s: float):
    """Time the oracle's feedforward on batches of 16 random rows until
    `budget_s` is spent.  Returns (flops, seconds, description)."""
    import numpy as np
    import oracle as orc
    x = inp["x"]
    w1, w3, w2 = (inp[k].double().numpy() for k in ("w1", "w3", "w2"))
    rng = np.random.default_rng(0)
    rows_done, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s or rows_done == 0:
        rows = np.sort(rng.choice(x.shape[0], size=16, replace=False))
        orc.ffn_rows(x[rows].double().numpy(), w1, w3, w2)
        rows_done += 16
    dt = time.perf_counter() - t0
    return 6.0 * rows_done * w["h"] * w["f"], dt, f"{rows_done} random rows, numpy float64 matmuls"


def run_ffn(args, w):
    """Blockwise gated feedforward of one host's tokens, weights resident."""
    import torch
    from ring_attention_fwd_gb300.inputs import make_ffn_inputs
    ws, rank, local = _dist()
    T, h, f, c = w["T"], w["h"], w["f"], w["block_rows"]
    flops = 6.0 * T * h * f
    cfg = {"workload": args.workload, "tokens": T, "hidden": h, "intermediate": f, "block_rows": c,
           "ffn": "gated (silu)", "l2": "weights 270 MB + X 134 MB, larger than L2, no flush",
           "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"}
    cores = len(os.sched_getaffinity(0))
    inp = make_ffn_inputs(T, h, f, w["seed"])
    if args.impl == "reference":
        if rank != 0:
            return
        per_step = max(1.0, 60.0 / max(1, args.steps + args.warmup))
        ffn_oracle_sample(inp, w, per_step / 4)
        tot_f = tot_t = 0.0
        desc = ""
        for _ in range(args.steps):
            fl, t, desc = ffn_oracle_sample(inp, w, per_step)
            tot_f += fl
            tot_t += t
        val = tot_f / tot_t / 1e12
        print(json.dumps({
            "impl": "reference", "metric": FFN_METRIC, "value": val, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)
        return

    import ring_attention_fwd_gb300 as ra
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = {k: v.cuda() for k, v in inp.items()}
    y = torch.empty_like(dev["x"])
    work = torch.empty(ra.ffn_workspace_bytes(T, h, f, c), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        ra.ffn(dev["x"], dev["w1"], dev["w3"], dev["w2"], c, y=y, workspace=work)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ra.check_device_status()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # The step is timed with no events between its launches (consecutive
    # launches overlap); a second pass records the library's per-kernel events.
    with ClockSampler(local) as clk:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
    ra.set_kernel_timing(True)
    for _ in range(args.steps):
        step()
    ktimes = ra.kernel_times()
    ra.set_kernel_timing(False)
    ra.check_device_status()
    total_ms = t0.elapsed_time(t1)
    if ws > 1:
        tt = torch.tensor([total_ms], device="cuda")
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(tt.item())
    ms_step = total_ms / args.steps
    per_kernel = {}
    for name, ms in ktimes:
        per_kernel.setdefault(name, []).append(ms)
    nblocks = -(-T // c)
    algo = {"ffn_up": 4.0 * c * h * f, "ffn_down": 2.0 * c * h * f}    # per launch (full blocks)
    kernels = {}
    for n, l in per_kernel.items():
        kernels[n] = {"launches": len(l), "ms": statistics.mean(l)}
        if n in algo:
            kernels[n]["tflops"] = algo[n] / (kernels[n]["ms"] * 1e-3) / 1e12
    burst, sustained, src = _peaks()
    dom = max(kernels, key=lambda n: kernels[n]["ms"] * kernels[n]["launches"])
    achieved = kernels[dom]["tflops"]
    tr = NCU_TRAFFIC.get(dom)
    traffic = tr["bytes_per_launch"] if tr and tr["sha256"] == _src_hash("ffn.cu") and \
        tr["workload"] == args.workload else None
    xh = inp["x"].pin_memory()
    yh = torch.empty_like(y, device="cpu").pin_memory()
    xs, ys = [dev["x"], torch.empty_like(dev["x"])], [y, torch.empty_like(y)]
    e2e_steps = max(8, args.steps)          # amortises the unhidden first upload and last download
    e2e_ms = pipelined_e2e(
        e2e_steps, stream, lambda b: [(xs[b], xh)],
        lambda b: ra.ffn(xs[b], dev["w1"], dev["w3"], dev["w2"], c, y=ys[b], workspace=work),
        lambda b: [(yh, ys[b])])
    line = {
        "metric": FFN_METRIC, "value": flops * ws / (ms_step * 1e-3) / 1e12, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random-init weights)",
        "config": cfg, "tokens_per_s": T * ws / (ms_step * 1e-3),
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": sustained, "unit": UNIT,
                     "frac": achieved / sustained, "traffic": traffic, "algorithmic_flops_per_launch": algo[dom],
                     "avg_launch_ms": kernels[dom]["ms"], "peak_kind": f"{src} sustained bf16 (burst {burst})",
                     "frac_of_burst": achieved / burst},
        "e2e": {"value": flops * ws / (e2e_ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": xh.numel() * xh.element_size(),
                "d2h_bytes_per_step": yh.numel() * yh.element_size(), "steps": e2e_steps,
                "copies": "overlapped with the neighbouring steps' compute on two copy streams (up, down); double-buffered"},
        "kernels": kernels, "kernels_note": "per-kernel times from a second pass with events between launches",
        "blocks_per_step": nblocks,
        "gpu_launches": len(ktimes),
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        fl, t, desc = ffn_oracle_sample(inp, w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": fl / t / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc + f"; {t:.1f} s"}
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_128k")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--heads", type=int, default=0,
                    help="run the workload with this many heads instead of its own (same per-head shape; "
                         "for profiling captures that must stay small)")
    ap.add_argument("--kernels-only", action="store_true",
                    help="time the kernels only: no end-to-end copies, merge or CPU baseline (profiling runs)")
    ap.add_argument("--oracle-full", action="store_true",
                    help="time the oracle on the whole workload (every head and row) for cpu_baseline instead of "
                         "a bounded sample; tens of minutes at 65536 tokens and beyond")
    ap.add_argument("--fwd-kernel", default="single", choices=["single", "pair"],
                    help="bf16 forward kernel: one CTA per SM (the library's default) or SM pairs")
    ap.add_argument("--balance", action="store_true",
                    help="report per-virtual-host work and time, striped vs contiguous (default workload balance_32k)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    from ring_attention_fwd_gb300.inputs import WORKLOADS
    if args.balance:
        if args.workload == "long_128k" and "--workload" not in sys.argv:
            args.workload = "balance_32k"
        run_balance(args)
        return
    from ring_attention_fwd_gb300.inputs import DECODE_WORKLOADS, FFN_WORKLOADS
    if args.workload in FFN_WORKLOADS:
        run_ffn(args, dict(FFN_WORKLOADS[args.workload]))
        return
    if args.workload in DECODE_WORKLOADS:
        run_decode(args, dict(DECODE_WORKLOADS[args.workload]))
        return
    from ring_attention_fwd_gb300.inputs import LONG_WORKLOADS
    w = dict(WORKLOADS[args.workload] if args.workload in WORKLOADS else LONG_WORKLOADS[args.workload])
    if args.heads > 0:
        w["H"] = args.heads
    if args.kernels_only:
        args.no_cpu_baseline = True
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
