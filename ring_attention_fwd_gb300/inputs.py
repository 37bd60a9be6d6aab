"""Seeded synthetic inputs for ring attention workloads.

This module only draws random numbers; it contains none of the attention
arithmetic.  Both the CUDA path's tests/bench and the CPU oracle consume the
tensors it returns, so the two sides see bit-identical inputs.

Recipe (fixed, so that every caller reproduces the same values):
  * one ``torch.Generator('cpu')`` seeded with ``seed``;
  * tensors drawn in the order Q, K, V, dO (dO only when requested);
  * inside a tensor, one ``randn(S, D)`` float32 draw per (b, h) slab, in
    row-major (b, h) order;
  * each slab is multiplied by ``scale`` (0.5 for the 131072-token workload:
    a power of two, so the product is exact) and then rounded to the storage
    dtype with round-to-nearest-even (``Tensor.to``).

The tensors are in *storage order* [B, H, S, D]: for the striped layout,
storage row ``p = i*c + r`` of a head holds token ``r*N + i``; the generator
does not care, it only fills storage rows.
"""
from __future__ import annotations

import torch

_DTYPES = {"bf16": torch.bfloat16, "f32": torch.float32}


def make_inputs(B: int, H: int, S: int, D: int, seed: int, *, dtype: str = "bf16",
                scale: float = 1.0, with_grad: bool = False) -> dict:
    """Return {'q','k','v'[, 'do']} CPU tensors of shape [B, H, S, D]."""
    if dtype not in _DTYPES:
        raise ValueError(f"dtype must be one of {sorted(_DTYPES)}")
    tdt = _DTYPES[dtype]
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    names = ["q", "k", "v"] + (["do"] if with_grad else [])
    out = {}
    for name in names:
        t = torch.empty((B, H, S, D), dtype=tdt)
        for b in range(B):
            for h in range(H):
                x = torch.randn((S, D), generator=g, dtype=torch.float32)
                if scale != 1.0:
                    x.mul_(scale)
                t[b, h].copy_(x.to(tdt))
        out[name] = t
    return out


# Peaked inputs: the structure below makes the running row maximum of the
# online softmax jump by a known amount, so that the O correction runs.
PEAK_A = 16.0      # query coordinate
PEAK_B = 8.0       # key coordinate per ring step (score step A*B/sqrt(128) = 11.3)
PEAK_PLANT = 40.0  # planted key coordinate (score A*40/sqrt(128) = 56.6)


def make_peaked_inputs(B: int, H: int, S: int, N: int, seed: int, mode: str = "ring") -> dict:
    """bf16 {'q','k','v','do'} [B, H, S, 128] whose scores grow along the ring.

    ``make_inputs`` (seeded, N(0,1)) first; then some coordinates of q and k
    are overwritten with fixed values (all exact in bf16), the rest stay
    random.  Storage block i holds rows [i*c, (i+1)*c), c = S/N.
      * ``ring`` (N <= 64): coordinate x < N of a query row in block i is
        PEAK_A if x == i, else 0; of a key row in block j it is
        PEAK_B * ((x - j) mod N).  The score of a block-i query and a block-j
        key is PEAK_A*PEAK_B*((i - j) mod N)/sqrt(128) plus the random part:
        it grows by 11.3 at every step of the ring order j = i, i-1, ...
      * ``tiles``: coordinate 0 of every query is PEAK_A and of a key at row
        r of its block PEAK_B * (r // 128): scores grow by 11.3 from one
        128-key tile to the next, inside every block.
      * ``planted``: coordinate 0 of every query is PEAK_A, of every key 0,
        except storage row 0 (block 0's first token, which every query sees,
        and which a contiguous causal sweep meets last) with PEAK_PLANT: that
        key's score exceeds every other by about 50.
    v and dO are left as drawn."""
    if S % N:
        raise ValueError("S must be a multiple of N")
    t = make_inputs(B, H, S, 128, seed, with_grad=True)
    q, k = t["q"], t["k"]
    c = S // N
    if mode == "ring":
        if N > 64:
            raise ValueError("ring mode needs N <= 64")
        blk = torch.arange(S) // c                     # storage block of each row
        x = torch.arange(N)
        q[..., :N] = torch.where(x[None, :] == blk[:, None], PEAK_A, 0.0).to(q.dtype)
        k[..., :N] = (PEAK_B * ((x[None, :] - blk[:, None]) % N)).to(k.dtype)
    elif mode == "tiles":
        q[..., 0] = PEAK_A
        k[..., 0] = (PEAK_B * ((torch.arange(S) % c) // 128)).to(k.dtype)
    elif mode == "planted":
        q[..., 0] = PEAK_A
        k[..., 0] = 0.0
        k[..., 0, 0] = PEAK_PLANT
    else:
        raise ValueError(f"unknown mode {mode!r}")
    return t


def as_float64(t: torch.Tensor):
    """Upcast a CPU tensor (bf16 or f32) to a float64 NumPy array, exactly."""
    return t.to(torch.float64).numpy()


# The five workloads the library is specified against.  Names say what each
# is; sizes are the workload's own.  ``seed`` is the workload's 1-based index.
WORKLOADS = {
    "tiny_f32": dict(B=1, H=1, S=256, D=64, N=4, causal=False, layout="contiguous",
                     dtype="f32", scale=1.0, seed=1, grad=False),
    "causal_8k": dict(B=1, H=8, S=8192, D=128, N=8, causal=True, layout="contiguous",
                      dtype="bf16", scale=1.0, seed=2, grad=False),
    "balance_32k": dict(B=1, H=16, S=32768, D=128, N=16, causal=True, layout="striped",
                        dtype="bf16", scale=1.0, seed=3, grad=False),
    "long_128k": dict(B=1, H=32, S=131072, D=128, N=32, causal=True, layout="contiguous",
                      dtype="bf16", scale=0.5, seed=4, grad=False),
    "fwdbwd_64k": dict(B=1, H=32, S=65536, D=128, N=16, causal=True, layout="striped",
                       dtype="bf16", scale=1.0, seed=5, grad=True),
}


# Beyond the specified workloads: a sequence in the million-token range the
# method exists for (1,048,576 tokens in 64 ring blocks of 16384, 4 heads).
# Same recipe; measured by `bench.py --workload long_1m`, and a 2-head copy is
# the long-sequence parity case of the tests.
LONG_WORKLOADS = {
    "long_1m": dict(B=1, H=4, S=1 << 20, D=128, N=64, causal=True, layout="contiguous",
                    dtype="bf16", scale=0.5, seed=8, grad=True),
}


def make_decode_inputs(B: int, H: int, S: int, D: int, seed: int, *, scale: float = 1.0) -> dict:
    """Return {'q' [B, H, D], 'k', 'v' [B, H, S, D]} bf16 CPU tensors for ring
    decode: one new query token per (b, h) and an S-row KV cache.

    Same recipe as ``make_inputs``: one generator seeded with ``seed``; q first
    (one ``randn(1, D)`` per (b, h) slab), then K, then V (one ``randn(S, D)``
    per slab), each times ``scale`` and rounded to bf16 (nearest even)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    out = {}
    for name, rows in (("q", 1), ("k", S), ("v", S)):
        t = torch.empty((B, H, rows, D), dtype=torch.bfloat16)
        for b in range(B):
            for h in range(H):
                x = torch.randn((rows, D), generator=g, dtype=torch.float32)
                if scale != 1.0:
                    x.mul_(scale)
                t[b, h].copy_(x.to(torch.bfloat16))
        out[name] = t
    out["q"] = out["q"][:, :, 0].contiguous()
    return out


# Ring decode workload: one token of a 256K-token context, 32 heads of 128
# (the 32-host, 256K-context serving example of the reading notes, §5.6).
DECODE_WORKLOADS = {
    "decode_256k": dict(B=1, H=32, S=262144, D=128, N=32, scale=1.0, seed=6),
}


def make_ffn_inputs(T: int, h: int, f: int, seed: int) -> dict:
    """Return {'x' [T, h], 'w1', 'w3' [f, h], 'w2' [h, f]} bf16 CPU tensors for
    the blockwise feedforward (random-init weights of that architecture).

    One generator seeded with ``seed``; drawn in the order x, w1, w3, w2, each
    one ``randn`` of its full shape; x as drawn, each weight times
    1/sqrt(fan_in) (fan_in = its second dimension) so activations stay O(1);
    then rounded to bf16 (nearest even)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    out = {}
    for name, shape in (("x", (T, h)), ("w1", (f, h)), ("w3", (f, h)), ("w2", (h, f))):
        t = torch.randn(shape, generator=g, dtype=torch.float32)
        if name != "x":
            t.mul_(1.0 / float(shape[1]) ** 0.5)
        out[name] = t.to(torch.bfloat16)
    return out


# Blockwise feedforward workload: the gated feedforward of a LLaMA-7B-shaped
# layer (hidden 4096, intermediate 11008) over one host's 16384 tokens, in
# blocks of 4096 rows (the ring block size of the 131072-token workload).
FFN_WORKLOADS = {
    "ffn_7b": dict(T=16384, h=4096, f=11008, block_rows=4096, seed=7),
}
