"""What the peaked inputs (``inputs.make_peaked_inputs``) force, computed from
the inputs alone in float64 on the CPU.

The forward kernel keeps a per-row reference maximum and rescales O (and l)
only when a new tile's row maximum exceeds it by more than 8 in log2 units
(a factor 2^8).  These helpers compute, for every query row, the row maximum of
each KV tile in the order the ring sweep meets them, and count the places
where that maximum jumps by more than the threshold after keys have already
been folded in -- each is a place where O must be rescaled for the result to
be right ([AQ] §分块注意力: m_new = max(m, rowmax S), alpha = e^(m - m_new)).
"""
from __future__ import annotations

import numpy as np

import oracle as orc

RESCALE_LOG2 = 8.0
KV_TILE = 128


def tile_maxima(q, k, N: int, causal: bool, layout: str) -> np.ndarray:
    """float64 [S, T]: for each query row, the maximum scaled score (log2
    units) of the T-th KV tile its sweep meets (ring order of blocks, tiles of
    128 keys ascending inside a block); -inf for tiles skipped or without a
    visible key.  T = N * ceil(c / 128)."""
    S, D = q.shape
    c = S // N
    nkt = -(-c // KV_TILE)
    pos = orc.token_positions(S, N, layout)
    out = np.full((S, N * nkt), -np.inf)
    for i in range(N):
        rows = np.arange(i * c, (i + 1) * c)
        for s, j in enumerate(orc.ring_order(i, N)):
            if causal and layout == orc.CONTIGUOUS and j > i:
                continue
            for kt in range(nkt):
                keys = np.arange(j * c + kt * KV_TILE, j * c + min(c, (kt + 1) * KV_TILE))
                sc = (q[rows] @ k[keys].T) / np.sqrt(D)
                sc = np.where(orc.visible(pos[rows], pos[keys], causal), sc, -np.inf)
                out[rows, s * nkt + kt] = sc.max(axis=1) / np.log(2.0)
    return out


def rescale_events(maxima: np.ndarray) -> np.ndarray:
    """Per row, the number of tiles whose maximum exceeds the running reference
    by more than the threshold after a finite reference exists (the reference
    follows the kernel's rule: it moves only on such a jump, or on the first
    finite maximum)."""
    S, T = maxima.shape
    ref = np.full(S, -np.inf)
    ev = np.zeros(S, dtype=np.int64)
    for t in range(T):
        m = maxima[:, t]
        jump = m > ref + RESCALE_LOG2
        ev += jump & np.isfinite(ref)
        ref = np.where(jump, m, ref)
    return ev


def blocks_seen(maxima: np.ndarray, N: int) -> np.ndarray:
    """Per row, how many KV blocks contribute at least one visible key."""
    S, T = maxima.shape
    return np.isfinite(maxima.reshape(S, N, T // N)).any(axis=2).sum(axis=1)


# (B, H, S, N, causal, layout, mode): shapes span several tiles, ragged tiles
# (c = 200, 900), one block (N = 1), both layouts, and causal and not.
PEAKED_CASES = [
    (1, 2, 1024, 4, True, "contiguous", "ring"),
    (1, 2, 1024, 4, True, "striped", "ring"),
    (1, 1, 1600, 8, True, "contiguous", "ring"),      # c = 200: ragged KV tiles and units
    (1, 1, 1600, 8, True, "striped", "ring"),
    (2, 1, 2048, 8, True, "striped", "ring"),
    (1, 2, 1024, 4, False, "contiguous", "ring"),
    (1, 1, 1024, 1, True, "contiguous", "tiles"),     # one block: the jumps are between its 8 tiles
    (1, 1, 900, 1, True, "contiguous", "tiles"),      # ragged last tile
    (1, 2, 1536, 6, True, "contiguous", "planted"),
    (1, 2, 1536, 6, True, "striped", "planted"),
]


def expected_events_ok(mode: str, maxima: np.ndarray, ev: np.ndarray, N: int) -> bool:
    """What each construction guarantees, row by row."""
    S = maxima.shape[0]
    if mode == "ring":       # every further block raises the maximum past the threshold
        return bool(np.all(ev == blocks_seen(maxima, N) - 1))
    if mode == "tiles":      # every further tile does
        return bool(np.all(ev == np.isfinite(maxima).sum(axis=1) - 1))
    c = S // N               # planted: every row outside block 0 meets it after other keys
    return bool(np.all(ev[c:] >= 1))


def _bf16(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float64).numpy()


def rounding_floor(q, k, v, do, o_ref, lse_ref, o_saved, lse_saved, N: int, causal: bool, layout: str):
    """Deviation of each gradient of ONE head caused by the backward's bf16
    rounding points alone, from a float64 emulation on the oracle's causal
    rule: P enters the dV product in bf16, dS = P (dP - D_vec) enters the dQ
    and dK products in bf16, and dQ, dK, dV are stored in bf16; everything else
    exact.  The emulated kernel starts from the saved state (o_saved,
    lse_saved); the reference gradient from (o_ref, lse_ref) -- the same
    state when the backward alone is judged, the exact forward state when the
    forward feeding the backward is (then D_vec's use of the bf16 O counts).
    Returns {name: (max abs deviation, Frobenius norm of the deviation)}.

    On peaked inputs the keys of one block share a large component that
    cancels in dQ = dS K (each row of dS sums to ~0) but not in its rounding
    error, which is why these inputs need this floor beside the tolerance of
    unstructured inputs."""
    S, D = q.shape
    pos = orc.token_positions(S, N, layout)
    s = q @ k.T / np.sqrt(D)
    dP = do @ v.T

    def state(o, lse):
        vis = orc.visible(pos, pos, causal) & np.isfinite(lse)[:, None]
        P = np.where(vis, np.exp(np.where(vis, s - lse[:, None], 0.0)), 0.0)
        return P, P * (dP - (do * o).sum(axis=1)[:, None])

    P, dS = state(o_ref, lse_ref)
    exact = {"dQ": dS @ k / np.sqrt(D), "dK": dS.T @ q / np.sqrt(D), "dV": P.T @ do}
    P, dS = state(o_saved, lse_saved)
    Pb, dSb = _bf16(P), _bf16(dS)
    rounded = {"dQ": _bf16(dSb @ k / np.sqrt(D)), "dK": _bf16(dSb.T @ q / np.sqrt(D)), "dV": _bf16(Pb.T @ do)}
    return {n: (float(np.abs(rounded[n] - exact[n]).max()), float(np.linalg.norm(rounded[n] - exact[n])))
            for n in exact}


def emulated_forward_o(q, k, v, N: int, causal: bool, layout: str):
    """The forward's output of ONE head with its bf16 rounding points
    emulated in float64: P = e^(s - rowmax) enters the P V product in bf16,
    the row sum stays unrounded, and O is stored in bf16."""
    S, D = q.shape
    pos = orc.token_positions(S, N, layout)
    s = np.where(orc.visible(pos, pos, causal), q @ k.T / np.sqrt(D), -np.inf)
    e = np.exp(s - s.max(axis=1)[:, None])
    return _bf16((_bf16(e) @ v) / e.sum(axis=1)[:, None])
