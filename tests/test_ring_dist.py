"""Multi-process ring forward on CPU (gloo): the K/V exchange protocol of
ring_attention_fwd_gb300.ring with the CPU oracle computing each block pair.

Each rank is one ring host.  The injected block compute checks that the K/V
block a rank holds in round s is exactly block (rank - s) mod N, then folds
the oracle's partial state for that pair; the final rows of every rank must
equal the oracle's full attention.  No GPU is involved."""
import datetime
import os
import socket
import tempfile

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as orc


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(S, D, seed):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((S, D)) for _ in range(3)]


def _worker(rank, world, port, S, D, causal, layout, outdir, mode):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=20))
    try:
        from ring_attention_fwd_gb300.ring import ring_forward
        q, k, v = _inputs(S, D, 5)
        c = S // world
        blk = lambda x, b: torch.from_numpy(x[b * c:(b + 1) * c].copy())[None, None]  # [1,1,c,D]
        seen = []

        def step(qq, kk, vv, n, i, j):
            assert torch.equal(kk, blk(k, j)) and torch.equal(vv, blk(v, j)), f"rank {i}: wrong block for {j}"
            seen.append(j)
            qf, kf, vf = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
            qf[i * c:(i + 1) * c] = qq[0, 0].numpy()
            kf[j * c:(j + 1) * c] = kk[0, 0].numpy()
            vf[j * c:(j + 1) * c] = vv[0, 0].numpy()
            o, l = orc.block_pair_attention(qf, kf, vf, i, j, n, causal, layout)
            return torch.from_numpy(o)[None, None], torch.from_numpy(l)[None, None]

        def merge(o, l, oj, lj):
            mo, ml = orc.lse_merge(o[0, 0].numpy(), l[0, 0].numpy(), oj[0, 0].numpy(), lj[0, 0].numpy())
            o[0, 0] = torch.from_numpy(mo)
            l[0, 0] = torch.from_numpy(ml)

        if mode == "leave" and rank == 1:
            return                       # this host leaves before its first send
        if mode == "late" and rank == 1:
            import time
            time.sleep(1.5)              # this host's blocks arrive late, but within the time-out
        try:
            o, l = ring_forward(blk(q, rank), blk(k, rank), blk(v, rank), causal=causal, layout=layout,
                                step=step, merge=merge,
                                timeout_s={"leave": 3.0, "late": 10.0}.get(mode))
        except Exception as e:           # noqa: BLE001 - reported to the parent
            with open(os.path.join(outdir, f"err{rank}.txt"), "w") as f:
                f.write(type(e).__name__ + ": " + str(e))
            return
        np.save(os.path.join(outdir, f"o{rank}.npy"), o[0, 0].numpy())
        np.save(os.path.join(outdir, f"l{rank}.npy"), l[0, 0].numpy())
        np.save(os.path.join(outdir, f"seen{rank}.npy"), np.array(seen))
    finally:
        if mode != "leave":
            dist.destroy_process_group()


@pytest.mark.parametrize("world,layout,causal", [(2, "contiguous", True), (2, "striped", True),
                                                 (4, "striped", True), (4, "contiguous", True),
                                                 (3, "contiguous", False)])
def test_ring_forward_gloo_matches_full_attention(world, layout, causal):
    S, D = 12 * world, 8
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_worker, args=(world, _free_port(), S, D, causal, layout, d, "ok"), nprocs=world, join=True)
        q, k, v = _inputs(S, D, 5)
        c = S // world
        fo, fl = orc.attention_rows(q, k, v, np.arange(S), world, causal, layout)
        for r in range(world):
            assert not os.path.exists(os.path.join(d, f"err{r}.txt")), open(os.path.join(d, f"err{r}.txt")).read()
            np.testing.assert_allclose(np.load(os.path.join(d, f"o{r}.npy")), fo[r * c:(r + 1) * c], atol=1e-12)
            np.testing.assert_allclose(np.load(os.path.join(d, f"l{r}.npy")), fl[r * c:(r + 1) * c], atol=1e-12)
            order = orc.ring_order(r, world)
            expect = [j for j in order if not (causal and layout == "contiguous" and j > r)]
            assert np.load(os.path.join(d, f"seen{r}.npy")).tolist() == expect


@pytest.mark.timeout(120)
def test_ring_forward_tolerates_a_late_host():
    """A host whose sends start 1.5 s late (inside the 10 s exchange limit)
    delays the ring but every rank still gets the exact result."""
    world, S, D = 3, 36, 8
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_worker, args=(world, _free_port(), S, D, True, "striped", d, "late"), nprocs=world, join=True)
        q, k, v = _inputs(S, D, 5)
        c = S // world
        fo, fl = orc.attention_rows(q, k, v, np.arange(S), world, True, "striped")
        for r in range(world):
            assert not os.path.exists(os.path.join(d, f"err{r}.txt")), open(os.path.join(d, f"err{r}.txt")).read()
            np.testing.assert_allclose(np.load(os.path.join(d, f"o{r}.npy")), fo[r * c:(r + 1) * c], atol=1e-12)
            np.testing.assert_allclose(np.load(os.path.join(d, f"l{r}.npy")), fl[r * c:(r + 1) * c], atol=1e-12)


@pytest.mark.timeout(120)
def test_ring_forward_reports_a_host_that_left():
    """A host that leaves before sending must surface as an error on its
    neighbour within the exchange time-out, not as a hang."""
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_worker, args=(2, _free_port(), 24, 8, True, "striped", d, "leave"), nprocs=2, join=True)
        assert os.path.exists(os.path.join(d, "err0.txt"))
        assert not os.path.exists(os.path.join(d, "o0.npy"))


# ------------------------------------------------------------------ ring decode
def _decode_inputs(B, H, S, D, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((B, H, D)), rng.standard_normal((B, H, S, D)), rng.standard_normal((B, H, S, D))


def _oracle_partial(q, k, v):
    """Oracle partial of one cache segment for every (b, h)."""
    B, H, D = q.shape
    o, l = np.zeros((B, H, D)), np.zeros((B, H))
    for b in range(B):
        for h in range(H):
            o[b, h], l[b, h] = orc.decode_attention(q[b, h], k[b, h], v[b, h])
    return o, l


def _decode_worker(rank, world, port, B, H, S, D, outdir, mode):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=20))
    try:
        from ring_attention_fwd_gb300.ring import ring_decode
        q, k, v = _decode_inputs(B, H, S, D, 11)
        blocks = orc.decode_blocks(S, world)
        partials = [_oracle_partial(q, k[:, :, a:b], v[:, :, a:b]) for (a, b) in blocks]
        a, b = blocks[rank]
        merged = []

        def step(qq, kk, vv):
            assert kk.shape[2] == b - a
            o, l = _oracle_partial(qq.numpy(), kk.numpy(), vv.numpy())
            return torch.from_numpy(o), torch.from_numpy(l)

        def merge(o, l, oj, lj):
            # which block's partial arrived (by value; empty partials compare equal to each other)
            hits = [j for j, (po, pl) in enumerate(partials)
                    if np.array_equal(pl, lj.numpy()) and np.array_equal(po, oj.numpy())]
            merged.append(hits)
            for bb in range(o.shape[0]):
                mo, ml = orc.lse_merge(o[bb].numpy(), l[bb].numpy(), oj[bb].numpy(), lj[bb].numpy())
                o[bb] = torch.from_numpy(mo)
                l[bb] = torch.from_numpy(ml)

        if mode == "leave" and rank == 1:
            return
        try:
            o, l = ring_decode(torch.from_numpy(q), torch.from_numpy(k[:, :, a:b].copy()),
                               torch.from_numpy(v[:, :, a:b].copy()), step=step, merge=merge,
                               timeout_s=3.0 if mode == "leave" else None, lse_dtype=torch.float64)
        except Exception as e:           # noqa: BLE001 - reported to the parent
            with open(os.path.join(outdir, f"err{rank}.txt"), "w") as f:
                f.write(type(e).__name__ + ": " + str(e))
            return
        np.save(os.path.join(outdir, f"o{rank}.npy"), o.numpy())
        np.save(os.path.join(outdir, f"l{rank}.npy"), l.numpy())
        with open(os.path.join(outdir, f"merged{rank}.txt"), "w") as f:
            f.write(repr(merged))
    finally:
        if mode != "leave":
            dist.destroy_process_group()


@pytest.mark.parametrize("world,S", [(2, 40), (4, 37), (3, 2)])
def test_ring_decode_gloo_matches_whole_cache(world, S):
    """Every rank ends with the decode of the whole cache; rank i merges the
    partials of blocks i-1, i-2, ... in that order (S=2 on 3 ranks: one empty block)."""
    B, H, D = 2, 2, 8
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_decode_worker, args=(world, _free_port(), B, H, S, D, d, "ok"), nprocs=world, join=True)
        q, k, v = _decode_inputs(B, H, S, D, 11)
        ro, rl = orc.decode_batch(q, k, v, world)
        blocks = orc.decode_blocks(S, world)
        for r in range(world):
            assert not os.path.exists(os.path.join(d, f"err{r}.txt")), open(os.path.join(d, f"err{r}.txt")).read()
            np.testing.assert_allclose(np.load(os.path.join(d, f"o{r}.npy")), ro, atol=1e-12)
            np.testing.assert_allclose(np.load(os.path.join(d, f"l{r}.npy")), rl, atol=1e-12)
            merged = eval(open(os.path.join(d, f"merged{r}.txt")).read())   # noqa: S307 - our own repr
            order = orc.ring_order(r, world)[1:]
            assert len(merged) == world - 1
            for hits, j in zip(merged, order):
                assert j in hits or (blocks[j][0] == blocks[j][1] and hits), (r, merged, order)


@pytest.mark.timeout(120)
def test_ring_decode_reports_a_host_that_left():
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_decode_worker, args=(2, _free_port(), 1, 1, 16, 4, d, "leave"), nprocs=2, join=True)
        assert os.path.exists(os.path.join(d, "err0.txt"))
        assert not os.path.exists(os.path.join(d, "o0.npy"))


# ------------------------------------------------------------------ ring backward
def _bwd_worker(rank, world, port, S, D, causal, layout, outdir, mode):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=20))
    try:
        from ring_attention_fwd_gb300.ring import ring_backward
        rng = np.random.default_rng(21)
        q, k, v, do = (rng.standard_normal((S, D)) for _ in range(4))
        o, lse = orc.attention_rows(q, k, v, np.arange(S), world, causal, layout)
        c = S // world
        blk = lambda x, b: torch.from_numpy(x[b * c:(b + 1) * c].copy())[None, None]
        seen = []

        def step(qq, kk, vv, oo, ll, dd, gq, gk, gv, n, i, j):
            assert torch.equal(kk, blk(k, j)) and torch.equal(vv, blk(v, j)), f"rank {i}: wrong block for {j}"
            assert gq.dtype == torch.float32 and gk.dtype == torch.float32
            # the round adds into a fresh partial: it never waits for the accumulators in flight
            assert not gk.any() and not gv.any(), f"rank {i}: round {j} got a non-zero dK/dV buffer"
            seen.append(j)
            a, b, cc = orc.block_pair_bwd(q, k, v, o, lse, do, i, j, n, causal, layout)
            gq[0, 0] += torch.from_numpy(a).float()
            gk[0, 0] += torch.from_numpy(b).float()
            gv[0, 0] += torch.from_numpy(cc).float()

        if mode == "leave" and rank == 1:
            return
        try:
            dq, dk, dv = ring_backward(blk(q, rank), blk(k, rank), blk(v, rank), blk(o, rank),
                                       torch.from_numpy(lse[rank * c:(rank + 1) * c].copy())[None, None],
                                       blk(do, rank), causal=causal, layout=layout, step=step,
                                       timeout_s=3.0 if mode == "leave" else None)
        except Exception as e:           # noqa: BLE001 - reported to the parent
            with open(os.path.join(outdir, f"err{rank}.txt"), "w") as f:
                f.write(type(e).__name__ + ": " + str(e))
            return
        for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
            np.save(os.path.join(outdir, f"{name}{rank}.npy"), t[0, 0].double().numpy())
        np.save(os.path.join(outdir, f"seen{rank}.npy"), np.array(seen))
    finally:
        if mode != "leave":
            dist.destroy_process_group()


@pytest.mark.parametrize("world,layout,causal", [(2, "contiguous", True), (3, "striped", True),
                                                 (4, "contiguous", True), (2, "contiguous", False)])
def test_ring_backward_gloo_matches_full_gradient(world, layout, causal):
    """Every rank ends with its rows of dQ, dK, dV of the whole sequence; the
    float32 accumulators limit agreement to ~1e-6 relative."""
    S, D = 8 * world, 6
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_bwd_worker, args=(world, _free_port(), S, D, causal, layout, d, "ok"), nprocs=world, join=True)
        rng = np.random.default_rng(21)
        q, k, v, do = (rng.standard_normal((S, D)) for _ in range(4))
        o, lse = orc.attention_rows(q, k, v, np.arange(S), world, causal, layout)
        ref = orc.attention_bwd_head(q, k, v, o, lse, do, world, causal, layout)
        c = S // world
        for r in range(world):
            assert not os.path.exists(os.path.join(d, f"err{r}.txt")), open(os.path.join(d, f"err{r}.txt")).read()
            for name, full in zip(("dq", "dk", "dv"), ref):
                np.testing.assert_allclose(np.load(os.path.join(d, f"{name}{r}.npy")), full[r * c:(r + 1) * c],
                                           atol=1e-5, rtol=1e-5)
            expect = [j for j in orc.ring_order(r, world) if not (causal and layout == "contiguous" and j > r)]
            assert np.load(os.path.join(d, f"seen{r}.npy")).tolist() == expect


@pytest.mark.timeout(120)
def test_ring_backward_reports_a_host_that_left():
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_bwd_worker, args=(2, _free_port(), 16, 4, True, "striped", d, "leave"), nprocs=2, join=True)
        assert os.path.exists(os.path.join(d, "err0.txt"))
        assert not os.path.exists(os.path.join(d, "dq0.npy"))
