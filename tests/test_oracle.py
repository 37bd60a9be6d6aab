"""Pins for the CPU oracle: what the pages and the mathematics fix, not the
oracle restated.  CPU only (no gpu marker)."""
import json
import math
import os

import numpy as np
import pytest

import oracle as orc

LAYOUTS = ["contiguous", "striped"]


def _rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


# ---------------------------------------------------------------- brute force
def _brute_force_head(q, k, v, N, causal, striped):
    """Scalar Python loops: softmax without max subtraction, direct sums.

    Token of storage row p: row r of block i is token i*c+r (contiguous) or
    r*N+i (striped) -- written here independently of the oracle.
    """
    S, D = len(q), len(q[0])
    c = S // N

    def tok(p):
        i, r = p // c, p % c
        return r * N + i if striped else p

    O, L = [], []
    for a in range(S):
        w = []
        for b in range(S):
            if causal and tok(b) > tok(a):
                w.append(0.0)
                continue
            dot = sum(q[a][x] * k[b][x] for x in range(D))
            w.append(math.exp(dot / math.sqrt(D)))
        tot = sum(w)
        O.append([sum(w[b] * v[b][x] for b in range(S)) / tot for x in range(D)])
        L.append(math.log(tot))
    return np.array(O), np.array(L)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S,N,D", [(8, 2, 4), (12, 3, 5), (16, 4, 8), (6, 1, 3)])
def test_brute_force_matches_both_forms(S, N, D, causal, layout):
    rng = np.random.default_rng(S * 100 + N * 10 + D + causal)
    q, k, v = (_rand(rng, 1, 1, S, D) for _ in range(3))
    ob, lb = _brute_force_head(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(), N, causal,
                               layout == "striped")
    on, ln = orc.naive_attention(q, k, v, N, causal, layout)
    orr, lr = orc.ring_attention(q, k, v, N, causal, layout)
    np.testing.assert_allclose(on[0, 0], ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ln[0, 0], lb, rtol=0, atol=1e-12)
    np.testing.assert_allclose(orr[0, 0], ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lr[0, 0], lb, rtol=0, atol=1e-12)


def test_demo_setup_of_the_explainer_agrees():
    """[AQ] §Python 演示: n=16, d=8, 4 devices, seed 42; the page expects the
    ring result to equal full attention for every device.  It prints no
    values, so this pin is agreement only."""
    np.random.seed(42)
    n, d, ndev = 16, 8, 4
    Q = np.random.randn(n, d)
    K = np.random.randn(n, d)
    V = np.random.randn(n, d)
    on, _ = orc.naive_attention(Q[None, None], K[None, None], V[None, None], ndev, False, "contiguous")
    b = n // ndev
    for dev in range(ndev):
        o, _ = orc.ring_block_attention(Q, K, V, dev, ndev, False, "contiguous")
        assert np.abs(o - on[0, 0, dev * b:(dev + 1) * b]).max() < 1e-14


# --------------------------------------------------------------- page fixtures
def test_striped_assignment_matches_page(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "striped_tokens_n4.json")))
    pos = orc.token_positions(g["S"], g["N"], "striped")
    c = g["S"] // g["N"]
    for i, toks in enumerate(g["tokens_per_device"]):
        assert pos[i * c:(i + 1) * c].tolist() == toks


def test_ring_order_matches_diagram(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "ring_diagram_n4.json")))
    N = g["N"]
    for step, held in g["block_held_at_step"].items():
        assert [orc.ring_order(i, N)[int(step)] for i in range(N)] == held
    # one step later, host (i+1) holds what host i held: i sends to i+1
    for i in range(N):
        dst = g["sends_to"][i]
        assert orc.ring_order(dst, N)[1] == orc.ring_order(i, N)[0]


def test_causal_block_work_matches_page(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "causal_work_100tok_n4.json")))
    w = orc.block_rectangle_work(g["S"], g["N"], g["layout"], g["causal"])
    assert w.tolist() == g["block_rectangle_work"]
    assert w[-1] // w[0] == g["ratio_last_to_first"]


def test_flop_convention_matches_pages(golden_dir):
    from ring_attention_fwd_gb300 import flops
    g = json.load(open(os.path.join(golden_dir, "block_pair_cost.json")))
    for case in g["cases"]:
        c, d = case["c"], case["d"]
        # one query block against one KV block, no mask: a 1-block sequence
        assert flops.fwd_flops(B=1, H=1, S=c, D=d, causal=False) == case["flops"]
        assert flops.kv_block_bytes(c, d) == case["kv_bytes"]


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("layout", LAYOUTS)
def test_equal_keys_give_prefix_mean(layout):
    """All keys equal -> uniform weights over the visible set: O(t) is the mean
    of the visible values and LSE = ln|visible| + s."""
    rng = np.random.default_rng(7)
    S, N, D = 24, 4, 6
    q = _rand(rng, 1, 1, S, D)
    krow = _rand(rng, D)
    k = np.broadcast_to(krow, (1, 1, S, D)).copy()
    v = _rand(rng, 1, 1, S, D)
    o, lse = orc.ring_attention(q, k, v, N, True, layout)
    pos = orc.token_positions(S, N, layout)
    by_token = np.empty((S, D))
    by_token[pos] = v[0, 0]
    for p in range(S):
        t = pos[p]
        np.testing.assert_allclose(o[0, 0, p], by_token[:t + 1].mean(axis=0), atol=1e-13)
        s = q[0, 0, p] @ krow / math.sqrt(D)
        assert abs(lse[0, 0, p] - (math.log(t + 1) + s)) < 1e-12


def test_zero_queries_non_causal_mean_and_log_count():
    rng = np.random.default_rng(8)
    S, N, D = 20, 5, 4
    q = np.zeros((1, 1, S, D))
    k, v = _rand(rng, 1, 1, S, D), _rand(rng, 1, 1, S, D)
    o, lse = orc.naive_attention(q, k, v, N, False, "contiguous")
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0].mean(axis=0), (S, D)), atol=1e-14)
    np.testing.assert_allclose(lse, math.log(S), atol=1e-14)


def test_equal_values_give_that_value():
    rng = np.random.default_rng(9)
    S, N, D = 16, 4, 5
    q, k = _rand(rng, 1, 1, S, D, scale=3.0), _rand(rng, 1, 1, S, D, scale=3.0)
    u = _rand(rng, D)
    v = np.broadcast_to(u, (1, 1, S, D)).copy()
    for layout in LAYOUTS:
        o, _ = orc.ring_attention(q, k, v, N, True, layout)
        np.testing.assert_allclose(o[0, 0], np.broadcast_to(u, (S, D)), atol=1e-13)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_first_token_sees_only_itself(layout):
    """Causal token 0 has a single visible key: O = v_0, LSE = q_0.k_0/sqrt(D)."""
    rng = np.random.default_rng(10)
    S, N, D = 16, 4, 8
    q, k, v = (_rand(rng, 1, 1, S, D) for _ in range(3))
    o, lse = orc.ring_attention(q, k, v, N, True, layout)
    p0 = int(np.where(orc.token_positions(S, N, layout) == 0)[0][0])
    np.testing.assert_allclose(o[0, 0, p0], v[0, 0, p0], atol=1e-15)
    assert abs(lse[0, 0, p0] - q[0, 0, p0] @ k[0, 0, p0] / math.sqrt(D)) < 1e-14


def test_single_block_ring_is_plain_softmax():
    rng = np.random.default_rng(11)
    q, k, v = (_rand(rng, 2, 2, 10, 4) for _ in range(3))
    for causal in (False, True):
        a = orc.ring_attention(q, k, v, 1, causal, "contiguous")
        b = orc.naive_attention(q, k, v, 1, causal, "striped")   # N=1: same map
        np.testing.assert_allclose(a[0], b[0], atol=1e-14)
        np.testing.assert_allclose(a[1], b[1], atol=1e-14)


# ------------------------------------------------------------------ invariants
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("causal", [False, True])
def test_block_order_invariance(layout, causal):
    """Any permutation of the KV blocks gives the same result ([FT] core
    insight; [CH] §4 first assumption)."""
    rng = np.random.default_rng(12)
    S, N, D = 48, 6, 8
    q, k, v = (_rand(rng, 1, 2, S, D, scale=2.0) for _ in range(3))
    ref = orc.ring_attention(q, k, v, N, causal, layout)
    for seed in range(4):
        perm_rng = np.random.default_rng(100 + seed)
        out = orc.ring_attention(q, k, v, N, causal, layout,
                                 order_fn=lambda i, n: list(perm_rng.permutation(n)))
        np.testing.assert_allclose(out[0], ref[0], atol=1e-13)
        np.testing.assert_allclose(out[1], ref[1], atol=1e-13)


def test_merge_of_key_halves_equals_whole():
    """Split the keys into two disjoint sets, attend to each, merge: equals
    attention over all keys ([FT] "Online Softmax" merge identity)."""
    rng = np.random.default_rng(13)
    S, D = 40, 8
    q, k, v = (_rand(rng, S, D, scale=2.0) for _ in range(3))
    whole_o, whole_l = orc.attention_rows(q, k, v, np.arange(S), 1, False, "contiguous")
    sel = rng.permutation(S)
    A, B = sel[:13], sel[13:]
    oa, la = orc.attention_rows(q, k[A], v[A], np.arange(S), 1, False, "contiguous")
    ob, lb = orc.attention_rows(q, k[B], v[B], np.arange(S), 1, False, "contiguous")
    om, lm = orc.lse_merge(oa, la, ob, lb)
    np.testing.assert_allclose(om, whole_o, atol=1e-13)
    np.testing.assert_allclose(lm, whole_l, atol=1e-13)
    # the denominators obey l = l1 e^{m1-m} + l2 e^{m2-m} with lse = m + ln l
    assert np.allclose(np.exp(lm), np.exp(la) + np.exp(lb), rtol=1e-13)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("causal", [False, True])
def test_block_pair_partials_merge_to_the_whole(layout, causal):
    """Host i's N partial states (one per KV block it meets on the ring),
    folded with the merge, give its rows of full attention; under contiguous
    causal masking the pairs j > i are empty (lse -inf)."""
    rng = np.random.default_rng(21)
    S, N, D = 30, 5, 6
    q, k, v = (_rand(rng, S, D, scale=2.0) for _ in range(3))
    c = S // N
    full_o, full_l = orc.attention_rows(q, k, v, np.arange(S), N, causal, layout)
    for i in range(N):
        o = np.zeros((c, D))
        lse = np.full(c, -np.inf)
        for j in orc.ring_order(i, N):
            oj, lj = orc.block_pair_attention(q, k, v, i, j, N, causal, layout)
            if causal and layout == "contiguous" and j > i:
                assert np.all(lj == -np.inf) and np.all(oj == 0)
            o, lse = orc.lse_merge(o, lse, oj, lj)
        np.testing.assert_allclose(o, full_o[i * c:(i + 1) * c], atol=1e-13)
        np.testing.assert_allclose(lse, full_l[i * c:(i + 1) * c], atol=1e-13)


def test_merge_edge_cases():
    o = np.arange(6.0).reshape(2, 3)
    ninf = np.array([-np.inf, -np.inf])
    om, lm = orc.lse_merge(o, ninf, 2 * o, ninf)
    assert np.all(om == 0) and np.all(lm == -np.inf)
    om, lm = orc.lse_merge(o, np.array([0.5, -1.0]), 2 * o, ninf)   # one side empty
    np.testing.assert_allclose(om, o)
    np.testing.assert_allclose(lm, [0.5, -1.0])
    om, lm = orc.lse_merge(o, np.array([1e4, 0.0]), 2 * o, np.array([1e4, 0.0]))  # huge, equal
    np.testing.assert_allclose(om, 1.5 * o)
    np.testing.assert_allclose(lm, [1e4 + math.log(2), math.log(2)])


def test_striped_equals_contiguous_after_unpermuting():
    rng = np.random.default_rng(14)
    S, N, D = 32, 4, 8
    q, k, v = (_rand(rng, 1, 1, S, D) for _ in range(3))
    pos = orc.token_positions(S, N, "striped")      # storage row -> token
    # token-order tensors for the contiguous run
    qt, kt, vt = (np.empty_like(x) for x in (q, k, v))
    for src, dst in ((q, qt), (k, kt), (v, vt)):
        dst[0, 0, pos] = src[0, 0]
    os_, ls_ = orc.ring_attention(q, k, v, N, True, "striped")
    oc, lc = orc.ring_attention(qt, kt, vt, N, True, "contiguous")
    np.testing.assert_allclose(os_[0, 0], oc[0, 0, pos], atol=1e-13)
    np.testing.assert_allclose(ls_[0, 0], lc[0, 0, pos], atol=1e-13)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_causal_future_keys_do_not_leak(layout):
    rng = np.random.default_rng(15)
    S, N, D = 32, 4, 4
    q, k, v = (_rand(rng, 1, 1, S, D) for _ in range(3))
    pos = orc.token_positions(S, N, layout)
    o1, l1 = orc.ring_attention(q, k, v, N, True, layout)
    cut = 20
    fut = pos > cut
    k2, v2 = k.copy(), v.copy()
    k2[0, 0, fut] += 5.0
    v2[0, 0, fut] -= 3.0
    o2, l2 = orc.ring_attention(q, k2, v2, N, True, layout)
    keep = pos <= cut
    np.testing.assert_array_equal(o1[0, 0, keep], o2[0, 0, keep])
    np.testing.assert_array_equal(l1[0, 0, keep], l2[0, 0, keep])
    assert not np.allclose(o1[0, 0, ~keep], o2[0, 0, ~keep])


def test_probability_rows_sum_to_one():
    rng = np.random.default_rng(16)
    S, N, D = 24, 3, 8
    q, k, v = (_rand(rng, S, D, scale=2.0) for _ in range(3))
    for layout in LAYOUTS:
        _, lse = orc.attention_rows(q, k, v, np.arange(S), N, True, layout)
        P = orc.attention._probabilities(q, k, lse, N, True, layout)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-14)


# ------------------------------------------------------------------- gradients
def _loss(q, k, v, do, N, causal, layout):
    o, _ = orc.naive_attention(q, k, v, N, causal, layout)
    return float((o * do).sum())


@pytest.mark.parametrize("layout,causal", [("contiguous", True), ("striped", True), ("contiguous", False)])
def test_backward_matches_finite_differences(layout, causal):
    rng = np.random.default_rng(17)
    S, N, D = 12, 3, 4
    q, k, v, do = (_rand(rng, 1, 1, S, D) for _ in range(4))
    o, lse = orc.naive_attention(q, k, v, N, causal, layout)
    dq, dk, dv = orc.attention_bwd(q, k, v, o, lse, do, N, causal, layout)
    # the chunked form (query rows 5 at a time: a ragged last chunk) is pinned the same way
    cq, ck, cv = orc.attention_bwd_head_chunked(q[0, 0], k[0, 0], v[0, 0], o[0, 0], lse[0, 0], do[0, 0], N, causal,
                                                layout, row_chunk=5)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv), ("q", q, cq[None, None]), ("k", k, ck[None, None]),
                       ("v", v, cv[None, None])):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            fp = _loss(args["q"], args["k"], args["v"], do, N, causal, layout)
            args[name] = xm
            fm = _loss(args["q"], args["k"], args["v"], do, N, causal, layout)
            num[idx] = (fp - fm) / (2 * h)
        np.testing.assert_allclose(g, num, atol=2e-8, err_msg=name)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_backward_sum_identities(layout):
    """Rows of P sum to 1 and rows of dS sum to 0, hence per head
    sum_k dK = 0 and sum_k dV = sum_q dO."""
    rng = np.random.default_rng(18)
    S, N, D = 64, 4, 16
    q, k, v, do = (_rand(rng, 1, 2, S, D) for _ in range(4))
    o, lse = orc.naive_attention(q, k, v, N, True, layout)
    dq, dk, dv = orc.attention_bwd(q, k, v, o, lse, do, N, True, layout)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), atol=1e-12)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("chunk", [1, 7, 64, 200])
def test_chunked_backward_equals_whole_head(layout, causal, chunk):
    """Taking the query rows a chunk at a time changes only the order of the
    dK/dV sums (rounding), for chunks of one row, ragged chunks, and one chunk
    larger than the sequence."""
    rng = np.random.default_rng(52)
    S, D, N = 64, 8, 4
    q, k, v, do = (_rand(rng, S, D) for _ in range(4))
    o, lse = orc.naive_attention(q[None, None], k[None, None], v[None, None], N, causal, layout)
    o, lse = o[0, 0], lse[0, 0]
    ref = orc.attention_bwd_head(q, k, v, o, lse, do, N, causal, layout)
    got = orc.attention_bwd_head_chunked(q, k, v, o, lse, do, N, causal, layout, row_chunk=chunk)
    for r, g in zip(ref, got):
        np.testing.assert_allclose(g, r, rtol=1e-12, atol=1e-12)


def test_dq_rows_match_full_backward():
    rng = np.random.default_rng(19)
    S, N, D = 40, 4, 8
    q, k, v, do = (_rand(rng, S, D) for _ in range(4))
    for layout in LAYOUTS:
        o, lse = orc.attention_rows(q, k, v, np.arange(S), N, True, layout)
        dq, _, _ = orc.attention_bwd_head(q, k, v, o, lse, do, N, True, layout)
        rows = np.array([0, 7, 13, 39])
        np.testing.assert_allclose(orc.attention_bwd_dq_rows(q, k, v, do, rows, N, True, layout),
                                   dq[rows], atol=1e-13)


def test_kv_rows_match_full_backward():
    rng = np.random.default_rng(20)
    S, N, D = 48, 4, 8
    q, k, v, do = (_rand(rng, S, D) for _ in range(4))
    for layout in LAYOUTS:
        for causal in (True, False):
            o, lse = orc.attention_rows(q, k, v, np.arange(S), N, causal, layout)
            _, dk, dv = orc.attention_bwd_head(q, k, v, o, lse, do, N, causal, layout)
            keys = np.array([0, 5, 12, 30, 47])
            gk, gv = orc.attention_bwd_kv_rows(q, k, v, do, keys, N, causal, layout, row_chunk=7)
            np.testing.assert_allclose(gk, dk[keys], atol=1e-13)
            np.testing.assert_allclose(gv, dv[keys], atol=1e-13)


def test_kv_rows_split_over_query_blocks_adds_up():
    """dK_j and dV_j accumulate one query block per ring round ([CH] §5.2):
    the parts over any partition of the query rows add up to the full
    backward's rows, and queries that see none of the keys add nothing."""
    rng = np.random.default_rng(21)
    S, N, D = 60, 5, 8
    c = S // N
    q, k, v, do = (_rand(rng, S, D) for _ in range(4))
    for layout in LAYOUTS:
        o, lse = orc.attention_rows(q, k, v, np.arange(S), N, True, layout)
        _, dk, dv = orc.attention_bwd_head(q, k, v, o, lse, do, N, True, layout)
        keys = np.array([1, 14, 30, 59])
        gk, gv = np.zeros((keys.size, D)), np.zeros((keys.size, D))
        for i in rng.permutation(N):
            pk, pv = orc.attention_bwd_kv_rows(q, k, v, do, keys, N, True, layout, row_chunk=5,
                                               query_rows=np.arange(i * c, (i + 1) * c))
            gk += pk
            gv += pv
        np.testing.assert_allclose(gk, dk[keys], atol=1e-13)
        np.testing.assert_allclose(gv, dv[keys], atol=1e-13)
    pos = orc.token_positions(S, N, "contiguous")
    early = np.nonzero(pos < 30)[0]      # contiguous causal: these queries cannot see key 30 or 59
    pk, pv = orc.attention_bwd_kv_rows(q, k, v, do, np.array([30, 59]), N, True, "contiguous", query_rows=early)
    assert not pk.any() and not pv.any()


# ------------------------------------------------------------- work per device
def test_product_pair_counter_matches_oracle():
    from ring_attention_fwd_gb300 import flops
    for S, N in ((16, 4), (96, 3), (2048, 16)):
        for layout in LAYOUTS:
            for causal in (True, False):
                assert flops.visible_pairs_per_block(S, N, layout, causal) == \
                    orc.visible_pairs_per_device(S, N, layout, causal).tolist()


def test_visible_pairs_brute_force_and_balance():
    for S, N in ((16, 4), (64, 8), (96, 3)):
        for layout in LAYOUTS:
            pos = orc.token_positions(S, N, layout)
            vis = orc.visible(pos, pos, True)
            brute = vis.sum(axis=1).reshape(N, S // N).sum(axis=1)
            assert orc.visible_pairs_per_device(S, N, layout, True).tolist() == brute.tolist()
            assert brute.sum() == S * (S + 1) // 2
    # contiguous: device i does i*c^2 + c(c+1)/2; striped: N c(c-1)/2 + c(i+1)
    S, N = 32768, 16
    c = S // N
    cont = orc.visible_pairs_per_device(S, N, "contiguous", True)
    strp = orc.visible_pairs_per_device(S, N, "striped", True)
    assert cont.tolist() == [i * c * c + c * (c + 1) // 2 for i in range(N)]
    assert strp.tolist() == [N * c * (c - 1) // 2 + c * (i + 1) for i in range(N)]
    assert cont.max() / cont.min() > 2 * N - 2 and strp.max() / strp.min() < 1.001


# ---------------------------------------------------------------- ring decode
def _brute_force_decode(q, k, v):
    """Scalar loops, no max subtraction: o = sum_t w_t v_t / sum_t w_t, w_t = e^{q.k_t/sqrt(D)}."""
    D = len(q)
    w = [math.exp(sum(q[x] * kt[x] for x in range(D)) / math.sqrt(D)) for kt in k]
    tot = sum(w)
    return np.array([sum(w[t] * v[t][x] for t in range(len(k))) / tot for x in range(D)]), math.log(tot)


@pytest.mark.parametrize("L,D", [(1, 3), (5, 4), (17, 8)])
def test_decode_brute_force(L, D):
    rng = np.random.default_rng(40 + L)
    q, k, v = _rand(rng, D), _rand(rng, L, D), _rand(rng, L, D)
    o, lse = orc.decode_attention(q, k, v)
    bo, bl = _brute_force_decode(q.tolist(), k.tolist(), v.tolist())
    np.testing.assert_allclose(o, bo, rtol=1e-12, atol=1e-12)
    assert abs(lse - bl) < 1e-12


@pytest.mark.parametrize("layout", LAYOUTS)
def test_decode_equals_last_row_of_causal_prefill(layout):
    """The newest token's decode output is the last token's row of full causal
    attention: its causal mask admits every earlier key."""
    rng = np.random.default_rng(41)
    S, D, N = 24, 8, 4
    q, k, v = _rand(rng, S, D), _rand(rng, S, D), _rand(rng, S, D)
    pos = orc.token_positions(S, N, layout)
    last = int(np.argmax(pos))                    # storage row of token S-1
    ro, rl = orc.attention_rows(q, k, v, [last], N, True, layout)
    o, lse = orc.decode_attention(q[last], k, v)
    np.testing.assert_allclose(o, ro[0], rtol=1e-12, atol=1e-12)
    assert abs(lse - rl[0]) < 1e-12


def test_decode_zero_query_is_mean_and_log_count():
    rng = np.random.default_rng(42)
    k, v = _rand(rng, 9, 4), _rand(rng, 9, 4)
    o, lse = orc.decode_attention(np.zeros(4), k, v)
    np.testing.assert_allclose(o, v.mean(axis=0), rtol=1e-13, atol=1e-13)
    assert abs(lse - math.log(9)) < 1e-13


def test_decode_huge_equal_scores_do_not_overflow():
    """Scores near 1e4 overflow exp() without the max subtraction; equal keys
    give the mean of V and lse = s + ln L exactly."""
    D, L = 4, 6
    q = np.full(D, 100.0)
    k = np.full((L, D), 50.0)                     # s = 4 * 5000 / 2 = 10000
    v = np.arange(L * D, dtype=float).reshape(L, D)
    o, lse = orc.decode_attention(q, k, v)
    np.testing.assert_allclose(o, v.mean(axis=0), rtol=1e-13)
    assert abs(lse - (10000.0 + math.log(L))) < 1e-9


def test_decode_blocks_partition_the_cache():
    for S in (1, 5, 64, 100):
        for N in (1, 3, 7, 128):
            blocks = orc.decode_blocks(S, N)
            assert len(blocks) == N
            c = -(-S // N)
            covered = []
            for j, (a, b) in enumerate(blocks):
                assert 0 <= a <= b <= S and b - a <= c
                covered += list(range(a, b))
            assert covered == list(range(S))


@pytest.mark.parametrize("S,N", [(1, 1), (10, 3), (33, 4), (7, 12), (64, 8)])
def test_ring_decode_blocks_merge_to_the_whole(S, N):
    """Per-block partials merged in the ring order equal the one-shot
    definition, also with short and empty trailing blocks (N > S)."""
    rng = np.random.default_rng(43 + S + N)
    D = 6
    q, k, v = _rand(rng, D, scale=2.0), _rand(rng, S, D), _rand(rng, S, D)
    o, lse = orc.ring_decode(q, k, v, N)
    ro, rl = orc.decode_attention(q, k, v)
    np.testing.assert_allclose(o, ro, rtol=1e-12, atol=1e-12)
    assert abs(lse - rl) < 1e-12
    for holder in range(N):                       # any host's ring order gives the same state
        ho, hl = orc.ring_decode(q, k, v, N, holder=holder)
        np.testing.assert_allclose(ho, ro, rtol=1e-12, atol=1e-12)
        assert abs(hl - rl) < 1e-12


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("causal", [False, True])
def test_block_pair_backward_sums_to_the_full_gradient(layout, causal):
    """Summing one query block's round contributions over all KV blocks gives
    its rows of dQ; summing one KV block's over all query blocks gives its rows
    of dK and dV (the full gradient is pinned by finite differences above)."""
    rng = np.random.default_rng(51)
    S, D, N = 24, 5, 4
    c = S // N
    q, k, v, do = (_rand(rng, S, D) for _ in range(4))
    o, lse = orc.naive_attention(q[None, None], k[None, None], v[None, None], N, causal, layout)
    o, lse = o[0, 0], lse[0, 0]
    dQ, dK, dV = orc.attention_bwd_head(q, k, v, o, lse, do, N, causal, layout)
    sq = np.zeros_like(dQ)
    sk = np.zeros_like(dK)
    sv = np.zeros_like(dV)
    for i in range(N):
        for j in range(N):
            a, b, cc = orc.block_pair_bwd(q, k, v, o, lse, do, i, j, N, causal, layout)
            sq[i * c:(i + 1) * c] += a
            sk[j * c:(j + 1) * c] += b
            sv[j * c:(j + 1) * c] += cc
            if causal and layout == "contiguous" and j > i:
                assert not a.any() and not b.any() and not cc.any()
    np.testing.assert_allclose(sq, dQ, atol=1e-12)
    np.testing.assert_allclose(sk, dK, atol=1e-12)
    np.testing.assert_allclose(sv, dV, atol=1e-12)


# ---------------------------------------------------------------- blockwise feedforward
def _brute_ffn(x, w1, w3, w2):
    """Scalar loops with math.exp: y_r = sum_j W2[o, j] * silu(a_j) * b_j."""
    out = []
    for row in x:
        hid = []
        for j in range(len(w1)):
            a = sum(w1[j][t] * row[t] for t in range(len(row)))
            b = sum(w3[j][t] * row[t] for t in range(len(row)))
            hid.append(a / (1.0 + math.exp(-a)) * b)
        out.append([sum(w2[o][j] * hid[j] for j in range(len(hid))) for o in range(len(w2))])
    return np.array(out)


def test_ffn_brute_force():
    rng = np.random.default_rng(61)
    T, h, f = 5, 4, 7
    x, w1, w3, w2 = _rand(rng, T, h), _rand(rng, f, h), _rand(rng, f, h), _rand(rng, h, f)
    np.testing.assert_allclose(orc.ffn_rows(x, w1, w3, w2), _brute_ffn(x.tolist(), w1.tolist(), w3.tolist(),
                                                                     w2.tolist()), rtol=1e-12, atol=1e-12)


def test_silu_closed_forms():
    assert orc.silu(0.0) == 0.0
    assert abs(orc.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert orc.silu(800.0) == 800.0                    # no overflow: sigmoid -> 1
    assert orc.silu(-800.0) == 0.0 or abs(orc.silu(-800.0)) < 1e-300
    a = np.linspace(-6, 6, 25)
    np.testing.assert_allclose(orc.silu(a) - orc.silu(-a), a, atol=1e-14)   # silu(a) - silu(-a) = a


def test_ffn_identity_weights_give_silu_times_x():
    rng = np.random.default_rng(62)
    x = _rand(rng, 6, 5)
    eye = np.eye(5)
    np.testing.assert_allclose(orc.ffn_rows(x, eye, eye, eye), orc.silu(x) * x, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("T,c", [(10, 3), (8, 8), (9, 20), (7, 1)])
def test_blockwise_ffn_equals_whole_sequence(T, c):
    rng = np.random.default_rng(63 + T)
    h, f = 4, 6
    x, w1, w3, w2 = _rand(rng, T, h), _rand(rng, f, h), _rand(rng, f, h), _rand(rng, h, f)
    np.testing.assert_allclose(orc.blockwise_ffn(x, w1, w3, w2, c), orc.ffn_rows(x, w1, w3, w2), atol=1e-13)
