"""LSE merge parity: CUDA ra_merge vs the oracle's merge, on partial states
the oracle computes over disjoint key sets."""
import numpy as np
import pytest
import torch

import oracle as orc
from gpu_helpers import max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import ring_attention_fwd_gb300 as ra
    assert torch.cuda.is_available()
    return ra


def _partials(S, D, seed):
    rng = np.random.default_rng(seed)
    q, k, v = (rng.standard_normal((S, D)) * 1.5 for _ in range(3))
    sel = rng.permutation(S)
    A, B = sel[: S // 3], sel[S // 3:]
    oa, la = orc.attention_rows(q, k[A], v[A], np.arange(S), 1, False, "contiguous")
    ob, lb = orc.attention_rows(q, k[B], v[B], np.arange(S), 1, False, "contiguous")
    return oa, la, ob, lb


@pytest.mark.parametrize("dtype,D,tol_o", [(torch.bfloat16, 128, 2e-2), (torch.float32, 128, 1e-5),
                                           (torch.bfloat16, 37, 2e-2), (torch.float32, 5, 1e-5)])
def test_merge_matches_oracle(ra, dtype, D, tol_o):
    S = 3000
    oa, la, ob, lb = _partials(S, D, seed=D)
    # inputs as the GPU holds them (rounded); the expected value uses the same rounded inputs
    ta = torch.from_numpy(oa).to(dtype)
    tb = torch.from_numpy(ob).to(dtype)
    la32 = torch.from_numpy(la).float()
    lb32 = torch.from_numpy(lb).float()
    ro, rl = orc.lse_merge(ta.double().numpy(), la32.double().numpy(), tb.double().numpy(),
                           lb32.double().numpy())
    ga, gla = ta.cuda(), la32.cuda()
    ra.merge(ga, gla, tb.cuda(), lb32.cuda())
    torch.cuda.synchronize()
    assert max_err(ga.double().cpu().numpy(), ro) <= tol_o
    assert max_err(gla.cpu().numpy(), rl) <= 2e-6 * max(1.0, float(np.abs(rl).max()))


@pytest.mark.parametrize("D,rows", [(128, 3000), (36, 511), (5, 100)])
def test_merge_f32_state_bf16_partial(ra, D, rows):
    """A float32 running state folding a bf16 partial (ring hosts keep their
    output in float32 across rounds): both vectorised (D % 4 == 0) and scalar
    paths, against the oracle's merge of the same rounded inputs."""
    oa, la, ob, lb = _partials(rows, D, seed=100 + D)
    ta = torch.from_numpy(oa).float()
    tb = torch.from_numpy(ob).to(torch.bfloat16)
    la32, lb32 = torch.from_numpy(la).float(), torch.from_numpy(lb).float()
    la32[::9] = -float("inf")
    lb32[::4] = -float("inf")
    ro, rl = orc.lse_merge(ta.double().numpy(), la32.double().numpy(), tb.double().numpy(), lb32.double().numpy())
    ga, gla = ta.cuda(), la32.cuda()
    ra.merge(ga, gla, tb.cuda(), lb32.cuda())
    torch.cuda.synchronize()
    assert ga.dtype == torch.float32
    assert max_err(ga.double().cpu().numpy(), ro) <= 1e-5
    assert max_err(gla.cpu().numpy(), rl) <= 2e-6 * max(1.0, float(np.abs(rl[np.isfinite(rl)]).max()))


def test_merge_edge_rows(ra):
    D = 16
    o_a = torch.arange(4 * D, dtype=torch.float32).view(4, D)
    o_b = -2 * o_a
    inf = float("inf")
    la = torch.tensor([-inf, 0.5, -inf, 30.0])
    lb = torch.tensor([-inf, -inf, -1.0, 30.0])
    ga, gla = o_a.cuda(), la.cuda()
    ra.merge(ga, gla, o_b.cuda(), lb.cuda())
    torch.cuda.synchronize()
    ro, rl = orc.lse_merge(o_a.double().numpy(), la.double().numpy(), o_b.double().numpy(), lb.double().numpy())
    assert max_err(ga.cpu().numpy(), ro) <= 1e-5
    assert max_err(gla.cpu().numpy(), rl) <= 1e-5
    assert torch.isneginf(gla[0]) and bool((ga[0] == 0).all())


def test_merge_unaligned_and_empty(ra):
    D = 128
    oa, la, ob, lb = _partials(257, D, seed=3)
    buf_a = torch.zeros(257 * D + 1, dtype=torch.bfloat16)
    buf_a[1:] = torch.from_numpy(oa).to(torch.bfloat16).flatten()
    tb = torch.from_numpy(ob).to(torch.bfloat16)
    ga = buf_a.cuda()
    view = ga[1:].view(257, D)          # 2-byte aligned: scalar path
    gla = torch.from_numpy(la).float().cuda()
    ra.merge(view, gla, tb.cuda(), torch.from_numpy(lb).float().cuda())
    torch.cuda.synchronize()
    ro, rl = orc.lse_merge(buf_a[1:].view(257, D).double().numpy(), torch.from_numpy(la).float().double().numpy(),
                           tb.double().numpy(), torch.from_numpy(lb).float().double().numpy())
    assert max_err(view.double().cpu().numpy(), ro) <= 2e-2
    assert float(ga[0].float().cpu()) == 0.0     # the element before the view is untouched
    e = torch.empty((0, D), dtype=torch.bfloat16, device="cuda")
    le = torch.empty((0,), dtype=torch.float32, device="cuda")
    ra.merge(e, le, e, le)
