"""Derivation of the limits on the backward's whole-sequence identities (CPU).

Every row of the softmax P sums to 1 and every row of dS = P * (dP - D_vec)
sums to 0, so per head and column  sum_k dK = 0  and  sum_k dV = sum_q dO.
The GPU tests check these over all keys of full-size outputs.  The kernels
depart from exact arithmetic at their bf16 rounding points: the forward's
output O (which D_vec = rowsum(dO * O) reads), P and dS entering the tensor
cores, and the bf16 dK and dV outputs.  This test rounds at those points in a
float64 emulation built on the oracle's causal rule, and checks that

  * the identities stay well inside SUM_DK_LIMIT / SUM_DV_LIMIT (measured
    ratios ~1e-2 for dK and ~5e-4 for dV, the same at 2048 and 8192 tokens:
    the errors are rounding noise, relative to the column norms);
  * zeroing the dK and dV rows of one key block (a dropped or misplaced block)
    pushes them far outside.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from gpu_helpers import SUM_DK_LIMIT, SUM_DV_LIMIT


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _ratios(dk, dv, do):
    rk = np.abs(dk.sum(0)) / np.linalg.norm(dk, axis=0)
    rv = np.abs(dv.sum(0) - do.sum(0)) / np.sqrt(np.linalg.norm(dv, axis=0) ** 2 + np.linalg.norm(do, axis=0) ** 2)
    return float(rk.max()), float(rv.max())


@pytest.mark.parametrize("S,N,layout,scale", [(2048, 8, "contiguous", 0.5), (2048, 16, "striped", 1.0)])
def test_sum_identity_limits_under_bf16_rounding(S, N, layout, scale):
    rng = np.random.default_rng(21)
    D = 128
    q, k, v, do = (_bf16(rng.standard_normal((S, D)) * (scale if i < 2 else 1.0)) for i in range(4))
    pos = orc.token_positions(S, N, layout)
    s = np.where(orc.visible(pos, pos, True), q @ k.T / np.sqrt(D), -np.inf)
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    P = e / e.sum(axis=1)[:, None]
    O = _bf16(P @ v)                                  # forward output, stored in bf16
    Dvec = (do * O).sum(axis=1)
    dV = _bf16(_bf16(P).T @ do)                       # P enters the MMA in bf16; bf16 output
    dS = _bf16(P * (do @ v.T - Dvec[:, None]))        # dS enters the MMA in bf16
    dK = _bf16(dS.T @ q / np.sqrt(D))
    rk, rv = _ratios(dK, dV, do)
    assert rk <= SUM_DK_LIMIT / 3 and rv <= SUM_DV_LIMIT / 10, (rk, rv)
    c = S // N
    blk = np.nonzero(np.arange(S) // c == 1)[0]       # storage rows of block 1
    dK[blk] = 0.0
    dV[blk] = 0.0
    rk2, rv2 = _ratios(dK, dV, do)
    assert rk2 >= 2 * SUM_DK_LIMIT and rv2 >= 2 * SUM_DV_LIMIT, (rk2, rv2)
