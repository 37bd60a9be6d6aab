"""CPU oracle for the blockwise feedforward -- TEST INFRASTRUCTURE ONLY (same
rules as ``oracle.attention``: only tests, smoke() and bench.py's CPU legs use
it).

What is computed, and the readings taken:

  * The feedforward acts on each host's own block only, so it runs block by
    block locally, and its largest activation is bounded per block
    ([CH] §5.2 last step, §5.3 "blockwise feedforward"; [CH] §3 on BPT, which
    makes both attention and feedforward blockwise).
  * The pages do not give the feedforward's form.  Their experiments use
    LLaMA-style models ([CH] experiment settings), whose feedforward is the
    gated one: Y = (silu(X W1^T) * (X W3^T)) W2^T, silu(a) = a / (1 + e^-a),
    with W1, W3 [f, h] and W2 [h, f] in the (out, in) layout of a linear layer.
    That is the reading here.
  * Blockwise: the T token rows are processed c at a time; the f-wide
    intermediate of one block is the only intermediate held at once.  Every
    row's result depends on that row alone, so the blockwise result equals the
    whole-sequence one; the GPU keeps the intermediate in bf16 (its storage
    dtype), the oracle in float64.

Pins: tests/test_oracle.py (the test_ffn_* functions).
"""
from __future__ import annotations

import numpy as np


def silu(a):
    """a * sigmoid(a), written to stay finite for large |a|."""
    a = np.asarray(a, dtype=np.float64)
    e = np.exp(-np.abs(a))
    sig = np.where(a >= 0, 1.0 / (1.0 + e), e / (1.0 + e))
    return a * sig


def ffn_rows(x, w1, w3, w2):
    """Gated feedforward of the rows of x [n, h]; returns [n, h] float64."""
    return (silu(x @ w1.T) * (x @ w3.T)) @ w2.T


def blockwise_ffn(x, w1, w3, w2, c: int):
    """Feedforward of x [T, h] computed c rows at a time."""
    T = x.shape[0]
    if c < 1:
        raise ValueError("block rows c must be >= 1")
    y = np.zeros((T, w2.shape[0]))
    for r0 in range(0, T, c):
        y[r0:r0 + c] = ffn_rows(x[r0:r0 + c], w1, w3, w2)
    return y
