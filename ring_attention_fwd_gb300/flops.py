"""FLOP and byte conventions used to report throughput.

* One query block against one KV block of c rows costs 2dc^2 FLOPs for the
  scores and 2dc^2 for probabilities times values, 4dc^2 in all; sending the
  K and V blocks moves 4cd bytes in bf16 ("Ring Attention with Blockwise
  Transformers for Near Infinite Context" notes, §5.4).
* Whole forward: 4*S^2*D*H*B, halved when causal (the reporting convention of
  this library; the exact causal count is 4*D*H*B*S(S+1)/2).
* Backward: five c^2*D contractions of 2 FLOPs per multiply-add (S, dV, dP,
  dK, dQ) against two in the forward, so 2.5x the forward count.
"""


def fwd_flops(B: int, H: int, S: int, D: int, causal: bool) -> int:
    f = 4 * S * S * D * H * B
    return f // 2 if causal else f


def fwd_flops_exact(B: int, H: int, S: int, D: int, causal: bool) -> int:
    pairs = S * (S + 1) // 2 if causal else S * S
    return 4 * D * H * B * pairs


def bwd_flops(B: int, H: int, S: int, D: int, causal: bool) -> int:
    return fwd_flops(B, H, S, D, causal) * 5 // 2


def visible_pairs_per_block(S: int, N: int, layout: str, causal: bool) -> list:
    """Visible (query, key) pairs whose query lies in block i (virtual host i).

    Causal, contiguous: block i holds tokens i*c .. i*c+c-1, token t sees t+1
    keys, so i*c^2 + c(c+1)/2.  Causal, striped: block i holds tokens r*N + i,
    so N*c(c-1)/2 + c(i+1).  Non-causal: c*S for every block.
    """
    c = S // N
    if not causal:
        return [c * S] * N
    if layout == "contiguous":
        return [i * c * c + c * (c + 1) // 2 for i in range(N)]
    return [N * c * (c - 1) // 2 + c * (i + 1) for i in range(N)]


def kv_block_bytes(c: int, d: int, elem_bytes: int = 2) -> int:
    """Bytes of one K block plus one V block of c rows: 2*c*d*elem (4cd in bf16)."""
    return 2 * c * d * elem_bytes
