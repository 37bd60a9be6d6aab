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


def kv_block_bytes(c: int, d: int, elem_bytes: int = 2) -> int:
    """Bytes of one K block plus one V block of c rows: 2*c*d*elem (4cd in bf16)."""
    return 2 * c * d * elem_bytes
