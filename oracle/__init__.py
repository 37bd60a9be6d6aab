"""CPU oracle (float64 NumPy) -- test infrastructure, never the product path."""
from .attention import (  # noqa: F401
    CONTIGUOUS, STRIPED, token_positions, visible, attention_rows, naive_attention,
    ring_order, ring_block_attention, ring_attention, lse_merge, attention_bwd,
    attention_bwd_head, attention_bwd_head_chunked, attention_bwd_dq_rows, attention_bwd_kv_rows, visible_pairs_per_device,
    block_rectangle_work, block_pair_attention, block_pair_bwd,
)
from .decode import decode_attention, decode_blocks, ring_decode, decode_batch  # noqa: F401
from .ffn import silu, ffn_rows, blockwise_ffn  # noqa: F401
