"""Float64 CPU oracle for SlimKV decode attention (test infrastructure only)."""
from .slimkv_oracle import (append_kv, beacon_positions, decode_attn, decode_attn_alibi, decode_attn_full_kv,
                            decode_attn_reconstruct, decode_attn_reconstruct_rope, prefill_attn, window_positions, gqa_attn, reconstruct_kv, rope, rope_angles, round_bf16,
                            softmax_weights)

__all__ = ["append_kv", "round_bf16", "beacon_positions", "window_positions", "decode_attn", "decode_attn_alibi",
           "decode_attn_full_kv",
           "decode_attn_reconstruct", "decode_attn_reconstruct_rope", "prefill_attn", "gqa_attn", "reconstruct_kv", "rope",
           "rope_angles", "softmax_weights"]
