"""Float64 CPU oracle for SlimKV decode attention (test infrastructure only)."""
from .slimkv_oracle import (decode_attn, decode_attn_full_kv, decode_attn_reconstruct,
                            gqa_attn, reconstruct_kv, rope, rope_angles, softmax_weights)

__all__ = ["decode_attn", "decode_attn_full_kv", "decode_attn_reconstruct", "gqa_attn",
           "reconstruct_kv", "rope", "rope_angles", "softmax_weights"]
