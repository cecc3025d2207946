"""GB300-native paged KV-cache attention (kv_store / attn_prefill_varlen / attn_decode_paged)."""
