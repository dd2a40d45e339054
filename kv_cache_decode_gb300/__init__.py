"""Single-token decode attention over a KV cache for GB300 (sm_103a)."""
