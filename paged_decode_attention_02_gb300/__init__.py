"""Decode attention over a paged KV cache for GB300 (sm_103a)."""
