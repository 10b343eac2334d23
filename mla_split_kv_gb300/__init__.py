"""MLA split-KV decode for GB300 (sm_103a)."""
