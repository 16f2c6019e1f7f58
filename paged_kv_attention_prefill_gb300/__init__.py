"""Paged-KV attention for GB300 (sm_103a): C-ABI library + thin binding."""
