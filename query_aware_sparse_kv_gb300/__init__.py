"""Query-aware sparse paged KV decode for GB300 (sm_103a)."""
