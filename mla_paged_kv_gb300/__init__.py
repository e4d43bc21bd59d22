"""MLA decode over a paged KV cache, GB300 (sm_103a) native."""
