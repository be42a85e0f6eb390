"""prefix_shared_kv_gb300: prefix-shared KV attention on a page-1 pool for sm_103a (GB300)."""
