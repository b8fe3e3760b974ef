"""paged_kv_extend_gb300: extend attention over a page-size-1 KV pool,
decode attention, unified KV-index construction and merge_state, as
hand-written CUDA kernels for sm_103a behind a C ABI (libpkx.so)."""
