"""Quest decode-time hot path for GB300 (sm_103a): paged fp16 KV cache with per-page key
min/max boxes, query-aware page scoring, per-head top-K page selection and split-K
sparse flash-decode, as a C-ABI library (``libquest.so``) with a thin ctypes binding."""
