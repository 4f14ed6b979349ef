"""kv_cache_append_rope_gb300: cached incremental causal attention with RoPE on
one GB300, behind the C ABI of libkvc.so (include/kvc.h).

``kvc`` holds the Python binding (same names as the C entry points, argument
marshalling only); ``workloads`` holds seeded synthetic input generators.
"""
