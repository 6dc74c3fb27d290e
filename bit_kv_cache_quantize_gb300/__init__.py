"""KVarN KV-cache hot path on GB300 (sm_103a): per-tile quantiser and paged
decode attention behind a C-ABI library (``libkvarn.so``).

``bit_kv_cache_quantize_gb300.kvarn`` is the Python binding of that library
(argument marshalling only); ``bit_kv_cache_quantize_gb300.inputs`` holds the
seeded synthetic workloads.
"""
