"""GB300-native decoding-time KV-cache eviction step (BeaconKV-style).

``decoding_kv_cache_gb300.kvc`` binds the C ABI of ``libkvc.so`` (declared in ``include/kvc.h``);
``decoding_kv_cache_gb300.inputs`` builds the seeded synthetic workloads;
``decoding_kv_cache_gb300.build`` compiles the CUDA library for sm_103a.
"""
__version__ = "0.1.0"
