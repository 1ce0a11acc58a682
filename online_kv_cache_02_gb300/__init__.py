"""GB300-native TurboQuant-style online KV-cache quantization and decode attention.

The compute path is libtq.so (CUDA for sm_103a) behind the C ABI in
include/tq.h; ``online_kv_cache_02_gb300.tq`` is its ctypes binding and
``online_kv_cache_02_gb300.workloads`` the seeded synthetic input generators.
Importing the package itself loads nothing.
"""
