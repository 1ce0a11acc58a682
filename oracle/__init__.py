"""fp64 CPU oracle for TurboQuant-style online KV-cache quantization and decode
attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call, link
or execute anything in this package: only the tests, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.

It shares no code with the CUDA library.  Both sides implement the same
published random generator (SplitMix64 + Box-Muller) independently, and both
receive the same seeded synthetic inputs from the workload generator module.

Sources (web pages, cited by title and section):
  [P2] "생각정리 209 (TurboQuant)", uiyeonassociation.blogspot.com -- the
       two-stage method: rotation + per-coordinate codebook (stage 1), QJL on
       the residual (stage 2), the 2/pi shrinkage of an MSE-only 1-bit quantizer.
  [P4] "[LLM Serving] TurboQuant란 무엇이며, 어떻게 KV Cache 양자화로 메모리를
       5배 줄일 수 있을까?", riverfrot.github.io -- §2.2 attention, §3.1 paged
       blocks, §4.1 random rotation, §4.2 Lloyd-Max codebook, §4.3 QJL,
       §4.4 distortion bounds.

Every function is pinned by a ``-m "not gpu"`` test in tests/test_oracle_*.py;
the quantization-quality end-to-end figures of the pages (cos-sim, NIAH) need
real model KV and are not reproducible here ("parity unpinned" for those only).
"""

from .rng import splitmix64_stream, uniform_stream, gaussian_stream
from .turboquant import (
    Codebook, lloyd_max_gaussian, lloyd_max_sphere, rotation_matrix, qjl_matrix,
    TQParams, make_params, assign_codes, quantize_vectors, estimate_scores,
    pack_k_records, pack_v_records, unpack_k_records, unpack_v_records,
    cache_block_bytes, write_paged, read_paged, decode_attention,
    exact_attention, quantize_exclusions, search, causal_attention,
)

__all__ = [
    "splitmix64_stream", "uniform_stream", "gaussian_stream",
    "Codebook", "lloyd_max_gaussian", "lloyd_max_sphere", "rotation_matrix", "qjl_matrix",
    "TQParams", "make_params", "assign_codes", "quantize_vectors", "estimate_scores",
    "pack_k_records", "pack_v_records", "unpack_k_records", "unpack_v_records",
    "cache_block_bytes", "write_paged", "read_paged", "decode_attention",
    "exact_attention", "search", "causal_attention", "quantize_exclusions",
]
