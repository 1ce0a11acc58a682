"""Seeded synthetic inputs shaped like the pages' workloads (no method arithmetic).

Shared by the tests, the bench and the oracle checks: the only code both the
CUDA path and the oracle consume.  numpy PCG64 streams keyed by
(config seed, purpose, index) so any sequence can be regenerated alone.

Workloads (Llama-3.1-8B: 32 query / 8 KV heads, Qwen2.5-7B: 28 / 4, head dim
128, as in [P4] §2.4):
  c1  single head, N=1024 keys/values fp32 N(0,1), key channels 0-3 x10,
      8 fp32 N(0,1) queries; 3-bit K + QJL, 3-bit V; seed 0
  c2  quantize-only append: 32 seq x 8 KV heads x 4096 tokens, bf16; K N(0,1)
      with channels 0-3 x10, V N(0,1); 3-bit + QJL / 3-bit; 16-token pages with
      a random permutation of the 8192 page ids; seed 1
  c3  decode, 16 seq x 32768 tokens, 32/8 heads; 3.5-bit K (4 bits on rotated
      channels 0-63, 3 on 64-127) + QJL, 3.5-bit V; bf16 queries; seed 2
  c4  decode, 64 seq, lengths uniform in [1024, 8192], 28/4 heads; 2.5-bit
      (3/2) K + QJL, 2.5-bit V; seed 3
  c5  decode, 4 seq x 131072 tokens, 32/8 heads, 3-bit + QJL / 3-bit, K
      channels 0-7 x8, 128 split-K chunks of 1024, new token appended per step;
      seed 4
K/V channel scaling acts on the original (unrotated) channels.  Values drawn
in fp32 and rounded to bf16 (round-to-nearest-even) where the config is bf16.
"""

from dataclasses import dataclass, replace

import numpy as np

PURPOSE_K, PURPOSE_V, PURPOSE_Q, PURPOSE_TABLE, PURPOSE_LENS, PURPOSE_NEWK, PURPOSE_NEWV = 1, 2, 3, 4, 5, 6, 7


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "decode" or "quantize"
    batch: int
    q_heads: int
    kv_heads: int
    seq_len: int              # fixed length (decode) or tokens appended (quantize)
    len_range: tuple = None   # (lo, hi) inclusive, overrides seq_len per sequence
    k_bits: tuple = (3, 3)
    v_bits: tuple = (3, 3)
    m: int = 128
    qjl: bool = True
    outlier_channels: int = 4
    outlier_scale: float = 10.0
    dtype: str = "bf16"
    seed: int = 0
    chunk: int = 0            # split-K chunk tokens (0: library picks)
    append: bool = True       # decode step appends one new token per sequence first
    codebook: str = "gaussian"   # density the codebooks are fitted to: "gaussian" or "sphere"

    def scaled(self, **kw):
        return replace(self, **kw)


WORKLOADS = {
    "c1": Workload("c1", "decode", 1, 8, 1, 1024, dtype="f32", seed=0, append=False),
    "c2": Workload("c2", "quantize", 32, 8, 8, 4096, seed=1),
    "c3": Workload("c3", "decode", 16, 32, 8, 32768, k_bits=(4, 3), v_bits=(4, 3), seed=2),
    "c4": Workload("c4", "decode", 64, 28, 4, 8192, len_range=(1024, 8192), k_bits=(3, 2), v_bits=(3, 2), seed=3),
    "c5": Workload("c5", "decode", 4, 32, 8, 131072, outlier_channels=8, outlier_scale=8.0, seed=4, chunk=1024),
}


def bf16_round(x):
    """Round fp32 values to the nearest bf16 (ties to even); returns fp32 holding bf16 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) >> 16 << 16
    return bits.astype(np.uint32).view(np.float32)


def _rng(w, purpose, index=0):
    return np.random.default_rng([w.seed, purpose, index])


def _finish(w, x):
    return bf16_round(x) if w.dtype == "bf16" else x.astype(np.float32)


def seq_lens(w):
    if w.len_range is None:
        return np.full(w.batch, w.seq_len, dtype=np.int32)
    lo, hi = w.len_range
    return _rng(w, PURPOSE_LENS).integers(lo, hi + 1, size=w.batch).astype(np.int32)


def kv_tokens(w, which, b, start=0, count=None):
    """K ("k") or V ("v") of sequence b, tokens [start, start+count): [count, H, d] fp32.

    Drawn per (sequence, token) so any token range can be regenerated alone.
    """
    count = (int(seq_lens(w)[b]) - start) if count is None else count
    purpose = PURPOSE_K if which == "k" else PURPOSE_V
    out = np.empty((count, w.kv_heads, 128), dtype=np.float32)
    # one stream per 1024-token block keeps regeneration cheap and exact
    blk0, blk1 = start // 1024, (start + count + 1023) // 1024
    for blk in range(blk0, blk1):
        g = _rng(w, purpose, b * 4096 + blk).standard_normal((1024, w.kv_heads, 128), dtype=np.float32)
        lo = max(start, blk * 1024)
        hi = min(start + count, (blk + 1) * 1024)
        out[lo - start:hi - start] = g[lo - blk * 1024:hi - blk * 1024]
    if which == "k" and w.outlier_channels:
        out[..., :w.outlier_channels] *= np.float32(w.outlier_scale)
    return _finish(w, out)


def new_tokens(w, which, step=0):
    """The token appended to every sequence at a decode step: [B, 1, H, d]."""
    purpose = PURPOSE_NEWK if which == "k" else PURPOSE_NEWV
    x = _rng(w, purpose, step).standard_normal((w.batch, 1, w.kv_heads, 128), dtype=np.float32)
    if which == "k" and w.outlier_channels:
        x[..., :w.outlier_channels] *= np.float32(w.outlier_scale)
    return _finish(w, x)


def queries(w, step=0):
    return _finish(w, _rng(w, PURPOSE_Q, step).standard_normal((w.batch, w.q_heads, 128), dtype=np.float32))


def pages_per_seq(w):
    extra = 1 if (w.kind == "decode" and w.append) else 0
    return (int(seq_lens(w).max()) + extra + 15) // 16


def block_table(w):
    """Random permutation of all physical page ids, pages_per_seq per sequence."""
    pps = pages_per_seq(w)
    perm = _rng(w, PURPOSE_TABLE).permutation(w.batch * pps).astype(np.int32)
    return perm.reshape(w.batch, pps)


def packed_bytes_per_token_head(w):
    """Bytes of one packed K + V record ([P4] §2.4 KV-size accounting, per token and KV head)."""
    kb = (64 * w.k_bits[0] + 64 * w.k_bits[1]) // 8 + (w.m // 8 + 2 if w.qjl else 0) + 2
    vb = (64 * w.v_bits[0] + 64 * w.v_bits[1]) // 8 + 2
    return kb + vb
