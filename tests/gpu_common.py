"""GPU-side test plumbing: run the library through its C ABI with torch-owned device memory."""

import math

import numpy as np
import torch

import oracle
from online_kv_cache_02_gb300 import tq
from online_kv_cache_02_gb300 import workloads as wl

from . import helpers as th

DEV = torch.device("cuda:0")
SENTINEL = 0xA5


def ctx_for(w, seed=None):
    cfg = tq.make_config(k_bits=w.k_bits, v_bits=w.v_bits, m=w.m, seed=w.seed if seed is None else seed,
                         k_qjl=w.qjl,
                         codebook=tq.TQ_CODEBOOK_SPHERE if w.codebook == "sphere" else tq.TQ_CODEBOOK_GAUSSIAN)
    return tq.tq_create_ex(cfg)


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    return t if dtype is None else t.to(dtype)


def input_tensor(x, dtype_name):
    """numpy fp32 (already bf16-valued for bf16) -> device tensor and the library dtype code."""
    if dtype_name == "bf16":
        return to_dev(x).to(torch.bfloat16), tq.TQ_BF16
    return to_dev(x), tq.TQ_F32


def alloc_caches(ctx, H, num_pages, fill=SENTINEL):
    kpb, vpb = tq.tq_cache_layout(ctx, H)
    kc = torch.full((num_pages * kpb,), fill, dtype=torch.uint8, device=DEV)
    vc = torch.full((num_pages * vpb,), fill, dtype=torch.uint8, device=DEV)
    return kc, vc


def gpu_quantize(ctx, K, V, dtype_name, start_pos, bt, num_pages, kc, vc, stream=None):
    """K, V numpy [B, T, H, d] (either may be None)."""
    X = K if K is not None else V
    B, T, H, _ = X.shape
    kd = input_tensor(K, dtype_name)[0] if K is not None else None
    vd = input_tensor(V, dtype_name)[0] if V is not None else None
    code = tq.TQ_BF16 if dtype_name == "bf16" else tq.TQ_F32
    tq.tq_quantize(ctx, kd, vd, code, B, T, H, to_dev(np.asarray(start_pos, np.int32)), to_dev(bt),
                   bt.shape[1], num_pages, kc if K is not None else None, vc if V is not None else None, stream)


def gpu_decode(ctx, Q, dtype_name, H, lens, max_seq_len, bt, num_pages, kc, vc, chunk=0, scale=None):
    B, Hq, _ = Q.shape
    qd, code = input_tensor(Q, dtype_name)
    n = tq.tq_workspace_size(ctx, B, Hq, max_seq_len, chunk)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device=DEV)
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device=DEV)
    tq.tq_decode_attention(ctx, qd, code, B, Hq, H, to_dev(np.asarray(lens, np.int32)), max_seq_len, to_dev(bt),
                           bt.shape[1], num_pages, kc, vc, chunk, th.scale_for() if scale is None else scale,
                           out, ws, n)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def oracle_cache_bytes(p, H, num_pages, kind):
    return np.full(num_pages * H * oracle.cache_block_bytes(p, kind), SENTINEL, dtype=np.uint8)


def seq_locations(bt, b, positions, H):
    pos = np.repeat(np.asarray(positions, dtype=np.int64), H)
    heads = np.tile(np.arange(H), len(positions))
    pages = bt[b, pos // 16].astype(np.int64)
    return pages, pos % 16, heads


def scale_default():
    return 1.0 / math.sqrt(128)


__all__ = ["DEV", "SENTINEL", "ctx_for", "to_dev", "input_tensor", "alloc_caches", "gpu_quantize", "gpu_decode",
           "oracle_cache_bytes", "seq_locations", "scale_default", "wl", "th", "tq", "oracle", "torch", "np"]
