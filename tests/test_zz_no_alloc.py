"""Decode without a caller workspace, for callers that cannot allocate device memory.

tq_decode_attention_noalloc keeps its scratch in a fixed array inside the
library instead of a workspace the caller allocates; callers such as code
running inside a custom allocator, or a runtime whose arena already owns the
whole device, have no way to make that allocation.  This file is collected
last so a failure here leaves every other test already run.  Two calls in a
row, on different sizes, must each give what the ordinary entry point gives:
the second call sees the first call's leftovers in the shared array.
"""

import math

import numpy as np
import pytest

from .gpu_common import alloc_caches, ctx_for, gpu_quantize, th, to_dev, torch, tq, wl

pytestmark = pytest.mark.gpu


def _setup(seed, B, H, lens):
    w = wl.Workload("t", "decode", B, 8, H, int(max(lens)), k_bits=(4, 3), v_bits=(4, 3), seed=seed)
    rng = np.random.default_rng(seed)
    pps = (int(max(lens)) + 15) // 16
    num_pages = B * pps
    bt = rng.permutation(num_pages).astype(np.int32).reshape(B, pps)
    T = int(max(lens))
    K = wl.bf16_round(rng.standard_normal((B, T, H, 128)).astype(np.float32))
    V = wl.bf16_round(rng.standard_normal((B, T, H, 128)).astype(np.float32))
    return w, bt, num_pages, K, V


def _both(ctx, Hq, H, lens, bt, num_pages, kc, vc, q, chunk):
    B = len(lens)
    lens_d = to_dev(np.asarray(lens, np.int32))
    bt_d = to_dev(bt)
    max_len = int(max(lens))
    scale = 1.0 / math.sqrt(128)
    n = tq.tq_workspace_size(ctx, B, Hq, max_len, chunk)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    ref = torch.full((B, Hq, 128), float("nan"), device="cuda")
    tq.tq_decode_attention(ctx, q, tq.TQ_BF16, B, Hq, H, lens_d, max_len, bt_d, bt.shape[1], num_pages, kc, vc,
                           chunk, scale, ref, ws, n)
    got = torch.full((B, Hq, 128), float("nan"), device="cuda")
    tq.tq_decode_attention_noalloc(ctx, q, tq.TQ_BF16, B, Hq, H, lens_d, max_len, bt_d, bt.shape[1], num_pages,
                                   kc, vc, chunk, scale, got)
    torch.cuda.synchronize()
    return ref.cpu().numpy(), got.cpu().numpy()


def test_noalloc_decode_matches_workspace_decode_twice():
    cases = [(7, 3, 2, 16, [700, 33, 5], 64), (8, 2, 1, 8, [90, 1], 16)]
    w0 = _setup(*cases[0][:3], cases[0][4])[0]
    ctx = ctx_for(w0)
    try:
        for seed, B, H, Hq, lens, chunk in cases:
            w, bt, num_pages, K, V = _setup(seed, B, H, lens)
            kc, vc = alloc_caches(ctx, H, num_pages)
            gpu_quantize(ctx, K, V, "bf16", [0] * B, bt, num_pages, kc, vc)
            q = to_dev(wl.bf16_round(np.random.default_rng(seed + 1).standard_normal((B, Hq, 128))
                                     .astype(np.float32))).to(torch.bfloat16)
            ref, got = _both(ctx, Hq, H, lens, bt, num_pages, kc, vc, q, chunk)
            assert np.all(np.isfinite(got))
            assert th.rel_err(got, ref).max() <= th.ATT_TOL
        assert tq.tq_check_device_status(ctx) == 0
    finally:
        tq.tq_destroy(ctx)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    w = wl.Workload("t", "decode", 1, 8, 1, 16, seed=0)
    ctx = ctx_for(w)
    try:
        B, Hq, H, max_len = 64, 32, 8, 1 << 20     # partials for 16-token chunks need far more than 16 MiB
        assert tq.tq_workspace_size(ctx, B, Hq, max_len, 16) > tq.NOALLOC_SCRATCH_BYTES
        kc, vc = alloc_caches(ctx, 1, 1)
        q = torch.zeros(B, Hq, 128, dtype=torch.bfloat16, device="cuda")
        out = torch.zeros(B, Hq, 128, dtype=torch.float32, device="cuda")
        lens = to_dev(np.full(B, 16, np.int32))
        bt = to_dev(np.zeros((B, 1), np.int32))
        with pytest.raises(tq.TQError) as e:
            tq.tq_decode_attention_noalloc(ctx, q, tq.TQ_BF16, B, Hq, H, lens, max_len, bt, 1, 1, kc, vc, 16,
                                           0.1, out)
        assert e.value.status == tq.TQ_ERR_WORKSPACE
        assert torch.count_nonzero(out).item() == 0
    finally:
        tq.tq_destroy(ctx)
