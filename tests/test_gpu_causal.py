"""GPU multi-query causal attention over the compressed cache against the oracle, through the C ABI.

[P4] riverfrot.github.io "TurboQuant란 무엇이며…", §2.3: every new token's K/V join the cache, and the query of
new token t attends over its own prefix.  Both sides read the same cache bytes (the oracle quantizes and packs
the synthetic K/V; the bytes go to the device unchanged); the GPU's output for every (sequence, new token, query
head) is compared with oracle.causal_attention at the attention bar, and T = 1 with the decode call.
"""

import numpy as np
import pytest

from .gpu_common import DEV, ctx_for, gpu_decode, input_tensor, oracle, to_dev, torch, tq, wl
from .test_gpu_decode import _oracle_setup
from . import helpers as th

pytestmark = pytest.mark.gpu


def _causal(w, starts, T, Hq, H, seed=0, chunk=0, qdtype=None, scale=None):
    starts = np.asarray(starts, dtype=np.int32)
    lens = starts + T                                   # the cache holds every new token's K/V
    p, bt, num_pages, kc, vc = _oracle_setup(w, lens, H, seed)
    rng = np.random.default_rng(seed + 7)
    B = len(starts)
    Q = rng.standard_normal((B, T, Hq, 128)).astype(np.float32)
    qd = qdtype or w.dtype
    if qd == "bf16":
        Q = wl.bf16_round(Q)
    scale = th.scale_for() if scale is None else scale
    max_len = int(lens.max())
    ctx = ctx_for(w)
    try:
        qt, code = input_tensor(Q, qd)
        n = tq.tq_causal_workspace_size(ctx, B, T, Hq, max_len, chunk)
        ws = torch.empty(n, dtype=torch.uint8, device=DEV)
        out = torch.full((B, T, Hq, 128), float("nan"), dtype=torch.float32, device=DEV)
        tq.tq_causal_attention(ctx, qt, code, B, T, Hq, H, to_dev(starts), max_len, to_dev(bt), bt.shape[1],
                               num_pages, to_dev(kc), to_dev(vc), chunk, scale, out, ws, n)
        torch.cuda.synchronize()
        assert tq.tq_check_device_status(ctx) == 0
        got = out.cpu().numpy()
    finally:
        tq.tq_destroy(ctx)
    want = oracle.causal_attention(p, Q.astype(np.float64), starts, bt, kc, vc, H, scale=scale)
    err = th.rel_err(got.reshape(-1, 128), want.reshape(-1, 128))
    assert np.all(np.isfinite(got))
    assert err.max() <= th.ATT_TOL, (float(err.max()), int(np.argmax(err)))
    return got, (p, bt, num_pages, kc, vc, Q)


LUT_CONFIGS = [((3, 3), (3, 3), True), ((4, 3), (4, 3), True), ((3, 2), (3, 2), True), ((4, 4), (4, 4), False),
               ((2, 2), (2, 2), True), ((4, 4), (2, 2), True)]


@pytest.mark.parametrize("kb,vb,qjl", LUT_CONFIGS)
def test_causal_bit_widths(kb, vb, qjl):
    w = wl.Workload("t", "decode", 3, 8, 2, 0, k_bits=kb, v_bits=vb, qjl=qjl, seed=3)
    _causal(w, starts=[0, 37, 200], T=7, Hq=8, H=2, seed=1)


@pytest.mark.parametrize("T,G,starts", [(1, 4, [0, 19, 300]), (7, 1, [5, 64]), (64, 4, [0, 130]), (64, 8, [17]),
                                        (33, 3, [250, 1, 96])])
def test_causal_lengths_and_groups(T, G, starts):
    H = 2
    w = wl.Workload("t", "decode", len(starts), G * H, H, 0, k_bits=(3, 3), v_bits=(3, 3), seed=5)
    _causal(w, starts=starts, T=T, Hq=G * H, H=H, seed=T + G)


def test_causal_small_chunks_span_many_pages():
    # chunks of 32 tokens: a query's prefix crosses many chunks, each merged by log-sum-exp
    w = wl.Workload("t", "decode", 2, 4, 1, 0, k_bits=(4, 3), v_bits=(4, 3), seed=2)
    _causal(w, starts=[100, 250], T=40, Hq=4, H=1, seed=9, chunk=32)


def test_causal_fp32_queries():
    w = wl.Workload("t", "decode", 2, 8, 2, 0, k_bits=(3, 3), v_bits=(3, 3), dtype="f32", seed=4)
    _causal(w, starts=[3, 90], T=12, Hq=8, H=2, seed=3)


def test_causal_one_token_equals_decode():
    """T = 1 is a decode step over start + 1 tokens (the causal path also adds q~'s fp16 low parts to the
    scores, so the two agree within the attention bar rather than bit for bit)."""
    w = wl.Workload("t", "decode", 3, 8, 2, 0, k_bits=(3, 3), v_bits=(3, 3), seed=6)
    starts = np.array([0, 40, 511], dtype=np.int32)
    got, (p, bt, num_pages, kc, vc, Q) = _causal(w, starts=starts, T=1, Hq=8, H=2, seed=12)
    ctx = ctx_for(w)
    try:
        dec = gpu_decode(ctx, Q[:, 0], "bf16", 2, starts + 1, int(starts.max()) + 1, bt, num_pages, to_dev(kc),
                         to_dev(vc))
    finally:
        tq.tq_destroy(ctx)
    assert th.rel_err(got[:, 0].reshape(-1, 128), dec.reshape(-1, 128)).max() <= th.ATT_TOL


def test_causal_rejects_scales_above_the_bar():
    """Causal attention runs on the tensor cores only: |softmax_scale| above 1/sqrt(d) is rejected before any
    launch (the pointers below are never read)."""
    w = wl.Workload("t", "decode", 1, 4, 1, 0, k_bits=(3, 3), v_bits=(3, 3), seed=1)
    ctx = ctx_for(w)
    try:
        for scale in (0.3, -0.1):
            st = tq.raw_status("tq_causal_attention", ctx, 16, tq.TQ_BF16, 1, 4, 4, 1, 16, 64, 16, 4, 4, 16, 16, 0,
                               scale, 16, 16, 1 << 30, None)
            assert st == tq.TQ_ERR_UNSUPPORTED
    finally:
        tq.tq_destroy(ctx)


def test_causal_unsupported_widths_are_rejected():
    w = wl.Workload("t", "decode", 1, 4, 1, 0, k_bits=(1, 1), v_bits=(1, 1), seed=1)
    ctx = ctx_for(w)
    try:
        st = tq.raw_status("tq_causal_attention", ctx, 16, tq.TQ_BF16, 1, 4, 4, 1, 16, 64, 16, 4, 4, 16, 16, 0,
                           0.1, 16, 16, 1 << 30, None)
        assert st == tq.TQ_ERR_UNSUPPORTED
    finally:
        tq.tq_destroy(ctx)


def test_causal_large_chunks_take_the_lookup_table_kernel():
    """Chunks above 1024 tokens run on the lookup-table kernel's causal instances (blocks of 8 query rows)
    instead of the tensor-core kernel; the same bar holds."""
    w = wl.Workload("t", "decode", 2, 8, 2, 0, k_bits=(3, 3), v_bits=(3, 3), seed=8)
    _causal(w, starts=[1500, 40], T=9, Hq=8, H=2, seed=4, chunk=2048)


def test_causal_many_query_blocks():
    """More than 128 query rows per (sequence, KV head): several row blocks of the tensor-core kernel, the last
    one ragged, with chunks that cut the prefix into several items."""
    w = wl.Workload("t", "decode", 2, 8, 2, 0, k_bits=(4, 3), v_bits=(4, 3), seed=9)
    _causal(w, starts=[700, 5], T=70, Hq=8, H=2, seed=6, chunk=256)


def test_causal_unaligned_queries():
    """A query tensor 2 bytes off a 16-byte boundary: the tensor-core path's query prep falls back to scalar
    loads (same results as from an aligned copy)."""
    import torch
    w = wl.Workload("t", "decode", 2, 8, 2, 0, k_bits=(3, 3), v_bits=(3, 3), seed=6)
    starts = np.array([20, 3], np.int32)
    T, Hq, H = 5, 8, 2
    lens = starts + T
    p, bt, num_pages, kc, vc = _oracle_setup(w, lens, H, 2)
    Q = wl.bf16_round(np.random.default_rng(8).standard_normal((2, T, Hq, 128)).astype(np.float32))
    ctx = ctx_for(w)
    try:
        big = torch.empty(Q.size + 1, dtype=torch.bfloat16, device=DEV)
        qt = big[1:].view(2, T, Hq, 128)
        qt.copy_(torch.from_numpy(Q).to(DEV).to(torch.bfloat16))
        assert qt.data_ptr() % 16 != 0
        n = tq.tq_causal_workspace_size(ctx, 2, T, Hq, int(lens.max()), 0)
        ws = torch.empty(n, dtype=torch.uint8, device=DEV)
        out = torch.full((2, T, Hq, 128), float("nan"), dtype=torch.float32, device=DEV)
        scale = th.scale_for()
        tq.tq_causal_attention(ctx, qt, tq.TQ_BF16, 2, T, Hq, H, to_dev(starts), int(lens.max()), to_dev(bt),
                               bt.shape[1], num_pages, to_dev(kc), to_dev(vc), 0, scale, out, ws, n)
        torch.cuda.synchronize()
        assert tq.tq_check_device_status(ctx) == 0
        got = out.cpu().numpy()
    finally:
        tq.tq_destroy(ctx)
    want = oracle.causal_attention(p, Q.astype(np.float64), starts, bt, kc, vc, H, scale=scale)
    assert th.rel_err(got.reshape(-1, 128), want.reshape(-1, 128)).max() <= th.ATT_TOL


def test_causal_bad_page_is_skipped_and_flagged():
    """A block-table entry outside [0, num_pages) in sequence 0's prefix: the kernel skips that page's tokens,
    flags the page bit, and sequence 1 (untouched) still matches the oracle."""
    import torch
    w = wl.Workload("t", "decode", 2, 8, 2, 0, k_bits=(4, 3), v_bits=(4, 3), seed=7)
    starts = np.array([90, 60], np.int32)
    T, Hq, H = 6, 8, 2
    lens = starts + T
    p, bt, num_pages, kc, vc = _oracle_setup(w, lens, H, 3)
    Q = wl.bf16_round(np.random.default_rng(11).standard_normal((2, T, Hq, 128)).astype(np.float32))
    bad = bt.copy()
    bad[0, 2] = num_pages + 7                            # positions 32..47 of sequence 0
    ctx = ctx_for(w)
    try:
        qt, code = input_tensor(Q, "bf16")
        n = tq.tq_causal_workspace_size(ctx, 2, T, Hq, int(lens.max()), 0)
        ws = torch.empty(n, dtype=torch.uint8, device=DEV)
        out = torch.full((2, T, Hq, 128), float("nan"), dtype=torch.float32, device=DEV)
        scale = th.scale_for()
        tq.tq_causal_attention(ctx, qt, code, 2, T, Hq, H, to_dev(starts), int(lens.max()), to_dev(bad),
                               bad.shape[1], num_pages, to_dev(kc), to_dev(vc), 0, scale, out, ws, n)
        torch.cuda.synchronize()
        flags = tq.tq_check_device_status(ctx)
        got = out.cpu().numpy()
    finally:
        tq.tq_destroy(ctx)
    assert flags & 1                                     # the page-id bit
    assert np.all(np.isfinite(got))
    want = oracle.causal_attention(p, Q.astype(np.float64), starts, bt, kc, vc, H, scale=scale)
    assert th.rel_err(got[1].reshape(-1, 128), want[1].reshape(-1, 128)).max() <= th.ATT_TOL
