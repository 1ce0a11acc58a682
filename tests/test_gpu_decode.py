"""GPU decode-attention parity against the oracle, through the C ABI.

Both sides read the same cache bytes: the oracle quantizes and packs the
synthetic K/V, the bytes go to the device unchanged, and the GPU's output is
compared with the oracle's two-pass fp64 softmax over the same records.
"""

import numpy as np
import pytest

from .gpu_common import (alloc_caches, ctx_for, gpu_decode, oracle, oracle_cache_bytes, seq_locations, th, to_dev,
                         torch, tq, wl)

pytestmark = pytest.mark.gpu


def _oracle_setup(w, lens, H, seed, kv=None):
    """Oracle-quantized caches for sequences of the given lengths; kv = (K, V) [B, L, H, 128] fp32 replaces
    the seeded N(0,1) draws."""
    rng = np.random.default_rng(seed)
    B = len(lens)
    pps = max(1, (int(max(lens)) + 15) // 16)
    num_pages = B * pps + 2
    bt = rng.permutation(num_pages)[:B * pps].astype(np.int32).reshape(B, pps)
    p = th.params_for(w)
    kc = oracle_cache_bytes(p, H, num_pages, "k")
    vc = oracle_cache_bytes(p, H, num_pages, "v")
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        if kv is None:
            K = rng.standard_normal((L, H, 128)).astype(np.float32)
            K[..., :w.outlier_channels] *= w.outlier_scale
            V = rng.standard_normal((L, H, 128)).astype(np.float32)
        else:
            K, V = kv[0][b, :L].astype(np.float32), kv[1][b, :L].astype(np.float32)
        if w.dtype == "bf16":
            K, V = wl.bf16_round(K), wl.bf16_round(V)
        pages, slots, heads = seq_locations(bt, b, np.arange(L), H)
        th.oracle_quantize_into(p, "k", kc, K.reshape(-1, 128), pages, slots, heads, H)
        th.oracle_quantize_into(p, "v", vc, V.reshape(-1, 128), pages, slots, heads, H)
    return p, bt, num_pages, kc, vc


def _check(w, lens, Hq, H, chunk=0, scale=None, seed=0, qdtype=None, kv=None, Q=None, tol=None):
    lens = np.asarray(lens, dtype=np.int32)
    p, bt, num_pages, kc, vc = _oracle_setup(w, lens, H, seed, kv)
    rng = np.random.default_rng(seed + 100)
    if Q is None:
        Q = rng.standard_normal((len(lens), Hq, 128)).astype(np.float32)
    qd = qdtype or w.dtype
    if qd == "bf16":
        Q = wl.bf16_round(Q)
    scale = th.scale_for() if scale is None else scale
    ctx = ctx_for(w)
    try:
        got = gpu_decode(ctx, Q, qd, H, lens, int(max(lens.max(), 1)), bt, num_pages, to_dev(kc), to_dev(vc),
                         chunk=chunk, scale=scale)
        assert tq.tq_check_device_status(ctx) == 0
    finally:
        tq.tq_destroy(ctx)
    ref = oracle.decode_attention(p, Q.astype(np.float64), lens, bt, kc, vc, H, scale=scale)
    err = th.rel_err(got, ref)
    assert np.all(np.isfinite(got))
    # The bar is 2e-3 at every scale: above 1/sqrt(d) the library runs its fp32 kernels (the
    # tensor-core path's fp16 operands would carry a logit error that grows with the scale).
    if tol is None:
        tol = th.ATT_TOL
    assert err.max() <= tol, (err.max(), np.unravel_index(err.argmax(), err.shape))
    return err.max()


BASE = wl.Workload("t", "decode", 1, 8, 1, 0, seed=0)


@pytest.mark.parametrize("kb,vb,qjl", [((3, 3), (3, 3), True), ((4, 3), (4, 3), True), ((3, 2), (3, 2), True),
                                       ((4, 4), (4, 4), True), ((2, 2), (2, 2), True), ((4, 4), (2, 2), True),
                                       ((3, 3), (3, 3), False), ((4, 3), (4, 3), False),
                                       ((2, 2), (4, 4), False), ((1, 1), (1, 1), True), ((4, 4), (2, 3), True)])
def test_decode_bit_configs(kb, vb, qjl):
    w = BASE.scaled(k_bits=kb, v_bits=vb, qjl=qjl, dtype="bf16")
    _check(w, [300, 17, 129], Hq=8, H=2, chunk=64, seed=1)


@pytest.mark.parametrize("G", [1, 2, 3, 4, 7, 8])
def test_decode_gqa_group_sizes(G):
    w = BASE.scaled(dtype="bf16")
    _check(w, [200, 45], Hq=2 * G, H=2, chunk=0, seed=G)


@pytest.mark.parametrize("chunk", [16, 48, 1024, 0])
def test_decode_chunking_is_invisible(chunk):
    w = BASE.scaled(dtype="bf16")
    _check(w, [1000, 1, 16, 33], Hq=4, H=1, chunk=chunk, seed=3)


@pytest.mark.parametrize("lens,chunk", [([8000, 7990], 64), ([8000, 7990], 16)])
@pytest.mark.parametrize("qjl", [True, False])
def test_decode_warp_counts(lens, chunk, qjl):
    """The persistent kernel runs 12 or 16 warps per CTA, whichever costs least for the launch's items
    (chunks x KV heads x sequences; on 152 SMs: 500 items -> 12, 2000 -> 16, which fill one wave of 16-warp
    CTAs but not of 12-warp ones); both agree with the oracle on the same 3.5-bit inputs, with and without the
    QJL term."""
    w = BASE.scaled(dtype="bf16", k_bits=(4, 3), v_bits=(4, 3), qjl=qjl)
    _check(w, lens, Hq=8, H=2, chunk=chunk, seed=6)


def test_decode_running_max_moves_within_chunks():
    """Logits that climb along the sequence (keys = noise + a ramp along query head 0's direction, 0 -> ~9 nats
    over each 1024-token chunk for that head, ramps of random sign and size for the other heads) and a late spike
    13 nats above everything before it: the running softmax max moves many times inside every chunk, several
    times by more than the kernel's 2^3 slack.  Bar: the standard 2e-3 (a missed or wrong rescale changes
    weights by 8x or more)."""
    w = BASE.scaled(dtype="bf16", k_bits=(4, 3), v_bits=(4, 3))
    rng = np.random.default_rng(77)
    B, H, Hq, L = 2, 2, 8, 3072
    Q = wl.bf16_round(rng.standard_normal((B, Hq, 128)).astype(np.float32))
    K = 0.3 * rng.standard_normal((B, L, H, 128)).astype(np.float32)
    V = rng.standard_normal((B, L, H, 128)).astype(np.float32)
    G = Hq // H
    t = np.arange(L)
    ramp = 9.0 * (t % 1024) / 1024.0                       # nats, restarting at each chunk
    for b in range(B):
        for h in range(H):
            qd = Q[b, h * G] / np.linalg.norm(Q[b, h * G])
            amp = ramp * np.sqrt(128) / np.linalg.norm(Q[b, h * G])     # key length giving `ramp` nats
            amp[L - 40] = 22.0 * np.sqrt(128) / np.linalg.norm(Q[b, h * G])
            K[b, :, h, :] += amp[:, None] * qd[None, :]
    K, V = wl.bf16_round(K), wl.bf16_round(V)
    logits = np.einsum("bhd,blhd->bhl", Q.reshape(B, H, G, 128)[:, :, 0], K) / np.sqrt(128)
    assert logits.max() > 20.0 and np.ptp(logits[:, :, :1024]) > 8.0     # the intended shape
    _check(w, [L, L - 7], Hq=Hq, H=H, chunk=1024, seed=7, kv=(K, V), Q=Q, tol=th.ATT_TOL)


@pytest.mark.parametrize("kb,vb", [((3, 3), (3, 3)), ((4, 3), (4, 3)), ((3, 2), (3, 2))])
def test_decode_sphere_codebook(kb, vb):
    """Codebooks fitted to the exact rotated-coordinate density: the decode tables take the context's
    centroids, so the parity bar is the standard one."""
    w = BASE.scaled(dtype="bf16", k_bits=kb, v_bits=vb, codebook="sphere")
    _check(w, [700, 33, 1], Hq=8, H=2, chunk=0, seed=8)


def test_decode_empty_and_single_token_sequences():
    w = BASE.scaled(dtype="f32")
    lens = [0, 1, 2, 0]
    _check(w, lens, Hq=4, H=2, chunk=16, seed=4)


def test_decode_fp32_queries_and_scale():
    w = BASE.scaled(dtype="f32")
    _check(w, [257, 90], Hq=4, H=2, chunk=32, scale=0.3, seed=5)
    _check(w, [257, 90], Hq=4, H=2, chunk=32, scale=0.0, seed=5)    # uniform weights


@pytest.mark.parametrize("scale", [1.0, -0.25, 0.09])
def test_decode_large_scales_keep_the_bar(scale):
    """|scale| above 1/sqrt(d) (0.0884) runs the fp32 kernels: the attention bar holds for sharp softmaxes too,
    for both bit layouts the tensor-core path would take."""
    _check(BASE.scaled(dtype="bf16", k_bits=(4, 3), v_bits=(4, 3)), [300, 17], Hq=8, H=2, scale=scale, seed=6)


def test_decode_config_c1():
    """Single head, N=1024 fp32 keys (channels 0-3 x10) and values, 8 fp32 queries, 3-bit + QJL."""
    w = wl.WORKLOADS["c1"]
    _check(w, [1024], Hq=8, H=1, chunk=0, seed=0)


def test_decode_bad_page_is_skipped_and_flagged():
    w = BASE.scaled(dtype="bf16")
    lens = np.array([40], np.int32)
    p, bt, num_pages, kc, vc = _oracle_setup(w, lens, 1, 9)
    bt_bad = bt.copy()
    bt_bad[0, 1] = num_pages + 5                 # tokens 16..31 point outside the cache
    Q = wl.bf16_round(np.random.default_rng(9).standard_normal((1, 4, 128)).astype(np.float32))
    ctx = ctx_for(w)
    try:
        got = gpu_decode(ctx, Q, "bf16", 1, lens, 40, bt_bad, num_pages, to_dev(kc), to_dev(vc), chunk=16)
        assert tq.tq_check_device_status(ctx) & 1
        # a length beyond max_seq_len is clamped and flagged
        gpu_decode(ctx, Q, "bf16", 1, np.array([48], np.int32), 40, bt, num_pages, to_dev(kc), to_dev(vc))
        assert tq.tq_check_device_status(ctx) & 4
    finally:
        tq.tq_destroy(ctx)
    # the skipped block simply does not take part
    keep = np.r_[0:16, 32:40]
    pages, slots = bt[0, keep // 16], keep % 16
    heads = np.zeros(len(keep), dtype=np.int64)
    kr = oracle.unpack_k_records(p, oracle.read_paged(p, "k", kc, pages, slots, heads, 1))
    vr = oracle.unpack_v_records(p, oracle.read_paged(p, "v", vc, pages, slots, heads, 1))
    ref = np.stack([oracle.turboquant.attend_one(p, Q[0, h].astype(np.float64), kr, vr, th.scale_for())
                    for h in range(4)])
    assert th.rel_err(got[0], ref).max() <= th.ATT_TOL


def test_workspace_too_small_is_rejected():
    w = BASE.scaled(dtype="bf16")
    ctx = ctx_for(w)
    try:
        kc, vc = alloc_caches(ctx, 1, 1)
        n = tq.tq_workspace_size(ctx, 1, 4, 16, 16)
        import torch
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        out = torch.empty(1, 4, 128, dtype=torch.float32, device="cuda")
        q = torch.zeros(1, 4, 128, dtype=torch.bfloat16, device="cuda")
        lens = to_dev(np.array([16], np.int32))
        bt = to_dev(np.zeros((1, 1), np.int32))
        with pytest.raises(tq.TQError) as e:
            tq.tq_decode_attention(ctx, q, tq.TQ_BF16, 1, 4, 1, lens, 16, bt, 1, 1, kc, vc, 16, 0.1, out, ws, n - 1)
        assert e.value.status == tq.TQ_ERR_WORKSPACE
        with pytest.raises(tq.TQError):
            tq.tq_decode_attention(ctx, q, tq.TQ_BF16, 1, 4, 3, lens, 16, bt, 1, 1, kc, vc, 16, 0.1, out, ws, n)
    finally:
        tq.tq_destroy(ctx)


@pytest.mark.parametrize("scale", [None, 0.5])
def test_append_decode_equals_separate_calls(scale):
    """The fused step equals quantize + decode over L + 1 (scale 0.5: both on the fp32 kernels)."""
    import torch
    from .gpu_common import gpu_quantize
    scale = th.scale_for() if scale is None else scale
    w = BASE.scaled(k_bits=(4, 3), v_bits=(4, 3), dtype="bf16")
    rng = np.random.default_rng(21)
    B, H, Hq = 3, 2, 8
    lens = np.array([40, 17, 5], np.int32)
    pps = 4
    num_pages = B * pps
    bt = rng.permutation(num_pages).astype(np.int32).reshape(B, pps)
    K = wl.bf16_round(rng.standard_normal((B, 40, H, 128)).astype(np.float32))
    V = wl.bf16_round(rng.standard_normal((B, 40, H, 128)).astype(np.float32))
    kn = wl.bf16_round(rng.standard_normal((B, 1, H, 128)).astype(np.float32))
    vn = wl.bf16_round(rng.standard_normal((B, 1, H, 128)).astype(np.float32))
    Q = wl.bf16_round(rng.standard_normal((B, Hq, 128)).astype(np.float32))
    ctx = ctx_for(w)
    try:
        outs, caches = [], []
        for fused in (True, False):
            kc, vc = alloc_caches(ctx, H, num_pages)
            for b in range(B):
                gpu_quantize(ctx, K[b:b + 1, :lens[b]], V[b:b + 1, :lens[b]], "bf16", [0], bt[b:b + 1], num_pages,
                             kc, vc)
            max_len = int(lens.max()) + 1
            n = tq.tq_workspace_size(ctx, B, Hq, max_len, 16)
            ws = torch.empty(n, dtype=torch.uint8, device="cuda")
            out = torch.zeros(B, Hq, 128, dtype=torch.float32, device="cuda")
            qd = to_dev(Q).to(torch.bfloat16)
            if fused:
                tq.tq_append_decode(ctx, to_dev(kn).to(torch.bfloat16), to_dev(vn).to(torch.bfloat16), qd, tq.TQ_BF16,
                                    B, Hq, H, to_dev(lens), max_len, to_dev(bt), pps, num_pages, kc, vc, 16,
                                    scale, out, ws, n)
            else:
                gpu_quantize(ctx, kn, vn, "bf16", lens, bt, num_pages, kc, vc)
                tq.tq_decode_attention(ctx, qd, tq.TQ_BF16, B, Hq, H, to_dev(lens + 1), max_len, to_dev(bt), pps,
                                       num_pages, kc, vc, 16, scale, out, ws, n)
            torch.cuda.synchronize()
            outs.append(out.cpu().numpy())
            caches.append((kc.cpu().numpy(), vc.cpu().numpy()))
        assert tq.tq_check_device_status(ctx) == 0
    finally:
        tq.tq_destroy(ctx)
    assert np.array_equal(caches[0][0], caches[1][0]) and np.array_equal(caches[0][1], caches[1][1])
    # the same kernels over the same bytes and chunks: the fused step's chaining (the query prep ends only
    # after the append) changes no result
    assert np.all(np.isfinite(outs[0]))
    assert np.array_equal(outs[0], outs[1])


def test_decode_chunk_choice():
    """tq_decode_chunk: a multiple of 16; full equal-length batches fill whole waves of warps; a batch of much
    shorter sequences (same max_seq_len) gets chunks no longer than the full batch's; decoding with it is
    what any other chunk gives (the chunking tests above)."""
    w = BASE.scaled(dtype="bf16", k_bits=(4, 3), v_bits=(4, 3))
    ctx = ctx_for(w)
    try:
        full = tq.tq_decode_chunk(ctx, 16, 32, 8, 16 * 32769, 32769)
        short = tq.tq_decode_chunk(ctx, 16, 32, 8, 16 * 6000, 32769)
        assert full % 16 == 0 and short % 16 == 0 and 256 <= short <= full
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        items = 16 * 8 * (-(-32769 // full))
        assert items % sms == 0 or items > 4 * sms
        with pytest.raises(tq.TQError):
            tq.tq_decode_chunk(ctx, 16, 32, 8, 16 * 32769 + 1, 32769)
    finally:
        tq.tq_destroy(ctx)


def test_decode_many_rows_use_the_warp_merge():
    """1,280 query rows (B = 40, 32/8 heads); lengths 0..47 and chunks of 16, so that rows merge up to three
    chunks (one warp per row in the merge, Pi staged in shared memory)."""
    rng = np.random.default_rng(31)
    lens = rng.integers(0, 48, size=40)
    lens[3] = 0
    w = BASE.scaled(k_bits=(4, 3), v_bits=(4, 3), dtype="bf16")
    _check(w, lens, 32, 8, chunk=16, seed=5)


def test_decode_merge_many_chunks():
    """Up to 69 chunks per row (lengths 1,100 / 700 / 5, chunks of 16): the merge gives a row eight warps, each
    merging two batches of chunks, and the row maximum and weight sum run over chunks past the first 32."""
    w = BASE.scaled(k_bits=(3, 3), v_bits=(3, 3), dtype="bf16")
    _check(w, [1100, 700, 5], 8, 2, chunk=16, seed=12)


def test_append_decode_many_rows_against_the_oracle():
    """The fused step at 1,024 query rows (B = 64, 16/4 heads): the append kernel writes the new token, the
    partials kernel covers all L + 1 positions.  The oracle quantizes the cached tokens; the library appends the
    new one; the oracle then decodes over all L + 1 from the bytes the library holds."""
    import torch
    w = BASE.scaled(k_bits=(3, 3), v_bits=(3, 3), dtype="bf16")
    rng = np.random.default_rng(41)
    B, H, Hq = 64, 4, 16
    lens = rng.integers(8, 60, size=B).astype(np.int32)            # cached tokens; the new one goes at lens[b]
    p, bt, num_pages, kc, vc = _oracle_setup(w, lens + 1, H, 9)
    pos = lens.astype(np.int64)
    kn = np.zeros((B, 1, H, 128), np.float32)
    vn = np.zeros((B, 1, H, 128), np.float32)
    # the new token's bf16 K/V: re-drawn here and written by the oracle at position lens[b], over what the setup put
    r2 = np.random.default_rng(43)
    for b in range(B):
        K = wl.bf16_round(r2.standard_normal((1, H, 128)).astype(np.float32))
        V = wl.bf16_round(r2.standard_normal((1, H, 128)).astype(np.float32))
        kn[b, 0], vn[b, 0] = K[0], V[0]
        pages, slots, heads = seq_locations(bt, b, [int(pos[b])], H)
        th.oracle_quantize_into(p, "k", kc, K.reshape(-1, 128), pages, slots, heads, H)
        th.oracle_quantize_into(p, "v", vc, V.reshape(-1, 128), pages, slots, heads, H)
    Q = wl.bf16_round(rng.standard_normal((B, Hq, 128)).astype(np.float32))
    scale = th.scale_for()
    ctx = ctx_for(w)
    try:
        kcd, vcd = to_dev(kc), to_dev(vc)
        max_len = int(lens.max()) + 1
        n = tq.tq_workspace_size(ctx, B, Hq, max_len, 16)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        tq.tq_append_decode(ctx, to_dev(kn).to(torch.bfloat16), to_dev(vn).to(torch.bfloat16),
                            to_dev(Q).to(torch.bfloat16), tq.TQ_BF16, B, Hq, H, to_dev(lens), max_len, to_dev(bt),
                            bt.shape[1], num_pages, kcd, vcd, 16, scale, out, ws, n)
        torch.cuda.synchronize()
        assert tq.tq_check_device_status(ctx) == 0
        got = out.cpu().numpy()
        kc_gpu, vc_gpu = kcd.cpu().numpy(), vcd.cpu().numpy()
    finally:
        tq.tq_destroy(ctx)
    # the oracle decodes the bytes the library holds (quantize exactness has its own tests; a value within the
    # 1e-6 band of a boundary may take the other code)
    ref = oracle.decode_attention(p, Q.astype(np.float64), lens + 1, bt, kc_gpu, vc_gpu, H, scale=scale)
    assert np.all(np.isfinite(got))
    assert th.rel_err(got, ref).max() <= th.ATT_TOL
