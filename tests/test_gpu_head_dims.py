"""Head dimensions other than 128 (d a multiple of 32 up to 256) on the GPU against the oracle, through the C ABI.

[P4] riverfrot.github.io "TurboQuant란 무엇이며…", §4.1-§4.3: nothing in the method fixes d; the rotation, the
QJL matrix and the codebook (fitted per (d, b) for the exact density) are drawn for the context's d.  Quantize:
every record field the GPU writes equals the oracle's (codes and signs bit for bit outside the exact-tie
exclusions, norms exactly, residual norms within one fp16 ulp).  Decode: the GPU's attention output over
oracle-written cache bytes is within the attention bar of the oracle's fp64 softmax.
"""

import math

import numpy as np
import pytest

from .gpu_common import DEV, oracle, oracle_cache_bytes, seq_locations, to_dev, torch, tq, wl
from . import helpers as th

pytestmark = pytest.mark.gpu


def _params(d, kb, vb, split, m, qjl, seed, codebook="gaussian"):
    return oracle.make_params(d=d, m=m, k_bits=kb, k_split=split, v_bits=vb, v_split=split, seed=seed, k_qjl=qjl,
                              codebook=codebook)


def _ctx(d, kb, vb, split, m, qjl, seed, codebook="gaussian"):
    cfg = tq.make_config(k_bits=kb, v_bits=vb, m=m, seed=seed, k_split=split, v_split=split, k_qjl=qjl, d=d,
                         codebook=tq.TQ_CODEBOOK_SPHERE if codebook == "sphere" else tq.TQ_CODEBOOK_GAUSSIAN)
    return tq.tq_create_ex(cfg)


def _draw(rng, shape, dtype, outliers=4):
    X = rng.standard_normal(shape).astype(np.float32)
    X[..., :outliers] *= 10
    return wl.bf16_round(X) if dtype == "bf16" else X


QUANT_CASES = [
    # d, k_bits, v_bits, split, m, qjl, dtype, codebook
    (256, (3, 3), (3, 3), 128, 128, True, "bf16", "gaussian"),
    (256, (4, 3), (4, 2), 128, 128, True, "f32", "gaussian"),
    (256, (2, 4), (1, 3), 64, 96, True, "bf16", "sphere"),
    (256, (4, 4), (4, 4), 256, 128, False, "bf16", "gaussian"),
    (64, (3, 2), (3, 2), 32, 64, True, "f32", "sphere"),
    (96, (4, 3), (3, 3), 32, 128, True, "bf16", "gaussian"),
    (32, (3, 3), (2, 2), 0, 32, True, "f32", "sphere"),
    (160, (1, 2), (4, 1), 96, 128, True, "bf16", "gaussian"),
]


@pytest.mark.parametrize("d,kb,vb,split,m,qjl,dtype,codebook", QUANT_CASES)
def test_quantize_records_match_oracle(d, kb, vb, split, m, qjl, dtype, codebook):
    B, T, H = 3, 21, 2
    starts = np.array([0, 7, 30], np.int32)
    seed = d + split + m
    rng = np.random.default_rng(seed)
    pps = (int(starts.max()) + T + 15) // 16
    num_pages = B * pps + 2
    bt = rng.permutation(num_pages)[:B * pps].astype(np.int32).reshape(B, pps)
    K = _draw(rng, (B, T, H, d), dtype)
    V = _draw(rng, (B, T, H, d), dtype, outliers=0)
    ctx = _ctx(d, kb, vb, split, m, qjl, seed, codebook)
    try:
        kpb, vpb = tq.tq_cache_layout(ctx, H)
        kc = torch.full((num_pages * kpb,), 0xA5, dtype=torch.uint8, device=DEV)
        vc = torch.full((num_pages * vpb,), 0xA5, dtype=torch.uint8, device=DEV)
        code = tq.TQ_BF16 if dtype == "bf16" else tq.TQ_F32
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        tq.tq_quantize(ctx, to_dev(K).to(tdt), to_dev(V).to(tdt), code, B, T, H, to_dev(starts), to_dev(bt), pps,
                       num_pages, kc, vc)
        torch.cuda.synchronize()
        assert tq.tq_check_device_status(ctx) == 0
        got = {"k": kc.cpu().numpy(), "v": vc.cpu().numpy()}
    finally:
        tq.tq_destroy(ctx)
    p = _params(d, kb, vb, split, m, qjl, seed, codebook)
    assert oracle.cache_block_bytes(p, "k") * H == kpb and oracle.cache_block_bytes(p, "v") * H == vpb
    pages, slots, heads = map(np.concatenate, zip(*[seq_locations(bt, b, starts[b] + np.arange(T), H)
                                                     for b in range(B)]))
    for kind, X in (("k", K), ("v", V)):
        want = oracle_cache_bytes(p, H, num_pages, kind)
        q, ex = th.oracle_quantize_into(p, kind, want, X.reshape(-1, d), pages, slots, heads, H)
        res = th.compare_records(p, kind, got[kind], q, ex, pages, slots, heads, H)
        th.assert_records_ok(res)
        mask = th.touched_mask(p, kind, got[kind].size, pages, slots, heads, H)
        assert np.all(got[kind][~mask] == 0xA5)


def _oracle_caches(p, d, lens, H, rng, dtype, num_pages, bt):
    kc = oracle_cache_bytes(p, H, num_pages, "k")
    vc = oracle_cache_bytes(p, H, num_pages, "v")
    for b, L in enumerate(lens):
        if L == 0:
            continue
        K = _draw(rng, (int(L), H, d), dtype)
        V = _draw(rng, (int(L), H, d), dtype, outliers=0)
        pages, slots, heads = seq_locations(bt, b, np.arange(int(L)), H)
        th.oracle_quantize_into(p, "k", kc, K.reshape(-1, d), pages, slots, heads, H)
        th.oracle_quantize_into(p, "v", vc, V.reshape(-1, d), pages, slots, heads, H)
    return kc, vc


def _decode_case(d, kb, vb, split, m, qjl, lens, Hq, H, chunk=0, qdtype="bf16", seed=0, noalloc=False):
    lens = np.asarray(lens, np.int32)
    rng = np.random.default_rng(seed)
    B = len(lens)
    pps = max(1, (int(lens.max()) + 15) // 16)
    num_pages = B * pps + 1
    bt = rng.permutation(num_pages)[:B * pps].astype(np.int32).reshape(B, pps)
    p = _params(d, kb, vb, split, m, qjl, seed)
    kc, vc = _oracle_caches(p, d, lens, H, rng, "bf16", num_pages, bt)
    Q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    if qdtype == "bf16":
        Q = wl.bf16_round(Q)
    scale = 1.0 / math.sqrt(d)
    max_len = int(max(lens.max(), 1))
    ctx = _ctx(d, kb, vb, split, m, qjl, seed)
    try:
        qt = to_dev(Q).to(torch.bfloat16) if qdtype == "bf16" else to_dev(Q)
        code = tq.TQ_BF16 if qdtype == "bf16" else tq.TQ_F32
        out = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device=DEV)
        if noalloc:
            tq.tq_decode_attention_noalloc(ctx, qt, code, B, Hq, H, to_dev(lens), max_len, to_dev(bt), pps,
                                           num_pages, to_dev(kc), to_dev(vc), chunk, scale, out)
        else:
            n = tq.tq_workspace_size(ctx, B, Hq, max_len, chunk)
            ws = torch.empty(n, dtype=torch.uint8, device=DEV)
            tq.tq_decode_attention(ctx, qt, code, B, Hq, H, to_dev(lens), max_len, to_dev(bt), pps, num_pages,
                                   to_dev(kc), to_dev(vc), chunk, scale, out, ws, n)
        torch.cuda.synchronize()
        assert tq.tq_check_device_status(ctx) == 0
        got = out.cpu().numpy()
    finally:
        tq.tq_destroy(ctx)
    want = oracle.decode_attention(p, Q.astype(np.float64), lens, bt, kc, vc, H, scale=scale)
    assert np.all(np.isfinite(got))
    err = th.rel_err(got.reshape(-1, d), want.reshape(-1, d))
    assert err.max() <= th.ATT_TOL, (float(err.max()), int(err.argmax()))
    return err.max()


@pytest.mark.parametrize("kb,vb,split,qjl", [((3, 3), (3, 3), 128, True), ((4, 3), (4, 3), 128, True),
                                             ((3, 2), (2, 2), 96, True), ((4, 4), (4, 4), 0, False),
                                             ((1, 2), (4, 1), 160, True)])
def test_decode_d256_bit_widths(kb, vb, split, qjl):
    _decode_case(256, kb, vb, split, 128, qjl, lens=[70, 1, 33], Hq=8, H=2, seed=sum(kb) + split)


@pytest.mark.parametrize("lens,Hq,H,chunk", [([0, 5, 300], 4, 4, 0), ([129], 8, 1, 32), ([17, 64, 2, 100], 6, 2, 16),
                                             ([511, 40], 16, 2, 128)])
def test_decode_d256_lengths_groups_chunks(lens, Hq, H, chunk):
    _decode_case(256, (3, 3), (3, 3), 128, 128, True, lens=lens, Hq=Hq, H=H, chunk=chunk, seed=len(lens) + Hq)


@pytest.mark.parametrize("d,m", [(64, 64), (96, 128), (32, 32), (192, 96)])
def test_decode_other_dims(d, m):
    _decode_case(d, (4, 3), (3, 3), (d // 64) * 32, m, True, lens=[45, 3], Hq=4, H=1, qdtype="f32", seed=d)


def test_decode_d256_noalloc():
    _decode_case(256, (3, 3), (3, 3), 128, 128, True, lens=[90, 31], Hq=8, H=4, noalloc=True, seed=4)


def test_append_decode_d256_matches_oracle():
    """The fused step at d = 256: the new token's K/V are quantized into the cache (records equal to the
    oracle's) and the query attends over the L + 1 tokens."""
    d, kb, vb, split, m, H, Hq = 256, (4, 3), (4, 3), 128, 128, 2, 8
    lens = np.array([40, 17, 0], np.int32)
    B = len(lens)
    rng = np.random.default_rng(31)
    pps = 4
    num_pages = B * pps
    bt = rng.permutation(num_pages).astype(np.int32).reshape(B, pps)
    p = _params(d, kb, vb, split, m, True, 31)
    kc, vc = _oracle_caches(p, d, lens, H, rng, "bf16", num_pages, bt)
    kn = _draw(rng, (B, 1, H, d), "bf16")
    vn = _draw(rng, (B, 1, H, d), "bf16", outliers=0)
    Q = wl.bf16_round(rng.standard_normal((B, Hq, d)).astype(np.float32))
    scale = 1.0 / math.sqrt(d)
    ctx = _ctx(d, kb, vb, split, m, True, 31)
    try:
        kcd, vcd = to_dev(kc), to_dev(vc)
        max_len = int(lens.max()) + 1
        n = tq.tq_workspace_size(ctx, B, Hq, max_len, 0)
        ws = torch.empty(n, dtype=torch.uint8, device=DEV)
        out = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device=DEV)
        tq.tq_append_decode(ctx, to_dev(kn).to(torch.bfloat16), to_dev(vn).to(torch.bfloat16),
                            to_dev(Q).to(torch.bfloat16), tq.TQ_BF16, B, Hq, H, to_dev(lens), max_len, to_dev(bt), pps,
                            num_pages, kcd, vcd, 0, scale, out, ws, n)
        torch.cuda.synchronize()
        assert tq.tq_check_device_status(ctx) == 0
        got, gk, gv = out.cpu().numpy(), kcd.cpu().numpy(), vcd.cpu().numpy()
    finally:
        tq.tq_destroy(ctx)
    pages, slots, heads = map(np.concatenate, zip(*[seq_locations(bt, b, [lens[b]], H) for b in range(B)]))
    for kind, X, cache, g in (("k", kn, kc, gk), ("v", vn, vc, gv)):
        q, ex = th.oracle_quantize_into(p, kind, cache, X.reshape(-1, d), pages, slots, heads, H)
        th.assert_records_ok(th.compare_records(p, kind, g, q, ex, pages, slots, heads, H))
    want = oracle.decode_attention(p, Q.astype(np.float64), lens + 1, bt, kc, vc, H, scale=scale)
    err = th.rel_err(got.reshape(-1, d), want.reshape(-1, d))
    assert err.max() <= th.ATT_TOL, float(err.max())


def test_d256_causal_and_search_are_unsupported():
    ctx = _ctx(256, (3, 3), (3, 3), 128, 128, True, 1)
    try:
        st = tq.raw_status("tq_causal_attention", ctx, 16, tq.TQ_BF16, 1, 4, 4, 1, 16, 64, 16, 4, 4, 16, 16, 0,
                           0.1, 16, 16, 1 << 30, None)
        assert st == tq.TQ_ERR_UNSUPPORTED
        st = tq.raw_status("tq_search", ctx, 16, tq.TQ_BF16, 1, 16, 16, 1, 16, 1, 16, 16, 16, 1 << 30, None)
        assert st == tq.TQ_ERR_UNSUPPORTED
    finally:
        tq.tq_destroy(ctx)
