"""The fused decode step's append kernel (one warp per new vector), through tq_append_decode.

[P4] riverfrot.github.io "TurboQuant란 무엇이며…", §2.3 (each step's new K/V
join the cache before the new query attends) and §4.1-§4.3 (the records the
append writes).  The new tokens' records are compared field by field with the
oracle's quantization of the same inputs, inside the 1e-6 decision bands too
where the vectors are placed there; every other cache byte must keep its
sentinel.
"""

import numpy as np
import pytest

from .gpu_common import SENTINEL, alloc_caches, ctx_for, oracle, seq_locations, th, to_dev, torch, tq, wl
from .test_gpu_quantize import _near_decision_vectors

pytestmark = pytest.mark.gpu


def _append(w, kn, vn, lens, H, Hq, bt, num_pages, seed=0):
    """tq_append_decode of kn/vn [B, 1, H, 128] at positions lens[b]; returns the caches and the output."""
    B = kn.shape[0]
    rng = np.random.default_rng(seed)
    Q = rng.standard_normal((B, Hq, 128)).astype(np.float32)
    if w.dtype == "bf16":
        Q = wl.bf16_round(Q)
    dt, code = (torch.bfloat16, tq.TQ_BF16) if w.dtype == "bf16" else (torch.float32, tq.TQ_F32)
    ctx = ctx_for(w)
    try:
        tq.tq_refine_counters(ctx, reset=True)
        kc, vc = alloc_caches(ctx, H, num_pages)
        max_len = int(lens.max()) + 1
        n = tq.tq_workspace_size(ctx, B, Hq, max_len, 0)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        tq.tq_append_decode(ctx, to_dev(kn).to(dt), to_dev(vn).to(dt), to_dev(Q).to(dt), code, B, Hq, H,
                            to_dev(lens), max_len, to_dev(bt), bt.shape[1], num_pages, kc, vc, 0, th.scale_for(),
                            out, ws, n)
        torch.cuda.synchronize()
        assert tq.tq_check_device_status(ctx) == 0
        refined = tq.tq_refine_counters(ctx)
        return kc.cpu().numpy(), vc.cpu().numpy(), out.cpu().numpy(), refined
    finally:
        tq.tq_destroy(ctx)


def _check_records(w, H, bt, lens, kn, vn, got_k, got_v, exact_bands=False):
    p = th.params_for(w)
    B = len(lens)
    pages, slots, heads = [], [], []
    for b in range(B):
        pg, sl, hd = seq_locations(bt, b, [int(lens[b])], H)
        pages.append(pg), slots.append(sl), heads.append(hd)
    pages, slots, heads = np.concatenate(pages), np.concatenate(slots), np.concatenate(heads)
    for kind, got, X in (("k", got_k, kn), ("v", got_v, vn)):
        q = oracle.quantize_vectors(p, X.reshape(-1, 128).astype(np.float64), kind)
        ex = oracle.quantize_exclusions(p, q, kind)
        res = th.compare_records(p, kind, got, q, ex, pages, slots, heads, H)
        if exact_bands:      # vectors placed in the bands on purpose: every decision, inside them too
            assert res["codes_mismatch"] == 0 and res["codes_mismatch_excluded"] == 0, res
            assert res["norm_mismatch"] == 0, res
            assert res.get("rnorm_ulp_max", 0) <= 1, res
            if kind == "k" and p.k_qjl:
                raw = oracle.read_paged(p, "k", got, pages, slots, heads, H)
                assert np.array_equal(oracle.unpack_k_records(p, raw)["signs"], q["signs"])
        else:
            th.assert_records_ok(res)
        # nothing outside the new records changed
        touched = th.touched_mask(p, kind, got.size, pages, slots, heads, H)
        assert np.all(got[~touched] == SENTINEL)


@pytest.mark.parametrize("kb,vb,qjl,dtype", [((4, 3), (4, 3), True, "bf16"), ((3, 3), (3, 3), True, "f32"),
                                             ((2, 2), (2, 2), False, "bf16"), ((4, 4), (2, 2), True, "bf16"),
                                             ((1, 2), (3, 1), True, "f32")])
def test_append_records_against_the_oracle(kb, vb, qjl, dtype):
    """37 sequences x 3 KV heads (111 vectors of each kind: the last CTA's warps partly idle), positions across
    page boundaries, N(0,1) tokens with the outlier channels of the workloads."""
    w = wl.WORKLOADS["c3"].scaled(k_bits=kb, v_bits=vb, qjl=qjl, dtype=dtype)
    rng = np.random.default_rng(7)
    B, H, Hq = 37, 3, 6
    lens = rng.integers(0, 64, size=B).astype(np.int32)
    lens[:4] = [0, 15, 16, 63]
    pps = 4
    num_pages = B * pps + 3
    bt = rng.permutation(num_pages)[:B * pps].astype(np.int32).reshape(B, pps)
    kn = rng.standard_normal((B, 1, H, 128)).astype(np.float32)
    kn[..., :w.outlier_channels] *= w.outlier_scale
    vn = rng.standard_normal((B, 1, H, 128)).astype(np.float32)
    if dtype == "bf16":
        kn, vn = wl.bf16_round(kn), wl.bf16_round(vn)
    got_k, got_v, out, _ = _append(w, kn, vn, lens, H, Hq, bt, num_pages)
    _check_records(w, H, bt, lens, kn, vn, got_k, got_v)
    assert np.all(np.isfinite(out))


def test_append_decisions_near_boundaries_are_exact():
    """New tokens whose exact quantization has a code within 3e-6 of a boundary or a sign bit with |z| < 1.5e-5
    ||r||, a zero vector and one whose fp16 norm is zero: the append re-decides them in fp64 and every record
    equals the oracle's, inside the 1e-6 bands too."""
    w = wl.Workload("t", "decode", 1, 1, 1, 64, k_bits=(3, 3), v_bits=(3, 3), dtype="bf16", seed=5)
    p = th.params_for(w)
    near_code, near_sign = _near_decision_vectors(p, 40, 40, seed=23)
    tiny = wl.bf16_round((np.random.default_rng(3).standard_normal((1, 128)) * 1e-9).astype(np.float32))
    X = np.concatenate([near_code, near_sign, np.zeros((1, 128)), tiny]).astype(np.float32)
    B = X.shape[0]
    H = 1
    kn = X.reshape(B, 1, H, 128)
    lens = np.full(B, 5, np.int32)
    bt = np.arange(B, dtype=np.int32)[:, None]
    got_k, got_v, _, refined = _append(w, kn, kn, lens, H, 4, bt, B)
    assert refined[0] >= 40 and refined[1] >= 40, refined
    _check_records(w, H, bt, lens, kn, kn, got_k, got_v, exact_bands=True)


def test_append_bad_page_is_flagged_and_others_written():
    """The new token of one sequence maps to a page id out of range: the append stores nothing for it and
    sets the device error word; the other sequences' records are written as the oracle's."""
    w = wl.WORKLOADS["c3"].scaled(k_bits=(3, 3), v_bits=(3, 3), qjl=True, dtype="bf16")
    rng = np.random.default_rng(9)
    B, H, Hq = 6, 2, 4
    lens = np.array([3, 17, 31, 40, 8, 22], np.int32)
    pps = 4
    num_pages = B * pps
    bt = rng.permutation(num_pages).astype(np.int32).reshape(B, pps)
    bad = 2
    bt[bad, lens[bad] // 16] = num_pages + 7           # the page of sequence 2's new token
    kn = wl.bf16_round(rng.standard_normal((B, 1, H, 128)).astype(np.float32))
    vn = wl.bf16_round(rng.standard_normal((B, 1, H, 128)).astype(np.float32))
    Q = wl.bf16_round(rng.standard_normal((B, Hq, 128)).astype(np.float32))
    ctx = ctx_for(w)
    try:
        kc, vc = alloc_caches(ctx, H, num_pages)
        n = tq.tq_workspace_size(ctx, B, Hq, int(lens.max()) + 1, 0)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        tq.tq_append_decode(ctx, to_dev(kn).to(torch.bfloat16), to_dev(vn).to(torch.bfloat16),
                            to_dev(Q).to(torch.bfloat16), tq.TQ_BF16, B, Hq, H, to_dev(lens), int(lens.max()) + 1,
                            to_dev(bt), pps, num_pages, kc, vc, 0, th.scale_for(), out, ws, n)
        torch.cuda.synchronize()
        assert tq.tq_check_device_status(ctx) != 0
        got_k, got_v = kc.cpu().numpy(), vc.cpu().numpy()
    finally:
        tq.tq_destroy(ctx)
    good = [b for b in range(B) if b != bad]
    p = th.params_for(w)
    pages, slots, heads = [], [], []
    for b in good:
        pg, sl, hd = seq_locations(bt, b, [int(lens[b])], H)
        pages.append(pg), slots.append(sl), heads.append(hd)
    pages, slots, heads = np.concatenate(pages), np.concatenate(slots), np.concatenate(heads)
    for kind, got, X in (("k", got_k, kn), ("v", got_v, vn)):
        q = oracle.quantize_vectors(p, X[good].reshape(-1, 128).astype(np.float64), kind)
        res = th.compare_records(p, kind, got, q, oracle.quantize_exclusions(p, q, kind), pages, slots, heads, H)
        th.assert_records_ok(res)
        touched = th.touched_mask(p, kind, got.size, pages, slots, heads, H)
        assert np.all(got[~touched] == SENTINEL)       # nothing written for the bad page, nor anywhere else
