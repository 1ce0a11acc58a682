"""GPU quantize parity against the oracle, through the C ABI."""

import numpy as np
import pytest

from .gpu_common import (alloc_caches, ctx_for, gpu_quantize, oracle, oracle_cache_bytes, seq_locations, th, tq,
                         wl)

pytestmark = pytest.mark.gpu

VARIANTS = [
    # k_bits, v_bits, qjl, m, dtype
    ((3, 3), (3, 3), True, 128, "f32"),
    ((3, 3), (3, 3), True, 128, "bf16"),
    ((4, 3), (4, 3), True, 128, "bf16"),
    ((3, 2), (3, 2), True, 128, "bf16"),
    ((1, 1), (2, 2), True, 64, "f32"),
    ((4, 4), (1, 4), False, 128, "bf16"),
    ((2, 4), (4, 1), True, 96, "f32"),
]


def _run_case(kb, vb, qjl, m, dtype, B=3, T=37, H=2, starts=(0, 5, 19), seed=11, codebook="gaussian"):
    w = wl.Workload("t", "quantize", B, H, H, T, k_bits=kb, v_bits=vb, qjl=qjl, m=m, dtype=dtype, seed=seed,
                    codebook=codebook)
    rng = np.random.default_rng(seed)
    pps = (max(starts) + T + 15) // 16
    num_pages = B * pps + 3
    bt = rng.permutation(num_pages)[:B * pps].astype(np.int32).reshape(B, pps)
    K = rng.standard_normal((B, T, H, 128)).astype(np.float32)
    K[..., :4] *= 10
    V = rng.standard_normal((B, T, H, 128)).astype(np.float32)
    if dtype == "bf16":
        K, V = wl.bf16_round(K), wl.bf16_round(V)
    ctx = ctx_for(w)
    try:
        kc, vc = alloc_caches(ctx, H, num_pages)
        gpu_quantize(ctx, K, V, dtype, starts, bt, num_pages, kc, vc)
        assert tq.tq_check_device_status(ctx) == 0
        got_k, got_v = kc.cpu().numpy(), vc.cpu().numpy()
    finally:
        tq.tq_destroy(ctx)
    p = th.params_for(w)
    for kind, X, got in (("k", K, got_k), ("v", V, got_v)):
        pages, slots, heads = [], [], []
        for b in range(B):
            pg, sl, hd = seq_locations(bt, b, starts[b] + np.arange(T), H)
            pages.append(pg), slots.append(sl), heads.append(hd)
        pages, slots, heads = map(np.concatenate, (pages, slots, heads))
        want = oracle_cache_bytes(p, H, num_pages, kind)
        q, ex = th.oracle_quantize_into(p, kind, want, X.reshape(-1, 128), pages, slots, heads, H)
        res = th.compare_records(p, kind, got, q, ex, pages, slots, heads, H)
        th.assert_records_ok(res)
        # addressing: bytes outside the written records are untouched
        mask = th.touched_mask(p, kind, got.size, pages, slots, heads, H)
        assert np.all(got[~mask] == 0xA5)
        # and written bytes equal the oracle's except where a residual norm may differ by one ulp
        diff = np.nonzero(got != want)[0]
        if kind == "v" or not qjl:
            assert diff.size == 0 or res["codes_mismatch_excluded"] > 0, res


@pytest.mark.parametrize("kb,vb,qjl,m,dtype", VARIANTS)
def test_quantize_matches_oracle(kb, vb, qjl, m, dtype):
    _run_case(kb, vb, qjl, m, dtype)


@pytest.mark.parametrize("kb,vb", [((3, 3), (3, 3)), ((4, 3), (4, 3)), ((4, 4), (2, 2)), ((1, 1), (1, 1))])
def test_quantize_sphere_codebook(kb, vb):
    """Codebooks fitted to the exact rotated-coordinate density: the same bit-exact record parity on the
    tensor-core path (and the SIMT path for 1 bit)."""
    _run_case(kb, vb, True, 128, "bf16", T=150, codebook="sphere")


def test_quantize_many_tiles_ragged_tail():
    # 1000 vectors per kind: 31 full tiles of 32 and a ragged tail of 8
    _run_case((3, 3), (3, 3), True, 128, "bf16", B=5, T=25, H=8, starts=(0, 16, 3, 40, 7), seed=5)


def test_append_one_token_at_a_time_equals_bulk():
    w = wl.Workload("t", "quantize", 2, 4, 4, 21, seed=2)
    rng = np.random.default_rng(2)
    B, T, H = 2, 21, 4
    pps = 2
    bt = np.array([[3, 0], [1, 2]], dtype=np.int32)
    K = wl.bf16_round(rng.standard_normal((B, T, H, 128)).astype(np.float32))
    V = wl.bf16_round(rng.standard_normal((B, T, H, 128)).astype(np.float32))
    ctx = ctx_for(w)
    try:
        kc1, vc1 = alloc_caches(ctx, H, 4)
        gpu_quantize(ctx, K, V, "bf16", [0, 0], bt, 4, kc1, vc1)
        kc2, vc2 = alloc_caches(ctx, H, 4)
        for t in range(T):
            gpu_quantize(ctx, K[:, t:t + 1], V[:, t:t + 1], "bf16", [t, t], bt, 4, kc2, vc2)
        assert tq.tq_check_device_status(ctx) == 0
        assert np.array_equal(kc1.cpu().numpy(), kc2.cpu().numpy())
        assert np.array_equal(vc1.cpu().numpy(), vc2.cpu().numpy())
    finally:
        tq.tq_destroy(ctx)


def test_zero_and_boundary_vectors():
    """A zero vector, a vector whose fp16 norm is zero, and vectors placed exactly on codebook boundaries.

    The 22 boundary vectors carry 16 boundary coordinates each: 352 exact
    re-decisions in one tile, more than one pass of the re-decision queue holds.
    """
    T = 24
    w = wl.Workload("t", "quantize", 1, 1, 1, T, dtype="f32", seed=0)
    p = th.params_for(w)
    cb = p.books[3]
    X = np.zeros((T, 128))
    for r in range(1, T - 1):
        u = np.random.default_rng(r).standard_normal(128)
        u[:16] = cb.boundaries[np.arange(16) % 7]
        u[16:] *= np.sqrt((128 - np.sum(u[:16] ** 2)) / np.sum(u[16:] ** 2))    # ||u||^2 = d, so u is kept
        X[r] = p.Pi.T @ (u * 3.0 / np.sqrt(128))                                # ||x|| = 3
    X[T - 1] = np.random.default_rng(99).standard_normal(128) * 1e-9     # ||x|| ~ 1e-8: fp16 norm 0
    X = X.astype(np.float32)
    K = X.reshape(1, T, 1, 128)
    bt = np.array([[0, 1]], dtype=np.int32)
    ctx = ctx_for(w)
    try:
        tq.tq_refine_counters(ctx, reset=True)
        kc, vc = alloc_caches(ctx, 1, 2)
        gpu_quantize(ctx, K, K, "f32", [0], bt, 2, kc, vc)
        assert tq.tq_check_device_status(ctx) == 0
        refined = tq.tq_refine_counters(ctx)
        got_k, got_v = kc.cpu().numpy(), vc.cpu().numpy()
    finally:
        tq.tq_destroy(ctx)
    assert refined[0] >= 2 * (T - 2) * 16
    pages, slots, heads = seq_locations(bt, 0, np.arange(T), 1)
    for kind, got in (("k", got_k), ("v", got_v)):
        q = oracle.quantize_vectors(p, X.astype(np.float64), kind)
        assert q["n16"][T - 1] == 0 and q["norm"][T - 1] > 0
        res = th.compare_records(p, kind, got, q, oracle.quantize_exclusions(p, q, kind), pages, slots, heads, 1)
        assert res["codes_mismatch"] == 0 and res["norm_mismatch"] == 0, res
        # the values within 1e-6 of a boundary were re-decided in fp64: they agree too
        assert res["codes_excluded"] >= (T - 2) * 16 and res["codes_mismatch_excluded"] == 0, res
        if kind == "k":
            assert res["signs_mismatch"] == 0, res


def _near_decision_vectors(p, n_code, n_sign, seed):
    """bf16-valued vectors whose exact quantization has a code within 3e-6 of a boundary (u units) or a sign bit
    with |z| < 1.5e-5 ||r|| -- decisions the fast tensor-core arithmetic cannot take for certain -- found by
    searching seeded N(0,1) draws with the oracle."""
    rng = np.random.default_rng(seed)
    near_code, near_sign = [], []
    for _ in range(200):
        if len(near_code) >= n_code and len(near_sign) >= n_sign:
            break
        X = wl.bf16_round(rng.standard_normal((8192, 128)).astype(np.float32)).astype(np.float64)
        q = oracle.quantize_vectors(p, X, "k")
        t = p.books[3].boundaries
        dist = np.min(np.abs(q["u"][:, :, None] - t[None, None, :]), axis=(1, 2))
        zmin = np.min(np.abs(q["z"]), axis=1) / q["rho"]
        near_code += list(X[dist < 3e-6])
        near_sign += list(X[(zmin < 1.5e-5) & (dist >= 3e-6)])
    assert len(near_code) >= n_code and len(near_sign) >= n_sign
    return np.array(near_code[:n_code]), np.array(near_sign[:n_sign])


def test_bf16_decisions_near_boundaries_are_exact():
    """The bf16 tensor-core path hands every decision inside its guard (code near a boundary, sign near zero) to
    exact double-float arithmetic.  Two tiles of vectors with a code near a boundary and two with a sign near
    zero give hundreds of such decisions at once -- more than the kernel's queue for them holds, so some are
    taken where they arise -- and every record still equals the oracle's, inside the 1e-6 bands too."""
    w = wl.Workload("t", "quantize", 1, 1, 1, 1024, k_bits=(3, 3), v_bits=(3, 3), seed=5)
    p = th.params_for(w)
    near_code, near_sign = _near_decision_vectors(p, 256, 256, seed=17)
    rest = wl.bf16_round(np.random.default_rng(18).standard_normal((512, 128)).astype(np.float32))
    X = np.concatenate([near_code, near_sign, rest]).astype(np.float32)
    T = X.shape[0]
    K = X.reshape(1, T, 1, 128)
    bt = np.arange(T // 16, dtype=np.int32)[None, :]
    ctx = ctx_for(w)
    try:
        tq.tq_refine_counters(ctx, reset=True)
        kc, vc = alloc_caches(ctx, 1, T // 16)
        gpu_quantize(ctx, K, K, "bf16", [0], bt, T // 16, kc, vc)
        assert tq.tq_check_device_status(ctx) == 0
        refined = tq.tq_refine_counters(ctx)
        got = {"k": kc.cpu().numpy(), "v": vc.cpu().numpy()}
    finally:
        tq.tq_destroy(ctx)
    assert refined[0] >= 2 * 256 and refined[1] >= 256, refined
    pages, slots, heads = seq_locations(bt, 0, np.arange(T), 1)
    for kind in ("k", "v"):
        q = oracle.quantize_vectors(p, X.astype(np.float64), kind)
        ex = oracle.quantize_exclusions(p, q, kind)
        res = th.compare_records(p, kind, got[kind], q, ex, pages, slots, heads, 1)
        assert res["codes_mismatch"] == 0 and res["codes_mismatch_excluded"] == 0 and res["norm_mismatch"] == 0, res
        if kind == "k":
            raw = oracle.read_paged(p, "k", got["k"], pages, slots, heads, 1)
            rec = oracle.unpack_k_records(p, raw)
            assert np.array_equal(rec["signs"], q["signs"])            # every sign bit, inside the band too
            assert res["rnorm_ulp_max"] <= 1, res


def test_out_of_range_pages_are_skipped_and_flagged():
    w = wl.Workload("t", "quantize", 2, 1, 1, 20, seed=3)
    rng = np.random.default_rng(3)
    K = wl.bf16_round(rng.standard_normal((2, 20, 1, 128)).astype(np.float32))
    bt = np.array([[0, 7], [1, 2]], dtype=np.int32)     # page 7 does not exist (3 pages)
    ctx = ctx_for(w)
    try:
        kc, vc = alloc_caches(ctx, 1, 3)
        gpu_quantize(ctx, K, K, "bf16", [0, 30], bt, 3, kc, vc)   # seq 1: positions 30.. exceed 2 pages
        flags = tq.tq_check_device_status(ctx)
        assert flags & 1 and flags & 2
        assert tq.tq_check_device_status(ctx) == 0               # cleared by the read
        got = kc.cpu().numpy()
    finally:
        tq.tq_destroy(ctx)
    p = th.params_for(w)
    # tokens 0..15 of seq 0 landed in page 0, positions 30-31 of seq 1 in page 2; nothing else was written
    pg0, sl0, hd0 = seq_locations(bt, 0, np.arange(16), 1)
    pg1, sl1, hd1 = seq_locations(bt, 1, np.array([30, 31]), 1)
    pages, slots, heads = np.r_[pg0, pg1], np.r_[sl0, sl1], np.r_[hd0, hd1]
    X = np.concatenate([K[0, :16, 0], K[1, :2, 0]]).astype(np.float64)
    q = oracle.quantize_vectors(p, X, "k")
    th.assert_records_ok(th.compare_records(p, "k", got, q, oracle.quantize_exclusions(p, q, "k"),
                                            pages, slots, heads, 1))
    mask = th.touched_mask(p, "k", got.size, pages, slots, heads, 1)
    assert np.all(got[~mask] == 0xA5)


def test_invalid_arguments_launch_nothing():
    w = wl.Workload("t", "quantize", 1, 1, 1, 4, seed=0)
    ctx = ctx_for(w)
    try:
        kc, vc = alloc_caches(ctx, 1, 1)
        bt = np.zeros((1, 1), np.int32)
        with pytest.raises(tq.TQError):
            gpu_quantize(ctx, np.zeros((1, 4, 1, 128), np.float32), None, "f32", [0], bt, 0, kc, vc)
        with pytest.raises(tq.TQError):
            tq.tq_quantize(ctx, kc, None, 7, 1, 1, 1, kc, kc, 1, 1, kc, None)
        assert np.all(kc.cpu().numpy() == 0xA5)
    finally:
        tq.tq_destroy(ctx)
