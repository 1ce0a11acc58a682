"""Inner-product search (the decode's two-stage estimate without softmax, then the k best per query)
against the oracle, through the C ABI.

Both sides read the same database bytes: the oracle quantizes and packs the vectors into one KV head's
K cache, the bytes go to the device unchanged.  Checked: every score (tq_search_scores, the arithmetic of
the path tq_search takes for that k) against the oracle's fp64 estimate; the returned top k as the exact
stable ranking of the GPU's own scores (index work: bit-exact); and the returned vectors against the
oracle's ranking up to the score tolerance.

Score bar: the tensor-core path (k <= 16, 2-4-bit key groups, m = 128) multiplies the decode's fp16
operands -- q~, u and the centroids rounded to fp16 (relative 2^-12 each), fp32 accumulation -- which an
fp64 emulation of that arithmetic puts at up to 5.8e-4 of the query's largest |score| on N(0,1) data with
outlier channels; the bar is 1.5e-3 of it.  The CUDA-core path (fp32 throughout) keeps 1e-4.
"""

import numpy as np
import pytest

from .gpu_common import DEV, ctx_for, input_tensor, oracle, th, to_dev, torch, tq, wl

pytestmark = pytest.mark.gpu


def _database(w, n, seed, perm_pages=True, X=None):
    rng = np.random.default_rng(seed)
    if X is None:
        X = rng.standard_normal((n, 128)).astype(np.float32)
        X[:, :w.outlier_channels] *= w.outlier_scale
    npg = (n + 15) // 16
    num_pages = npg + 3
    row = (rng.permutation(num_pages)[:npg] if perm_pages else np.arange(npg)).astype(np.int32)
    p = th.params_for(w)
    cache = np.zeros(num_pages * oracle.cache_block_bytes(p, "k"), dtype=np.uint8)
    th.oracle_quantize_into(p, "k", cache, X, row[np.arange(n) // 16].astype(np.int64), np.arange(n) % 16,
                            np.zeros(n, dtype=np.int64), 1)
    return p, X, row, num_pages, cache


def _tensor_core_path(w, k):
    return k <= 16 and w.m == 128 and all(2 <= b <= 4 for b in w.k_bits)


def _search(ctx, Q, dtype, row, num_pages, cache, n, k):
    nq = Q.shape[0]
    qd, code = input_tensor(Q, dtype)
    kc, bt = to_dev(cache), to_dev(row)
    ws_n = tq.tq_search_workspace_size(ctx, nq, n, k)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=DEV)
    ts = torch.full((nq, k), float("nan"), dtype=torch.float32, device=DEV)
    ti = torch.full((nq, k), -1, dtype=torch.int32, device=DEV)
    tq.tq_search(ctx, qd, code, nq, kc, bt, num_pages, n, k, ts, ti, ws, ws_n)
    ws0_n = tq.tq_search_workspace_size(ctx, nq, n, 0)
    ws0 = torch.empty(ws0_n, dtype=torch.uint8, device=DEV)
    sc = torch.full((nq, n), float("nan"), dtype=torch.float32, device=DEV)
    tq.tq_search_scores(ctx, qd, code, nq, kc, bt, num_pages, n, k, sc, ws0, ws0_n)
    torch.cuda.synchronize()
    return ts.cpu().numpy(), ti.cpu().numpy(), sc.cpu().numpy()


def _check(w, n, nq, k, dtype="bf16", seed=0, X=None, Q=None):
    p, X, row, num_pages, cache = _database(w, n, seed, X=X)
    if Q is None:
        Q = np.random.default_rng(seed + 1).standard_normal((nq, 128)).astype(np.float32)
    if dtype == "bf16":
        Q = wl.bf16_round(Q)
    ctx = ctx_for(w)
    try:
        ts, ti, scores = _search(ctx, Q, dtype, row, num_pages, cache, n, k)
        assert tq.tq_check_device_status(ctx) == 0
    finally:
        tq.tq_destroy(ctx)
    want, wtop, wvals = oracle.search(p, Q.astype(np.float64), row, cache, n, k)
    scale = np.abs(want).max(axis=1, keepdims=True)
    tol = (1.5e-3 if _tensor_core_path(w, k) else 1e-4) * scale
    # every score
    assert np.all(np.abs(scores - want) <= tol), float(np.max(np.abs(scores - want) / scale))
    # the returned k: the exact stable ranking of the GPU's own scores
    mine = np.argsort(-scores, axis=1, kind="stable")[:, :k]
    assert np.array_equal(ti, mine)
    assert np.array_equal(ts, np.take_along_axis(scores, ti, axis=1))
    # against the oracle: each returned vector scores within tol of the oracle's k-th best or above
    got_true = np.take_along_axis(want, ti.astype(np.int64), axis=1)
    assert np.all(got_true >= wvals[:, -1:] - 2 * tol)
    return ti, wtop


@pytest.mark.parametrize("kb,qjl", [((3, 3), True), ((4, 3), True), ((3, 2), True), ((2, 2), False)])
def test_search_matches_oracle(kb, qjl):
    w = wl.Workload("s", "search", 1, 1, 1, 0, k_bits=kb, qjl=qjl, seed=4)
    _check(w, 1000, 13, 10)


def test_search_ragged_sizes_and_full_k():
    """One query, a database of 37 vectors (a partial page), every vector returned; fp32 queries; 2049
    vectors (two scoring blocks, the second with one vector) and 9 queries (two query groups)."""
    w = wl.Workload("s", "search", 1, 1, 1, 0, k_bits=(3, 3), seed=5)
    _check(w, 37, 1, 37, dtype="f32", seed=1)
    _check(w, 2049, 9, 5, seed=2)


def test_search_finds_scaled_copies():
    """Each query's scaled copy in the database ranks first on the GPU as in the oracle."""
    w = wl.Workload("s", "search", 1, 1, 1, 0, k_bits=(3, 3), seed=6)
    rng = np.random.default_rng(11)
    Q = rng.standard_normal((5, 128)).astype(np.float32)
    X = rng.standard_normal((700, 128)).astype(np.float32)
    where = rng.choice(700, 5, replace=False)
    X[where] = 4.0 * Q
    ti, wtop = _check(w, 700, 5, 3, dtype="f32", seed=3, X=X, Q=Q)
    assert np.array_equal(ti[:, 0], where) and np.array_equal(wtop[:, 0], where)


@pytest.mark.parametrize("kb,qjl", [((4, 4), True), ((2, 4), True), ((4, 2), False), ((3, 4), True)])
def test_search_tensor_core_bit_widths(kb, qjl):
    w = wl.Workload("s", "search", 1, 1, 1, 0, k_bits=kb, qjl=qjl, seed=9)
    _check(w, 1500, 7, 16)


@pytest.mark.parametrize("kb", [(4, 3), (3, 3)])
def test_search_several_query_blocks(kb):
    """130 queries: three blocks of up to 64 on the tensor-core path (the last one ragged), 3000 vectors
    (24 tiles of 128, the last partial); 4/3-bit keys run one epilogue group, 3-bit keys two (each block's
    shared bars cleared before it)."""
    w = wl.Workload("s", "search", 1, 1, 1, 0, k_bits=kb, seed=10)
    _check(w, 3000, 130, 16, seed=5)


@pytest.mark.parametrize("k", [16, 40])
def test_search_ties_keep_the_lowest_indices(k):
    """One vector copied to 700 positions spread over the whole database (many tiles and CTAs): its copies
    have bit-identical records and scores, rank first for a query along it, and the cut inside the tie group
    keeps the lowest indices in order -- on both paths (k = 16 tensor cores, k = 40 CUDA cores)."""
    w = wl.Workload("s", "search", 1, 1, 1, 0, k_bits=(3, 3), seed=11)
    rng = np.random.default_rng(21)
    n = 20000
    X = rng.standard_normal((n, 128)).astype(np.float32)
    Q = rng.standard_normal((2, 128)).astype(np.float32)
    where = np.sort(rng.choice(n, 700, replace=False))
    X[where] = 6.0 * Q[0]
    ti, wtop = _check(w, n, 2, k, dtype="f32", seed=4, X=X, Q=Q)
    assert np.array_equal(ti[0], where[:k]) and np.array_equal(wtop[0], where[:k])


def test_search_bad_page_and_arguments():
    """A page id out of range: its vectors score -inf (never ranked above a real one) and the device
    error word is set; bad arguments and a short workspace are rejected before any launch."""
    w = wl.Workload("s", "search", 1, 1, 1, 0, k_bits=(3, 3), seed=7)
    p, X, row, num_pages, cache = _database(w, 64, 3)
    row = row.copy()
    row[1] = num_pages + 5                          # vectors 16..31
    Q = wl.bf16_round(np.random.default_rng(4).standard_normal((3, 128)).astype(np.float32))
    ctx = ctx_for(w)
    try:
        ts, ti, scores = _search(ctx, Q, "bf16", row, num_pages, cache, 64, 48)
        assert tq.tq_check_device_status(ctx) != 0
        assert np.all(np.isneginf(scores[:, 16:32]))
        assert not np.any((ti >= 16) & (ti < 32))
        qd, code = input_tensor(Q, "bf16")
        ws = torch.empty(tq.tq_search_workspace_size(ctx, 3, 64, 8), dtype=torch.uint8, device=DEV)
        out_s = torch.empty(3, 8, device=DEV)
        out_i = torch.empty(3, 8, dtype=torch.int32, device=DEV)
        kc, bt = to_dev(cache), to_dev(row)
        for k_top, n_db, ws_n in ((0, 64, ws.numel()), (65, 64, ws.numel()), (1025, 2000, ws.numel()),
                                  (8, 64, ws.numel() - 1), (8, num_pages * 16 + 1, ws.numel())):
            with pytest.raises(tq.TQError):
                tq.tq_search(ctx, qd, code, 3, kc, bt, num_pages, n_db, k_top, out_s, out_i, ws, ws_n)
    finally:
        tq.tq_destroy(ctx)


@pytest.mark.parametrize("k,bad_pages", [(8, (0, 2)), (40, (0, 2)), (16, (0, 1, 2))])
def test_search_bad_pages_and_too_few_finite_scores(k, bad_pages):
    """Out-of-range page ids in a 50-vector database: their vectors score -inf and the device error word is
    set.  When fewer than k scores are finite (k = 40 with 18 finite on the CUDA-core path, k = 16 with 2
    finite on the tensor-core path) the rest of the answer is the -inf vectors in index order."""
    w = wl.Workload("s", "search", 1, 1, 1, 0, k_bits=(3, 3), seed=8)
    p, X, row, num_pages, cache = _database(w, 50, 6)
    row = row.copy()
    for j, pg in enumerate(bad_pages):
        row[pg] = num_pages + 1 + j if j % 2 == 0 else -3
    Q = wl.bf16_round(np.random.default_rng(7).standard_normal((3, 128)).astype(np.float32))
    ctx = ctx_for(w)
    try:
        ts, ti, scores = _search(ctx, Q, "bf16", row, num_pages, cache, 50, k)
        assert tq.tq_check_device_status(ctx) & 1
    finally:
        tq.tq_destroy(ctx)
    bad = np.concatenate([np.arange(16 * pg, 16 * pg + 16) for pg in bad_pages])
    finite = 50 - bad.size
    assert np.all(np.isneginf(scores[:, bad])) and np.all(np.isfinite(np.delete(scores, bad, axis=1)))
    assert np.array_equal(ti, np.argsort(-scores, axis=1, kind="stable")[:, :k])
    assert np.array_equal(ts, np.take_along_axis(scores, ti, axis=1))
    if k > finite:
        assert np.array_equal(ti[:, finite:], np.tile(bad[:k - finite], (3, 1)))


def test_query_count_beyond_the_grid_is_rejected_before_launch():
    """nq above 65535 x 8 queries returns TQ_ERR_UNSUPPORTED before anything runs (the pointers are never read)."""
    ctx = ctx_for(wl.WORKLOADS["c2"])
    try:
        st = tq.raw_status("tq_search", ctx, 256, tq.TQ_BF16, 65535 * 8 + 1, 256, 256, 1, 16, 1, 256, 256, 256,
                           1 << 40, None)
        assert st == tq.TQ_ERR_UNSUPPORTED
        st = tq.raw_status("tq_search", ctx, 256, tq.TQ_BF16, 65535 * 8, 256, 256, 1, 16, 1, 256, 256, 256, 0, None)
        assert st == tq.TQ_ERR_WORKSPACE          # at the limit: the next check (workspace) answers
    finally:
        tq.tq_destroy(ctx)
