"""Pins for the oracle's rotation, quantizer, QJL estimator, packing and attention."""

import math
import os

import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import turboquant as tq

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
D = 128


@pytest.fixture(scope="module")
def p3():
    return oracle.make_params(d=D, m=128, k_bits=(3, 3), v_bits=(3, 3), seed=0)


# --- rotation ---------------------------------------------------------------

@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_rotation_is_orthogonal(d):
    Pi = oracle.rotation_matrix(d, 0)
    assert Pi.shape == (d, d)
    assert np.max(np.abs(Pi.T @ Pi - np.eye(d))) < 1e-12
    assert np.max(np.abs(Pi @ Pi.T - np.eye(d))) < 1e-12


@pytest.mark.parametrize("d", [32, 128, 256])
def test_rotation_is_the_positive_diagonal_qr_factor(d):
    Pi = oracle.rotation_matrix(d, 0)
    g = oracle.gaussian_stream(0, 1, d * d).reshape(d, d)
    R = Pi.T @ g
    assert np.max(np.abs(np.tril(R, -1))) < 1e-11
    assert np.all(np.diag(R) > 0)
    assert np.allclose(Pi[:, 0], g[:, 0] / np.linalg.norm(g[:, 0]), atol=1e-14)


def test_rotation_spreads_coordinates_like_the_sphere():
    """Over seeds, coordinates of Pi e_1 have std 1/sqrt(d) and kurtosis 3d/(d+2)."""
    d = 32
    vals = np.concatenate([oracle.rotation_matrix(d, s)[:, 0] for s in range(400)])
    assert abs(vals.std() * math.sqrt(d) - 1.0) < 0.03
    kurt = stats.kurtosis(vals, fisher=False)
    assert abs(kurt - 3.0 * d / (d + 2)) < 0.12
    # heavy outlier channels are flattened: kurtosis of a spiky vector before/after rotation
    x = np.zeros(128)
    x[:4] = 10.0
    x[4:] = np.random.default_rng(0).standard_normal(124)
    y = oracle.rotation_matrix(128, 1) @ x
    assert stats.kurtosis(x, fisher=False) > 10 and stats.kurtosis(y, fisher=False) < 4.5


# --- quantizer --------------------------------------------------------------

def _unit_vectors(n, d, seed):
    x = np.random.default_rng(seed).standard_normal((n, d))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


@pytest.mark.parametrize("d,n,closed_6dp", [(64, 100000, 0.639111), (128, 100000, 0.637864), (256, 50000, 0.637242)])
def test_two_over_pi_shrinkage_one_bit(d, n, closed_6dp):
    """MSE-only 1-bit: E<q, x^>/<q, x> = sqrt(d) sqrt(2/pi) Gamma(d/2) / (sqrt(pi) Gamma((d+1)/2)), which falls
    to 2/pi = 0.63662 as d grows."""
    p = oracle.make_params(d=d, k_bits=(1, 1), v_bits=(1, 1), seed=3, k_qjl=False)
    closed = math.sqrt(d) * math.sqrt(2 / math.pi) * math.exp(
        math.lgamma(d / 2) - math.lgamma((d + 1) / 2)) / math.sqrt(math.pi)
    assert abs(closed - closed_6dp) < 1e-6 and 2 / math.pi < closed < 2 / math.pi * (1 + 1 / d)
    X = _unit_vectors(n, d, 5)
    q = oracle.quantize_vectors(p, X, "v")
    Xhat = tq.dequantize_values(p, {"codes": q["codes"], "n16": np.linalg.norm(X, axis=1)}) @ p.Pi
    ratio = np.sum(X * Xhat, axis=1)          # <x, x^> / ||x||^2 with ||x|| = 1
    se = ratio.std() / math.sqrt(ratio.size)
    assert abs(ratio.mean() - closed) < 4 * se + 1e-12
    # and with a general query: E<q, x^> = closed * <q, x> (linear in q)
    qv = np.random.default_rng(6).standard_normal(d)
    num = Xhat @ qv
    den = X @ qv
    slope = np.sum(num * den) / np.sum(den * den)
    assert abs(slope - closed) < 0.01


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("d", [128, 256])
def test_distortion_per_bit(bits, d):
    """||x - x^||^2 / ||x||^2 on random unit vectors tracks the Gaussian Lloyd-Max MSE."""
    p = oracle.make_params(d=d, k_bits=(bits, bits), v_bits=(bits, bits), seed=2, k_qjl=False)
    X = _unit_vectors(4000, d, bits)
    q = oracle.quantize_vectors(p, X, "v")
    Yhat = tq.dequantize_values(p, {"codes": q["codes"], "n16": np.ones(len(X))})
    err = np.sum((q["y"] - Yhat) ** 2, axis=1).mean()
    gauss = p.books[bits].mse()
    assert abs(err / gauss - 1.0) < 0.03
    assert 4.0 ** -bits <= err <= math.sqrt(3) * math.pi / 2 * 4.0 ** -bits


# The 3-bit Gaussian Lloyd-Max boundaries (Max 1960, tests/golden/max1960_gaussian.txt), to 4 decimals:
# 0, +-0.5006, +-1.0500, +-1.7480.  Codes below are counted by hand from those values.
def test_codes_on_between_and_just_below_boundaries(p3):
    """code = #{k : u >= t_k}: on a boundary -> the upper cell, one ulp below -> the lower cell."""
    t = p3.books[3].boundaries
    assert np.allclose(t, [-1.7480, -1.0500, -0.5006, 0.0, 0.5006, 1.0500, 1.7480], atol=1e-4)
    on = oracle.assign_codes(t, t)
    below = oracle.assign_codes(np.nextafter(t, -np.inf), t)
    above = oracle.assign_codes(np.nextafter(t, np.inf), t)
    assert on.tolist() == [1, 2, 3, 4, 5, 6, 7]
    assert below.tolist() == [0, 1, 2, 3, 4, 5, 6]
    assert above.tolist() == [1, 2, 3, 4, 5, 6, 7]
    between = [-9.0, -2.0, -1.5, -0.8, -0.3, 0.3, 0.8, 1.5, 2.0, 9.0, -0.0]
    assert oracle.assign_codes(between, t).tolist() == [0, 0, 1, 2, 3, 4, 5, 6, 7, 7, 4]
    # 1 bit: the single boundary 0 -> negative 0, non-negative 1; 2 bits: 0, +-0.9816 (Max 1960)
    t1, t2 = p3.books.get(1) or oracle.lloyd_max_gaussian(1), oracle.lloyd_max_gaussian(2)
    assert oracle.assign_codes([-1e-300, 0.0, 1e-300], t1.boundaries).tolist() == [0, 1, 1]
    assert oracle.assign_codes([-1.0, -0.9, -1e-9, 0.0, 0.9, 1.0], t2.boundaries).tolist() == [0, 1, 1, 2, 2, 3]


def test_quantize_assigns_exact_u_end_to_end():
    """Identity rotation, d = 64, x with sixteen entries +-2 and the rest 0: ||x|| = 8 and u = sqrt(64) x / 8 = x
    exactly, so the codes through quantize_vectors are known by hand (3 bits: u = -2 -> 0, u = 0 -> 4 (tie up),
    u = 2 -> 7); keys: n16 = 8 and r~ = y - c[code] exactly representable."""
    import dataclasses
    p = oracle.make_params(d=64, m=32, k_bits=(3, 3), k_split=32, v_bits=(3, 3), v_split=32, seed=0)
    p = dataclasses.replace(p, Pi=np.eye(64))
    x = np.zeros(64)
    x[:8] = 2.0
    x[8:16] = -2.0
    q = oracle.quantize_vectors(p, x[None, :], "k")
    assert q["norm"][0] == 8.0 and q["n16"][0] == 8.0
    assert np.array_equal(q["u"][0], x)
    assert q["codes"][0].tolist() == [7] * 8 + [0] * 8 + [4] * 48
    c = p.books[3].centroids
    want_r = x - np.array([c[7]] * 8 + [c[0]] * 8 + [c[4]] * 48)     # y - (n16/sqrt(d)) c[code] with y = x, n16/sqrt(d) = 1
    assert np.array_equal(q["r"][0], want_r)


def test_quantize_exclusions_by_hand():
    """Codes within eps = 1e-6 of a boundary and signs with |z| < eps rho are excluded; one excluded code
    excludes every sign bit of its vector."""
    p = oracle.make_params(d=D, m=128, k_bits=(3, 3), v_bits=(3, 3), seed=0)
    t = p.books[3].boundaries
    U = np.full((3, D), 0.25)                   # 0.25: more than 0.25 from every 3-bit boundary
    U[0, 5] = t[4] + 5e-7                        # inside the band
    U[0, 70] = t[1] - 9.9e-7                     # inside
    U[1, 9] = t[6] + 2e-6                        # outside
    U[1, 100] = t[3] - 1.01e-6                   # outside (boundary 0)
    rho = np.array([2.0, 4.0, 1.0])
    Z = np.full((3, 128), 0.5)
    Z[1, 3] = 3.9e-6                             # |z| < 1e-6 * 4
    Z[1, 77] = -4.1e-6                           # not
    Z[2, 0] = -0.0                               # |z| = 0 < 1e-6
    Z[2, 127] = 1.1e-6                           # not (rho = 1)
    ex = oracle.quantize_exclusions(p, {"u": U, "z": Z, "rho": rho}, "k")
    want_codes = np.zeros((3, D), dtype=bool)
    want_codes[0, [5, 70]] = True
    assert np.array_equal(ex["codes"], want_codes)
    want_signs = np.zeros((3, 128), dtype=bool)
    want_signs[0, :] = True                      # vector 0 has excluded codes
    want_signs[1, 3] = True
    want_signs[2, 0] = True
    assert np.array_equal(ex["signs"], want_signs)
    ex_v = oracle.quantize_exclusions(p, {"u": U}, "v")
    assert "signs" not in ex_v and np.array_equal(ex_v["codes"], want_codes)


def test_zero_vector(p3):
    q = oracle.quantize_vectors(p3, np.zeros((1, D)), "k")
    assert np.all(q["codes"] == 4)                      # u = 0 sits on the middle boundary -> upper
    assert q["n16"][0] == 0 and q["rho16"][0] == 0
    assert np.all(q["signs"] == 1)                      # S * 0 = 0 -> sign bit set


@pytest.mark.parametrize("d,m", [(128, 128), (256, 96)])
def test_two_stage_estimator_is_unbiased(d, m):
    """Mean over many Gaussian projections of the stage-2 estimate equals <q, x> exactly."""
    rng = np.random.default_rng(11)
    p = oracle.make_params(d=d, m=m, k_bits=(2, 2), k_split=d // 2, v_bits=(2, 2), v_split=d // 2, seed=4)
    x = rng.standard_normal(d)
    x[:4] *= 10
    qv = rng.standard_normal(d)
    q = oracle.quantize_vectors(p, x[None, :], "k")
    r = q["r"][0]
    rho = float(np.linalg.norm(r))
    qt = p.Pi @ qv
    exact = float(qv @ x)
    n_draws = 2000
    est = np.empty(n_draws)
    mse_only = None
    for i in range(n_draws):
        S = rng.standard_normal((p.m, d))
        pp = tq.TQParams(**{**p.__dict__, "S": S})
        z = S @ r
        rec = {"codes": q["codes"], "n16": q["n16"], "signs": (z >= 0).astype(np.uint8)[None, :],
               "rho16": np.array([rho])}
        est[i] = tq.estimate_scores(pp, qt, S @ qt, rec)[0]
        if mse_only is None:
            pq = tq.TQParams(**{**p.__dict__, "k_qjl": False})
            mse_only = tq.estimate_scores(pq, qt, None, rec)[0]
    var = ((math.pi / 2) * (qt @ qt) * rho ** 2 - (qt @ r) ** 2) / p.m
    z = (est.mean() - exact) / math.sqrt(var / n_draws)
    assert abs(z) < 4.5
    assert abs(est.var() / var - 1) < 0.15
    # stage 1 alone misses exactly the residual term <qt, r>
    assert abs(mse_only + qt @ r - exact) < 1e-9


# --- packing and the paged cache -------------------------------------------

def _golden_bytes(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [int(t, 16) for ln in f if not ln.startswith("#") for t in ln.split()]


def test_pack_hand_example_3bit():
    p = oracle.make_params(d=D, k_bits=(3, 3), v_bits=(3, 3), seed=0)
    codes = np.zeros((1, D), dtype=np.int64)
    codes[0, :8] = np.arange(8)
    raw = tq._pack_codes(p, codes, "v")
    assert raw[0, :3].tolist() == _golden_bytes("pack_b3_codes_0to7.txt") and raw.shape == (1, 48)


def test_pack_hand_example_4bit():
    p = oracle.make_params(d=D, k_bits=(4, 4), v_bits=(4, 4), seed=0)
    codes = np.full((1, D), 8, dtype=np.int64)
    codes[0, :4] = [0, 7, 8, 15]
    raw = tq._pack_codes(p, codes, "v")
    assert raw[0, :2].tolist() == _golden_bytes("pack_b4_sign_magnitude.txt") and raw.shape == (1, 64)


def _format_integer(codes, bits_per_channel):
    """The code area as one integer, from the format's definition written group by group."""
    acc, base = 0, 0
    groups = []
    j = 0
    while j < len(codes):           # consecutive channels of equal width form a group
        b = int(bits_per_channel[j])
        k = j
        while k < len(codes) and int(bits_per_channel[k]) == b:
            k += 1
        groups.append((b, [int(c) for c in codes[j:k]]))
        j = k
    for b, cs in groups:
        if b == 3:
            for o in range(0, len(cs), 8):
                c = cs[o:o + 8]
                octet = sum(c[i] << (4 * i) for i in range(6))
                for q in range(3):
                    octet |= ((c[6] >> q) & 1) << (8 * q + 3)
                    octet |= ((c[7] >> q) & 1) << (8 * q + 7)
                acc |= octet << (base + 3 * o)
        elif b == 4:
            for i, c in enumerate(cs):
                acc |= ((c - 8) if c >= 8 else (15 - c)) << (base + 4 * i)
        else:
            for i, c in enumerate(cs):
                acc |= c << (base + b * i)
        base += b * len(cs)
    return acc, base


@pytest.mark.parametrize("kb,vb", [((3, 3), (3, 3)), ((4, 3), (4, 3)), ((3, 2), (3, 2)), ((1, 1), (2, 4)),
                                   ((4, 4), (2, 2))])
def test_pack_matches_format_definition(kb, vb):
    p = oracle.make_params(d=D, k_bits=kb, v_bits=vb, seed=0)
    rng = np.random.default_rng(1)
    for kind in ("k", "v"):
        cb = p.channel_bits(kind)
        codes = np.stack([rng.integers(0, 1 << int(b), size=5) for b in cb], axis=1)
        raw = tq._pack_codes(p, codes, kind)
        for row in range(5):
            acc, nbits = _format_integer(codes[row], cb)
            assert bytes(raw[row]) == acc.to_bytes(nbits // 8, "little")
        assert np.array_equal(tq._unpack_codes(p, raw, kind), codes)


def test_sign_bit_order(p3):
    signs = np.zeros((1, 128), dtype=np.uint8)
    signs[0, [0, 9, 127]] = 1
    rec = oracle.pack_k_records(p3, {"codes": np.zeros((1, D), dtype=np.int64), "n16": np.ones(1),
                                     "signs": signs, "rho16": np.ones(1)})
    w = rec["signs"][0].view("<u4")
    assert w.tolist() == [1 | (1 << 9), 0, 0, 1 << 31]


@pytest.mark.parametrize("kb,vb,kbytes,vbytes", [((3, 3), (3, 3), 1088, 800), ((4, 3), (4, 3), 1216, 928),
                                                  ((3, 2), (3, 2), 960, 672)])
def test_block_sizes(kb, vb, kbytes, vbytes):
    """Per token-head: 3-bit 68+50 B, 3.5-bit 76+58 B, 2.5-bit 60+42 B; 16 slots per block."""
    p = oracle.make_params(d=D, k_bits=kb, v_bits=vb, seed=0)
    assert oracle.cache_block_bytes(p, "k") == kbytes and oracle.cache_block_bytes(p, "v") == vbytes


def test_paged_roundtrip_through_permuted_block_table(p3):
    rng = np.random.default_rng(2)
    B, H, T = 3, 2, 37
    maxp = 4
    perm = rng.permutation(B * maxp)
    bt = perm.reshape(B, maxp).astype(np.int32)
    X = rng.standard_normal((B, T, H, D))
    q = oracle.quantize_vectors(p3, X.reshape(-1, D), "k")
    rec = oracle.pack_k_records(p3, q)
    bb = oracle.cache_block_bytes(p3, "k")
    cache = np.zeros(B * maxp * H * bb, dtype=np.uint8)
    bi, ti, hi = np.meshgrid(np.arange(B), np.arange(T), np.arange(H), indexing="ij")
    pages = bt[bi.ravel(), ti.ravel() // 16]
    slots = ti.ravel() % 16
    oracle.write_paged(p3, "k", cache, rec, pages, slots, hi.ravel(), H)
    back = oracle.read_paged(p3, "k", cache, pages, slots, hi.ravel(), H)
    for k in rec:
        assert np.array_equal(np.asarray(back[k]).view(np.uint8), np.asarray(rec[k]).view(np.uint8))
    # the byte address of one field follows the block layout by hand
    b, t, h = 2, 21, 1
    page = bt[b, t // 16]
    off = page * H * bb + h * bb + 16 * 48 + 16 * 16 + (t % 16) * 2
    n16 = np.frombuffer(cache[off:off + 2].tobytes(), dtype=np.float16)[0]
    assert n16 == np.float16(q["n16"][(b * T + t) * H + h])


# --- attention ----------------------------------------------------------------

def _records(p, K, V):
    return (oracle.unpack_k_records(p, oracle.pack_k_records(p, oracle.quantize_vectors(p, K, "k"))),
            oracle.unpack_v_records(p, oracle.pack_v_records(p, oracle.quantize_vectors(p, V, "v"))))


def test_attention_single_token_returns_dequantized_value(p3):
    rng = np.random.default_rng(3)
    K, V, qv = rng.standard_normal((1, D)), rng.standard_normal((1, D)), rng.standard_normal(D)
    kr, vr = _records(p3, K, V)
    o = tq.attend_one(p3, qv, kr, vr, 1 / math.sqrt(D))
    vq = oracle.quantize_vectors(p3, V, "v")
    want = p3.Pi.T @ (vq["n16"][0] / math.sqrt(D) * p3.books[3].centroids[vq["codes"][0]])
    assert np.allclose(o, want, atol=1e-14)


def test_attention_identical_keys_average_values(p3):
    rng = np.random.default_rng(4)
    K = np.repeat(rng.standard_normal((1, D)), 17, axis=0)
    V = rng.standard_normal((17, D))
    kr, vr = _records(p3, K, V)
    o = tq.attend_one(p3, rng.standard_normal(D), kr, vr, 1 / math.sqrt(D))
    want = p3.Pi.T @ tq.dequantize_values(p3, vr).mean(axis=0)
    assert np.allclose(o, want, atol=1e-13)


def test_attention_token_order_does_not_matter(p3):
    rng = np.random.default_rng(5)
    K, V, qv = rng.standard_normal((17, D)), rng.standard_normal((17, D)), rng.standard_normal(D)
    kr, vr = _records(p3, K, V)
    perm = rng.permutation(17)
    o1 = tq.attend_one(p3, qv, kr, vr, 0.1)
    o2 = tq.attend_one(p3, qv, {k: v[perm] for k, v in kr.items()}, {k: v[perm] for k, v in vr.items()}, 0.1)
    assert np.allclose(o1, o2, atol=1e-13)


@pytest.mark.parametrize("qjl", [False, True])
@pytest.mark.parametrize("n", [2, 3, 17, 64])
def test_attention_approaches_exact_attention_with_more_bits(n, qjl):
    """The quantized path converges to textbook fp64 attention as bits grow.

    At 8 bits the per-coordinate error is about sqrt(2.7 * 4**-8) ~ 6e-3 of the
    coordinate scale, so the output must agree to ~1% RMS; each extra pair of bits
    must shrink the error, and 1-bit codes must be visibly worse.
    """
    rng = np.random.default_rng(n)
    K, V, qv = rng.standard_normal((n, D)), rng.standard_normal((n, D)), rng.standard_normal(D)
    ref = oracle.exact_attention(qv, K, V, 1 / math.sqrt(D))
    errs = {}
    for bits in (1, 2, 4, 8):
        p = oracle.make_params(d=D, m=128, k_bits=(bits, bits), v_bits=(bits, bits), seed=6, k_qjl=qjl)
        kr, vr = _records(p, K, V)
        o = tq.attend_one(p, qv, kr, vr, 1 / math.sqrt(D))
        errs[bits] = np.linalg.norm(o - ref) / np.linalg.norm(ref)
    assert errs[8] < 1.5e-2
    assert errs[8] < errs[4] < errs[2]
    assert errs[1] > 0.1


def test_decode_attention_gqa_and_paging(p3):
    rng = np.random.default_rng(7)
    B, Hq, Hk, maxp = 2, 4, 2, 3
    lens = np.array([37, 5])
    bt = rng.permutation(B * maxp).reshape(B, maxp).astype(np.int32)
    kbb, vbb = oracle.cache_block_bytes(p3, "k"), oracle.cache_block_bytes(p3, "v")
    kc = np.zeros(B * maxp * Hk * kbb, np.uint8)
    vc = np.zeros(B * maxp * Hk * vbb, np.uint8)
    Ks, Vs = {}, {}
    for b in range(B):
        for h in range(Hk):
            K = rng.standard_normal((lens[b], D))
            V = rng.standard_normal((lens[b], D))
            Ks[b, h], Vs[b, h] = K, V
            pages, slots = tq.token_locations(bt, b, np.arange(lens[b]))
            heads = np.full(lens[b], h)
            oracle.write_paged(p3, "k", kc, oracle.pack_k_records(p3, oracle.quantize_vectors(p3, K, "k")), pages, slots, heads, Hk)
            oracle.write_paged(p3, "v", vc, oracle.pack_v_records(p3, oracle.quantize_vectors(p3, V, "v")), pages, slots, heads, Hk)
    Q = rng.standard_normal((B, Hq, D))
    out = oracle.decode_attention(p3, Q, lens, bt, kc, vc, Hk)
    for b in range(B):
        for h in range(Hq):
            kr, vr = _records(p3, Ks[b, h // 2], Vs[b, h // 2])
            assert np.allclose(out[b, h], tq.attend_one(p3, Q[b, h], kr, vr, 1 / math.sqrt(D)), atol=1e-13)


# ---------------------------------------------------------------------------
# inner-product search (the vector-search use of the same estimate)
# ---------------------------------------------------------------------------

def _search_db(p, X, perm=None):
    n = X.shape[0]
    npg = (n + 15) // 16
    row = np.arange(npg) if perm is None else np.asarray(perm)[:npg]
    cache = np.zeros((int(row.max()) + 1) * oracle.cache_block_bytes(p, "k"), dtype=np.uint8)
    q = oracle.quantize_vectors(p, X, "k")
    pages, slots = row[np.arange(n) // 16], np.arange(n) % 16
    oracle.write_paged(p, "k", cache, oracle.pack_k_records(p, q), pages, slots, np.zeros(n, dtype=np.int64), 1)
    return row, cache


def test_search_ranks_scaled_copies_first():
    """A database holding 4x each query among random vectors: the estimate <q, 4q> = 4||q||^2 dwarfs every
    other score, so each query's best hit is its own copy."""
    p = oracle.make_params(k_bits=(3, 3), seed=3)
    rng = np.random.default_rng(5)
    Q = rng.standard_normal((6, 128))
    X = rng.standard_normal((300, 128))
    where = rng.choice(300, 6, replace=False)
    X[where] = 4.0 * Q
    row, cache = _search_db(p, X)
    scores, top, vals = oracle.search(p, Q, row, cache, 300, 3)
    assert np.array_equal(top[:, 0], where)
    assert np.all(np.diff(vals, axis=1) <= 0)
    # the estimate of <q, 4q> is within the quantization error of the exact value
    exact = 4.0 * np.sum(Q * Q, axis=1)
    assert np.all(np.abs(vals[:, 0] - exact) < 0.1 * exact)


def test_search_ties_by_index_and_block_table_indirection():
    """Duplicate vectors have equal estimates and rank by lower index; a permuted block table reads back
    the same database."""
    p = oracle.make_params(k_bits=(4, 3), seed=2)
    rng = np.random.default_rng(8)
    X = rng.standard_normal((100, 128))
    X[[10, 40, 70]] = 3.0 * X[5]
    Q = X[5:6] / np.linalg.norm(X[5])
    row, cache = _search_db(p, X)
    s1, top, _ = oracle.search(p, Q, row, cache, 100, 4)
    assert list(top[0, :3]) == [10, 40, 70] and s1[0, 10] == s1[0, 40] == s1[0, 70]
    perm = np.random.default_rng(9).permutation(20)
    row2, cache2 = _search_db(p, X, perm)
    s2, top2, _ = oracle.search(p, Q, row2, cache2, 100, 4)
    assert np.array_equal(s1, s2) and np.array_equal(top, top2)


# ---------------------------------------------------------------------------
# multi-query causal attention over the compressed cache (many new tokens)
# ---------------------------------------------------------------------------

def _causal_setup(p, K, V, perm=None):
    """K, V [B, L, H, d] written through a block table (identity or permuted pages)."""
    B, L, H, _ = K.shape
    pps = (L + 15) // 16
    npages = B * pps
    order = np.arange(npages) if perm is None else np.asarray(perm)
    bt = order.reshape(B, pps)
    kc = np.zeros(npages * H * oracle.cache_block_bytes(p, "k"), dtype=np.uint8)
    vc = np.zeros(npages * H * oracle.cache_block_bytes(p, "v"), dtype=np.uint8)
    for b in range(B):
        pos = np.repeat(np.arange(L), H)
        heads = np.tile(np.arange(H), L)
        pages, slots = bt[b, pos // 16].astype(np.int64), pos % 16
        for kind, X, cache in (("k", K, kc), ("v", V, vc)):
            q = oracle.quantize_vectors(p, X[b].reshape(-1, 128), kind)
            rec = oracle.pack_k_records(p, q) if kind == "k" else oracle.pack_v_records(p, q)
            oracle.write_paged(p, kind, cache, rec, pages, slots, heads, H)
    return bt, kc, vc


def test_causal_attention_masks_the_future():
    """A query at position s+t sees positions <= s+t only: changing a later key or value leaves it unchanged,
    changing an earlier one does not; a permuted block table reads back the same result."""
    p = oracle.make_params(k_bits=(3, 3), v_bits=(3, 3), seed=1)
    rng = np.random.default_rng(12)
    B, L, H, Hq, T = 2, 40, 2, 4, 6
    K, V = rng.standard_normal((B, L, H, 128)), rng.standard_normal((B, L, H, 128))
    start = np.array([30, 34])                       # new tokens at start .. start + T - 1 (< L)
    Q = rng.standard_normal((B, T, Hq, 128))
    bt, kc, vc = _causal_setup(p, K, V)
    base = oracle.causal_attention(p, Q, start, bt, kc, vc, H)
    K2, V2 = K.copy(), V.copy()
    K2[0, 33] += 5.0                                 # position 33 of sequence 0: seen by t >= 3 only
    V2[0, 33] -= 5.0
    bt2, kc2, vc2 = _causal_setup(p, K2, V2)
    other = oracle.causal_attention(p, Q, start, bt2, kc2, vc2, H)
    assert np.array_equal(other[0, :3], base[0, :3]) and np.array_equal(other[1], base[1])
    assert np.all(np.abs(other[0, 3:] - base[0, 3:]).max(axis=-1) > 1e-6)
    perm = np.random.default_rng(3).permutation(B * ((L + 15) // 16))
    bt3, kc3, vc3 = _causal_setup(p, K, V, perm)
    assert np.array_equal(oracle.causal_attention(p, Q, start, bt3, kc3, vc3, H), base)


def test_causal_attention_approaches_exact_at_four_bits():
    """Against textbook causal softmax attention over the unquantized keys and values (each query against its
    own prefix), the error of the compressed result about halves per bit (the reconstruction error of a
    Lloyd-Max code falls about 2x per bit in norm); measured 0.79 / 0.40 / 0.20 at 2 / 3 / 4 bits here, where
    averaging over 64 random values makes the exact output small."""
    rng = np.random.default_rng(13)
    B, L, H, Hq, T = 1, 64, 1, 2, 4
    K, V = rng.standard_normal((B, L, H, 128)), rng.standard_normal((B, L, H, 128))
    start = np.array([L - T])
    Q = rng.standard_normal((B, T, Hq, 128))
    errs = {}
    for bits in (2, 3, 4):
        p = oracle.make_params(k_bits=(bits, bits), v_bits=(bits, bits), seed=2)
        bt, kc, vc = _causal_setup(p, K, V)
        got = oracle.causal_attention(p, Q, start, bt, kc, vc, H)
        e = 0.0
        for t in range(T):
            n = int(start[0]) + t + 1
            for h in range(Hq):
                want = oracle.exact_attention(Q[0, t, h], K[0, :n, 0], V[0, :n, 0], 1.0 / math.sqrt(128))
                e = max(e, np.max(np.abs(got[0, t, h] - want)) / np.max(np.abs(want)))
        errs[bits] = e
    assert errs[2] > errs[3] > errs[4] and errs[4] < 0.25
    assert 1.6 < errs[2] / errs[3] < 2.5 and 1.6 < errs[3] / errs[4] < 2.5
