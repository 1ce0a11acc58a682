"""Plain fp64 restatement of the TurboQuant quantize and decode-attention path.

TEST INFRASTRUCTURE ONLY -- see the package docstring.  The steps follow the
pages' order: random rotation, per-coordinate Lloyd-Max codes, residual, 1-bit
QJL sketch of the residual, then attention with the two-stage inner-product
estimate.  numpy primitives (matmul, QR, searchsorted, packbits, exp) serve as
steps; nothing is blocked, fused or reordered beyond the formulas written here.

Readings where the pages are silent (each listed in the project's design notes):
  * codebook density: N(0,1) in unit-variance units, u = sqrt(d) * y / ||x||
    ([P4] §4.2 says the rotated coordinate is Beta-distributed, close to
    Gaussian at high d); Lloyd iteration on the positive half, mirrored.
  * codes are 0-based and ascending; a value equal to a boundary rounds up.
  * QJL acts in the rotated domain: signs of S * r~ with r~ = y - y^ and the
    query side uses S * (Pi q); the estimator constant sqrt(pi/2)/m.
  * the stage-1 reconstruction, and so the residual, use the stored fp16 norm;
    codes use the exact norm.  sign(0) counts as +1 (bit set).
  * a zero vector has u = 0 (codes land on the upper side of the 0 boundary).
"""

import math
from dataclasses import dataclass, field

import numpy as np
from scipy import special

from .rng import gaussian_stream

PAGE = 16  # tokens per cache page (block table granularity, [P4] §3.1)


# ---------------------------------------------------------------------------
# Stage 1 ingredients: rotation and codebook
# ---------------------------------------------------------------------------

def rotation_matrix(d, seed):
    """Pi: Haar-random orthogonal d x d ([P4] §4.1 "random orthogonal matrix R").

    G (d x d, stream 1, row-major) -> G = QR (Householder, numpy/LAPACK) ->
    Pi = Q diag(sign R_ii), the unique QR factor with a positive R diagonal.
    """
    g = gaussian_stream(seed, 1, d * d).reshape(d, d)
    q, r = np.linalg.qr(g)
    s = np.sign(np.diag(r))
    s[s == 0] = 1.0
    return q * s[None, :]


def qjl_matrix(m, d, seed):
    """S: m x d with i.i.d. N(0,1) entries (stream 2, row-major), [P4] §4.3."""
    return gaussian_stream(seed, 2, m * d).reshape(m, d)


def _phi(t):
    return math.exp(-0.5 * t * t) / math.sqrt(2.0 * math.pi)


def _upper_tail(t):
    """Q(t) = P(Z > t) for Z ~ N(0,1)."""
    return 0.5 * math.erfc(t / math.sqrt(2.0))


@dataclass
class Codebook:
    bits: int
    centroids: np.ndarray      # 2**b ascending
    boundaries: np.ndarray     # 2**b - 1 ascending, boundary k between centroid k and k+1
    iterations: int = 0

    def mse(self):
        """Per-coordinate distortion E[(Z - Q(Z))^2] for Z ~ N(0,1).

        Per cell (a, b): P0 = P(a<Z<b), M1 = phi(a) - phi(b),
        M2 = P0 + a phi(a) - b phi(b); the cell contributes M2 - 2c M1 + c^2 P0.
        """
        t = [-math.inf] + list(self.boundaries) + [math.inf]
        total = 0.0
        for k, c in enumerate(self.centroids):
            a, b = t[k], t[k + 1]
            p0 = _tail_or(a, 1.0) - _tail_or(b, 0.0)
            m1 = _phi_or0(a) - _phi_or0(b)
            m2 = p0 + _tphi_or0(a) - _tphi_or0(b)
            total += m2 - 2.0 * c * m1 + c * c * p0
        return total


def _tail_or(t, at_minus_inf):
    if t == math.inf:
        return 0.0
    if t == -math.inf:
        return at_minus_inf
    return _upper_tail(t)


def _phi_or0(t):
    return 0.0 if math.isinf(t) else _phi(t)


def _tphi_or0(t):
    return 0.0 if math.isinf(t) else t * _phi(t)


def lloyd_max_gaussian(bits, tol=1e-15, max_iter=200000):
    """Lloyd-Max 2**b-level quantizer for N(0,1) ([P4] §4.2).

    Lloyd's two conditions, iterated: each boundary is the midpoint of its two
    centroids, each centroid is the conditional mean of its cell,
    E[Z | a < Z < b] = (phi(a) - phi(b)) / (Phi(b) - Phi(a)).  The density is
    symmetric, so the iteration runs on the positive half (cells [t_k, t_{k+1})
    with t_0 = 0) and the result is mirrored; the middle boundary is exactly 0.
    """
    if bits < 1:
        raise ValueError("bits >= 1")
    key = (bits, tol, max_iter)
    if key in _BOOKS:
        return _BOOKS[key]
    h = 1 << (bits - 1)
    a = (np.arange(h) + 0.5) * 3.0 / h   # any increasing start
    it = 0
    for it in range(1, max_iter + 1):
        lo = np.concatenate([[0.0], 0.5 * (a[:-1] + a[1:])])    # cell k = [lo_k, hi_k)
        hi = np.concatenate([lo[1:], [np.inf]])
        phi_hi = np.where(np.isinf(hi), 0.0, np.exp(-0.5 * np.where(np.isinf(hi), 0.0, hi) ** 2))
        num = (np.exp(-0.5 * lo ** 2) - phi_hi) / math.sqrt(2.0 * math.pi)
        den = 0.5 * (special.erfc(lo / math.sqrt(2.0)) - special.erfc(hi / math.sqrt(2.0)))
        new = num / den
        delta = np.max(np.abs(new - a))
        a = new
        if delta <= tol:
            break
    pos_t = 0.5 * (a[:-1] + a[1:])
    centroids = np.concatenate([-a[::-1], a])
    boundaries = np.concatenate([-pos_t[::-1], [0.0], pos_t])
    _BOOKS[key] = Codebook(bits, centroids, boundaries, it)
    return _BOOKS[key]


_BOOKS = {}


def lloyd_max_sphere(bits, d, tol=1e-15, max_iter=200000):
    """Lloyd-Max 2**b-level quantizer for the exact density of one coordinate of
    a randomly rotated vector in unit-variance units ([P4] §4.2: the rotated
    coordinate follows a Beta distribution, close to N(0,1) at high d).

    u = sqrt(d) z with z a coordinate of a uniform point on the unit sphere of
    R^d, so z^2 ~ Beta(1/2, (d-1)/2).  For u >= 0:
      P(U >= u)   = I_{1 - u^2/d}((d-1)/2, 1/2) / 2   (regularized incomplete beta),
      E[U; U >= u] = sqrt(d) Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2) (d-1)) (1 - u^2/d)^((d-1)/2).
    The same two Lloyd conditions and positive-half iteration as
    lloyd_max_gaussian; the last cell ends at sqrt(d).
    """
    if bits < 1 or d < 4:
        raise ValueError("bits >= 1, d >= 4")
    key = ("sphere", bits, d, tol, max_iter)
    if key in _BOOKS:
        return _BOOKS[key]
    rd = math.sqrt(d)
    cmom = rd * math.exp(special.gammaln(d / 2.0) - special.gammaln((d - 1) / 2.0)) / math.sqrt(math.pi) / (d - 1)

    def tail(u):
        z2 = np.minimum(u / rd, 1.0) ** 2
        return 0.5 * special.betainc((d - 1) / 2.0, 0.5, 1.0 - z2)

    def moment(u):
        z2 = np.minimum(u / rd, 1.0) ** 2
        return cmom * (1.0 - z2) ** ((d - 1) / 2.0)

    h = 1 << (bits - 1)
    a = (np.arange(h) + 0.5) * min(3.0, rd) / h     # every starting cell inside the support (0, sqrt(d))
    it = 0
    for it in range(1, max_iter + 1):
        lo = np.concatenate([[0.0], 0.5 * (a[:-1] + a[1:])])
        hi = np.concatenate([lo[1:], [rd]])
        new = (moment(lo) - moment(hi)) / (tail(lo) - tail(hi))
        delta = np.max(np.abs(new - a))
        a = new
        if delta <= tol:
            break
    pos_t = 0.5 * (a[:-1] + a[1:])
    centroids = np.concatenate([-a[::-1], a])
    boundaries = np.concatenate([-pos_t[::-1], [0.0], pos_t])
    _BOOKS[key] = Codebook(bits, centroids, boundaries, it)
    return _BOOKS[key]


# ---------------------------------------------------------------------------
# Parameters
# ---------------------------------------------------------------------------

@dataclass
class TQParams:
    d: int
    m: int
    k_bits: tuple          # (bits on channels < k_split, bits on the rest)
    k_split: int
    v_bits: tuple
    v_split: int
    k_qjl: bool
    seed: int
    Pi: np.ndarray = field(repr=False)
    S: np.ndarray = field(repr=False)
    books: dict = field(repr=False)   # bits -> Codebook

    def channel_bits(self, kind):
        bits, split = (self.k_bits, self.k_split) if kind == "k" else (self.v_bits, self.v_split)
        return np.array([bits[0]] * split + [bits[1]] * (self.d - split))

    def code_bits(self, kind):
        return int(self.channel_bits(kind).sum())


def make_params(d=128, m=128, k_bits=(3, 3), k_split=64, v_bits=(3, 3), v_split=64,
                seed=0, k_qjl=True, codebook="gaussian"):
    """Everything the method draws or precomputes once: Pi, S and the codebooks
    (codebook "gaussian": N(0,1) Lloyd-Max; "sphere": the exact rotated-coordinate
    density, lloyd_max_sphere)."""
    Pi = rotation_matrix(d, seed)
    S = qjl_matrix(m, d, seed)
    if codebook == "sphere":
        books = {b: lloyd_max_sphere(b, d) for b in set(k_bits) | set(v_bits)}
    elif codebook == "gaussian":
        books = {b: lloyd_max_gaussian(b) for b in set(k_bits) | set(v_bits)}
    else:
        raise ValueError(codebook)
    return TQParams(d, m, tuple(k_bits), k_split, tuple(v_bits), v_split, bool(k_qjl),
                    int(seed), Pi, S, books)


def _centroid_table(params, kind):
    """Per-channel (centroids, boundaries) lists for the channel's bit-width."""
    cb = params.channel_bits(kind)
    return [params.books[int(b)] for b in cb]


# ---------------------------------------------------------------------------
# Quantize (stage 1 + stage 2)
# ---------------------------------------------------------------------------

def fp16_round(x):
    """Round-to-nearest-even to IEEE half, returned as fp64 values."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def assign_codes(u, boundaries):
    """Code of each unit-variance coordinate u: the number of boundaries t_k with u >= t_k
    ([P4] §4.2: a value falls in the cell between two boundaries; a value exactly on a
    boundary goes to the upper cell)."""
    u = np.asarray(u, dtype=np.float64)
    t = np.asarray(boundaries, dtype=np.float64)
    return np.sum(u[..., None] >= t, axis=-1).astype(np.int64)


def quantize_vectors(params, X, kind):
    """Quantize rows of X (n x d, any float dtype, taken exactly into fp64).

    [P2] stage 1 / [P4] §4.1-§4.2: y = Pi x, u = sqrt(d) y / ||x||,
    code_j = #{k : u_j >= t_k}.  For keys ([P2] stage 2, [P4] §4.3):
    n16 = fp16(||x||), r~ = y - (n16/sqrt(d)) c[code], z = S r~,
    sign_i = [z_i >= 0], rho16 = fp16(||r~||).
    """
    X = np.asarray(X, dtype=np.float64)
    d = params.d
    norm = np.sqrt(np.sum(X * X, axis=1))
    Y = X @ params.Pi.T
    safe = np.where(norm > 0, norm, 1.0)
    U = np.where(norm[:, None] > 0, math.sqrt(d) * Y / safe[:, None], 0.0)
    books = _centroid_table(params, kind)
    codes = np.empty(U.shape, dtype=np.int64)
    chat = np.empty(U.shape)
    for j in range(d):
        bk = books[j]
        codes[:, j] = assign_codes(U[:, j], bk.boundaries)
        chat[:, j] = bk.centroids[codes[:, j]]
    n16 = fp16_round(norm)
    out = {"codes": codes, "norm": norm, "n16": n16, "u": U, "y": Y}
    if kind == "k" and params.k_qjl:
        R = Y - (n16 / math.sqrt(d))[:, None] * chat
        Z = R @ params.S.T
        rho = np.sqrt(np.sum(R * R, axis=1))
        out.update(signs=(Z >= 0).astype(np.uint8), z=Z, rho=rho, rho16=fp16_round(rho), r=R)
    return out


def quantize_exclusions(params, q, kind, eps=1e-6):
    """Positions where finite-precision arithmetic may legitimately disagree.

    A code is excluded when its unit-variance coordinate lies within eps of one
    of its codebook boundaries.  A sign bit is excluded when |z_i| < eps * rho
    (its projection is within eps of the sign boundary in unit-variance units
    of z, whose spread is rho), or when any code of the same vector is
    excluded (the residual depends on all codes).
    """
    books = _centroid_table(params, kind)
    U = q["u"]
    code_ex = np.zeros(U.shape, dtype=bool)
    for j in range(params.d):
        t = books[j].boundaries
        code_ex[:, j] = np.min(np.abs(U[:, j:j + 1] - t[None, :]), axis=1) < eps
    res = {"codes": code_ex}
    if "z" in q:
        sign_ex = np.abs(q["z"]) < eps * q["rho"][:, None]
        sign_ex |= code_ex.any(axis=1)[:, None]
        res["signs"] = sign_ex
    return res


# ---------------------------------------------------------------------------
# Packed records and the paged cache
# ---------------------------------------------------------------------------
# Record format (this project's spec; the pages fix only "b-bit codes, signs,
# norms, 16-token blocks"):
#   codes: one bit stream per vector (byte k holds stream bits 8k..8k+7, least
#          significant first).  Channels [0, split) form the first group
#          (b_hi bits each), channels [split, d) the second (b_lo bits); each
#          group holds its channels' *stored values* in order:
#            b = 1, 2: value of group channel c at group bits [b*c, b*c + b).
#            b = 3:    channels in octets of 8 (24 bits, octet o at group bit
#                      24*o); octet channel i < 6 at octet bits 4i..4i+2,
#                      channel 6 at octet bits 3, 11, 19 and channel 7 at
#                      bits 7, 15, 23 (value bits 0, 1, 2 in that order).
#            b = 4:    value of group channel c at group bits [4c, 4c + 4).
#          The stored value is the code itself for b <= 3; for b = 4 it is
#          sign-magnitude: code >= 8 -> code - 8, code < 8 -> 8 + (7 - code)
#          (bit 3 set for the negative half, bits 0-2 the rank of |centroid|).
#   signs: m bits, projection i at byte i//8, bit i%8 (so 32 per uint32 word).
#   norms: IEEE half.
# Block (one page, one KV head), structure of arrays over the 16 slots:
#   K: codes[16][cbk] | signs[16][m/8] | n16[16] | rho16[16]
#   V: codes[16][cbv] | n16[16]
# Page = H_kv consecutive blocks; cache = pages consecutively.

def code_bytes(params, kind):
    return params.code_bits(kind) // 8


def cache_block_bytes(params, kind):
    if kind == "k":
        sb = params.m // 8 if params.k_qjl else 0
        rb = 2 if params.k_qjl else 0
        return PAGE * (code_bytes(params, "k") + sb + 2 + rb)
    return PAGE * (code_bytes(params, "v") + 2)


def code_bit_positions(params, kind):
    """pos[j][q]: stream bit of bit q of channel j's stored value (format above)."""
    bits, split = (params.k_bits, params.k_split) if kind == "k" else (params.v_bits, params.v_split)
    pos = []
    for j in range(params.d):
        if j < split:
            base, c, b = 0, j, bits[0]
        else:
            base, c, b = split * bits[0], j - split, bits[1]
        if b == 3:
            ob, i = base + 24 * (c // 8), c % 8
            if i < 6:
                pos.append([ob + 4 * i + q for q in range(3)])
            else:
                pos.append([ob + 4 * (2 * q + (i - 6)) + 3 for q in range(3)])
        else:
            pos.append([base + b * c + q for q in range(b)])
    return pos


def stored_value(code, b):
    """The b-bit value written for a code (identity except sign-magnitude at b = 4)."""
    code = np.asarray(code)
    if b != 4:
        return code
    return np.where(code >= 8, code - 8, 8 + (7 - code))


def code_from_stored(value, b):
    value = np.asarray(value)
    if b != 4:
        return value
    return np.where(value & 8, 7 - (value & 7), 8 + value)


def _pack_codes(params, codes, kind):
    cb = params.channel_bits(kind)
    pos = code_bit_positions(params, kind)
    bits = np.zeros((codes.shape[0], int(cb.sum())), dtype=np.uint8)
    for j in range(params.d):
        v = stored_value(codes[:, j], int(cb[j]))
        for q, p in enumerate(pos[j]):
            bits[:, p] = (v >> q) & 1
    return np.packbits(bits, axis=1, bitorder="little")


def _unpack_codes(params, raw, kind):
    cb = params.channel_bits(kind)
    pos = code_bit_positions(params, kind)
    bits = np.unpackbits(raw, axis=1, bitorder="little").astype(np.int64)
    codes = np.zeros((raw.shape[0], params.d), dtype=np.int64)
    for j in range(params.d):
        v = np.zeros(raw.shape[0], dtype=np.int64)
        for q, p in enumerate(pos[j]):
            v |= bits[:, p] << q
        codes[:, j] = code_from_stored(v, int(cb[j]))
    return codes


def pack_k_records(params, q):
    rec = {"codes": _pack_codes(params, q["codes"], "k"), "n16": q["n16"].astype(np.float16)}
    if params.k_qjl:
        rec["signs"] = np.packbits(q["signs"], axis=1, bitorder="little")
        rec["rho16"] = q["rho16"].astype(np.float16)
    return rec


def pack_v_records(params, q):
    return {"codes": _pack_codes(params, q["codes"], "v"), "n16": q["n16"].astype(np.float16)}


def unpack_k_records(params, rec):
    out = {"codes": _unpack_codes(params, rec["codes"], "k"),
           "n16": rec["n16"].astype(np.float64)}
    if params.k_qjl:
        out["signs"] = np.unpackbits(rec["signs"], axis=1, bitorder="little")[:, :params.m]
        out["rho16"] = rec["rho16"].astype(np.float64)
    return out


def unpack_v_records(params, rec):
    return {"codes": _unpack_codes(params, rec["codes"], "v"),
            "n16": rec["n16"].astype(np.float64)}


def _block_fields(params, kind):
    """(name, bytes per slot) in block order."""
    if kind == "k":
        f = [("codes", code_bytes(params, "k"))]
        if params.k_qjl:
            f.append(("signs", params.m // 8))
        f.append(("n16", 2))
        if params.k_qjl:
            f.append(("rho16", 2))
        return f
    return [("codes", code_bytes(params, "v")), ("n16", 2)]


def _as_bytes(name, arr):
    if name in ("n16", "rho16"):
        return np.asarray(arr, dtype=np.float16).view(np.uint8).reshape(-1, 2)
    return np.asarray(arr, dtype=np.uint8)


def write_paged(params, kind, cache, rec, pages, slots, heads, num_kv_heads):
    """Store records (one row per vector) at (page, slot, head) in the cache bytes."""
    bb = cache_block_bytes(params, kind)
    page_stride = num_kv_heads * bb
    base = np.asarray(pages, dtype=np.int64) * page_stride + np.asarray(heads, dtype=np.int64) * bb
    slots = np.asarray(slots, dtype=np.int64)
    off = 0
    for name, nb in _block_fields(params, kind):
        data = _as_bytes(name, rec[name])
        for k in range(nb):
            cache[base + off + slots * nb + k] = data[:, k]
        off += PAGE * nb
    return cache


def read_paged(params, kind, cache, pages, slots, heads, num_kv_heads):
    """Inverse of write_paged: gather records at (page, slot, head)."""
    bb = cache_block_bytes(params, kind)
    page_stride = num_kv_heads * bb
    base = np.asarray(pages, dtype=np.int64) * page_stride + np.asarray(heads, dtype=np.int64) * bb
    slots = np.asarray(slots, dtype=np.int64)
    rec = {}
    off = 0
    for name, nb in _block_fields(params, kind):
        data = np.stack([cache[base + off + slots * nb + k] for k in range(nb)], axis=1)
        if name in ("n16", "rho16"):
            rec[name] = data.copy().view(np.float16).reshape(-1)
        else:
            rec[name] = data
        off += PAGE * nb
    return rec


def token_locations(block_table, b, positions):
    """Physical (page, slot) of token positions of sequence b ([P4] §3.1 blocks)."""
    positions = np.asarray(positions, dtype=np.int64)
    return block_table[b, positions // PAGE].astype(np.int64), positions % PAGE


# ---------------------------------------------------------------------------
# Decode attention
# ---------------------------------------------------------------------------

def estimate_scores(params, qt, uq, krec):
    """Two-stage estimate of <q, k> for every cached key ([P2] stage 2, [P4] §4.3).

    qt = Pi q, uq = S Pi q.  Stage 1: <qt, (n16/sqrt(d)) c[code]>.  Stage 2:
    sqrt(pi/2)/m * rho16 * sum_i uq_i * (+1 if sign bit else -1).
    """
    d = params.d
    books = _centroid_table(params, "k")
    C = np.empty(krec["codes"].shape)
    for j in range(d):
        C[:, j] = books[j].centroids[krec["codes"][:, j]]
    s = (krec["n16"] / math.sqrt(d)) * (C @ qt)
    if params.k_qjl:
        pm = 2.0 * krec["signs"].astype(np.float64) - 1.0
        s = s + math.sqrt(math.pi / 2.0) / params.m * krec["rho16"] * (pm @ uq)
    return s


def dequantize_values(params, vrec):
    """Stage-1 reconstruction of values in the rotated domain, (n16/sqrt(d)) c[code]."""
    books = _centroid_table(params, "v")
    C = np.empty(vrec["codes"].shape)
    for j in range(params.d):
        C[:, j] = books[j].centroids[vrec["codes"][:, j]]
    return (vrec["n16"] / math.sqrt(params.d))[:, None] * C


def attend_one(params, q, krec, vrec, scale):
    """One query against one sequence's records: estimated scores, two-pass
    softmax ([P4] §2.2 and §4.3 softmax(QK^T/sqrt(d))), weighted sum of the
    dequantized values, inverse rotation back to the original basis."""
    n = krec["n16"].shape[0]
    if n == 0:
        return np.zeros(params.d)
    qt = params.Pi @ q
    uq = params.S @ qt
    logits = scale * estimate_scores(params, qt, uq, krec)
    mx = np.max(logits)
    p = np.exp(logits - mx)
    p /= np.sum(p)
    ot = p @ dequantize_values(params, vrec)
    return params.Pi.T @ ot


def decode_attention(params, q, seq_lens, block_table, k_cache, v_cache, num_kv_heads,
                     scale=None, pairs=None):
    """Decode attention for q [B, Hq, d] over the paged caches.

    Query head h reads KV head h // (Hq / H_kv).  `pairs` optionally restricts
    the work to a list of (b, h) for sampled checks; other rows stay zero.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    group = Hq // num_kv_heads
    out = np.zeros((B, Hq, d))
    todo = pairs if pairs is not None else [(b, h) for b in range(B) for h in range(Hq)]
    cache_rec = {}
    for b, h in todo:
        hk = h // group
        key = (b, hk)
        if key not in cache_rec:
            L = int(seq_lens[b])
            pages, slots = token_locations(block_table, b, np.arange(L))
            heads = np.full(L, hk)
            kr = unpack_k_records(params, read_paged(params, "k", k_cache, pages, slots, heads, num_kv_heads))
            vr = unpack_v_records(params, read_paged(params, "v", v_cache, pages, slots, heads, num_kv_heads))
            cache_rec[key] = (kr, vr)
        kr, vr = cache_rec[key]
        out[b, h] = attend_one(params, q[b, h], kr, vr, scale)
    return out


def causal_attention(params, q, start_pos, block_table, k_cache, v_cache, num_kv_heads, scale=None):
    """Multi-query causal attention over the compressed cache ([P4] §2.3: a new
    token's query attends over every cached token, the new tokens' K/V having
    been appended first).  q [B, T, Hq, d] holds the queries of T new tokens at
    positions start_pos[b] + t; token t attends over positions 0 .. start_pos[b] + t
    of sequence b (the cache already holds all of them).  Decode is T = 1.
    """
    q = np.asarray(q, dtype=np.float64)
    B, T, Hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    group = Hq // num_kv_heads
    out = np.zeros((B, T, Hq, d))
    for b in range(B):
        last = int(start_pos[b]) + T                     # positions 0 .. last - 1 are needed
        pages, slots = token_locations(block_table, b, np.arange(last))
        for hk in range(num_kv_heads):
            heads = np.full(last, hk)
            kr = unpack_k_records(params, read_paged(params, "k", k_cache, pages, slots, heads, num_kv_heads))
            vr = unpack_v_records(params, read_paged(params, "v", v_cache, pages, slots, heads, num_kv_heads))
            for t in range(T):
                n = int(start_pos[b]) + t + 1
                kt = {key: val[:n] for key, val in kr.items()}
                vt = {key: val[:n] for key, val in vr.items()}
                for h in range(hk * group, (hk + 1) * group):
                    out[b, t, h] = attend_one(params, q[b, t, h], kt, vt, scale)
    return out


def search(params, q, block_table_row, k_cache, n_db, k_top):
    """Inner-product search over a quantized key database ([P2] "생각정리 209
    (TurboQuant)": the vector-search use; [P4] §4.3: the two-stage estimate).

    The database is one KV head's K cache: vector t at page block_table_row[t // 16],
    slot t % 16.  Returns the [nq, n_db] estimated inner products and the k_top
    best per query, best first, equal scores by lower index.
    """
    q = np.asarray(q, dtype=np.float64)
    pages = np.asarray(block_table_row, dtype=np.int64)[np.arange(n_db) // PAGE]
    slots = np.arange(n_db) % PAGE
    krec = unpack_k_records(params, read_paged(params, "k", k_cache, pages, slots, np.zeros(n_db, dtype=np.int64), 1))
    scores = np.empty((q.shape[0], n_db))
    for i in range(q.shape[0]):
        qt = params.Pi @ q[i]
        scores[i] = estimate_scores(params, qt, params.S @ qt, krec)
    order = np.argsort(-scores, axis=1, kind="stable")[:, :k_top]
    return scores, order, np.take_along_axis(scores, order, axis=1)


def exact_attention(q, K, V, scale):
    """Textbook softmax(q K^T * scale) V in fp64, for pins only."""
    logits = scale * (K @ q)
    p = np.exp(logits - np.max(logits))
    p /= p.sum()
    return p @ V
