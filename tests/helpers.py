"""Shared helpers for the GPU parity tests: oracle-built caches and field-wise comparison.

Parity bars (the readings of the target tolerances these tests apply):
  * codes and sign bits bit-exact, except codes whose unit-variance value is
    within 1e-6 of a boundary and the signs of such vectors (and signs with
    |S r| < 1e-6 ||r||); the excluded count must stay <= 1e-4 of all codes
  * fp16 key/value norms bit-exact (they feed the residual, so the GPU decides
    them from an exact double-float norm)
  * fp16 residual norm within one fp16 ulp (a stored floating-point value)
  * page/slot addressing bit-exact: every byte the oracle did not write stays
    as it was
  * attention output: max_j |o_j - o*_j| / max_j |o*_j| <= 2e-3 per vector
"""

import math

import numpy as np

import oracle
from oracle import turboquant as otq

ATT_TOL = 2e-3


def params_for(w, seed=None):
    return oracle.make_params(d=128, m=w.m, k_bits=w.k_bits, v_bits=w.v_bits, seed=w.seed if seed is None else seed,
                              k_qjl=w.qjl, codebook=w.codebook)


def locations(block_table, b_idx, pos, h_idx):
    pages = block_table[b_idx, pos // 16].astype(np.int64)
    return pages, pos % 16, h_idx


def oracle_quantize_into(p, kind, cache, X, pages, slots, heads, H):
    """Quantize rows of X with the oracle and write them into the byte cache; returns (q, excl)."""
    q = oracle.quantize_vectors(p, X, kind)
    rec = oracle.pack_k_records(p, q) if kind == "k" else oracle.pack_v_records(p, q)
    oracle.write_paged(p, kind, cache, rec, pages, slots, heads, H)
    return q, oracle.quantize_exclusions(p, q, kind)


def compare_records(p, kind, got_cache, want_q, excl, pages, slots, heads, H):
    """Field-wise comparison of GPU-written records against the oracle's quantization."""
    raw = oracle.read_paged(p, kind, got_cache, pages, slots, heads, H)
    rec = oracle.unpack_k_records(p, raw) if kind == "k" else oracle.unpack_v_records(p, raw)
    res = {}
    cm = rec["codes"] != want_q["codes"]
    res["codes_total"] = cm.size
    res["codes_excluded"] = int(excl["codes"].sum())
    res["codes_mismatch"] = int((cm & ~excl["codes"]).sum())
    res["codes_mismatch_excluded"] = int((cm & excl["codes"]).sum())
    res["norm_mismatch"] = int((rec["n16"] != want_q["n16"]).sum())
    if kind == "k" and p.k_qjl:
        sm = rec["signs"] != want_q["signs"]
        res["signs_mismatch"] = int((sm & ~excl["signs"]).sum())
        res["signs_excluded"] = int(excl["signs"].sum())
        got = rec["rho16"].astype(np.float16).view(np.uint16).astype(np.int64)
        want = want_q["rho16"].astype(np.float16).view(np.uint16).astype(np.int64)
        res["rnorm_ulp_max"] = int(np.max(np.abs(got - want))) if got.size else 0
        res["rnorm_ulp_count"] = int(np.sum(got != want))
    return res


def assert_records_ok(res):
    assert res["codes_mismatch"] == 0, res
    assert res["norm_mismatch"] == 0, res
    assert res["codes_excluded"] <= 1e-4 * res["codes_total"] + 1, res
    if "signs_mismatch" in res:
        assert res["signs_mismatch"] == 0, res
        assert res["rnorm_ulp_max"] <= 1, res


def rel_err(got, ref):
    """Per output vector: max_j |got - ref| / max_j |ref| (rows of zeros must match exactly)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref), axis=-1)
    num = np.max(np.abs(got - ref), axis=-1)
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), num)


def scale_for(d=128):
    return 1.0 / math.sqrt(d)


def touched_mask(p, kind, nbytes, pages, slots, heads, H):
    """Boolean mask of cache bytes the records at these locations occupy."""
    mask = np.zeros(nbytes, dtype=bool)
    bb = oracle.cache_block_bytes(p, kind)
    base = np.asarray(pages) * H * bb + np.asarray(heads) * bb
    off = 0
    for name, nb in otq._block_fields(p, kind):
        for k in range(nb):
            mask[base + off + np.asarray(slots) * nb + k] = True
        off += 16 * nb
    return mask
