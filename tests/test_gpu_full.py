"""Full-size workloads in the launch configuration bench.py times, checked on samples.

The GPU quantizes the whole synthetic history and runs one bench step (append a
token, decode).  For sampled sequences and KV heads the oracle quantizes the same
inputs itself: the GPU-written records must match its codes/signs/norms, and the
GPU's attention output for the query heads of those KV heads must match the
oracle's decode of its own records within 2e-3.
"""

import math

import numpy as np
import pytest

import bench

from .gpu_common import oracle, seq_locations, th, tq, wl
from .gpu_common import torch

pytestmark = pytest.mark.gpu


def _check_sequence(w, db, b, heads, stats):
    p = th.params_for(w)
    L = int(db.lens[b])
    G = w.q_heads // w.kv_heads
    kc, vc = db.kc.cpu().numpy(), db.vc.cpu().numpy()
    out = db.out.cpu().numpy()
    for h in heads:
        K = np.concatenate([wl.kv_tokens(w, "k", b)[:, h], wl.new_tokens(w, "k")[b, :, h]]).astype(np.float64)
        V = np.concatenate([wl.kv_tokens(w, "v", b)[:, h], wl.new_tokens(w, "v")[b, :, h]]).astype(np.float64)
        pos = np.arange(L + 1)
        pages, slots = db.bt[b, pos // 16].astype(np.int64), pos % 16
        hh = np.full(L + 1, h)
        recs = {}
        for kind, X, cache in (("k", K, kc), ("v", V, vc)):
            q = oracle.quantize_vectors(p, X, kind)
            ex = oracle.quantize_exclusions(p, q, kind)
            res = th.compare_records(p, kind, cache, q, ex, pages, slots, hh, w.kv_heads)
            th.assert_records_ok(res)
            stats["codes"] += res["codes_total"]
            stats["excluded"] += res["codes_excluded"]
            rec = oracle.pack_k_records(p, q) if kind == "k" else oracle.pack_v_records(p, q)
            recs[kind] = oracle.unpack_k_records(p, rec) if kind == "k" else oracle.unpack_v_records(p, rec)
        Q = wl.queries(w)[b].astype(np.float64)
        for g in range(G):
            hq = h * G + g
            ref = oracle.turboquant.attend_one(p, Q[hq], recs["k"], recs["v"], 1.0 / math.sqrt(128))
            err = th.rel_err(out[b, hq], ref)
            stats["max_err"] = max(stats["max_err"], float(err))
            assert err <= th.ATT_TOL, (w.name, b, hq, float(err))


@pytest.mark.parametrize("name,samples", [("c3", [(15, [0, 7])]), ("c4", [(0, [3]), (63, [0])]),
                                          ("c5", [(3, [5])])])
def test_decode_workload_full_size(name, samples):
    w = wl.WORKLOADS[name]
    stream = torch.cuda.current_stream()
    db = bench.DecodeBench(w, torch, tq)
    try:
        db.step(stream)
        db.step(stream)      # a second step overwrites the same appended slot with the same token
        torch.cuda.synchronize()
        assert tq.tq_check_device_status(db.ctx) == 0
        stats = {"codes": 0, "excluded": 0, "max_err": 0.0}
        for b, heads in samples:
            _check_sequence(w, db, b, heads, stats)
        assert stats["excluded"] <= 1e-4 * stats["codes"], stats
        print(name, stats)
    finally:
        db.close()


def test_quantize_workload_full_size():
    w = wl.WORKLOADS["c2"]
    stream = torch.cuda.current_stream()
    qb = bench.QuantizeBench(w, torch, tq)
    try:
        qb.step(stream)
        torch.cuda.synchronize()
        assert tq.tq_check_device_status(qb.ctx) == 0
        p = th.params_for(w)
        kc, vc = qb.kc.cpu().numpy(), qb.vc.cpu().numpy()
        total = excluded = 0
        for b, h in ((0, 0), (31, 7), (17, 3)):
            pages, slots, hh = seq_locations(qb.bt, b, np.arange(w.seq_len), w.kv_heads)
            sel = hh == h
            for kind, cache in (("k", kc), ("v", vc)):
                X = wl.kv_tokens(w, kind, b)[:, h].astype(np.float64)
                q = oracle.quantize_vectors(p, X, kind)
                ex = oracle.quantize_exclusions(p, q, kind)
                res = th.compare_records(p, kind, cache, q, ex, pages[sel], slots[sel], hh[sel], w.kv_heads)
                th.assert_records_ok(res)
                total += res["codes_total"]
                excluded += res["codes_excluded"]
        assert excluded <= 1e-4 * total
    finally:
        qb.close()
