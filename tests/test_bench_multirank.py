"""bench.py's multi-rank host logic on CPU, as two gloo ranks.

The decode and quantize work shards with no collective (weak scaling: every
rank runs its own replica); the only cross-rank steps are the barrier and the
max-over-ranks of the timed region, and the reference arm printing on rank 0
alone.  Those run here with world size 2 over gloo on 127.0.0.1.
"""

import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # each rank timed its own replica; all of them must report the slowest one
        ms = bench.max_over_ranks(10.0 + 3.0 * rank, dist, "cpu")
        dist.barrier()
        # the weak-scaling value: units all ranks processed / the slowest rank's time
        bytes_per_rank = 1000 * (rank + 1)
        total = torch.tensor([float(bytes_per_rank)])
        dist.all_reduce(total)
        value = float(total.item()) / (ms * 1e-3) / 1e9
        # reference arm: rank 0 alone prints its line (a short oracle run); other ranks exit without output
        out = io.StringIO()
        if rank != 0:
            with redirect_stdout(out):
                bench.run_reference(bench.parse(["--impl", "reference", "--steps", "1", "--warmup", "0",
                                                 "--config", "c3"]))
        q.put((rank, ms, value, out.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        rank, ms, value, out = q.get(timeout=120)
        res[rank] = (ms, value, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == res[1][0] == 13.0
    assert res[0][1] == res[1][1] == pytest.approx(3000.0 / 13e-3 / 1e9)
    assert res[1][2] == ""          # non-zero ranks of the reference arm print nothing


def test_single_process_time_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, None, "cpu") == 7.5


def test_reference_line_is_one_json_object(monkeypatch, capsys):
    """Rank 0 of the reference arm prints one JSON line with the contract's keys (a short oracle sample)."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    bench.run_reference(bench.parse(["--impl", "reference", "--steps", "1", "--warmup", "0", "--config", "c3",
                                     "--cpu-workers", "2"]))
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "cpu_baseline", "e2e", "config"):
        assert key in rec
    assert rec["impl"] == "reference" and rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["value"] > 0


def test_cpu_baseline_pool_reports_cores_and_rates():
    """The oracle pool behind cpu_baseline: spawn-started workers, every worker at once and one alone, and the
    quantize rate on c2 slices (extrapolated and labelled so)."""
    sys.path.insert(0, ROOT)
    import bench
    from online_kv_cache_02_gb300 import workloads as wl
    w = wl.WORKLOADS["c3"].scaled(batch=1, seq_len=512)
    pool = bench.OraclePool(w, 2)
    try:
        rec = bench.cpu_baseline(pool, w, seconds=0.5)
        assert rec["cores"] == 2 and rec["kind"] == "oracle" and rec["value"] > 0
        assert rec["single_core"]["cores"] == 1 and rec["single_core"]["value"] > 0
        assert rec["cpu_model"] and rec["host_cores"] >= 1
        q = pool.quantize_rates()
        assert q["cores"] == 2 and q["value"] > 0 and q["single_core"]["value"] > 0
        assert "extrapolated" in q["sample"] and "extrapolated" in q["single_core"]["sample"]
    finally:
        pool.close()
