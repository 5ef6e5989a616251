"""Host-side bench logic: the max-over-ranks / sum-over-ranks reduction on
world_size-2 gloo process groups, and the CPU reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t, u = bench.aggregate(elapsed_s=1.0 + rank, units_local=10.0 * (rank + 1))
        bench.barrier()
        q.put((rank, t, u, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, u, env in out:
        assert t == 2.0 and u == 30.0
        assert env == (rank, 2, 0)


def test_aggregate_without_process_group_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(1.5, 7.0) == (1.5, 7.0)


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1", "--workload", "router_small"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=120, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_shape_rows_carry_the_sustained_rate():
    """Each per-shape row reports the back-to-back time without PDL and, when
    measured, the PDL-chain time, both as µs per launch and as a fraction of
    the peak from the same algorithmic bytes; the flush cross-check when
    given."""
    sys.path.insert(0, ROOT)
    import types
    import bench
    import skinny_inputs as si
    cases = si.projection_cases()[:2]
    plans = [dict(backend=1, consumer=1, split_k=1, block_n=4, grid_x=528, grid_y=1),
             dict(backend=4, consumer=2, split_k=8, block_n=64, grid_x=8, grid_y=33)]
    wl = types.SimpleNamespace(cases=cases, plans=plans)
    rows = bench.shape_rows(wl, [10.0, 20.0], 6788.3, flushed=[(12.0, 11.0, 13.0)] * 2, chained=[8.0, 16.0])
    assert [r["kernel"] for r in rows] == ["dotprod", "tmem_gemm"]
    for r, c, iso, ch in zip(rows, cases, (10.0, 20.0), (8.0, 16.0)):
        assert r["us_per_launch"] == iso and r["chained_pdl"]["us_per_launch"] == ch
        assert r["frac_of_peak"] == pytest.approx(c.algorithmic_bytes / iso / 1e3 / 6788.3, abs=1e-4)
        assert r["chained_pdl"]["frac_of_peak"] == pytest.approx(c.algorithmic_bytes / ch / 1e3 / 6788.3, abs=1e-4)
        assert r["flush_us"] == {"median": 12.0, "p10": 11.0, "p90": 13.0}
    assert "chained_pdl" not in bench.shape_rows(wl, [10.0, 20.0], 6788.3)[0]
