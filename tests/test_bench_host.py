"""Host-side logic of the benchmark (no GPU): byte accounting, the
multi-rank reduction (world size 2 over gloo on CPU, as torchrun would launch
the replicas), and the CPU-oracle reference arm."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_algorithmic_bytes_moonep():
    b = bench.algorithmic_bytes(4096, 7168, 64, 8, 4096 * 8)
    # dispatch: read x once (58.72 MB) + tok_map, write 8 rows per token (469.76 MB)
    assert b["dispatch"] == 4096 * 7168 * 2 + 4096 * 8 * 8 + 32768 * 7168 * 2
    assert abs(b["dispatch"] / 1e6 - 528.74) < 0.01
    # combine: read 8 rows per token + map + weights, write one row per token
    assert abs(b["combine"] / 1e6 - 528.87) < 0.01
    assert 0.5e6 < b["plan"] < 0.6e6


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    t, b = bench.aggregate(10.0 + rank, 100.0 * (rank + 1), world)
    q.put((rank, t, b, bench.dist_env()))
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    import socket

    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, b, env in got:
        assert t == 11.0          # max over ranks
        assert b == 300.0         # sum over ranks
        assert env == (2, rank, rank)


def test_single_rank_aggregate_is_identity():
    assert bench.aggregate(5.0, 7.0, 1) == (5.0, 7.0)


@pytest.mark.timeout(300)
def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["metric"] == bench.METRIC
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.timeout(300)
def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1"], capture_output=True, text=True,
                       timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_pinned_core_restores_affinity():
    before = os.sched_getaffinity(0)
    with bench.PinnedCore() as pin:
        assert os.sched_getaffinity(0) == {pin.core}
        assert pin.core == max(before)
    assert os.sched_getaffinity(0) == before


def test_host_cpu_model_is_named():
    assert isinstance(bench.host_cpu_model(), str) and bench.host_cpu_model()


@pytest.mark.parametrize("name,S", [("tiny", None), ("dedup", 0), ("dedup", 1), ("dedup", 40),
                                    ("fp8small", 4)])
def test_oracle_calls_per_config(name, S):
    """The CPU leg's per-call timing over each workload kind: every call runs
    and reports its algorithmic bytes (the dedup workload adds the group
    plan and the two dedup calls)."""
    import workloads
    wl = workloads.make(name, seed=3, S=S) if S is not None else workloads.make(name, seed=3)
    calls = bench._oracle_calls(wl)
    want = {"plan", "dispatch", "combine"}
    if name == "dedup":
        want |= {"group_plan", "dispatch_dedup", "combine_dedup"}
    assert set(calls) == want
    res = bench._time_calls(calls)
    for k, v in res.items():
        assert v["us"] > 0 and v["algorithmic_bytes"] >= 0, k
    if S not in (0,):
        assert res["dispatch"]["algorithmic_bytes"] > 0
