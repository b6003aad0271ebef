"""Host logic of bench.py on the CPU: algorithmic bytes, the step's launch list,
the row sharding of the multi-GPU path and its max-over-ranks timing (two gloo
ranks), and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_silu_moe_decode_bytes_match_page():
    # Megatron-LM PR "Size MoE activation kernel grid to the row count",
    # "What changed and why": 9.44 MB moved for 2048 rows at d = 768.
    with open(os.path.join(ROOT, "tests", "golden", "page_numbers.json")) as f:
        p = json.load(f)["silu_moe_decode_bytes"]
    assert round(bench.silu_bytes(p["M"], p["d"]) / 1e6, 2) == p["printed_MB"]


def test_gelu_bytes_read_gate_up_once_write_once():
    assert bench.gelu_bytes(2048, 16384) == 2048 * (2 * 16384 + 16384) * 2 == 201326592


def test_step_launch_list():
    L = bench.workload_launches()
    gelu = [x for x in L if x["op"] == "gelu"]
    assert len(gelu) == 6 * 5 * 2 and len(L) == 64
    assert {x["z"] for x in gelu} == {0.0, 1.6448536269514722}
    # z is the outer loop: the first 30 launches are z = 0
    assert all(x["z"] == 0.0 for x in gelu[:30])
    only = bench.workload_launches((2048, 16384))
    assert len(only) == 2 and all(x["T"] == 2048 for x in only)


@pytest.mark.parametrize("T,world", [(2048, 1), (2048, 2), (2049, 2), (7, 4), (3, 8), (0, 2)])
def test_shard_rows_partition(T, world):
    seen = []
    for r in range(world):
        s, n = bench.shard_rows(T, world, r)
        assert n >= 0
        seen.extend(range(s, s + n))
    assert seen == list(range(T))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        t = bench.max_over_ranks(1.0 + rank, world, None)
        s, n = bench.shard_rows(2049, world, rank)
        q.put((rank, t, s, n))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_and_sharding_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.0, 2.0]           # both see the slowest rank
    assert res[0][2:] == (0, 1025) and res[1][2:] == (1025, 1024)


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, GATED_ACT_REF_BUDGET_S="4")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True,
                       env=env, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["metric"] == bench.METRIC and j["unit"] == "GB/s"
    assert j["value"] > 0 and j["cpu_baseline"]["kind"] == "oracle"
    assert j["e2e"]["h2d_bytes_per_step"] == 0


def test_cpu_model_names_arm_cores(monkeypatch):
    import builtins
    import io
    real_open = builtins.open

    def fake_open(path, *a, **k):
        if path == "/proc/cpuinfo":
            return io.StringIO("processor\t: 0\nCPU implementer\t: 0x41\nCPU part\t: 0xd4f\n")
        return real_open(path, *a, **k)

    monkeypatch.setattr(builtins, "open", fake_open)
    name = bench.cpu_model()
    assert "Neoverse-V2" in name and "0xd4f" in name
