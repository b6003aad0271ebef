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
    # the same workload as the CUDA arm's line; the sample is in cpu_baseline
    assert j["config"]["workload"] == bench.STEP_WORKLOAD
    launches = bench.workload_launches(None, None)
    assert j["config"]["bytes_per_step"] == sum(L["bytes"] for L in launches)
    assert j["config"]["launches_per_step"] == len(launches) == 64
    assert f"first min(T, {j['config']['sample_rows_per_launch']}) rows" in \
        j["cpu_baseline"]["sample"]


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


def _synthetic_full_record() -> dict:
    """A whole-step record shaped like run_ours' (every per-shape and widened
    row present, long numbers), to size the printed line."""
    import workloads as W
    rows = []
    for L in bench.workload_launches():
        rows.append({"op": L["op"], "T": L["T"], "d": L["d"], "z": L["z"],
                     "kernel": "gelu_cta_rows<1024,4,true>", "us": 123.456, "GBps": 6543.2,
                     "frac_of_measured": 0.9671, "frac_of_spec_8TBps": 0.8179,
                     "x_floor": 12.345, "launches_in_graph": 200,
                     **({"stream_us": 121.234, "x_stream": 1.018, "copy_us": 119.876,
                         "x_copy": 1.029} if L["op"] == "gelu" else {})})
    widened = [dict(rows[0], op=L["op"]) for L in bench.extra_launches()]
    return {
        "metric": bench.METRIC, "value": 4818.3, "unit": "GB/s", "n_gpus": 1, "steps": 200,
        "warmup": 10, "ms_per_step": 0.56512, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": bench.STEP_WORKLOAD, "launches_per_step": 64,
                   "bytes_per_step": 2699599872, "l2": "no flush: every launch has its own "
                   "buffers (2.7 GB per step, 129 MB L2)",
                   "parallelism": "rows sharded over 1 GPU(s), no collective",
                   "launch_floor_us": 0.353},
        "roofline": {"bound": "hbm", "kernel": "gelu_pipe_rows<16,8>", "achieved": 6084.1,
                     "peak": 6766.0, "unit": "GB/s", "frac": 0.8992, "peak_source": "measured",
                     "frac_of_spec_8TBps": 0.7605, "launches_per_step": 6,
                     "bytes_per_launch_avg": 234881024, "avg_launch_us": 35.932,
                     "time_share": 0.3811, "traffic": 203587211},
        "e2e": {"value": 270.123, "unit": "GB/s", "ms_per_step": 9.9943, "steps": 10,
                "reps_ms": [9.9, 10.0, 10.1], "h2d_bytes_per_step": 1799733248,
                "d2h_bytes_per_step": 899866624, "link_ceiling": 282.1, "frac_of_link": 0.9576,
                "pipeline": "3 streams", "link": {"value": 282.1}},
        "e2e_host_direct": {"value": 255.432, "unit": "GB/s", "frac_of_link": 0.8912},
        "gpu_launches": 12800,
        "clocks": {"sm_mhz": 2070, "sm_max_mhz": 2070, "reasons": ["sw_power_cap"],
                   "samples": 123, "source": "nvml"},
        "per_shape": rows, "widened_rows": widened,
        "cpu_baseline": {"value": 6.0916, "unit": "GB/s", "cores": 16, "kind": "oracle",
                         "sample": "3 full step(s) of the workload (64 launches, 2699599872 "
                                   "algorithmic bytes each) through the fp64 C oracle, OpenMP "
                                   "over rows; 1.33 s wall",
                         "sample_short": "3 whole step(s) on 16 threads, 1.3 s",
                         "single_core": {"value": 0.452, "unit": "GB/s", "cores": 1},
                         "cpu_model": "aarch64 Neoverse-V2", "nproc": 16},
        "_z": W.Z95,
    }


def test_bench_line_is_short_and_last(capsys, tmp_path):
    """The driver keeps only the tail of stdout: the line must be the last one
    and short enough to survive a tail of a few KB whole."""
    full = _synthetic_full_record()
    detail = tmp_path / "detail.json"
    bench.emit(full, str(detail))
    out = capsys.readouterr().out
    last = out.rstrip("\n").splitlines()[-1]
    assert len(last.encode()) <= 2048, len(last)
    j = json.loads(last)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "dtype", "config", "roofline", "e2e", "cpu_baseline",
              "gpu_launches", "clocks"):
        assert k in j, k
    assert j["config"]["workload"] == bench.STEP_WORKLOAD
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in j["roofline"]
    assert j["e2e"]["h2d_bytes_per_step"] > 0 and j["e2e"]["d2h_bytes_per_step"] > 0
    for k in ("value", "unit", "cores", "kind", "sample"):
        assert k in j["cpu_baseline"]
    assert set(j["targets"]) == {"cols"} | {f"{T}x{d}" for T, d in bench.TARGET_SHAPES}
    assert set(j["decode"]) == {"cols"} | {f"{T}x{d}" for T, d in bench.DECODE_SHAPES}
    # the side file keeps every row
    back = json.loads(detail.read_text())
    assert len(back["per_shape"]) == 64 and len(back["widened_rows"]) == len(bench.extra_launches())


def test_workload_name_of_both_arms():
    args = bench.parse_args([])
    assert bench.workload_name(args, bench.workload_launches()) == bench.STEP_WORKLOAD
    args = bench.parse_args(["--only", "2048,16384"])
    assert bench.workload_name(args, bench.workload_launches(args.only)) == \
        "gelu_and_mul_sparse T=2048 d=16384"
    args = bench.parse_args(["--only-silu", "2048"])
    L = bench.workload_launches(None, args.only_silu)
    assert bench.workload_name(args, L) == "silu_and_mul M=2048 d=768"
