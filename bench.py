#!/usr/bin/env python
"""Throughput of the fused gated activations on GB300: achieved HBM GB/s and
us/launch over the T x d sweep.

One step = one pass over the whole workload, every launch through the C ABI:
  * gelu_and_mul_sparse for every T in {1, 8, 64, 256, 1024, 2048} x
    d in {2048, 4096, 8192, 16384, 32768} x z in {0, 1.6448536269514722}
    (exactly T rows each; i.i.d. N(0,1) bf16, seed 7919 T + d);
  * silu_and_mul for the MoE decode rows M in {1024, 2048, 4096, 16384}, d = 768.
The step runs as CUDA graphs (the way both pages' frameworks run these
activations): graph A holds the launches of the dominant kernel, graph B the
rest; CUDA events on the launching stream bracket each replay, which gives the
step time and the dominant kernel's average launch time.  A separate table
gives every shape's us/launch from a graph of N launches over rotating buffers.

Algorithmic bytes: gelu T*3d*2 (gate+up read once, output written once),
silu M*3d*2.  Every launch of a step has its own input and output buffers
(2.6 GB per step against a 129 MB L2), so every launch reads HBM and no L2
flush is needed.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Multi-GPU (weak scaling, rows sharded, no collective on the data path):
  python -m torch.distributed.run --nproc-per-node N --master-addr 127.0.0.1 ... bench.py --gpus N
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s (and % of GB300 peak) and µs/launch vs T×d sweep"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
SPEC_HBM_GBS = 8000.0


# ----------------------------------------------------------------- host logic
def gelu_bytes(T: int, d: int) -> int:
    """Algorithmic bytes of one gelu_and_mul_sparse call: read 4d, write 2d per row."""
    return T * 3 * d * 2


def silu_bytes(M: int, d: int) -> int:
    """Algorithmic bytes of one silu_and_mul call: read 4d, write 2d per row."""
    return M * 3 * d * 2


def shard_rows(T: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous row block [start, start + count) of rank `rank` out of `world`."""
    base, extra = divmod(T, world)
    start = rank * base + min(rank, extra)
    return start, base + (1 if rank < extra else 0)


def workload_launches(only: tuple | None = None, only_silu: int | None = None) -> list[dict]:
    """The step's launch list: gelu over (z, T, d), then silu over M.  `only`
    keeps one gelu shape, `only_silu` one silu row count (profiling runs)."""
    import workloads as W
    if only_silu:
        return [{"op": "silu", "T": only_silu, "d": W.SILU_D, "z": None,
                 "bytes": silu_bytes(only_silu, W.SILU_D)}]
    out = []
    for z in W.SWEEP_Z:
        for T in W.SWEEP_T:
            for d in W.SWEEP_D:
                if only and (only[0], only[1]) != (T, d):
                    continue
                if only and len(only) > 2 and only[2] != z:
                    continue
                out.append({"op": "gelu", "T": T, "d": d, "z": z, "bytes": gelu_bytes(T, d)})
    if not only:
        for M in W.SILU_M:
            out.append({"op": "silu", "T": M, "d": W.SILU_D, "z": None,
                        "bytes": silu_bytes(M, W.SILU_D)})
    return out


def extra_launches() -> list[dict]:
    """Widened rows, measured per shape (not part of the timed step): the
    bounded silu at the MoE page's case (a 16384-row buffer bound with 2048
    live rows, and fully live), dense gelu_and_mul, squared_relu, the sparse
    GELU on fp16/fp32 rows and in native-rounding mode."""
    import workloads as W
    d = W.SILU_D
    return [
        {"op": "silu_bounded", "T": 16384, "d": d, "live": 2048, "z": None,
         "bytes": silu_bytes(2048, d)},
        {"op": "silu_bounded", "T": 16384, "d": d, "live": 16384, "z": None,
         "bytes": silu_bytes(16384, d)},
        {"op": "gelu_dense", "T": 2048, "d": 16384, "z": None, "bytes": gelu_bytes(2048, 16384)},
        {"op": "gelu_dense", "T": 64, "d": 8192, "z": None, "bytes": gelu_bytes(64, 8192)},
        {"op": "squared_relu", "T": 2048, "d": d, "z": None, "bytes": 2048 * d * 2 * 2},
        {"op": "squared_relu", "T": 16384, "d": d, "z": None, "bytes": 16384 * d * 2 * 2},
        {"op": "gelu_f16", "T": 2048, "d": 16384, "z": W.Z95, "bytes": gelu_bytes(2048, 16384)},
        {"op": "gelu_f32", "T": 2048, "d": 16384, "z": W.Z95,
         "bytes": 2 * gelu_bytes(2048, 16384)},
        {"op": "gelu_f32", "T": 64, "d": 8192, "z": W.Z95, "bytes": 2 * gelu_bytes(64, 8192)},
        {"op": "gelu_native", "T": 2048, "d": 16384, "z": W.Z95,
         "bytes": gelu_bytes(2048, 16384)},
        {"op": "gelu_native", "T": 64, "d": 8192, "z": W.Z95, "bytes": gelu_bytes(64, 8192)},
    ]


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


def _code_only(text: str) -> str:
    """Source text without comments and whitespace (the hash tracks code only)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return re.sub(r"\s+", "", text)


def kernel_sources_hash() -> str:
    """Hash of the library's CUDA/C++ code (comments and whitespace ignored)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_activation_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f)) as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def load_traffic(kernel: str, algorithmic_bytes: float) -> float | None:
    """DRAM bytes (read + write) of one launch of `kernel` moving
    `algorithmic_bytes`, from the committed ncu capture of that kernel scaled
    by algorithmic bytes; None when there is no capture or the kernel sources
    changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            j = json.load(f)
    except Exception:
        return None
    if j.get("csrc_sha256_16") != kernel_sources_hash():
        return None
    ent = j.get("kernels", {}).get(kernel)
    if ent is None:
        return None
    return float(ent["traffic_per_algorithmic_byte"]) * algorithmic_bytes


# ----------------------------------------------------------------- clocks (NVML, read only)
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML in a thread (read-only)."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.samples: list[tuple[int, int]] = []
        self.max_mhz = None
        self.period = period_s
        self.ok = False
        self._stop = threading.Event()
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None)
            self.reasons_fn = fn or self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = True
        except OSError:
            pass

    def _sample(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) == 0 and \
                self.reasons_fn(self.h, ctypes.byref(r)) == 0:
            self.samples.append((int(c.value), int(r.value)))

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self._stop.set()
            self._t.join()
            self._sample()

    def summary(self) -> dict:
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml unavailable"}
        busy = [s for s in self.samples if not (s[1] & 0x1)] or self.samples
        mask = 0
        for _, r in busy:
            mask |= r
        reasons = [n for b, n in self.REASONS.items() if mask & b]
        return {"sm_mhz": statistics.median(s[0] for s in busy), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(busy), "source": "nvml"}


# ----------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None:
            dist.barrier(device_ids=[device])
        else:
            dist.barrier()


def max_over_ranks(x: float, world: int, device: str | None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- inputs
def rank_input(launch: dict, world: int, rank: int):
    """CPU bf16 input of one launch for this rank (rank 0 at N=1: the config's own input)."""
    import workloads as W
    T, d = launch["T"], launch["d"]
    if launch["op"] in ("gelu", "gelu_native"):
        seed = W.sweep_seed(T, d) + 1000003 * rank
        return W.iid(T, d, seed=seed, z=launch["z"]).x
    x = W.silu(T, d) if rank == 0 else None
    if x is None:
        import torch
        g = torch.Generator().manual_seed(3 + T + 1000003 * rank)
        x = torch.randn((T, 2 * d), generator=g).to(torch.bfloat16)
    return x


def kernel_name(plan: dict) -> str:
    v = plan["variant"]
    if v == "warp_rows":
        return f"gelu_warp_rows<{plan['vec_per_thread']}>"
    if v == "cta_row":
        cl = "true" if plan["cluster"] > 1 else "false"
        return f"gelu_cta_rows<{plan['threads']},{plan['vec_per_thread']},{cl}>"
    if v == "scalar":
        return "gelu_scalar_rows"
    if v == "tma_rows":
        return f"gelu_tma_rows<{plan['threads']},4>"
    if v == "pipe_rows":
        return f"gelu_pipe_rows<{plan['threads'] // 32 - 1},{plan['vec_per_thread']}>"
    if v == "split_rows":
        return f"gelu_split_rows<{plan['threads']},{plan['vec_per_thread']}> x{plan['cluster']}"
    return v


# ----------------------------------------------------------------- our arm
_WORKSPACE = {}


def _workspace(ga, device):
    """One zeroed row-ticket workspace per device.  Every launch of the bench
    on a device runs on one stream at a time, so they may share it."""
    key = str(device)
    if key not in _WORKSPACE:
        _WORKSPACE[key] = ga.new_workspace(device)
    return _WORKSPACE[key]


def _launch(ga, L, x, out):
    op = L["op"]
    if op == "gelu":
        ws = _workspace(ga, x.device) if x.is_cuda else None
        ga.gelu_and_mul_sparse(x, L["z"], d=L["d"], out=out, workspace=ws)
    elif op == "silu":
        ga.silu_and_mul(x, out=out)
    elif op == "silu_bounded":
        ga.silu_and_mul_bounded(x, L["n_rows"], out=out)
    elif op == "gelu_dense":
        ga.gelu_and_mul(x, d=L["d"], out=out)
    elif op == "squared_relu":
        ga.squared_relu(x, out=out)
    elif op in ("gelu_f16", "gelu_f32"):
        ga.gelu_and_mul_sparse(x, L["z"], d=L["d"], out=out)
    elif op == "gelu_native":
        ga.gelu_and_mul_sparse_native(x, L["z"], d=L["d"], out=out)
    else:
        raise ValueError(op)


def _in_width(L) -> int:
    return L["d"] if L["op"] == "squared_relu" else 2 * L["d"]


def _dtype_of(L):
    import torch
    return {"gelu_f16": torch.float16, "gelu_f32": torch.float32}.get(L["op"], torch.bfloat16)


def per_shape_times(ga, launches, dev, peak_gbs, reps=5) -> tuple[list, float]:
    """us/launch of every shape: a CUDA graph of N launches whose inputs and
    outputs rotate through a 1.5 GB / 0.75 GB arena (consecutive launches touch
    fresh memory; a window is reused only after >1 GB of traffic), median of
    `reps` replays.  Also the per-launch time of the library's empty kernel
    (same launch attributes) in the same harness: the launch floor."""
    import torch
    arena_in = torch.empty(768 << 20, dtype=torch.bfloat16, device=dev).normal_()
    arena_out = torch.empty(384 << 20, dtype=torch.bfloat16, device=dev)

    def timed_graph(fns):
        for f in fns[:2]:
            f()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for f in fns:
                f()
        g.replay()
        ts = []
        for _ in range(reps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) / len(fns))
        del g
        return statistics.median(ts)

    floor_ms = timed_graph([lambda: ga.noop() for _ in range(200)])
    rows = []
    seen = {}
    for L in launches:
        key = (L["op"], L["T"], L["d"], L["z"], L.get("live"))
        if key in seen:
            continue
        T, d = L["T"], L["d"]
        if L["op"] == "silu_bounded":
            L["n_rows"] = torch.tensor([L["live"]], dtype=torch.int32, device=dev)
        dt = _dtype_of(L)
        a_in, a_out = arena_in.view(dt), arena_out.view(dt)     # same bytes, reinterpreted
        n_in, n_out = T * _in_width(L), T * d
        win = max(1, min(a_in.numel() // n_in, a_out.numel() // n_out))
        N = int(min(200, max(20, win)))
        fns = []
        for i in range(N):
            w = i % win
            x = a_in[w * n_in:(w + 1) * n_in].view(T, _in_width(L))
            o = a_out[w * n_out:(w + 1) * n_out].view(T, d)
            fns.append(lambda x=x, o=o, L=L: _launch(ga, L, x, o))
        t = timed_graph(fns)
        seen[key] = t
        gbs = L["bytes"] / (t * 1e-3) / 1e9
        floor = floor_ms + L["bytes"] / (peak_gbs * 1e9) * 1e3
        row = {"op": L["op"], "T": T, "d": d, "z": L["z"], "kernel": L.get("kernel", L["op"]),
               "us": round(t * 1e3, 3), "GBps": round(gbs, 1),
               "frac_of_measured": round(gbs / peak_gbs, 4),
               "frac_of_spec_8TBps": round(gbs / SPEC_HBM_GBS, 4),
               "x_floor": round(t / floor, 3), "launches_in_graph": N,
               "rows_per_s": round(L.get("live", T) / (t * 1e-3), 1)}
        if "live" in L:
            row["live_rows"] = L["live"]
        if L["op"] in ("gelu", "silu"):
            # a floor this library did not write: device-to-device
            # cudaMemcpyAsync nodes (torch's copy_ of contiguous bytes) that
            # read and write half the launch's bytes each, so the same
            # read + write traffic, from and to the same rotating windows
            half = L["bytes"] // 2
            b_in, b_out = arena_in.view(torch.uint8), arena_out.view(torch.uint8)
            cwin = max(1, min(b_in.numel() // half, b_out.numel() // half))
            cfns = [lambda s=b_in[(i % cwin) * half:((i % cwin) + 1) * half],
                    o=b_out[(i % cwin) * half:((i % cwin) + 1) * half]: o.copy_(s)
                    for i in range(N)]
            tc = timed_graph(cfns)
            row["copy_us"] = round(tc * 1e3, 3)
            row["x_copy"] = round(t / tc, 3)
        if L["op"] == "gelu":
            # the same bytes through a purely elementwise kernel (dense
            # gelu_and_mul: no reduction): what streaming these rows costs
            sfns = [lambda x=arena_in[(i % win) * n_in:((i % win) + 1) * n_in].view(T, 2 * d),
                    o=arena_out[(i % win) * n_out:((i % win) + 1) * n_out].view(T, d):
                    ga.gelu_and_mul(x, d=d, out=o) for i in range(N)]
            ts = timed_graph(sfns)
            row["stream_us"] = round(ts * 1e3, 3)
            row["x_stream"] = round(t / ts, 3)
        rows.append(row)
    del arena_in, arena_out
    torch.cuda.synchronize()
    return rows, floor_ms * 1e3


def run_ours(args, world, rank, local):
    import torch
    import gated_activation_gb300 as ga

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    launches = workload_launches(args.only, args.only_silu)
    if args.native:   # profiling: the same launches in native-rounding mode
        for L in launches:
            L["op"] = "gelu_native"
    peaks = load_peaks()

    # inputs: seeded on the CPU and copied once to HBM; every launch has its own
    # input and output buffer, so nothing a launch reads was touched by the
    # step's earlier launches and consecutive steps are >2.5 GB apart
    host_in, dev_in, dev_out = {}, [], []
    for L in launches:
        key = (L["op"], L["T"], L["d"])
        L["key"] = key
        if key not in host_in:
            host_in[key] = rank_input(L, world, rank)
        dev_in.append(host_in[key].to(dev))
        dev_out.append(torch.empty((L["T"], L["d"]), dtype=torch.bfloat16, device=dev))
    for i, L in enumerate(launches):
        if L["op"] == "gelu":
            L["plan"] = ga.gelu_and_mul_sparse_plan(dev_in[i], d=L["d"], workspace=True)
            L["kernel"] = kernel_name(L["plan"])
        elif L["op"] == "gelu_native":
            L["plan"] = ga.gelu_and_mul_sparse_native_plan(dev_in[i], d=L["d"])
            L["kernel"] = kernel_name(L["plan"]) + " native"
        else:
            L["plan"] = None
            L["kernel"] = "silu_vec"
    for i, L in enumerate(launches):        # eager pass: loads modules, checks every call
        _launch(ga, L, dev_in[i], dev_out[i])
    torch.cuda.synchronize()

    profiling = bool(args.only or args.only_silu)
    shapes, floor_us = per_shape_times(ga, launches + ([] if profiling else extra_launches()),
                                       dev, peaks["hbm_gbs"]) \
        if not args.no_per_shape else ([], None)
    shapes_step = [r for r in shapes if r["op"] in ("gelu", "silu")]
    widened = [r for r in shapes if r["op"] not in ("gelu", "silu")]

    # the dominant kernel (largest total time per step, from the per-shape table
    # when present, else from bytes) runs as graph A, everything else as graph B
    def weight(i, L):
        if shapes_step:
            for r in shapes_step:
                if (r["op"], r["T"], r["d"], r["z"]) == (L["op"], L["T"], L["d"], L["z"]):
                    return r["us"]
        return L["bytes"]
    tot: dict[str, float] = {}
    for i, L in enumerate(launches):
        tot[L["kernel"]] = tot.get(L["kernel"], 0.0) + weight(i, L)
    dom = max(tot, key=tot.get)
    idx_a = [i for i, L in enumerate(launches) if L["kernel"] == dom]
    idx_b = [i for i, L in enumerate(launches) if L["kernel"] != dom]

    graphs = []
    for idx in (idx_a, idx_b):
        if not idx:
            graphs.append(None)
            continue
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in idx:
                _launch(ga, launches[i], dev_in[i], dev_out[i])
        graphs.append(g)

    def step(ev):
        ev[0].record()
        if graphs[0] is not None:
            graphs[0].replay()
        ev[1].record()
        if graphs[1] is not None:
            graphs[1].replay()
        ev[2].record()

    scratch_ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for _ in range(args.warmup):
        step(scratch_ev)
    torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world, local)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for k in range(args.steps):
            step(evs[k])
        torch.cuda.synchronize()
    barrier(world, local)

    step_ms = [e[0].elapsed_time(e[2]) for e in evs]
    dom_ms = [e[0].elapsed_time(e[1]) for e in evs]
    ms = max_over_ranks(statistics.fmean(step_ms), world, dev)
    bytes_step = sum(L["bytes"] for L in launches)
    value = world * bytes_step / (ms * 1e-3) / 1e9

    b_dom = sum(launches[i]["bytes"] for i in idx_a)
    t_dom = statistics.fmean(dom_ms) / len(idx_a)          # ms per launch
    achieved = (b_dom / len(idx_a)) / (t_dom * 1e-3) / 1e9
    traffic = load_traffic(dom, b_dom / len(idx_a))
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peaks["source"],
                "frac_of_spec_8TBps": round(achieved / SPEC_HBM_GBS, 4),
                "launches_per_step": len(idx_a), "bytes_per_launch_avg": b_dom // len(idx_a),
                "avg_launch_us": round(t_dom * 1e3, 3),
                "time_share": round(statistics.fmean(dom_ms) / statistics.fmean(step_ms), 4),
                "traffic": None if traffic is None else round(traffic)}

    e2e = run_e2e(args, launches, host_in, world, local, dev)
    e2e_direct = run_e2e_host_direct(args, launches, host_in, world, local, dev)
    link = link_ceiling(e2e["h2d_bytes_per_step"], e2e["d2h_bytes_per_step"], dev)
    for rec in (e2e, e2e_direct):
        rec["link_ceiling"] = link["value"]
        rec["frac_of_link"] = round(rec["value"] / world / link["value"], 4)
    e2e["link"] = link

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(launches, host_in)

    full = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_name(args, launches),
                       "launches_per_step": len(launches), "bytes_per_step": bytes_step,
                       "l2": "no flush: every launch has its own buffers (2.7 GB per step, "
                             "129 MB L2)",
                       "parallelism": f"rows sharded over {world} GPU(s), no collective",
                       "launch_floor_us": None if floor_us is None else round(floor_us, 3)},
            "roofline": roofline, "e2e": e2e, "e2e_host_direct": e2e_direct,
            "gpu_launches": len(launches) * args.steps,
            "clocks": clk.summary(), "per_shape": shapes_step, "widened_rows": widened}
    if cpu is not None:
        full["cpu_baseline"] = cpu
    if rank == 0:
        emit(full, args.detail)


STEP_WORKLOAD = ("gelu_and_mul_sparse T{1,8,64,256,1024,2048} x d{2048..32768} x z{0,1.645} "
                 "+ silu_and_mul M{1024,2048,4096,16384} d768")
# the shapes north of T*d = 2048*8192 (the bandwidth target) and the decode
# shapes (d = 8192) that the compact line summarises
TARGET_SHAPES = ((1024, 16384), (1024, 32768), (2048, 8192), (2048, 16384), (2048, 32768))
DECODE_SHAPES = ((1, 8192), (8, 8192), (64, 8192))
LINE_LIMIT = 2000


def workload_name(args, launches) -> str:
    """config.workload of both arms: the step's sweep, or the one shape that a
    profiling run (--only, --only-silu) times."""
    if args.only:
        return f"gelu_and_mul_sparse T={args.only[0]} d={args.only[1]}"
    if args.only_silu:
        return f"silu_and_mul M={args.only_silu} d={launches[0]['d']}"
    return STEP_WORKLOAD


def _shape_row(rows, T, d, z):
    for r in rows:
        if r["op"] == "gelu" and r["T"] == T and r["d"] == d and r["z"] == z:
            return r
    return None


def compact_line(full: dict) -> dict:
    """The one stdout line: the contract's keys and a short summary of the
    per-shape table (the full record goes to the --detail file)."""
    import workloads as W
    keep = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "gpu_launches")
    line = {k: full[k] for k in keep if k in full}
    c = full["config"]
    line["config"] = {k: c[k] for k in ("workload", "bytes_per_step", "l2", "parallelism",
                                        "launch_floor_us") if k in c}
    r = full["roofline"]
    line["roofline"] = {k: r[k] for k in ("bound", "kernel", "achieved", "peak", "unit", "frac",
                                          "traffic", "avg_launch_us", "peak_source") if k in r}
    e = full["e2e"]
    line["e2e"] = {k: e[k] for k in ("value", "unit", "h2d_bytes_per_step",
                                     "d2h_bytes_per_step", "frac_of_link") if k in e}
    if "e2e_host_direct" in full:
        line["e2e"]["host_direct"] = full["e2e_host_direct"]["value"]
    if "cpu_baseline" in full:
        cb = full["cpu_baseline"]
        line["cpu_baseline"] = {"value": cb["value"], "unit": cb["unit"], "cores": cb["cores"],
                                "kind": cb["kind"], "sample": cb.get("sample_short", cb["sample"]),
                                "one_core": cb.get("single_core", {}).get("value")}
    ck = full["clocks"]
    line["clocks"] = {"sm_mhz": ck.get("sm_mhz"), "sm_max_mhz": ck.get("sm_max_mhz"),
                      "reasons": ck.get("reasons", [])}
    rows = full.get("per_shape") or []
    if rows:
        # [us, fraction of 8 TB/s, time / device-to-device copy of the same bytes]
        tg = {}
        for T, d in TARGET_SHAPES:
            x = _shape_row(rows, T, d, W.Z95)
            if x:
                tg[f"{T}x{d}"] = [x["us"], x["frac_of_spec_8TBps"], x.get("x_copy")]
        line["targets"] = {"cols": ["us", "of_8TBps", "x_copy"], **tg}
        # [us, time / (empty launch + bytes at the measured peak), time / copy]
        dc = {}
        for T, d in DECODE_SHAPES:
            x = _shape_row(rows, T, d, W.Z95)
            if x:
                dc[f"{T}x{d}"] = [x["us"], x["x_floor"], x.get("x_copy")]
        line["decode"] = {"cols": ["us", "x_floor", "x_copy"], **dc}
        sl = {f"{x['T']}": [x["us"], x["x_floor"], x.get("x_copy")]
              for x in rows if x["op"] == "silu" and x["T"] in (1024, 2048)}
        if sl:
            line["silu_d768"] = {"cols": ["us", "x_floor", "x_copy"], **sl}
        gel = [x for x in rows if x["op"] == "gelu" and "stream_us" in x]
        if gel:
            fused = sum(x["us"] for x in gel)
            line["vs_copy"] = round(fused / sum(x["copy_us"] for x in gel), 3)
            line["vs_stream"] = round(fused / sum(x["stream_us"] for x in gel), 3)
    nat = [x for x in full.get("widened_rows") or []
           if x["op"] == "gelu_native" and x["T"] == 2048]
    if nat:
        line["native_2048x16384"] = {"us": nat[0]["us"], "frac": nat[0]["frac_of_measured"]}
    line["detail"] = "per-shape and widened-row tables: bench.py --detail FILE"
    return line


def emit(full: dict, detail_path: str | None) -> str:
    """Write the full record to `detail_path` (if given) and print the compact
    line, the last line of stdout.  Returns the printed text."""
    if detail_path:
        with open(detail_path, "w") as f:
            json.dump(full, f, indent=1)
    text = json.dumps(compact_line(full), separators=(",", ":"))
    if len(text) > LINE_LIMIT:
        print(f"warning: bench line is {len(text)} bytes", file=sys.stderr)
    print(text, flush=True)
    return text


def run_e2e(args, launches, host_in, world, local, dev) -> dict:
    """Same metric through the public call with host buffers: every step copies
    each launch's input host->device from pinned memory and its output back,
    pipelined over three streams (copy in / compute / copy out) so the copies
    of one launch overlap the kernels of its neighbours."""
    import torch
    import gated_activation_gb300 as ga
    n = len(launches)
    pin_in = {k: v.pin_memory() for k, v in host_in.items()}
    pin_out = [torch.empty((L["T"], L["d"]), dtype=torch.bfloat16).pin_memory() for L in launches]
    d_in = [torch.empty(tuple(host_in[L["key"]].shape), dtype=torch.bfloat16, device=dev)
            for L in launches]
    d_out = [torch.empty((L["T"], L["d"]), dtype=torch.bfloat16, device=dev) for L in launches]
    h2d = sum(host_in[L["key"]].numel() * 2 for L in launches)
    d2h = sum(L["T"] * L["d"] * 2 for L in launches)
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_k = [torch.cuda.Event() for _ in range(n)]
    ev_out = [torch.cuda.Event() for _ in range(n)]
    first = [True]

    def step():
        for i, L in enumerate(launches):
            with torch.cuda.stream(s_in):
                if not first[0]:
                    s_in.wait_event(ev_k[i])            # previous kernel i done reading
                d_in[i].copy_(pin_in[L["key"]], non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(ev_in[i])
                if not first[0]:
                    s_comp.wait_event(ev_out[i])        # previous output i copied out
                _launch(ga, L, d_in[i], d_out[i])
                ev_k[i].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_k[i])
                pin_out[i].copy_(d_out[i], non_blocking=True)
                ev_out[i].record(s_out)
        first[0] = False

    steps = max(1, min(args.steps, args.e2e_steps))
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()

    def timed() -> float:
        barrier(world, local)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for s in (s_in, s_comp, s_out):
            s.wait_event(a)
        for _ in range(steps):
            step()
        for s in (s_in, s_comp, s_out):
            cur.wait_stream(s)
        b.record(cur)
        torch.cuda.synchronize()
        barrier(world, local)
        return max_over_ranks(a.elapsed_time(b) / steps, world, dev)

    return _e2e_record(launches, world, steps, h2d, d2h, timed,
                       pipeline="3 streams: H2D / kernels / D2H, pinned host buffers")


E2E_REPS = 3


def _e2e_record(launches, world, steps, h2d, d2h, timed, **extra) -> dict:
    """Time `steps` end-to-end steps E2E_REPS times; the line carries the
    median (host memory traffic of other tenants moves single runs by 10-20%)."""
    reps = sorted(timed() for _ in range(E2E_REPS))
    ms = reps[len(reps) // 2]
    bytes_step = sum(L["bytes"] for L in launches)
    return {"value": round(world * bytes_step / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
            "ms_per_step": round(ms, 4), "steps": steps, "reps_ms": [round(r, 4) for r in reps],
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, **extra}


def link_ceiling(h2d: int, d2h: int, dev) -> dict:
    """What the CPU-GPU link itself carries for this step's mix of directions:
    copy-engine copies between page-locked host and device buffers, H2D and D2H
    at once on two streams in the step's byte ratio, plus each direction alone.
    The end-to-end figures above cannot beat the first number."""
    import torch
    unit = 256 << 20
    n_in = unit
    n_out = max(16, int(unit * d2h / max(h2d, 1)) // 16 * 16)
    hi = torch.empty(n_in, dtype=torch.uint8).pin_memory()
    ho = torch.empty(n_out, dtype=torch.uint8).pin_memory()
    di = torch.empty(n_in, dtype=torch.uint8, device=dev)
    do = torch.empty(n_out, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn, reps=5):
        fn()
        torch.cuda.synchronize()
        cur = torch.cuda.current_stream()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for s in (s1, s2):
            s.wait_event(a)
        for _ in range(reps):
            fn()
        for s in (s1, s2):
            cur.wait_stream(s)
        b.record(cur)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e-3 / reps

    def up():
        with torch.cuda.stream(s1):
            di.copy_(hi, non_blocking=True)

    def down():
        with torch.cuda.stream(s2):
            ho.copy_(do, non_blocking=True)

    def both():
        up()
        down()

    # best of three timings each: the ceiling is what the link can carry, and a
    # stray stall in one timing (seen once as half the one-direction rate for
    # both directions at once) must not lower it
    t_both, t_up, t_down = (min(timed(fn) for _ in range(3)) for fn in (both, up, down))
    return {"value": round((n_in + n_out) / t_both / 1e9, 1), "unit": "GB/s",
            "h2d_alone": round(n_in / t_up / 1e9, 1), "d2h_alone": round(n_out / t_down / 1e9, 1),
            "mix_h2d_to_d2h": round(h2d / max(d2h, 1), 3),
            "method": "cudaMemcpyAsync between page-locked host and device buffers, "
                      "both directions at once in the step's byte ratio"}


def run_e2e_host_direct(args, launches, host_in, world, local, dev) -> dict:
    """The same public calls given page-locked HOST buffers directly: the
    kernels read each input and write each output over the CPU-GPU link in
    place, so no copy is issued.  The bytes crossing the link per step equal
    the explicit-copy path's."""
    import torch
    import gated_activation_gb300 as ga
    pin_in = {k: v.pin_memory() for k, v in host_in.items()}
    pin_out = [torch.empty((L["T"], L["d"]), dtype=torch.bfloat16).pin_memory() for L in launches]
    h2d = sum(host_in[L["key"]].numel() * 2 for L in launches)
    d2h = sum(L["T"] * L["d"] * 2 for L in launches)

    def step():
        for i, L in enumerate(launches):
            _launch(ga, L, pin_in[L["key"]], pin_out[i])

    steps = max(1, min(args.steps, args.e2e_steps))
    for _ in range(2):
        step()
    torch.cuda.synchronize()

    def timed() -> float:
        barrier(world, local)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            step()
        b.record()
        torch.cuda.synchronize()
        barrier(world, local)
        return max_over_ranks(a.elapsed_time(b) / steps, world, dev)

    return _e2e_record(launches, world, steps, h2d, d2h, timed,
                       transfer="kernels read the inputs from and write the results to "
                                "page-locked host buffers in place (NVLink-C2C); no copy is issued")


# ----------------------------------------------------------------- the oracle on host cores
def _oracle_pass(o, launches, host_in, rows: int | None, nthreads: int = 0) -> int:
    """Run the fp64 oracle over (the first `rows` rows of) every launch on
    `nthreads` OpenMP threads (0: the default); return bytes."""
    import workloads as W
    done = 0
    for L in launches:
        x = host_in[L["key"]]
        r = x.shape[0] if rows is None else min(rows, x.shape[0])
        bits = W.to_bits(x[:r])
        if L["op"] in ("gelu", "gelu_native"):
            o.gelu_and_mul_sparse(bits, d=L["d"], z=L["z"], nthreads=nthreads)
            done += gelu_bytes(r, L["d"])
        else:
            o.silu_and_mul(bits, d=L["d"], nthreads=nthreads)
            done += silu_bytes(r, L["d"])
    return done


def cpu_model() -> str:
    """The host CPU's name, from /proc/cpuinfo where the kernel gives one."""
    import platform
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        info = ""
    for key in ("model name", "Model name", "Hardware"):
        for line in info.splitlines():
            if line.startswith(key) and ":" in line:
                return line.split(":", 1)[1].strip()
    parts = {line.split(":", 1)[0].strip(): line.split(":", 1)[1].strip()
             for line in info.splitlines() if ":" in line}
    if "CPU implementer" in parts:   # Arm: implementer and part number
        impl, part = parts["CPU implementer"], parts.get("CPU part", "?")
        # Arm Ltd (0x41) cores by their MIDR part numbers
        known = {"0xd0c": "Neoverse-N1", "0xd40": "Neoverse-V1", "0xd49": "Neoverse-N2",
                 "0xd4f": "Neoverse-V2", "0xd8e": "Neoverse-N3", "0xd84": "Neoverse-V3"}
        name = known.get(part.lower()) if impl.lower() == "0x41" else None
        return f"{platform.machine()} {name + ' ' if name else ''}(implementer {impl} part {part})"
    return platform.machine() or "unknown"


def cpu_baseline(launches, host_in) -> dict:
    """The oracle on the host cores: whole steps on every core until about 1 s of
    wall time (about 16 core-seconds on a 16-core host), and a bounded sample on
    one core (the first R rows of every launch, R doubled until a pass takes 4 s)."""
    import oracle
    o = oracle.default()
    cores = o.max_threads()
    passes, b, dt = 0, 0, 0.0
    t0 = time.perf_counter()
    while passes < 8 and (passes == 0 or dt < 1.0):
        b += _oracle_pass(o, launches, host_in, None)
        passes += 1
        dt = time.perf_counter() - t0
    R, b1, dt1 = 1, 0, 0.0
    while True:
        t1 = time.perf_counter()
        b1 = _oracle_pass(o, launches, host_in, R, nthreads=1)
        dt1 = max(time.perf_counter() - t1, 1e-6)
        if dt1 >= 4.0 or R >= 2048:
            break
        R *= 2
    _oracle_pass(o, launches[:1], host_in, 1, nthreads=cores)   # restore the thread count
    return {"value": round(b / dt / 1e9, 4), "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"{passes} full step(s) of the workload ({len(launches)} launches, "
                      f"{b // passes} algorithmic bytes each) through the fp64 C oracle, "
                      f"OpenMP over rows; {dt:.2f} s wall",
            "single_core": {"value": round(b1 / dt1 / 1e9, 4), "unit": UNIT, "cores": 1,
                            "sample": f"first min(T, {R}) rows of each launch ({b1} algorithmic "
                                      f"bytes); {dt1:.2f} s wall"},
            "sample_short": f"{passes} whole step(s) on {cores} threads, {dt:.1f} s",
            "cpu_model": cpu_model(), "nproc": os.cpu_count()}


def run_reference(args, world, rank):
    """The oracle as the reference arm (rank 0 only), on a bounded sample per step."""
    if rank != 0:
        return
    import oracle
    o = oracle.default()
    launches = workload_launches(args.only, args.only_silu)
    host_in = {}
    for L in launches:
        key = (L["op"], L["T"], L["d"])
        L["key"] = key
        if key not in host_in:
            host_in[key] = rank_input(L, 1, 0)
    # size the per-step sample (first R rows of every launch) so the run ends in minutes
    total = args.steps + args.warmup
    budget = float(os.environ.get("GATED_ACT_REF_BUDGET_S", "120"))
    t0 = time.perf_counter()
    _oracle_pass(o, launches, host_in, 1)
    t1 = max(time.perf_counter() - t0, 1e-4)
    R = 1
    while R < 2048 and (2 * R) * t1 * 1.2 * total < budget:
        R *= 2
    for _ in range(args.warmup):
        _oracle_pass(o, launches, host_in, R)
    times, nbytes = [], 0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        nbytes = _oracle_pass(o, launches, host_in, R)
        times.append(time.perf_counter() - t0)
    ms = statistics.fmean(times) * 1e3
    value = nbytes / (ms * 1e-3) / 1e9
    sample = (f"first min(T, {R}) rows of each of the {len(launches)} launches per step "
              f"({nbytes} algorithmic bytes), fp64 C oracle, OpenMP over rows")
    line = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": workload_name(args, launches),
                       "launches_per_step": len(launches),
                       "bytes_per_step": sum(L["bytes"] for L in launches),
                       "parallelism": "the oracle on rank 0's host cores",
                       "sample_rows_per_launch": R},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": o.max_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--detail", default=None, metavar="FILE",
                    help="also write the full record (per-shape and widened-row tables) here")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-shape", action="store_true",
                    help="skip the per-shape us/launch table (profiling runs)")
    ap.add_argument("--only", type=lambda s: tuple(float(v) if "." in v else int(v)
                                                   for v in s.split(",")), default=None,
                    help="time one gelu shape T,d[,z] (profiling); not a bench line")
    ap.add_argument("--native", action="store_true",
                    help="with --only: the launches in native-rounding mode (profiling)")
    ap.add_argument("--only-silu", type=int, default=None, metavar="M",
                    help="time one silu_and_mul row count M (profiling); not a bench line")
    a = ap.parse_args(argv)
    if a.warmup < 3 and a.impl == "ours":
        ap.error("--warmup must be >= 3")
    if a.native and not a.only:
        ap.error("--native needs --only T,d")
    return a


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_setup(args)
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
