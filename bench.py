"""Benchmark of the sparse MLA decode on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

One step is one decode call over the whole workload (every row, head and key:
gather, QK, row-max exchange, P, PV, split merge, epilogue). The default
workload is the throughput decode configuration, the largest of the five that
one GPU takes (B=256 rows, H=128 heads, top-k 2048 with every row full, a
1048576-row E4M3 pool of 604 MB, 1% of the pool rows scaled x8 before
quantisation); ``--config`` selects the others (tiny, latency, dsa, dense) and
the top-k select.

Timing: W untimed warm-up steps, then K timed steps between a barrier and
torch.cuda.synchronize() on both sides. L2 is flushed before every step by
writing a buffer twice the L2 size and then reading another one (no dirty
line is left to be written back during the decode); each decode call is
bracketed by CUDA
events on the stream it is launched on, so ``ms_per_step`` is decode time only.
``value`` is the gathered-KV throughput (576 bytes per (row, key)) of all
ranks; ``e2e`` is the same metric through the public call with the step's
inputs (q, indices, counts) copied from pinned host memory and its outputs
(out, lse) copied back inside the timed region (the cache pool is resident).

Besides the mean, the line gives the median of the flushed calls and, under
``graph``, the warm per-call time of 100 back-to-back calls captured in one
CUDA graph.

``--impl reference`` times the CPU oracle (the plain C restatement of the
method) on the host cores, the only reference this method has, on a fixed
row sample of the workload sized to about a second per step.

With N > 1 (torchrun, one process per GPU) every rank decodes its own replica
of the workload; there is no data-path collective. Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("sparse MLA decode µs/call and gathered-KV GB/s; % of HBM/FP8-MMA roofline")
UNIT = "GB/s"
DEFAULT_CONFIG = "throughput"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

WORKLOAD_TEXT = {
    "tiny": "tiny: B=2 rows, H=16, top-k 64, counts {64,37}, pool 4096x576 E4M3",
    "latency": "latency decode: B=5 verify rows, H=64, top-k 256 (counts U[200,256], one row "
               "count 0), pool 65536x576 E4M3",
    "dsa": "DSA decode: B=64, H=128, top-k 2048 (counts U[1,2048], 4 rows 0), pool 262144x576 "
           "E4M3, half of each row's keys from a 4096-row window",
    "throughput": "throughput decode: B=256, H=128, top-k 2048 full, pool 1048576x576 E4M3, "
                  "1% of rows x8",
    "dense": "dense-as-sparse: 32 requests x 4 causal rows, L U[1024,8192], H=16, pool "
             "262144x576 E4M3 shuffled",
    "topk": "top-k select (the decode's index producer): 64 rows of bf16 logits, row lengths "
            "U[1024,65536] of 65536, top-k 2048",
}
TOPK_METRIC = "top-k select µs/call and bf16-logit GB/s; % of HBM roofline"


def peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "source": "measured (MEASURED_PEAKS.json)"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "source": "fallback (no MEASURED_PEAKS.json)"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", rank=rank, world_size=world)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(value: float, world: int, device) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(bytes_per_rank: int, ms_local: float, world: int, device) -> tuple[float, float]:
    """Replicas: every rank moved bytes_per_rank in its own time; the job time
    is the slowest rank's and the job throughput all ranks' bytes over it.
    Returns (ms of the slowest rank, GB/s of the whole job)."""
    ms = reduce_max(ms_local, world, device)
    return ms, world * bytes_per_rank / (ms * 1e-3) / 1e9


def workload_stats(case) -> dict:
    from sparse_mla_decode_gb300 import inputs
    return inputs.algorithmic_bytes(case)


def run_gpu(args, world, rank, local) -> dict | None:
    import torch
    from sparse_mla_decode_gb300 import binding, inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    case = inputs.config(args.config)
    stats = workload_stats(case)
    bf16q = args.query == "bf16"
    if bf16q:  # the query is read as bf16: twice the bytes
        stats["total"] += stats["q"]
        stats["q"] *= 2
    # Rows that come in groups sharing one index list (the dense-as-sparse
    # workload's four causal rows per request) go through the grouped call
    # (the bf16-query call takes rows one by one).
    group = 1 if bf16q else ROW_GROUP.get(args.config, 1)
    plan = binding.smd_plan_grouped(case.B, case.H, case.W, group).as_dict()
    # Where the library's workspace plan (the spread kernel) applies, the
    # workspace entry point is timed with a workspace of the size it asks for.
    ws_bytes = binding.smd_workspace_bytes_grouped(case.B, case.H, case.W, group)
    if ws_bytes > 0:
        plan = binding.smd_plan_grouped(case.B, case.H, case.W, group, ws_bytes).as_dict()
    if bf16q:  # with the workspace it asks for (the spread kernel where it applies)
        ws_bytes = binding.smd_workspace_bytes_bf16q(case.B, case.H, case.W)
        plan = binding.smd_plan_bf16q(case.B, case.H, case.W, ws_bytes).as_dict()

    q = torch.from_numpy(case.q8).to(dev)
    q16 = torch.from_numpy(case.q16.view(np.int16)).to(dev).view(torch.bfloat16)
    kv = torch.from_numpy(case.kv8).to(dev)
    idx = torch.from_numpy(case.indices).to(dev)
    cnt = torch.from_numpy(case.counts).to(dev)
    out = torch.empty((case.B, case.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((case.B, case.H), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    # L2 flush: write a buffer twice the L2 size, then read another one of that
    # size, so that no dirty line of the write is left to be written back
    # inside the timed region.
    flush_w = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    flush = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream

    workspace = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    ptrs = (q.data_ptr(), kv.data_ptr(), case.N, idx.data_ptr(), case.W, cnt.data_ptr(),
            case.B, case.H, case.sm_scale, case.q_scale, case.k_scale, out.data_ptr(),
            lse.data_ptr(), status.data_ptr(), sptr)

    gptrs = ptrs[:8] + (group,) + ptrs[8:]
    bptrs = (q16.data_ptr(),) + ptrs[1:8] + (case.sm_scale, case.k_scale) + ptrs[11:]

    def decode(st=sptr):
        if bf16q and ws_bytes > 0:
            rc = binding.smd_sparse_mla_decode_bf16q_ws(*bptrs[:-1], workspace.data_ptr(), ws_bytes,
                                                        st)
        elif bf16q:
            rc = binding.smd_sparse_mla_decode_bf16q(*bptrs[:-1], st)
        elif group > 1 and ws_bytes > 0:
            rc = binding.smd_sparse_mla_decode_grouped_ws(*gptrs[:-1], workspace.data_ptr(),
                                                          ws_bytes, st)
        elif group > 1:
            rc = binding.smd_sparse_mla_decode_grouped(*gptrs[:-1], st)
        elif ws_bytes > 0:
            rc = binding.smd_sparse_mla_decode_ws(*ptrs[:-1], workspace.data_ptr(), ws_bytes, st)
        else:
            rc = binding.smd_sparse_mla_decode(*ptrs[:-1], st)
        if rc != 0:
            raise binding.SmdError(rc, "decode")

    def l2_flush():
        flush_w.zero_()
        torch.sum(flush, dim=0, out=flush_out)

    # Warm-up (also JIT/module load).
    for _ in range(max(args.warmup, 3)):
        l2_flush()
        decode()
    torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local).start() if rank == 0 else None
    time.sleep(0.2 if sampler else 0)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        l2_flush()
        starts[i].record(stream)
        decode()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t0
    clocks = sampler.stop() if sampler else None
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_local = float(np.mean(times_ms))
    ms, value = aggregate(stats["kv_gathered"], ms_local, world, dev)
    graph = graph_timing(decode, dev)

    # ---- end to end through the public call: host buffers in, host buffers out
    # (smd_sparse_mla_decode_host copies q, indices and counts in and out and
    # lse back, pipelined with the decode).
    hq = (torch.from_numpy(case.q16.view(np.int16)).view(torch.bfloat16) if bf16q
          else torch.from_numpy(case.q8)).pin_memory()
    hidx = torch.from_numpy(case.indices).pin_memory()
    hcnt = torch.from_numpy(case.counts).pin_memory()
    hout = torch.empty((case.B, case.H, 512), dtype=torch.bfloat16).pin_memory()
    hlse = torch.empty((case.B, case.H), dtype=torch.float32).pin_memory()
    host_ws_bytes = binding.smd_workspace_bytes_host(case.B, case.H, case.W, group, bf16q)
    host_ws = torch.empty(max(host_ws_bytes, 16), dtype=torch.uint8, device=dev)
    host_chunks = binding.smd_plan_host(case.B, case.H, case.W, group, bf16q)

    def e2e_step():
        binding.sparse_mla_decode_host(hq, kv, hidx, hcnt, case.sm_scale, case.q_scale,
                                       case.k_scale, out=hout, lse=hlse, status=status,
                                       workspace=host_ws, row_group=group, bf16_query=bf16q)

    for _ in range(max(args.warmup, 3)):
        l2_flush()
        e2e_step()
    torch.cuda.synchronize()
    e_starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        l2_flush()
        e_starts[i].record(stream)
        e2e_step()
        e_ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = reduce_max(float(np.mean([s.elapsed_time(e) for s, e in zip(e_starts, e_ends)])),
                        world, dev)
    h2d = hq.numel() * hq.element_size() + hidx.numel() * 4 + hcnt.numel() * 4
    d2h = hout.numel() * 2 + hlse.numel() * 4

    if rank != 0:
        return None

    pk = peaks()
    gathered = stats["kv_gathered"]
    e2e_value = world * gathered / (e2e_ms * 1e-3) / 1e9
    achieved = stats["total"] / (ms * 1e-3) / 1e9
    fp8_peak_tflops, fp8_source = fp8_peak(pk)
    t_hbm = stats["total"] / (pk["hbm_gbs"] * 1e9)
    t_tc = stats["flops"] / (fp8_peak_tflops * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    traffic = load_traffic(args.config + ("_bf16q" if bf16q else ""), plan["kernel"])
    roofline = {
        "bound": bound,
        "achieved": round(achieved, 2) if bound == "hbm" else round(
            stats["flops"] / (ms * 1e-3) / 1e12, 3),
        "peak": pk["hbm_gbs"] if bound == "hbm" else fp8_peak_tflops,
        "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
        "traffic": traffic,
        "kernel": KERNEL_FILES[plan["kernel"]][0],
        "algorithmic_bytes": stats["total"],
        "algorithmic_flops": stats["flops"],
        "t_roof_us": round(max(t_hbm, t_tc) * 1e6, 4),
        "frac_of_roofline_time": round(max(t_hbm, t_tc) / (ms * 1e-3), 5),
        "peak_source": pk["source"] + ("" if bound == "hbm" else "; " + fp8_source),
        "tensor_peak_tflops": round(fp8_peak_tflops, 1),
        "tensor_frac": round(stats["flops"] / (ms * 1e-3) / 1e12 / fp8_peak_tflops, 5),
        "tensor_peak_source": fp8_source,
    }
    roofline["frac"] = round(roofline["achieved"] / roofline["peak"], 5)
    cpu = (cpu_baseline(case, stats, args.cpu_seconds, bf16q) if world == 1 or rank == 0
           else None)
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 6),
        "us_per_call": round(ms * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("bf16 query split into E4M3 hi + lo; fp8_e4m3 cache (fp32 accumulate)"
                  if bf16q else "fp8_e4m3 (fp32 accumulate)"),
        "data": "synthetic (seeded numpy PCG64; E4M3 per-tensor scaled)",
        "config": {
            "workload": WORKLOAD_TEXT[args.config],
            "name": args.config,
            "query": "bf16 (split)" if bf16q else "e4m3 (per-tensor scale)",
            "B": case.B, "H": case.H, "top_k": case.W, "pool_rows": case.N,
            "gathered_keys": case.gathered_rows(), "unique_rows": case.unique_rows(),
            "l2": "flushed before every timed step (write of a 2x-L2 buffer, then read of another, outside the events)",
            "plan": plan,
            "row_group": group,
            "workspace_bytes": int(ws_bytes),
            "parallelism": f"replicas x{world}",
        },
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "us_per_call": round(e2e_ms * 1e3, 3),
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "call": "smd_sparse_mla_decode_host", "row_chunks": int(host_chunks),
                "note": ("q, indices, counts H2D from pinned memory and out, lse D2H inside the "
                         "call, pipelined with the decode over row chunks; pool resident")},
        # per step: the decode kernel, plus the query-split kernel before the
        # spread kernel when the query is bf16
        "gpu_launches": args.steps * (2 if bf16q and plan["kernel"] == 5 else 1),
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 4),
        "us_median": round(float(np.median(times_ms)) * 1e3, 3),
        "graph": graph,
    }
    return line


# Per kernel: its name and the sources compiled into it (the .cu first, then
# the headers with device code or layout constants); a committed ncu summary
# counts for the current build only if it hashes the same files.
_COMMON = ("smd_internal.h", "smd_ptx.cuh")
KERNEL_FILES = {
    1: ("mma_decode_kernel", ("smd_mma.cu",) + _COMMON + ("smd_qsplit.cuh", "smd_tree.cuh")),
    2: ("tc_decode_kernel", ("smd_tc.cu",) + _COMMON + ("smd_tc_common.cuh", "smd_tree.cuh")),
    3: ("group_decode_kernel", ("smd_group.cu",) + _COMMON + ("smd_tree.cuh",)),
    4: ("tcg_decode_kernel", ("smd_tcg.cu",) + _COMMON + ("smd_tc_common.cuh", "smd_tree.cuh")),
    5: ("tcs_decode_kernel", ("smd_tcs.cu",) + _COMMON + ("smd_qsplit.cuh", "smd_tc_common.cuh",
                                                          "smd_tree.cuh")),
    "topk": ("topk_select_kernel", ("smd_topk.cu",) + _COMMON),
}


def source_digest(sources) -> str:
    """sha256[:16] over the kernel's source files, concatenated in order."""
    import hashlib
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(ROOT, "sparse_mla_decode_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# Workloads whose rows come in groups sharing one index list (rows per group).
ROW_GROUP = {"dense": 4}


def load_traffic(config: str, kernel: int = 1):
    """dram bytes per launch from the committed ncu summary of this kernel and
    workload; None unless it was taken on the current kernel sources."""
    name, sources = KERNEL_FILES[kernel]
    path = os.path.join(ROOT, "profiles", f"{name}_{config}.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("kernel_source_sha256_16") != source_digest(sources):
            return None
        return d.get("dram_bytes_per_launch")
    except Exception:
        return None


def oracle_rows(case, flops_per_core: float) -> np.ndarray:
    """A fixed row sample of the workload small enough for one oracle call to
    do about flops_per_core per host core (the whole workload if it is)."""
    import oracle
    cores = oracle.max_threads()
    per_row = 2 * case.H * 1088 * max(1, int(case.clamped_counts().mean()))
    budget_rows = max(1, int(flops_per_core * cores / max(per_row, 1)))
    if budget_rows >= case.B:
        return np.arange(case.B)
    return np.sort(np.random.default_rng(0).choice(case.B, size=budget_rows, replace=False))


def cpu_baseline(case, stats, seconds: float, bf16q: bool = False) -> dict:
    """The oracle, as it stands, on the host cores: repeats of the whole
    workload (or a row sample of it) for about `seconds`."""
    import oracle
    cores = oracle.max_threads()
    # A row sample small enough for one call to take a few seconds at most.
    rows = oracle_rows(case, 4e9)
    q8, idx, cnt = case.q8[rows], case.indices[rows], case.counts[rows]
    gathered = 576 * int(np.clip(cnt.astype(np.int64), 0, case.W).sum())
    reps, t_total = 0, 0.0
    while t_total < seconds or reps < 1:
        t0 = time.perf_counter()
        if bf16q:
            oracle.sparse_mla_decode_bf16q(case.q16[rows], case.kv8, idx, cnt, case.sm_scale,
                                           case.k_scale, threads=cores)
        else:
            oracle.sparse_mla_decode(q8, case.kv8, idx, cnt, case.sm_scale, case.q_scale,
                                     case.k_scale, threads=cores)
        t_total += time.perf_counter() - t0
        reps += 1
    per_call = t_total / reps
    sample = (f"{len(rows)} of {case.B} rows, {reps} repeats" if len(rows) < case.B
              else f"whole workload, {reps} repeats")
    return {"value": round(gathered / per_call / 1e9, 6), "unit": UNIT, "cores": cores,
            "kind": "oracle", "sample": sample, "us_per_call_sample": round(per_call * 1e6, 1)}


def graph_timing(call, dev, calls: int = 100, replays: int = 5):
    """The secondary timing: `calls` back-to-back calls captured in one CUDA
    graph (no L2 flush between them: warm), replayed `replays` times; per-call
    microseconds of the fastest and the median replay. None if the capture
    fails."""
    import torch
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            call(side.cuda_stream)
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream(dev).cuda_stream
            for _ in range(calls):
                call(cs)
        g.replay()
        torch.cuda.synchronize()
        per = []
        for _ in range(replays):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            per.append(e0.elapsed_time(e1) * 1e3 / calls)
        return {"calls": calls, "us_per_call_min": round(min(per), 3),
                "us_per_call_median": round(float(np.median(per)), 3),
                "note": "warm back-to-back calls in one CUDA graph, no L2 flush"}
    except Exception as exc:  # a capture that fails (e.g. an older PyTorch) is reported, not fatal
        torch.cuda.synchronize()
        return {"error": str(exc)[:200]}


FP8_PEAK_FILE = os.path.join(ROOT, "profiles", "tcgen05_fp8_mma_peak.json")


def fp8_peak(pk: dict) -> tuple[float, str]:
    """The FP8 tensor peak (TFLOP/s) for the roofline: the committed
    measurement of the tcgen05 kind::f8f6f4 rate probe (bench.py
    --measure-fp8-peak on this part), else 2 x the measured BF16 peak."""
    try:
        with open(FP8_PEAK_FILE) as f:
            d = json.load(f)
        return float(d["tflops_median"]), ("builder-measured tcgen05 kind::f8f6f4 rate "
                                           "(profiles/tcgen05_fp8_mma_peak.json)")
    except Exception:
        return 2.0 * pk["bf16_tflops"], "FP8 = 2 x measured BF16 (nominal ratio)"


def measure_fp8_peak(args) -> dict:
    """The FP8 tensor-pipe rate probe (smd_fp8_mma_probe): one CTA per SM
    issuing M128 N256 K32 E4M3 MMAs back to back; CUDA events around each
    launch, clocks sampled meanwhile."""
    import torch
    from sparse_mla_decode_gb300 import binding
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    iters = 20000
    for _ in range(max(args.warmup, 3)):
        ctas = binding.smd_fp8_mma_probe(iters, status.data_ptr(), stream.cuda_stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(0).start()
    time.sleep(0.2)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for a, b in ev:
        a.record(stream)
        binding.smd_fp8_mma_probe(iters, status.data_ptr(), stream.cuda_stream)
        b.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    ms = [a.elapsed_time(b) for a, b in ev]
    flops = ctas * iters * 2 * 128 * 256 * 32
    return {"what": "tcgen05.mma.cta_group::1.kind::f8f6f4 E4M3 x E4M3 -> FP32, M128 N256 K32, "
                    "K-major SW128 operands, one issuing thread per SM, back to back",
            "ctas": ctas, "mma_per_cta": iters, "flops_per_launch": flops,
            "launches": args.steps, "ms_median": round(float(np.median(ms)), 4),
            "ms_min": round(float(np.min(ms)), 4),
            "tflops_median": round(flops / (float(np.median(ms)) * 1e-3) / 1e12, 1),
            "tflops_max": round(flops / (float(np.min(ms)) * 1e-3) / 1e12, 1),
            "clocks": clocks}


def topk_bytes(case) -> dict:
    """Bytes the select must move at least once: the logits before each row's
    end, the index list and the counts."""
    ends = np.minimum(np.maximum(case.row_ends.astype(np.int64), 0), case.L)
    read = 2 * int(ends.sum())
    written = 4 * case.B * case.K + 4 * case.B
    return {"logits": read, "out": written, "total": read + written}


def run_topk(args, world, rank, local) -> dict | None:
    """The select on the GPU: one step = one smd_topk_select call over every row."""
    import torch
    from sparse_mla_decode_gb300 import binding, inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    case = inputs.topk_config()
    stats = topk_bytes(case)
    x = torch.from_numpy(case.logits.view(np.int16)).to(dev).view(torch.bfloat16)
    ends = torch.from_numpy(case.row_ends).to(dev)
    idx = torch.empty((case.B, case.K), dtype=torch.int32, device=dev)
    cnt = torch.empty((case.B,), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush_w = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    flush = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    ptrs = (x.data_ptr(), case.L, ends.data_ptr(), case.B, case.L, case.K, idx.data_ptr(),
            cnt.data_ptr(), status.data_ptr(), stream.cuda_stream)

    def select(st=stream.cuda_stream):
        rc = binding.smd_topk_select(*ptrs[:-1], st)
        if rc != 0:
            raise binding.SmdError(rc, "select")

    def l2_flush():
        flush_w.zero_()
        torch.sum(flush, dim=0, out=flush_out)

    for _ in range(max(args.warmup, 3)):
        l2_flush()
        select()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local).start() if rank == 0 else None
    time.sleep(0.2 if sampler else 0)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        l2_flush()
        starts[i].record(stream)
        select()
        stops[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t0
    clocks = sampler.stop() if sampler else None
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    times_ms = [a.elapsed_time(b) for a, b in zip(starts, stops)]
    ms_local = float(np.mean(times_ms))
    ms, value = aggregate(stats["logits"], ms_local, world, dev)
    graph = graph_timing(select, dev)

    # end to end through smd_topk_select_host: logits and row ends in pinned
    # host memory, indices and counts back there (read and written in place)
    hx = torch.from_numpy(case.logits.view(np.int16)).pin_memory().view(torch.bfloat16)
    he = torch.from_numpy(case.row_ends).pin_memory()
    hidx = torch.empty((case.B, case.K), dtype=torch.int32).pin_memory()
    hcnt = torch.empty((case.B,), dtype=torch.int32).pin_memory()
    host_ws = torch.empty(max(binding.smd_workspace_bytes_topk_host(case.B, case.L, case.K), 16),
                          dtype=torch.uint8, device=dev)

    def e2e_step():
        binding.topk_select_host(hx, case.K, row_ends=he, indices=hidx, counts=hcnt,
                                 status=status, workspace=host_ws, device=dev)

    for _ in range(max(args.warmup, 3)):
        l2_flush()
        e2e_step()
    torch.cuda.synchronize()
    e_starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_stops = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        l2_flush()
        e_starts[i].record(stream)
        e2e_step()
        e_stops[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = reduce_max(float(np.mean([a.elapsed_time(b) for a, b in zip(e_starts, e_stops)])),
                        world, dev)
    if rank != 0:
        return None
    pk = peaks()
    achieved = stats["total"] / (ms * 1e-3) / 1e9
    cpu = topk_cpu_baseline(case, stats, args.cpu_seconds)
    return {
        "metric": TOPK_METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 6),
        "us_per_call": round(ms * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 keys (u16 integer compares)",
        "data": "synthetic (seeded numpy PCG64 normal logits, bf16)",
        "config": {"workload": WORKLOAD_TEXT["topk"], "name": "topk", "B": case.B, "L": case.L,
                   "top_k": case.K,
                   "l2": "flushed before every timed step (write of a 2x-L2 buffer, then read of another, outside the events)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 5),
                     "traffic": load_traffic("topk", "topk"),
                     "kernel": "topk_select_kernel", "algorithmic_bytes": stats["total"],
                     "t_roof_us": round(stats["total"] / (pk["hbm_gbs"] * 1e9) * 1e6, 4),
                     "peak_source": pk["source"]},
        "cpu_baseline": cpu,
        "e2e": {"value": round(world * stats["logits"] / (e2e_ms * 1e-3) / 1e9, 3), "unit": UNIT,
                "us_per_call": round(e2e_ms * 1e3, 3),
                "h2d_bytes_per_step": int(hx.numel() * 2 + he.numel() * 4),
                "d2h_bytes_per_step": int(hidx.numel() * 4 + hcnt.numel() * 4),
                "call": "smd_topk_select_host",
                "note": ("logits and row ends in pinned host memory, indices and counts back "
                         "there; the select reads and writes them in place over the C2C link")},
        "gpu_launches": args.steps, "clocks": clocks, "wall_s_timed_region": round(wall, 4),
        "us_median": round(float(np.median(times_ms)) * 1e3, 3), "graph": graph,
    }


def topk_cpu_baseline(case, stats, seconds: float) -> dict:
    """The select oracle (numpy, one core) on the whole workload, repeated for
    about `seconds`."""
    from oracle import topk as otk
    reps, t_total = 0, 0.0
    while t_total < seconds or reps < 1:
        t0 = time.perf_counter()
        otk.topk_select(case.logits, case.K, case.row_ends)
        t_total += time.perf_counter() - t0
        reps += 1
    per_call = t_total / reps
    return {"value": round(stats["logits"] / per_call / 1e9, 6), "unit": UNIT, "cores": 1,
            "kind": "oracle", "sample": f"whole workload, {reps} repeats",
            "us_per_call_sample": round(per_call * 1e6, 1)}


def run_topk_reference(args, world, rank) -> dict | None:
    if rank != 0:
        return None
    from oracle import topk as otk
    from sparse_mla_decode_gb300 import inputs
    case = inputs.topk_config()
    stats = topk_bytes(case)
    for _ in range(args.warmup):
        otk.topk_select(case.logits, case.K, case.row_ends)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        otk.topk_select(case.logits, case.K, case.row_ends)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * float(np.mean(times))
    value = stats["logits"] / (ms * 1e-3) / 1e9
    return {
        "impl": "reference", "metric": TOPK_METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "us_per_call": round(ms * 1e3, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u16 keys (numpy oracle)", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT["topk"], "name": "topk", "B": case.B, "L": case.L,
                   "top_k": case.K},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "whole workload per step"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_reference(args, world, rank) -> dict | None:
    if rank != 0:
        return None
    from sparse_mla_decode_gb300 import inputs
    case = inputs.config(args.config)
    import oracle
    cores = oracle.max_threads()
    # Each step decodes a fixed row sample sized to about a second of the
    # host's cores (the whole workload where that is less).
    rows = oracle_rows(case, 1e9)
    q8, q16, idx, cnt = case.q8[rows], case.q16[rows], case.indices[rows], case.counts[rows]
    gathered = 576 * int(np.clip(cnt.astype(np.int64), 0, case.W).sum())
    sample = (f"{len(rows)} of {case.B} rows (a fixed seeded sample) per step"
              if len(rows) < case.B else "whole workload per step")

    def step():
        if args.query == "bf16":
            oracle.sparse_mla_decode_bf16q(q16, case.kv8, idx, cnt, case.sm_scale, case.k_scale,
                                           threads=cores)
        else:
            oracle.sparse_mla_decode(q8, case.kv8, idx, cnt, case.sm_scale, case.q_scale,
                                     case.k_scale, threads=cores)

    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    ms = 1e3 * float(np.mean(times))
    value = gathered / (ms * 1e-3) / 1e9
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "us_per_call": round(ms * 1e3, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 sums, fp32 logits (CPU oracle)",
        "data": "synthetic (seeded numpy PCG64)",
        "config": {"workload": WORKLOAD_TEXT[args.config], "name": args.config,
                   "B": case.B, "H": case.H, "top_k": case.W, "pool_rows": case.N},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--impl", default="smd", choices=["smd", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--query", default="e4m3", choices=["e4m3", "bf16"],
                    help="bf16: the bf16-query call (query split into E4M3 hi + lo)")
    ap.add_argument("--measure-fp8-peak", action="store_true",
                    help="time the FP8 tensor-pipe rate probe instead (one JSON line)")
    args = ap.parse_args(argv)
    if args.measure_fp8_peak:
        print(json.dumps(measure_fp8_peak(args)), flush=True)
        return
    world, rank, local = (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
                          int(os.environ.get("LOCAL_RANK", "0")))
    if args.impl == "reference":
        if args.steps > 50 and args.config != "tiny":
            args.steps = 50
        line = (run_topk_reference(args, world, rank) if args.config == "topk"
                else run_reference(args, world, rank))
    else:
        world, rank, local = dist_setup(args.gpus)
        line = (run_topk(args, world, rank, local) if args.config == "topk"
                else run_gpu(args, world, rank, local))
    if line is not None:
        print(json.dumps(line), flush=True)
    if args.impl != "reference" and world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
