"""Per-phase timeline of one decode call, from the tracing build's stamps.

    python -m sparse_mla_decode_gb300.phases --config throughput [--reps 5]

Loads the tracing variant of the library (SMD_TRACE_BUILD=1; built in-tree on
first use, -DSMD_TRACE), runs the workload's decode as bench.py does (inputs
resident on the device, the workspace the call asks for, the L2 flushed
before every call), and prints, for the last call, the median and 90th
percentile over the kernel's CTAs (the spread kernel: over its items, per
round) of the time from the CTA's first stamp to the end of each phase, plus
the span of the launch, then how the SMs were used: the SMs that ran rows,
the share of the span an SM was running one, the gaps between consecutive
rows on one SM (a CTA's exit to the next CTA's first stamp there; the spread
kernel: one item's end to the next one's start) and the idle time after an
SM's last row. The stamps are %globaltimer readings taken by one thread at
the end of each phase, and %smid at entry (smd_trace.cuh); the tracing build
computes the same results as the normal one.
"""
from __future__ import annotations

import argparse
import os

import numpy as np

PHASES = {
    1: ["entry", "keys staged", "query landed", "logits", "row maximum", "PV", "partials in", "end"],
    2: ["entry", "keys staged", "own maximum", "row maximum", "P", "O", "partials pushed",
        "partials in", "merged", "end"],
    5: ["item start", "keys staged", "own maximum", "row maximum", "P", "O", "partials written",
        "partials in", "end", "sums merged", "columns merged", "output staged"],
}
KERNEL_NAME = {1: "mma_decode_kernel", 2: "tc_decode_kernel", 5: "tcs_decode_kernel"}
ROW_GROUP = {"dense": 4}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--config", default="throughput",
                    choices=["tiny", "latency", "dsa", "throughput", "dense"])
    ap.add_argument("--reps", type=int, default=5)
    args = ap.parse_args(argv)
    os.environ["SMD_TRACE_BUILD"] = "1"

    import torch
    from . import binding, inputs

    if binding.smd_trace_enabled() != 1:
        raise SystemExit("the loaded library is not the tracing build")
    dev = torch.device("cuda", 0)
    case = inputs.config(args.config)
    G = ROW_GROUP.get(args.config, 1)
    q, kv, idx, cnt = (torch.from_numpy(a).to(dev) for a in (case.q8, case.kv8, case.indices,
                                                               case.counts))
    nb = binding.smd_workspace_bytes_grouped(case.B, case.H, case.W, G)
    ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device=dev) if nb > 0 else None
    plan = binding.smd_plan_grouped(case.B, case.H, case.W, G, nb).as_dict()
    kern = plan["kernel"]
    if kern not in PHASES:
        raise SystemExit(f"kernel {kern} of this workload keeps no phase table")
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(2 * 129 * 2 ** 20 // 4, device=dev)
    times = []
    for rep in range(args.reps):
        flush.zero_()
        if rep == args.reps - 1:
            torch.cuda.synchronize()
            assert binding.smd_trace_clear(kern) == binding.SMD_OK
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        binding.sparse_mla_decode(q, kv, idx, cnt, case.sm_scale, case.q_scale, case.k_scale,
                                  status=st, workspace=ws, row_group=G)
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1e3)
    if int(st.item()) != 0:
        raise SystemExit(f"device status {binding.smd_status_str(int(st.item()))}")
    rows, slots = 8192, 32
    buf = np.zeros(rows * slots, np.uint64)
    assert binding.smd_trace_read(kern, buf.ctypes.data, buf.size) == binding.SMD_OK
    t = buf.reshape(rows, slots).astype(np.int64)
    names = PHASES[kern]
    print(f"{KERNEL_NAME[kern]} on the {args.config} workload: plan {plan}")
    print(f"event time of the traced call {times[-1]:.1f} us (median of {args.reps}: "
          f"{np.median(times):.1f} us)")
    groups = [("all CTAs", np.arange(rows))]
    if kern == 5:
        groups = [(f"round {r}", np.arange(r, rows, 4)) for r in range(4)]
    for label, sel in groups:
        tt = t[sel]
        tt = tt[tt[:, 0] != 0]
        if len(tt) == 0:
            continue
        start = tt[:, 0]
        end_col = names.index("end")
        span = (tt[:, end_col].max() - start.min()) / 1e3 if (tt[:, end_col] != 0).any() else float("nan")
        print(f"\n{label}: {len(tt)} rows, span {span:.1f} us (first start to last end)")
        print("| phase ended | median (us) | p90 (us) |")
        print("|---|---|---|")
        for k, name in enumerate(names):
            v = tt[:, k]
            okm = v != 0
            if okm.sum() == 0:
                continue
            d = (v[okm] - start[okm]) / 1e3
            print(f"| {name} | {np.median(d):.2f} | {np.percentile(d, 90):.2f} |")
    occupancy(t, names.index("end"))
    return 0


def occupancy(t: np.ndarray, end_col: int) -> None:
    """Per-SM use over the launch: rows with both stamps, grouped by the SM
    id in the last slot."""
    t = t[(t[:, 0] != 0) & (t[:, end_col] != 0)]
    if len(t) == 0:
        return
    t0, t1 = t[:, 0].min(), t[:, end_col].max()
    span = (t1 - t0) / 1e3
    sm = t[:, -1]
    busy, gaps, tail = [], [], []
    for s in np.unique(sm):
        rows = t[sm == s]
        rows = rows[np.argsort(rows[:, 0])]
        ent, end = rows[:, 0], rows[:, end_col]
        busy.append((end - ent).sum() / 1e3)
        gaps.extend(((ent[1:] - end[:-1]) / 1e3).tolist())
        tail.append((t1 - end[-1]) / 1e3)
    busy = np.array(busy)
    print(f"\nSMs that ran rows: {len(busy)}; an SM ran a row {100 * busy.mean() / span:.1f} % of the "
          f"span on average (busy {busy.mean():.1f} of {span:.1f} us)")
    if gaps:
        g = np.array(gaps)
        print(f"gaps between consecutive rows on one SM: {len(g)}, median {np.median(g):.2f} us, "
              f"mean {g.mean():.2f} us, {g.sum() / len(busy):.1f} us per SM")
    print(f"idle after an SM's last row: median {np.median(tail):.1f} us, mean {np.mean(tail):.1f} us")


if __name__ == "__main__":
    raise SystemExit(main())
