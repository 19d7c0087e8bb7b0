"""The tracing build (-DSMD_TRACE, SMD_TRACE_BUILD=1): its kernels give the
normal build's bits, and every traced kernel stamps its phases in order.
Each check runs in a child process, since a process loads one variant."""
from __future__ import annotations

import os
import subprocess
import sys

import numpy as np
import pytest

from sparse_mla_decode_gb300 import inputs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, numpy as np, torch
from sparse_mla_decode_gb300 import binding, inputs
name, G, out_path = sys.argv[1], int(sys.argv[2]), sys.argv[3]
case = inputs.config(name)
dev = torch.device("cuda", 0)
q, kv, idx, cnt = (torch.from_numpy(a).to(dev) for a in (case.q8, case.kv8, case.indices, case.counts))
nb = binding.smd_workspace_bytes_grouped(case.B, case.H, case.W, G)
ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device=dev) if nb > 0 else None
st = torch.zeros(1, dtype=torch.int32, device=dev)
kern = binding.smd_plan_grouped(case.B, case.H, case.W, G, nb).kernel
traced = binding.smd_trace_enabled() == 1
if traced:
    assert binding.smd_trace_clear(kern) == 0
out, lse = binding.sparse_mla_decode(q, kv, idx, cnt, case.sm_scale, case.q_scale, case.k_scale,
                                     status=st, workspace=ws, row_group=G)
torch.cuda.synchronize()
assert int(st.item()) == 0
stamps = np.zeros(8192 * 32, np.uint64)
if traced:
    assert binding.smd_trace_read(kern, stamps.ctypes.data, stamps.size) == 0
np.savez(out_path, out=out.view(torch.int16).cpu().numpy(), lse=lse.view(torch.int32).cpu().numpy(),
         stamps=stamps, kern=kern)
"""


def run_child(name, G, traced, path):
    env = dict(os.environ)
    env["SMD_TRACE_BUILD"] = "1" if traced else "0"
    r = subprocess.run([sys.executable, "-c", CHILD, name, str(G), path], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    return np.load(path)


# Phase slots that every CTA (or item) of these workloads stamps, in order.
ORDERED = {1: [0, 1, 2, 3, 4, 5, 7], 2: [0, 1, 2, 3, 4, 5, 6, 7, 8, 9], 5: [0, 1, 2, 3, 4, 5, 8]}


@pytest.mark.parametrize("name,G", [("latency", 1), ("throughput", 1), ("dsa", 1), ("dense", 4)])
def test_tracing_build_bits_and_phase_order(cuda, tmp_path, name, G):
    plain = run_child(name, G, False, str(tmp_path / "plain.npz"))
    traced = run_child(name, G, True, str(tmp_path / "traced.npz"))
    assert np.array_equal(plain["out"], traced["out"]), f"{name}: out bits"
    assert np.array_equal(plain["lse"], traced["lse"]), f"{name}: lse bits"
    t = traced["stamps"].reshape(8192, 32).astype(np.int64)
    rows = t[t[:, 0] != 0]
    assert len(rows) > 0
    cols = ORDERED[int(traced["kern"])]
    seq = rows[:, cols]
    assert (seq > 0).all(), f"{name}: a phase without a stamp"
    assert (np.diff(seq, axis=1) >= 0).all(), f"{name}: phases out of order"
    # The last slot holds the SM each row ran on.
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert ((rows[:, 31] >= 0) & (rows[:, 31] < sms)).all(), f"{name}: SM ids"


def test_phases_tool_prints_the_timeline(cuda):
    env = dict(os.environ)
    r = subprocess.run([sys.executable, "-m", "sparse_mla_decode_gb300.phases", "--config", "latency",
                        "--reps", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    assert "mma_decode_kernel" in r.stdout and "| end |" in r.stdout
    assert "SMs that ran rows" in r.stdout
