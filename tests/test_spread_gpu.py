"""GPU parity of the spread tcgen05 kernel (SMD_KERNEL_TC_SPREAD): a row's
keys in pieces of at most 512 over any CTAs of a cooperative grid, maxima
and partials through the caller's workspace. Checked against the CPU oracle,
bit for bit against the cluster kernel where both split a row the same way,
bit for bit across grid sizes (rounds and units that straddle two rounds),
on rows longer than a cluster holds, with a workspace full of garbage and
reused, and through the timeout path."""
from __future__ import annotations

import numpy as np
import pytest

from sparse_mla_decode_gb300 import inputs
from test_parity_gpu import check, oracle_decode, to_dev

pytestmark = pytest.mark.gpu

SPREAD = 5
TC = 2


def workspace_for(case, dev, fill=None):
    import torch
    from sparse_mla_decode_gb300 import binding
    # the spread plan's size, also where the automatic plan would not take it
    n = binding.smd_workspace_bytes_ex(case.B, case.H, case.W, dict(kernel=SPREAD))
    assert n > 0
    if fill is None:
        return torch.zeros(n, dtype=torch.uint8, device=dev)
    g = torch.Generator(device=dev).manual_seed(fill)
    return torch.randint(0, 256, (n,), dtype=torch.uint8, device=dev, generator=g)


def spread(case, dev, tensors=None, ws=None, plan=None, expect_status=0):
    import torch
    from sparse_mla_decode_gb300 import binding
    q, kv, idx, cnt = tensors if tensors is not None else to_dev(case, dev)
    ws = workspace_for(case, dev) if ws is None else ws
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    force = dict(kernel=SPREAD)
    force.update(plan or {})
    out, lse = binding.sparse_mla_decode(q, kv, idx, cnt, case.sm_scale, case.q_scale,
                                         case.k_scale, status=status, plan=force, workspace=ws)
    torch.cuda.synchronize()
    assert int(status.item()) == expect_status, binding.smd_status_str(int(status.item()))
    return out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy()


SHAPES = [
    # (B, H, W, N, counts): one piece, several, ragged piece boundaries, empty
    # rows, more than a cluster holds (W > 2048), H < 128 and H = 256.
    (4, 128, 2048, 20000, [2048, 1, 0, 1537]),
    (3, 128, 1100, 9000, [513, 1024, 1100]),
    (2, 128, 9000, 40000, [9000, 6001]),
    (3, 64, 1500, 8000, [1500, 700, 0]),
    (2, 256, 700, 5000, [700, 512]),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}H{s[1]}W{s[2]}" for s in SHAPES])
def test_spread_matches_the_oracle(cuda, shape):
    B, H, W, N, counts = shape
    case = inputs.random_case(B * 13 + W, B=B, H=H, W=W, N=N, counts=counts, heavy_frac=0.02)
    out_g, lse_g = spread(case, cuda)
    out_o, lse_o = oracle_decode(case)
    check(out_g, lse_g, out_o, lse_o, f"spread {shape}")


@pytest.mark.parametrize("H", [16, 48, 80, 112])
def test_head_counts_below_128_on_both_unit_widths(cuda, H):
    """Rows of fewer than 128 heads: up to 64 lanes take the narrow form of the
    spread kernel (partials strided by the lanes, slices landed by bulk copies
    for more than four pieces), more take the wide one (stride 128, padding
    lanes). Ragged rows of up to 9 pieces; the oracle, and the cluster kernel's
    bits on the rows it holds (up to 2048 keys)."""
    import torch
    from sparse_mla_decode_gb300 import binding
    counts = [4500, 1, 0, 2048, 1537, 700]
    case = inputs.random_case(900 + H, B=6, H=H, W=4500, N=30000, counts=counts, heavy_frac=0.02)
    t = to_dev(case, cuda)
    out_s, lse_s = spread(case, cuda, tensors=t)
    out_o, lse_o = oracle_decode(case)
    check(out_s, lse_s, out_o, lse_o, f"spread H={H}")
    # the rows the cluster kernel holds (W <= 2048), decoded by it alone
    short = [1, 2, 3, 4, 5]
    sub = inputs.Case(case.name, case.q8[short], case.kv8, case.indices[short, :2048],
                      case.counts[short], case.sm_scale, case.q_scale, case.k_scale,
                      q16=case.q16[short])
    st = torch.zeros(1, dtype=torch.int32, device=cuda)
    q, kv, idx, cnt = to_dev(sub, cuda)
    out_c, lse_c = binding.sparse_mla_decode(q, kv, idx, cnt, sub.sm_scale, sub.q_scale,
                                             sub.k_scale, status=st, plan=dict(kernel=TC))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    out_c = out_c.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(out_c, out_s[short]), f"H={H}: out bits, spread vs cluster"
    assert np.array_equal(lse_c.cpu().numpy().view(np.uint32), lse_s[short].view(np.uint32)), \
        f"H={H}: lse bits, spread vs cluster"


@pytest.mark.parametrize("W", [1024, 2048])
def test_spread_is_the_cluster_kernel_where_they_split_alike(cuda, W):
    """Full rows: the cluster kernel's split (W / 512) is every row's piece
    count, so both sum the same keys in the same order: identical bits."""
    case = inputs.random_case(70 + W, B=5, H=128, W=W, N=30000, counts=[W] * 5)
    t = to_dev(case, cuda)
    from test_parity_gpu import gpu_decode
    out_c, lse_c = gpu_decode(case, cuda, plan=dict(kernel=TC), tensors=t)
    out_s, lse_s = spread(case, cuda, tensors=t)
    assert np.array_equal(out_s, out_c)
    assert np.array_equal(lse_s.view(np.uint32), lse_c.view(np.uint32))


def test_spread_grid_changes_no_bits(cuda):
    """The grid only lays pieces out: with 5 CTAs most rows straddle two
    rounds; identical bits on every grid."""
    rng = np.random.default_rng(71)
    counts = rng.integers(0, 2049, size=24).tolist()
    counts[3] = 0
    counts[4] = 2048
    case = inputs.random_case(71, B=24, H=128, W=2048, N=60000, counts=counts)
    t = to_dev(case, cuda)
    ref = spread(case, cuda, tensors=t)
    for grid in (4, 5, 17, 152):
        out, lse = spread(case, cuda, tensors=t, plan=dict(grid_x=grid))
        assert np.array_equal(out, ref[0]), grid
        assert np.array_equal(lse.view(np.uint32), ref[1].view(np.uint32)), grid
    rows = [0, 3, 4, 11, 23]
    out_o, lse_o = oracle_decode(case, rows)
    check(ref[0][rows], ref[1][rows], out_o, lse_o, "spread grid")


def test_spread_longest_rows(cuda):
    """32 pieces of 512 keys: the longest row the spread kernel takes."""
    case = inputs.random_case(72, B=1, H=128, W=16384, N=70000, counts=[16384])
    out_g, lse_g = spread(case, cuda)
    out_o, lse_o = oracle_decode(case)
    check(out_g, lse_g, out_o, lse_o, "spread 16384")


def test_spread_workspace_garbage_and_reuse(cuda):
    """The workspace needs no initialisation, and every call leaves its flags
    consumed: random bytes first, then the same workspace twice more."""
    case = inputs.random_case(73, B=6, H=128, W=2048, N=30000, counts=[2048, 900, 1, 0, 1600, 513])
    t = to_dev(case, cuda)
    ws = workspace_for(case, cuda, fill=5)
    first = spread(case, cuda, tensors=t, ws=ws)
    for _ in range(2):
        again = spread(case, cuda, tensors=t, ws=ws)
        assert np.array_equal(again[0], first[0])
        assert np.array_equal(again[1].view(np.uint32), first[1].view(np.uint32))
    out_o, lse_o = oracle_decode(case)
    check(first[0], first[1], out_o, lse_o, "spread garbage workspace")


def test_spread_timeout_is_reported_and_the_context_survives(cuda):
    from sparse_mla_decode_gb300 import binding
    case = inputs.random_case(74, B=3, H=128, W=1500, N=9000, counts=[1500, 600, 1200])
    t = to_dev(case, cuda)
    ws = workspace_for(case, cuda)
    spread(case, cuda, tensors=t, ws=ws, plan=dict(inject_stall=1, wait_budget_us=2000),
           expect_status=binding.SMD_ERR_TIMEOUT)
    ws.zero_()
    out_g, lse_g = spread(case, cuda, tensors=t, ws=ws)
    out_o, lse_o = oracle_decode(case)
    check(out_g, lse_g, out_o, lse_o, "spread after a timeout")


def test_dsa_config_through_the_workspace_call(cuda):
    """The DSA workload at full size through smd_sparse_mla_decode_ws, in the
    plan bench.py times; every row against the oracle."""
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.config("dsa")
    t = to_dev(case, cuda)
    nbytes = binding.smd_workspace_bytes(case.B, case.H, case.W)
    assert binding.smd_plan_ws(case.B, case.H, case.W).kernel == SPREAD
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=cuda)
    from test_parity_gpu import gpu_decode
    out_g, lse_g = gpu_decode(case, cuda, tensors=t, workspace=ws)
    out_o, lse_o = oracle_decode(case)  # every row
    check(out_g, lse_g, out_o, lse_o, "dsa spread")
    n = case.clamped_counts()
    assert np.all(np.isneginf(lse_g[n == 0])) and np.all(np.isfinite(lse_g[n > 0]))


def test_spread_call_replays_in_a_cuda_graph(cuda):
    """Captured once, replayed three times on one workspace: every replay gives
    the eager call's bits (each call's flags are zeroed by their readers, so
    the captured tokens never meet a stale flag)."""
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.random_case(75, B=5, H=128, W=2048, N=30000, counts=[2048, 700, 0, 1537, 2000])
    q, kv, idx, cnt = to_dev(case, cuda)
    ws = workspace_for(case, cuda, fill=7)
    ref = spread(case, cuda, tensors=(q, kv, idx, cnt), ws=ws)
    out = torch.empty((case.B, case.H, 512), dtype=torch.bfloat16, device=cuda)
    lse = torch.empty((case.B, case.H), dtype=torch.float32, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    side = torch.cuda.Stream(cuda)
    side.wait_stream(torch.cuda.current_stream(cuda))
    with torch.cuda.stream(side):
        binding.sparse_mla_decode(q, kv, idx, cnt, case.sm_scale, case.q_scale, case.k_scale,
                                  out=out, lse=lse, status=status, plan=dict(kernel=SPREAD),
                                  workspace=ws)
    torch.cuda.current_stream(cuda).wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.sparse_mla_decode(q, kv, idx, cnt, case.sm_scale, case.q_scale, case.k_scale,
                                  out=out, lse=lse, status=status, plan=dict(kernel=SPREAD),
                                  workspace=ws)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), ref[0])
        assert np.array_equal(lse.cpu().numpy().view(np.uint32), ref[1].view(np.uint32))
