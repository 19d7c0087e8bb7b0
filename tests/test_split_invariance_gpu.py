"""The GPU is bit-exact to itself across split and tile variants.

Each kernel family cuts a row's keys into fixed leaves by list position (512
keys on the tcgen05 kernels; 64 * ceil(n / 1024) keys, at most 16 leaves, on
the warp-MMA kernels), sums every leaf from zero in one order and combines the
leaves by one pairwise tree. A plan (cluster size, CTAs per row, the spread
over a cooperative grid, 16-head tiles, the resident-key window, the DSMEM or
L2 exchange, the batch a row comes in) only decides which CTA evaluates which
subtree, so every plan the library accepts gives the same output and LSE bits
for a row. The two families (warp MMA, tcgen05) agree within the parity
tolerance only. Ragged counts put leaf, chunk and k-step boundaries inside
CTAs, and empty CTAs beside full ones.
"""
from __future__ import annotations

import numpy as np
import pytest

from sparse_mla_decode_gb300 import inputs
from test_parity_gpu import check, gpu_decode, oracle_decode, to_dev

pytestmark = pytest.mark.gpu

MMA, TC, MMA_GROUP, TC_GROUP, SPREAD = 1, 2, 3, 4, 5


def same_bits(a, b, what):
    assert np.array_equal(a[0], b[0]), f"{what}: out bits differ"
    assert np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32)), f"{what}: lse bits differ"


def try_decode(case, dev, plan, tensors, workspace=None, row_group=1):
    """The decode under a forced plan, or None when the plan is refused
    (SMD_ERR_PLAN: it does not fit this shape)."""
    import torch
    from sparse_mla_decode_gb300 import binding
    q, kv, idx, cnt = tensors
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    try:
        out, lse = binding.sparse_mla_decode(q, kv, idx, cnt, case.sm_scale, case.q_scale,
                                             case.k_scale, status=status, plan=plan,
                                             workspace=workspace, row_group=row_group)
    except binding.SmdError as e:
        assert e.status == binding.SMD_ERR_PLAN, e
        return None
    torch.cuda.synchronize()
    assert int(status.item()) == 0, binding.smd_status_str(int(status.item()))
    return out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy()


def spread_workspace(case, dev, G=1):
    import torch
    from sparse_mla_decode_gb300 import binding
    B = case.B // G if G > 1 else case.B
    H = 128 if G > 1 else case.H
    n = binding.smd_workspace_bytes_ex(B, H, case.W, dict(kernel=SPREAD))
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=dev)


def l2_workspace(dev):
    import torch
    from sparse_mla_decode_gb300 import binding
    n = binding.smd_workspace_bytes_ex(256, 128, 2048, dict(kernel=TC))
    return torch.zeros(n, dtype=torch.uint8, device=dev)


MMA_CASES = [
    # (B, H, W, N, counts): 16 leaves of 64 keys; 16 of 128; 4 of 64; 16 of 192
    # (leaves that are not a power-of-two multiple of the 64-key chunk).
    (8, 32, 1000, 9000, [1000, 999, 513, 64, 63, 1, 0, 700]),
    (4, 16, 2048, 20000, [2048, 1025, 1024, 130]),
    (5, 64, 256, 4000, [256, 255, 129, 0, 33]),
    (3, 16, 3000, 20000, [3000, 2049, 191]),
]


@pytest.mark.parametrize("shape", MMA_CASES, ids=[f"B{s[0]}H{s[1]}W{s[2]}" for s in MMA_CASES])
def test_warp_mma_every_split_tile_and_window(cuda, shape):
    B, H, W, N, counts = shape
    case = inputs.random_case(900 + W, B=B, H=H, W=W, N=N, counts=counts, heavy_frac=0.02)
    t = to_dev(case, cuda)
    ref, ran = None, set()
    for split in (1, 2, 4, 8, 16):
        for tiles in (1, 2):
            for window in (64, 128, 256):
                got = try_decode(case, cuda, dict(kernel=MMA, split=split, tiles=tiles,
                                                  window=window), t)
                if got is None:
                    continue
                ran.add(split)
                if ref is None:
                    ref = got
                    out_o, lse_o = oracle_decode(case)
                    check(got[0], got[1], out_o, lse_o, f"mma {shape}")
                else:
                    same_bits(got, ref, f"mma split {split} tiles {tiles} window {window}")
    assert len(ran) >= 4, ran
    # the automatic plan too
    same_bits(gpu_decode(case, cuda, tensors=t), ref, "mma automatic plan")


def test_warp_mma_bf16_query_every_split(cuda):
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.random_case(905, B=4, H=32, W=1000, N=8000, counts=[1000, 517, 64, 0])
    q16 = torch.from_numpy(case.q16.view(np.int16)).to(cuda).view(torch.bfloat16)
    kv, idx, cnt = (torch.from_numpy(a).to(cuda) for a in (case.kv8, case.indices, case.counts))
    ref = None
    for split in (1, 2, 4, 8, 16):
        status = torch.zeros(1, dtype=torch.int32, device=cuda)
        try:
            out, lse = binding.sparse_mla_decode_bf16q(q16, kv, idx, cnt, case.sm_scale,
                                                       case.k_scale, status=status,
                                                       plan=dict(kernel=MMA, split=split))
        except binding.SmdError as e:
            assert e.status == binding.SMD_ERR_PLAN
            continue
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = (out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy())
        if ref is None:
            ref = got
        else:
            same_bits(got, ref, f"bf16 query split {split}")
    assert ref is not None


TC_CASES = [
    # (B, H, W, N, counts, splits): one leaf; two; three of four (an empty CTA).
    (4, 128, 512, 6000, [512, 300, 1, 0], (1, 2, 4)),
    (6, 128, 1024, 9000, [1024, 1000, 513, 512, 511, 0], (2, 4)),
    (4, 128, 2048, 20000, [2048, 1537, 1100, 129], (4,)),
    (3, 64, 1100, 7000, [1100, 600, 0], (4,)),
]


@pytest.mark.parametrize("shape", TC_CASES, ids=[f"B{s[0]}H{s[1]}W{s[2]}" for s in TC_CASES])
def test_tcgen05_every_split_exchange_and_the_spread_kernel(cuda, shape):
    B, H, W, N, counts, splits = shape
    case = inputs.random_case(910 + W + H, B=B, H=H, W=W, N=N, counts=counts, heavy_frac=0.02)
    t = to_dev(case, cuda)
    l2 = l2_workspace(cuda)
    ref = None
    for split in splits:
        for ws in (None, l2):
            got = try_decode(case, cuda, dict(kernel=TC, split=split), t, workspace=ws)
            assert got is not None, split
            if ref is None:
                ref = got
                out_o, lse_o = oracle_decode(case)
                check(got[0], got[1], out_o, lse_o, f"tc {shape}")
            else:
                same_bits(got, ref, f"tc split {split} l2 {ws is not None}")
    # the spread kernel: pieces over a cooperative grid, partials through L2
    sw = spread_workspace(case, cuda)
    for grid in (0, 3, 7, 152):
        plan = dict(kernel=SPREAD) if grid == 0 else dict(kernel=SPREAD, grid_x=grid)
        got = try_decode(case, cuda, plan, t, workspace=sw)
        if got is None:
            continue
        same_bits(got, ref, f"spread grid {grid}")


def test_tcgen05_spread_kernel_long_rows_every_grid(cuda):
    """Rows of up to 32 leaves (only the spread kernel takes them): the tree is
    five levels deep; grids of 32 .. 152 CTAs give one set of bits."""
    case = inputs.random_case(920, B=3, H=128, W=16384, N=70000, counts=[16384, 9001, 4097])
    t = to_dev(case, cuda)
    sw = spread_workspace(case, cuda)
    ref = try_decode(case, cuda, dict(kernel=SPREAD), t, workspace=sw)
    for grid in (32, 45, 100):
        same_bits(try_decode(case, cuda, dict(kernel=SPREAD, grid_x=grid), t, workspace=sw), ref,
                  f"spread grid {grid}")
    rows = [1, 2]
    out_o, lse_o = oracle_decode(case, rows)
    check(ref[0][rows], ref[1][rows], out_o, lse_o, "spread 32 leaves")


def _subset(case, rows):
    rows = np.asarray(rows)
    return inputs.Case(case.name + "-sub", case.q8[rows], case.kv8, case.indices[rows],
                       case.counts[rows], case.sm_scale, case.q_scale, case.k_scale)


BATCH_CASES = [
    # (H, W, N): tcgen05 (cluster; spread with a workspace), warp MMA
    # (latency-like), warp MMA with 16 leaves of 128 keys.
    (128, 2048, 60000),
    (64, 256, 20000),
    (16, 2000, 30000),
]


@pytest.mark.parametrize("shape", BATCH_CASES, ids=[f"H{s[0]}W{s[1]}" for s in BATCH_CASES])
def test_rows_give_the_same_bits_in_any_batch(cuda, shape):
    """The same rows decoded inside a batch of 200 and of 4: the plans differ
    (split, cluster vs spread kernel), the bits do not."""
    from sparse_mla_decode_gb300 import binding
    H, W, N = shape
    rng = np.random.default_rng(930 + H)
    counts = rng.integers(0, W + 1, size=200)
    counts[1] = 0
    counts[2] = W
    big = inputs.random_case(930 + H, B=200, H=H, W=W, N=N, counts=counts.tolist(), heavy_frac=0.01)
    small = _subset(big, [0, 1, 2, 3])
    tb, ts = to_dev(big, cuda), to_dev(small, cuda)
    pb, ps = binding.smd_plan(200, H, W), binding.smd_plan(4, H, W)
    out_b, lse_b = gpu_decode(big, cuda, tensors=tb)
    out_s, lse_s = gpu_decode(small, cuda, tensors=ts)
    same_bits((out_b[:4], lse_b[:4]), (out_s, lse_s), f"batch 200 vs 4 {shape}")
    if H % 128 != 0:
        assert (pb.split, pb.grid_x) != (ps.split, ps.grid_x)  # the plans differ
    else:
        # with a workspace the small batch goes to the spread kernel
        wb, ws_ = spread_workspace(big, cuda), spread_workspace(small, cuda)
        assert binding.smd_plan_ws(4, H, W).kernel == SPREAD
        assert binding.smd_plan_ws(200, H, W).kernel == TC
        got_b = gpu_decode(big, cuda, tensors=tb, workspace=wb)
        got_s = gpu_decode(small, cuda, tensors=ts, workspace=ws_)
        same_bits((got_b[0][:4], got_b[1][:4]), got_s, "workspace calls, batch 200 vs 4")
        same_bits(got_s, (out_s, lse_s), "spread vs cluster, batch 4")
    out_o, lse_o = oracle_decode(small)
    check(out_s, lse_s, out_o, lse_o, f"batch subset {shape}")


def test_row_groups_every_split_and_kernel_layout(cuda):
    """Groups of 4 rows sharing one list (ragged counts): the tcgen05 group
    kernel at every cluster size it takes, the spread kernel with groups at
    several grids; and the warp-MMA group kernel at every split and ring it
    takes."""
    case = inputs.grouped_case(940, 2, 4, 16, 1100, 12000, [1100, 1099, 700, 2, 0, 300, 301, 64])
    t = to_dev(case, cuda)
    ref = None
    for split in (4, 8, 16):
        got = try_decode(case, cuda, dict(kernel=TC_GROUP, split=split), t, row_group=4)
        assert got is not None
        if ref is None:
            ref = got
            out_o, lse_o = oracle_decode(case)
            check(got[0], got[1], out_o, lse_o, "tc groups")
        else:
            same_bits(got, ref, f"tc groups split {split}")
    sw = spread_workspace(case, cuda, G=4)
    for grid in (0, 5, 30):
        plan = dict(kernel=SPREAD) if grid == 0 else dict(kernel=SPREAD, grid_x=grid)
        got = try_decode(case, cuda, plan, t, workspace=sw, row_group=4)
        assert got is not None
        same_bits(got, ref, f"spread groups grid {grid}")
    mref, ran = None, set()
    for split in (1, 2, 4, 8, 16):
        for window in (64, 128):
            got = try_decode(case, cuda, dict(kernel=MMA_GROUP, split=split, window=window), t,
                             row_group=4)
            if got is None:
                continue
            ran.add(split)
            if mref is None:
                mref = got
                check(got[0], got[1], ref[0], ref[1], "warp-MMA groups vs tcgen05 groups")
            else:
                same_bits(got, mref, f"warp-MMA groups split {split} window {window}")
    assert ran >= {4, 8, 16}, ran


def test_row_groups_on_tcgen05_are_the_per_row_decode(cuda):
    """Within the tcgen05 family a row sees exactly its own leaves whether it
    is decoded alone (one row's 16 heads on the per-row kernel) or in a group
    of 4 sharing one list, so the bits agree."""
    case = inputs.grouped_case(941, 2, 4, 16, 1100, 12000, [1100, 1099, 700, 2, 0, 300, 301, 64])
    t = to_dev(case, cuda)
    per_row = try_decode(case, cuda, dict(kernel=TC), t)
    grouped = try_decode(case, cuda, dict(kernel=TC_GROUP), t, row_group=4)
    same_bits(grouped, per_row, "tcgen05 groups vs per row")
