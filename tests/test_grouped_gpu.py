"""GPU parity of the grouped decode (smd_sparse_mla_decode_grouped): rows in
groups of 2 or 4 that share one index list, gathered once per group, on both
group kernels (tcgen05 where G x H is 32 or 64 lanes, warp MMA always). Each
row's result is checked against the CPU oracle (which knows nothing about
groups), against the per-row decode, across ring sizes (identical bits) and
splits, and the contract check and the timeout path are exercised."""
from __future__ import annotations

import numpy as np
import pytest

from sparse_mla_decode_gb300 import inputs
from test_parity_gpu import check, oracle_decode, to_dev

pytestmark = pytest.mark.gpu

MMA_GROUP = 3
TC_GROUP = 4


def kernels(G, H, W):
    """The group kernels that take these shapes."""
    return [MMA_GROUP, TC_GROUP] if G * H in (32, 64) and W <= 8192 else [MMA_GROUP]


def grouped(case, dev, G, plan=None, tensors=None, expect_status=0):
    import torch
    from sparse_mla_decode_gb300 import binding
    q, kv, idx, cnt = tensors if tensors is not None else to_dev(case, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = binding.sparse_mla_decode(q, kv, idx, cnt, case.sm_scale, case.q_scale,
                                         case.k_scale, status=status, plan=plan, row_group=G)
    torch.cuda.synchronize()
    assert int(status.item()) == expect_status, binding.smd_status_str(int(status.item()))
    return out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy()


SHAPES = [
    # (R, G, H, W, N, counts): ragged chunk and split boundaries; empty rows;
    # the longest list in any row of the group, not only the last.
    (3, 4, 16, 700, 9000, None),
    (2, 4, 16, 129, 3000, [1, 64, 65, 129, 0, 0, 0, 0]),
    (2, 4, 32, 300, 5000, [300, 12, 299, 5, 64, 63, 62, 61]),
    (4, 2, 16, 2048, 20000, None),
    (3, 2, 48, 97, 2000, [97, 96, 0, 33, 1, 2]),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"R{s[0]}G{s[1]}H{s[2]}W{s[3]}" for s in SHAPES])
def test_grouped_matches_the_oracle_and_the_per_row_decode(cuda, shape):
    R, G, H, W, N, counts = shape
    case = inputs.grouped_case(10 * R + G + W, R, G, H, W, N, counts)
    t = to_dev(case, cuda)
    out_o, lse_o = oracle_decode(case)
    from test_parity_gpu import gpu_decode
    out_r, lse_r = gpu_decode(case, cuda, tensors=t)
    for kern in kernels(G, H, W):
        out_g, lse_g = grouped(case, cuda, G, plan=dict(kernel=kern), tensors=t)
        check(out_g, lse_g, out_o, lse_o, f"grouped kernel {kern} {shape}")
        check(out_g, lse_g, out_r, lse_r, f"grouped kernel {kern} vs per-row {shape}")


@pytest.mark.parametrize("kern,split", [(MMA_GROUP, s) for s in (1, 2, 4, 8, 16)] +
                         [(TC_GROUP, s) for s in (4, 8, 16)])
def test_grouped_every_split(cuda, kern, split):
    """1100 keys are 9 leaves of 128: the warp-MMA group kernel with groups of
    4 keeps at most 4 leaves a CTA (two TMEM stack levels of 64 floats), so
    splits 1 and 2 are refused as a plan, not computed."""
    from sparse_mla_decode_gb300 import binding
    case = inputs.grouped_case(41, 2, 4, 16, 1100, 12000, [1100, 1099, 700, 2, 0, 300, 301, 64])
    t = to_dev(case, cuda)
    if kern == MMA_GROUP and split < 4:
        with pytest.raises(binding.SmdError) as e:
            grouped(case, cuda, 4, plan=dict(kernel=kern, split=split), tensors=t)
        assert e.value.status == binding.SMD_ERR_PLAN
        return
    out_o, lse_o = oracle_decode(case)
    out_g, lse_g = grouped(case, cuda, 4, plan=dict(kernel=kern, split=split), tensors=t)
    check(out_g, lse_g, out_o, lse_o, f"grouped kernel {kern} split {split}")


def test_tc_groups_up_to_8192_keys(cuda):
    """Sixteen CTAs per cluster, 512 keys each, ragged last CTAs."""
    case = inputs.grouped_case(46, 2, 4, 16, 8192, 40000, [8192, 8191, 8190, 8189, 5000, 5001, 4999, 0])
    t = to_dev(case, cuda)
    out_g, lse_g = grouped(case, cuda, 4, plan=dict(kernel=TC_GROUP), tensors=t)
    out_o, lse_o = oracle_decode(case)
    check(out_g, lse_g, out_o, lse_o, "tc groups 8192")


def test_grouped_ring_size_changes_no_bits(cuda):
    """The warp-MMA group kernel's ring size (64-key slots) only lays work
    out: identical bits."""
    case = inputs.grouped_case(42, 3, 4, 16, 900, 10000)
    t = to_dev(case, cuda)
    ref = grouped(case, cuda, 4, plan=dict(kernel=MMA_GROUP, split=4, window=64), tensors=t)
    for window in (128, 192, 256):
        out, lse = grouped(case, cuda, 4, plan=dict(kernel=MMA_GROUP, split=4, window=window),
                           tensors=t)
        assert np.array_equal(out, ref[0]), window
        assert np.array_equal(lse.view(np.uint32), ref[1].view(np.uint32)), window


def test_group_of_one_is_the_per_row_decode(cuda):
    case = inputs.grouped_case(43, 2, 4, 16, 200, 3000)
    t = to_dev(case, cuda)
    from test_parity_gpu import gpu_decode
    out_1, lse_1 = grouped(case, cuda, 1, tensors=t)
    out_r, lse_r = gpu_decode(case, cuda, tensors=t)
    assert np.array_equal(out_1, out_r)
    assert np.array_equal(lse_1.view(np.uint32), lse_r.view(np.uint32))


@pytest.mark.parametrize("kern", [MMA_GROUP, TC_GROUP])
def test_rows_that_do_not_share_their_list_are_reported(cuda, kern):
    """One row of the second group reads a key its group's longest list does
    not hold: the call reports SMD_ERR_GROUP; the first group is unaffected."""
    from sparse_mla_decode_gb300 import binding
    case = inputs.grouped_case(44, 2, 4, 16, 256, 4000, [256, 255, 254, 253, 200, 256, 100, 7])
    case.indices[6, 50] = (case.indices[5, 50] + 1) % case.N
    t = to_dev(case, cuda)
    out_g, lse_g = grouped(case, cuda, 4, plan=dict(kernel=kern), tensors=t,
                           expect_status=binding.SMD_ERR_GROUP)
    out_o, lse_o = oracle_decode(case, rows=[0, 1, 2, 3])
    check(out_g[:4], lse_g[:4], out_o, lse_o, f"grouped kernel {kern}, the group that keeps the contract")


@pytest.mark.parametrize("kern", [MMA_GROUP, TC_GROUP])
def test_grouped_timeout_is_reported_and_the_context_survives(cuda, kern):
    from sparse_mla_decode_gb300 import binding
    case = inputs.grouped_case(45, 2, 4, 16, 600, 4000)
    t = to_dev(case, cuda)
    grouped(case, cuda, 4, plan=dict(kernel=kern, inject_stall=1, wait_budget_us=2000, split=4),
            tensors=t, expect_status=binding.SMD_ERR_TIMEOUT)
    out_g, lse_g = grouped(case, cuda, 4, plan=dict(kernel=kern), tensors=t)
    out_o, lse_o = oracle_decode(case)
    check(out_g, lse_g, out_o, lse_o, f"grouped kernel {kern} after a timeout")


def test_dense_as_sparse_full_size_sampled_rows(cuda):
    """The dense-as-sparse workload at full size through the grouped call, in
    the plan bench.py times and on the other group kernel; sampled requests
    against the oracle."""
    case = inputs.config("dense")
    t = to_dev(case, cuda)
    rows = np.concatenate([4 * r + np.arange(4) for r in range(0, 32, 4)])  # 8 requests, 32 rows
    out_o, lse_o = oracle_decode(case, rows)
    for plan in (None, dict(kernel=MMA_GROUP)):
        out_g, lse_g = grouped(case, cuda, 4, plan=plan, tensors=t)
        check(out_g[rows], lse_g[rows], out_o, lse_o, f"dense grouped sampled {plan}")


# ---- row groups on the spread tcgen05 kernel (smd_sparse_mla_decode_grouped_ws) ----------

SPREAD = 5


def grouped_ws(case, dev, G, tensors=None, plan=None, expect_status=0):
    """The grouped workspace call; the spread kernel unless `plan` says otherwise."""
    import torch
    from sparse_mla_decode_gb300 import binding
    # the spread kernel's size: one unit per group, like B / G rows of 128 heads
    nb = binding.smd_workspace_bytes_ex(case.B // G, 128, case.W, dict(kernel=SPREAD))
    assert nb > 0
    ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
    plan = dict(kernel=SPREAD) if plan is None else plan
    q, kv, idx, cnt = tensors if tensors is not None else to_dev(case, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = binding.sparse_mla_decode(q, kv, idx, cnt, case.sm_scale, case.q_scale,
                                         case.k_scale, status=status, plan=plan, row_group=G,
                                         workspace=ws)
    torch.cuda.synchronize()
    assert int(status.item()) == expect_status, binding.smd_status_str(int(status.item()))
    return out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy()


@pytest.mark.parametrize("shape", SHAPES, ids=[f"R{s[0]}G{s[1]}H{s[2]}W{s[3]}" for s in SHAPES])
def test_groups_on_the_spread_kernel(cuda, shape):
    R, G, H, W, N, counts = shape
    case = inputs.grouped_case(10 * R + G + W, R, G, H, W, N, counts)
    t = to_dev(case, cuda)
    out_o, lse_o = oracle_decode(case)
    out_g, lse_g = grouped_ws(case, cuda, G, tensors=t)
    check(out_g, lse_g, out_o, lse_o, f"grouped spread {shape}")
    from sparse_mla_decode_gb300 import binding
    # with a workspace the automatic plan takes the spread kernel wherever it
    # fits (G x H <= 128 lanes, lists of at most 16384 keys)
    assert binding.smd_plan_grouped(case.B, H, W, G, 1 << 40).kernel == SPREAD


def test_groups_on_the_spread_kernel_grid_changes_no_bits(cuda):
    case = inputs.grouped_case(47, 6, 4, 16, 5000, 40000,
                               [5000, 4999, 4000, 12, 0, 0, 0, 0, 700, 701, 702, 703,
                                2048, 2047, 10, 1, 3000, 3000, 3000, 3000, 513, 1, 0, 512])
    t = to_dev(case, cuda)
    ref = grouped_ws(case, cuda, 4, tensors=t)
    for grid in (10, 31, 152):
        out, lse = grouped_ws(case, cuda, 4, tensors=t, plan=dict(kernel=SPREAD, grid_x=grid))
        assert np.array_equal(out, ref[0]), grid
        assert np.array_equal(lse.view(np.uint32), ref[1].view(np.uint32)), grid
    out_o, lse_o = oracle_decode(case)
    check(ref[0], ref[1], out_o, lse_o, "grouped spread grid")


def test_groups_on_the_spread_kernel_report_a_broken_contract(cuda):
    from sparse_mla_decode_gb300 import binding
    case = inputs.grouped_case(44, 2, 4, 16, 256, 4000, [256, 255, 254, 253, 200, 256, 100, 7])
    case.indices[6, 50] = (case.indices[5, 50] + 1) % case.N
    t = to_dev(case, cuda)
    out_g, lse_g = grouped_ws(case, cuda, 4, tensors=t, expect_status=binding.SMD_ERR_GROUP)
    out_o, lse_o = oracle_decode(case, rows=[0, 1, 2, 3])
    check(out_g[:4], lse_g[:4], out_o, lse_o, "grouped spread, the group that keeps the contract")


def test_groups_longer_than_the_row_group_kernel_takes(cuda):
    """Lists of 12000 keys: the workspace call's automatic plan is the spread
    kernel (the row-group tcgen05 kernel stops at 8192)."""
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.grouped_case(48, 2, 4, 16, 12000, 60000, [12000, 11999, 9000, 3, 500, 0, 0, 0])
    nb = binding.smd_workspace_bytes_grouped(case.B, case.H, case.W, 4)
    assert nb > 0 and binding.smd_plan_grouped(case.B, 16, 12000, 4, nb).kernel == SPREAD
    q, kv, idx, cnt = to_dev(case, cuda)
    ws = torch.zeros(nb, dtype=torch.uint8, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    out, lse = binding.sparse_mla_decode(q, kv, idx, cnt, case.sm_scale, case.q_scale,
                                         case.k_scale, status=status, row_group=4, workspace=ws)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    out_o, lse_o = oracle_decode(case)
    check(out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy(), out_o, lse_o,
          "grouped spread 12000")


def test_dense_as_sparse_on_the_spread_kernel_sampled(cuda):
    case = inputs.config("dense")
    out_g, lse_g = grouped_ws(case, cuda, 4)
    rows = np.concatenate([4 * r + np.arange(4) for r in range(2, 32, 4)])  # 8 other requests
    out_o, lse_o = oracle_decode(case, rows)
    check(out_g[rows], lse_g[rows], out_o, lse_o, "dense grouped spread")
