"""GPU parity of the tcgen05 kernel (128 heads per CTA, TMA gather4, TMEM
accumulators) against the CPU oracle, at chunk and split boundaries, and
with fewer than 128 heads (the remaining TMEM lanes are padding)."""
from __future__ import annotations

import numpy as np
import pytest

from sparse_mla_decode_gb300 import inputs
from test_parity_gpu import check, gpu_decode, oracle_decode, to_dev

pytestmark = pytest.mark.gpu

TC = 2
MMA = 1

SHAPES = [
    # (B, H, W, N, counts): counts straddle the 32-key k-steps, the 128-key
    # chunks, the 512-key CTA share and the split boundaries.
    (4, 128, 129, 3000, [1, 127, 128, 129]),
    (3, 128, 512, 5000, [0, 511, 512]),
    (4, 128, 1024, 9000, [513, 1000, 1024, 2]),
    (3, 128, 2048, 20000, [2048, 2047, 1537]),
    (2, 256, 300, 4000, [300, 31]),
    (5, 128, 40, 200, [40, 0, -3, 33, 7]),
]


@pytest.fixture(scope="module")
def workspace(cuda):
    import torch
    from sparse_mla_decode_gb300 import binding
    nbytes = binding.smd_workspace_bytes_ex(256, 128, 2048, dict(kernel=2))
    return torch.empty(nbytes // 4, dtype=torch.float32, device=cuda)


@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}H{s[1]}W{s[2]}" for s in SHAPES])
def test_tc_random_shapes(cuda, shape, workspace):
    """Both exchanges of the split partials (DSMEM, and L2 through the
    workspace) match the oracle and give identical bits (same sum order)."""
    B, H, W, N, counts = shape
    case = inputs.random_case(300 + W, B=B, H=H, W=W, N=N, counts=counts, heavy_frac=0.02)
    t = to_dev(case, cuda)
    out_g, lse_g = gpu_decode(case, cuda, dict(kernel=TC), tensors=t)
    out_o, lse_o = oracle_decode(case)
    check(out_g, lse_g, out_o, lse_o, f"tc {shape}")
    out_w, lse_w = gpu_decode(case, cuda, dict(kernel=TC), tensors=t, workspace=workspace)
    check(out_w, lse_w, out_o, lse_o, f"tc l2 {shape}")
    assert np.array_equal(out_w, out_g)
    assert np.array_equal(lse_w.view(np.uint32), lse_g.view(np.uint32))


def test_tc_l2_exchange_over_many_waves(cuda, workspace):
    """800 CTAs on 152 SMs: workspace slots are reused wave after wave."""
    case = inputs.random_case(320, B=200, H=128, W=2048, N=50000, heavy_frac=0.01)
    t = to_dev(case, cuda)
    out_w, lse_w = gpu_decode(case, cuda, dict(kernel=TC), tensors=t, workspace=workspace)
    out_g, lse_g = gpu_decode(case, cuda, tensors=t)
    assert np.array_equal(out_w, out_g)
    assert np.array_equal(lse_w.view(np.uint32), lse_g.view(np.uint32))
    rows = [0, 57, 199]
    out_o, lse_o = oracle_decode(case, rows)
    check(out_w[rows], lse_w[rows], out_o, lse_o, "tc l2 waves")


@pytest.mark.parametrize("split", [1, 2, 4])
def test_tc_every_split(cuda, split, workspace):
    case = inputs.random_case(310, B=3, H=128, W=512, N=6000, counts=[512, 300, 0],
                              heavy_frac=0.02)
    for ws in (None, workspace):
        out_g, lse_g = gpu_decode(case, cuda, dict(kernel=TC, split=split), workspace=ws)
        out_o, lse_o = oracle_decode(case)
        check(out_g, lse_g, out_o, lse_o, f"tc split {split} ws {ws is not None}")


def test_tc_and_mma_kernels_agree(cuda):
    case = inputs.random_case(311, B=2, H=128, W=700, N=5000, counts=[700, 260], heavy_frac=0.05)
    t = to_dev(case, cuda)
    out_t, lse_t = gpu_decode(case, cuda, dict(kernel=TC), tensors=t)
    out_m, lse_m = gpu_decode(case, cuda, dict(kernel=MMA), tensors=t)
    check(out_t, lse_t, out_m, lse_m, "tc vs mma")


def test_tc_is_deterministic(cuda):
    case = inputs.random_case(312, B=4, H=128, W=2048, N=30000, counts=[2048, 1000, 5, 0])
    t = to_dev(case, cuda)
    a = gpu_decode(case, cuda, dict(kernel=TC), tensors=t)
    b = gpu_decode(case, cuda, dict(kernel=TC), tensors=t)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32))


def test_tc_timeout_reports_status(cuda):
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.random_case(313, B=2, H=128, W=600, N=3000, counts=[600, 10])
    q, kv, idx, cnt = to_dev(case, cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    binding.sparse_mla_decode(q, kv, idx, cnt, case.sm_scale, case.q_scale, case.k_scale,
                              status=status,
                              plan=dict(kernel=TC, inject_stall=1, wait_budget_us=2000))
    torch.cuda.synchronize()
    assert int(status.item()) == binding.SMD_ERR_TIMEOUT
    out_g, lse_g = gpu_decode(case, cuda, dict(kernel=TC), tensors=(q, kv, idx, cnt))
    out_o, lse_o = oracle_decode(case)
    check(out_g, lse_g, out_o, lse_o, "tc after timeout")


FEW_HEADS = [
    # (B, H, W, N, counts, split): H < 128 fills part of the 128 TMEM lanes; the
    # query tile then reaches into the next row's heads (or past the tensor).
    (5, 64, 256, 65536, [256, 200, 0, 231, 17], 1),
    (3, 16, 64, 4096, [64, 37, 1], 1),
    (4, 48, 600, 7000, [600, 513, 129, 0], 2),
    (2, 112, 1100, 9000, [1100, 64], 4),
]


@pytest.mark.parametrize("shape", FEW_HEADS, ids=[f"B{s[0]}H{s[1]}W{s[2]}S{s[5]}" for s in FEW_HEADS])
def test_tc_fewer_than_128_heads(cuda, shape, workspace):
    """The padding lanes' results are never stored; the real ones match the
    oracle, and the warp-MMA kernel, for both exchanges."""
    B, H, W, N, counts, split = shape
    case = inputs.random_case(330 + H, B=B, H=H, W=W, N=N, counts=counts, heavy_frac=0.02)
    t = to_dev(case, cuda)
    out_o, lse_o = oracle_decode(case)
    out_g, lse_g = gpu_decode(case, cuda, dict(kernel=TC, split=split), tensors=t)
    check(out_g, lse_g, out_o, lse_o, f"tc few heads {shape}")
    if split > 1:
        out_w, lse_w = gpu_decode(case, cuda, dict(kernel=TC, split=split), tensors=t,
                                  workspace=workspace)
        assert np.array_equal(out_w, out_g)
        assert np.array_equal(lse_w.view(np.uint32), lse_g.view(np.uint32))
    out_m, lse_m = gpu_decode(case, cuda, dict(kernel=MMA), tensors=t)
    check(out_g, lse_g, out_m, lse_m, f"tc vs mma few heads {shape}")
