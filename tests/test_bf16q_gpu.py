"""GPU parity of the bf16-query decode (smd_sparse_mla_decode_bf16q): each
(row, head) query split on the GPU into E4M3 hi + lo at its own power-of-two
scale, both halves through QK. Checked against the oracle's bf16-query
decode, bit for bit across layout variants, bit for bit against the E4M3
decode where the query is E4M3 already (lo = 0), on the full latency and
DSA workloads, and through the timeout path."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from sparse_mla_decode_gb300 import inputs
from test_parity_gpu import check, gpu_decode, to_dev

pytestmark = pytest.mark.gpu


def q16_dev(case, dev):
    import torch
    return torch.from_numpy(case.q16.view(np.int16)).to(dev).view(torch.bfloat16)


def bf16q_decode(case, dev, plan=None, tensors=None, q16=None, expect_status=0):
    import torch
    from sparse_mla_decode_gb300 import binding
    _, kv, idx, cnt = tensors if tensors is not None else to_dev(case, dev)
    q = q16 if q16 is not None else q16_dev(case, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = binding.sparse_mla_decode_bf16q(q, kv, idx, cnt, case.sm_scale, case.k_scale,
                                               status=status, plan=plan)
    torch.cuda.synchronize()
    assert int(status.item()) == expect_status, binding.smd_status_str(int(status.item()))
    return out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy()


def oracle_bf16q(case, rows=None):
    if rows is None:
        o16, _, lse, _ = oracle.sparse_mla_decode_bf16q(case.q16, case.kv8, case.indices,
                                                        case.counts, case.sm_scale, case.k_scale)
        return o16, lse.astype(np.float32)
    rows = np.asarray(rows)
    o16, _, lse, _ = oracle.sparse_mla_decode_bf16q(case.q16[rows], case.kv8, case.indices[rows],
                                                    case.counts[rows], case.sm_scale, case.k_scale)
    return o16, lse.astype(np.float32)


SHAPES = [
    (2, 16, 64, 4096, [64, 37]),
    (5, 64, 256, 20000, [256, 200, 0, 255, 1]),
    (3, 128, 700, 9000, [700, 1, 513]),
    (2, 32, 3000, 20000, [3000, 1999]),   # several windows per CTA
    (4, 48, 129, 2000, [129, 128, 0, -3]),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}H{s[1]}W{s[2]}" for s in SHAPES])
def test_bf16q_matches_the_oracle(cuda, shape):
    B, H, W, N, counts = shape
    case = inputs.random_case(B * 31 + W, B=B, H=H, W=W, N=N, counts=counts, heavy_frac=0.02)
    out_g, lse_g = bf16q_decode(case, cuda)
    out_o, lse_o = oracle_bf16q(case)
    check(out_g, lse_g, out_o, lse_o, f"bf16q {shape}")


def test_bf16q_layout_variants_are_bit_identical(cuda):
    case = inputs.random_case(95, B=3, H=32, W=900, N=10000, counts=[900, 431, 77])
    t = to_dev(case, cuda)
    ref = bf16q_decode(case, cuda, plan=dict(split=2, tiles=1, window=64), tensors=t)
    for tiles, window in ((2, 64), (1, 128), (1, 192)):
        out, lse = bf16q_decode(case, cuda, plan=dict(split=2, tiles=tiles, window=window),
                                tensors=t)
        assert np.array_equal(out, ref[0]), (tiles, window)
        assert np.array_equal(lse.view(np.uint32), ref[1].view(np.uint32)), (tiles, window)
    for split in (1, 4, 8):
        out, lse = bf16q_decode(case, cuda, plan=dict(split=split), tensors=t)
        out_o, lse_o = oracle_bf16q(case)
        check(out, lse, out_o, lse_o, f"bf16q split {split}")


@pytest.mark.parametrize("shift", [0, -4])
def test_bf16q_of_an_e4m3_query_is_the_e4m3_decode(cuda, shift):
    """A query of E4M3 values times 2^shift with 448 x 2^shift in every (row,
    head): lo = 0 and k = -shift, so the split decode adds zeros to the same
    accumulators and scales by the same lambda: the E4M3 decode's bits."""
    import torch
    case = inputs.random_case(96, B=3, H=16, W=300, N=4000, counts=[300, 5, 0])
    q8 = case.q8.copy()
    q8[:, :, 11] = 0x7E
    e4 = torch.from_numpy(q8).view(torch.float8_e4m3fn).to(torch.float32) * 2.0 ** shift
    q16 = e4.to(torch.bfloat16).to(cuda)
    t = to_dev(case, cuda)
    t = (torch.from_numpy(q8).to(cuda),) + t[1:]
    out_s, lse_s = bf16q_decode(case, cuda, tensors=t, q16=q16, plan=dict(kernel=1))
    case_e = inputs.Case(case.name, q8, case.kv8, case.indices, case.counts, case.sm_scale,
                         2.0 ** shift, case.k_scale)
    out_e, lse_e = gpu_decode(case_e, cuda, plan=dict(kernel=1), tensors=t)
    assert np.array_equal(out_s, out_e)
    assert np.array_equal(lse_s.view(np.uint32), lse_e.view(np.uint32))


def test_bf16q_latency_config(cuda):
    case = inputs.config("latency")
    out_g, lse_g = bf16q_decode(case, cuda)
    out_o, lse_o = oracle_bf16q(case)
    check(out_g, lse_g, out_o, lse_o, "bf16q latency")


def test_bf16q_dsa_config_sampled(cuda):
    case = inputs.config("dsa")
    out_g, lse_g = bf16q_decode(case, cuda)
    zero = np.where(case.counts == 0)[0][:1].tolist()
    rows = [0, 9, 63] + zero
    out_o, lse_o = oracle_bf16q(case, rows)
    check(out_g[rows], lse_g[rows], out_o, lse_o, "bf16q dsa")


def test_bf16q_timeout_is_reported_and_the_context_survives(cuda):
    from sparse_mla_decode_gb300 import binding
    case = inputs.random_case(97, B=2, H=16, W=64, N=1000, counts=[64, 10])
    t = to_dev(case, cuda)
    bf16q_decode(case, cuda, tensors=t, plan=dict(inject_stall=1, wait_budget_us=2000),
                 expect_status=binding.SMD_ERR_TIMEOUT)
    out_g, lse_g = bf16q_decode(case, cuda, tensors=t)
    out_o, lse_o = oracle_bf16q(case)
    check(out_g, lse_g, out_o, lse_o, "bf16q after a timeout")


# ---- the split query on the spread tcgen05 kernel (smd_sparse_mla_decode_bf16q_ws) ------

SPREAD = 5


def bf16q_ws(case, dev, tensors=None, plan=None, expect_status=0):
    import torch
    from sparse_mla_decode_gb300 import binding
    nb = binding.smd_workspace_bytes_bf16q(case.B, case.H, case.W)
    assert nb > 0
    ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    _, kv, idx, cnt = tensors if tensors is not None else to_dev(case, dev)
    out, lse = binding.sparse_mla_decode_bf16q(q16_dev(case, dev), kv, idx, cnt, case.sm_scale,
                                               case.k_scale, status=status, plan=plan,
                                               workspace=ws)
    torch.cuda.synchronize()
    assert int(status.item()) == expect_status, binding.smd_status_str(int(status.item()))
    return out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy()


SPREAD_SHAPES = [
    # (B, H, W, N, counts): one piece (no exchange), several, ragged, empty rows, a long row, H = 256
    (3, 128, 300, 4000, [300, 0, 129]),
    (4, 128, 2048, 20000, [2048, 1537, 513, 1]),
    (2, 128, 9000, 40000, [9000, 4097]),
    (2, 256, 700, 5000, [700, 512]),
]


@pytest.mark.parametrize("shape", SPREAD_SHAPES, ids=[f"B{s[0]}H{s[1]}W{s[2]}" for s in SPREAD_SHAPES])
def test_bf16q_on_the_spread_kernel_matches_the_oracle(cuda, shape):
    from sparse_mla_decode_gb300 import binding
    B, H, W, N, counts = shape
    case = inputs.random_case(B * 17 + W, B=B, H=H, W=W, N=N, counts=counts, heavy_frac=0.02)
    assert binding.smd_plan_bf16q(B, H, W, 1 << 40).kernel == SPREAD
    out_g, lse_g = bf16q_ws(case, cuda)
    out_o, lse_o = oracle_bf16q(case)
    check(out_g, lse_g, out_o, lse_o, f"bf16q spread {shape}")


def test_bf16q_spread_grid_changes_no_bits(cuda):
    case = inputs.random_case(99, B=10, H=128, W=2048, N=30000,
                              counts=[2048, 5, 0, 1400, 700, 2048, 513, 1, 1999, 900])
    t = to_dev(case, cuda)
    ref = bf16q_ws(case, cuda, tensors=t)
    for grid in (4, 9, 152):
        out, lse = bf16q_ws(case, cuda, tensors=t, plan=dict(kernel=SPREAD, grid_x=grid))
        assert np.array_equal(out, ref[0]), grid
        assert np.array_equal(lse.view(np.uint32), ref[1].view(np.uint32)), grid


def test_bf16q_spread_dsa_config_sampled(cuda):
    case = inputs.config("dsa")
    out_g, lse_g = bf16q_ws(case, cuda)
    zero = np.where(case.counts == 0)[0][:1].tolist()
    rows = [0, 9, 63] + zero
    out_o, lse_o = oracle_bf16q(case, rows)
    check(out_g[rows], lse_g[rows], out_o, lse_o, "bf16q spread dsa")


def test_bf16q_spread_timeout_is_reported_and_the_context_survives(cuda):
    from sparse_mla_decode_gb300 import binding
    case = inputs.random_case(100, B=3, H=128, W=1500, N=9000, counts=[1500, 600, 1200])
    t = to_dev(case, cuda)
    bf16q_ws(case, cuda, tensors=t, plan=dict(kernel=SPREAD, inject_stall=1, wait_budget_us=2000),
             expect_status=binding.SMD_ERR_TIMEOUT)
    out_g, lse_g = bf16q_ws(case, cuda, tensors=t)
    out_o, lse_o = oracle_bf16q(case)
    check(out_g, lse_g, out_o, lse_o, "bf16q spread after a timeout")


def test_bf16q_spread_throughput_config_sampled(cuda):
    """256 rows of 2048 keys: 1024 pieces in seven rounds over the cooperative
    grid, four pieces a unit exchanging partials; sampled rows of every round
    and piece position against the oracle."""
    from sparse_mla_decode_gb300 import binding
    case = inputs.config("throughput")
    assert binding.smd_plan_bf16q(case.B, case.H, case.W,
                                  binding.smd_workspace_bytes_bf16q(case.B, case.H, case.W)
                                  ).kernel == binding.SMD_KERNEL_TC_SPREAD
    out_g, lse_g = bf16q_ws(case, cuda)
    rows = [0, 37, 38, 151, 152, 255]
    out_o, lse_o = oracle_bf16q(case, rows)
    check(out_g[rows], lse_g[rows], out_o, lse_o, "bf16q spread throughput")
