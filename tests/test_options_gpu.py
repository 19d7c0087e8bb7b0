"""smd_decode (the options-struct call) on the GPU: each combination of
options gives, bit for bit, the out and LSE of the specialised entry point it
stands for (those are checked against the oracle by the other parity tests),
and one case per variant is checked against the oracle here as well."""
from __future__ import annotations

import numpy as np
import pytest

from sparse_mla_decode_gb300 import inputs
from test_parity_gpu import check, oracle_decode

pytestmark = pytest.mark.gpu


def bits(out, lse):
    import torch
    torch.cuda.synchronize()
    return (out.view(torch.int16).cpu().numpy().view(np.uint16),
            lse.cpu().numpy().view(np.uint32))


def dev_case(case, dev, bf16=False):
    import torch
    q = torch.from_numpy(case.q16.view(np.int16)).to(dev).view(torch.bfloat16) if bf16 \
        else torch.from_numpy(case.q8).to(dev)
    return (q, torch.from_numpy(case.kv8).to(dev), torch.from_numpy(case.indices).to(dev),
            torch.from_numpy(case.counts).to(dev))


def status_of(dev):
    import torch
    return torch.zeros(1, dtype=torch.int32, device=dev)


def assert_same(a, b, what):
    assert np.array_equal(a[0], b[0]), f"{what}: out bits"
    assert np.array_equal(a[1], b[1]), f"{what}: lse bits"


@pytest.mark.parametrize("name", ["tiny", "latency", "dsa"])
def test_default_and_workspace_options(cuda, name):
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.config(name)
    q, kv, idx, cnt = dev_case(case, cuda)
    args = (q, kv, idx, cnt, case.sm_scale, case.q_scale, case.k_scale)
    st = status_of(cuda)
    ref = bits(*binding.sparse_mla_decode(*args, status=st))
    got = bits(*binding.decode(*args, status=st))
    assert_same(got, ref, f"{name}: default options")
    nb = binding.smd_decode_workspace_bytes(case.B, case.H, case.W)
    assert nb == binding.smd_workspace_bytes(case.B, case.H, case.W)
    ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device=cuda)
    ref_ws = bits(*binding.sparse_mla_decode(*args, status=st, workspace=ws))
    got_ws = bits(*binding.decode(*args, status=st, workspace=ws))
    assert_same(got_ws, ref_ws, f"{name}: workspace")
    assert int(st.item()) == 0
    rows = [0, case.B - 1]
    out_o, lse_o = oracle_decode(case, rows)
    check(got_ws[0][rows], got_ws[1][rows].view(np.float32), out_o, lse_o, f"{name} via smd_decode")


def test_forced_plans(cuda):
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.random_case(71, B=6, H=128, W=1500, N=20000, counts=[1500, 1, 0, 700, 1024, 513])
    q, kv, idx, cnt = dev_case(case, cuda)
    args = (q, kv, idx, cnt, case.sm_scale, case.q_scale, case.k_scale)
    st = status_of(cuda)
    for force in (dict(kernel=binding.SMD_KERNEL_TC, split=4), dict(kernel=binding.SMD_KERNEL_MMA, split=8),
                  dict(kernel=binding.SMD_KERNEL_TC_SPREAD)):
        nb = binding.smd_decode_workspace_bytes(case.B, case.H, case.W, binding.smd_options(force=force))
        ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device=cuda) if nb else None
        ref = bits(*binding.sparse_mla_decode(*args, status=st, plan=force, workspace=ws))
        got = bits(*binding.decode(*args, status=st, plan=force, workspace=ws))
        assert_same(got, ref, f"forced {force}")
    assert int(st.item()) == 0


@pytest.mark.parametrize("name,ws", [("latency", False), ("dsa", True)])
def test_bf16_query_option(cuda, name, ws):
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.config(name)
    q16, kv, idx, cnt = dev_case(case, cuda, bf16=True)
    st = status_of(cuda)
    w = None
    if ws:
        o = binding.smd_options(query_type=binding.SMD_QUERY_BF16)
        w = torch.zeros(binding.smd_decode_workspace_bytes(case.B, case.H, case.W, o),
                        dtype=torch.uint8, device=cuda)
    ref = bits(*binding.sparse_mla_decode_bf16q(q16, kv, idx, cnt, case.sm_scale, case.k_scale,
                                                status=st, workspace=w))
    # q_scale is not used with a bf16 query: any value gives the same bits.
    got = bits(*binding.decode(q16, kv, idx, cnt, case.sm_scale, 123.0, case.k_scale, status=st,
                               workspace=w))
    assert_same(got, ref, f"{name}: bf16 query")
    assert int(st.item()) == 0


@pytest.mark.parametrize("ws", [False, True])
def test_row_group_option(cuda, ws):
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.grouped_case(72, 6, 4, 16, 3000, 30000)
    q, kv, idx, cnt = dev_case(case, cuda)
    args = (q, kv, idx, cnt, case.sm_scale, case.q_scale, case.k_scale)
    st = status_of(cuda)
    w = None
    if ws:
        o = binding.smd_options(row_group=4)
        w = torch.zeros(binding.smd_decode_workspace_bytes(case.B, case.H, case.W, o),
                        dtype=torch.uint8, device=cuda)
    ref = bits(*binding.sparse_mla_decode(*args, status=st, row_group=4, workspace=w))
    got = bits(*binding.decode(*args, status=st, row_group=4, workspace=w))
    assert_same(got, ref, f"row groups, workspace {ws}")
    assert int(st.item()) == 0
    rows = [0, 3, case.B - 1]
    out_o, lse_o = oracle_decode(case, rows)
    check(got[0][rows], got[1][rows].view(np.float32), out_o, lse_o, "row groups via smd_decode")


def test_library_scratch_option(cuda):
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.random_case(73, B=40, H=128, W=2048, N=40000, counts=[2048] * 39 + [0])
    q, kv, idx, cnt = dev_case(case, cuda)
    st = status_of(cuda)
    out = torch.empty((case.B, case.H, 512), dtype=torch.bfloat16, device=cuda)
    lse = torch.empty((case.B, case.H), dtype=torch.float32, device=cuda)
    rc = binding.smd_sparse_mla_decode_noalloc(
        q.data_ptr(), kv.data_ptr(), case.N, idx.data_ptr(), case.W, cnt.data_ptr(), case.B,
        case.H, case.sm_scale, case.q_scale, case.k_scale, out.data_ptr(), lse.data_ptr(),
        st.data_ptr(), torch.cuda.current_stream(cuda).cuda_stream)
    assert rc == binding.SMD_OK
    ref = bits(out, lse)
    got = bits(*binding.decode(q, kv, idx, cnt, case.sm_scale, case.q_scale, case.k_scale,
                               status=st, library_scratch=True))
    assert_same(got, ref, "library scratch")
    assert int(st.item()) == 0


def test_invalid_options_launch_nothing(cuda):
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.config("tiny")
    q, kv, idx, cnt = dev_case(case, cuda)
    out = torch.full((case.B, case.H, 512), 7.0, dtype=torch.bfloat16, device=cuda)
    lse = torch.full((case.B, case.H), 7.0, dtype=torch.float32, device=cuda)
    for kw, status in ((dict(reserved=1), binding.SMD_ERR_SHAPE),
                       (dict(row_group=2, query_type=binding.SMD_QUERY_BF16), binding.SMD_ERR_PLAN)):
        rc = binding.smd_decode(q.data_ptr(), kv.data_ptr(), case.N, idx.data_ptr(), case.W,
                                cnt.data_ptr(), case.B, case.H, case.sm_scale, case.q_scale,
                                case.k_scale, out.data_ptr(), lse.data_ptr(),
                                binding.smd_options(**kw), torch.cuda.current_stream(cuda).cuda_stream)
        assert rc == status
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())
