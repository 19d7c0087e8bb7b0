"""GPU checks of the host-buffer decode (smd_sparse_mla_decode_host): q, the
index list and the counts come from host memory, out and lse go back to it,
pipelined with the decode over row chunks. One chunk gives the bits of the
device call on all rows; several chunks give the bits of the device call on
each chunk's rows (the workspace call when the whole batch's plan is the
spread kernel, else the call without a workspace). Also checked against the
oracle, with pageable host memory, on a side stream, for grouped rows and
for the bf16 query."""
from __future__ import annotations

import numpy as np
import pytest

from sparse_mla_decode_gb300 import inputs
from test_parity_gpu import check, gpu_decode, oracle_decode, to_dev

pytestmark = pytest.mark.gpu


def host_decode(case, dev, chunks=0, row_group=1, bf16=False, pinned=True, stream=None,
                copies=0):
    import torch
    from sparse_mla_decode_gb300 import binding
    kv = torch.from_numpy(case.kv8).to(dev)
    if bf16:
        q = torch.from_numpy(case.q16.view(np.int16)).view(torch.bfloat16)
    else:
        q = torch.from_numpy(case.q8)
    idx = torch.from_numpy(case.indices)
    cnt = torch.from_numpy(case.counts)
    out = torch.empty((case.B, case.H, 512), dtype=torch.bfloat16)
    lse = torch.empty((case.B, case.H), dtype=torch.float32)
    if pinned:
        q, idx, cnt, out, lse = (t.pin_memory() for t in (q, idx, cnt, out, lse))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    # Garbage in the staging area: nothing may depend on its contents.
    nb = binding.smd_workspace_bytes_host(case.B, case.H, case.W, row_group, bf16, chunks)
    ws = torch.full((max(nb, 16),), 0xA5, dtype=torch.uint8, device=dev)
    torch.cuda.current_stream(dev).synchronize()  # the fill; the call may go on another stream
    binding.sparse_mla_decode_host(q, kv, idx, cnt, case.sm_scale, case.q_scale, case.k_scale,
                                   out=out, lse=lse, status=status, workspace=ws,
                                   row_group=row_group, bf16_query=bf16, chunks=chunks,
                                   stream=stream, copies=copies)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, binding.smd_status_str(int(status.item()))
    return out.view(torch.int16).numpy().view(np.uint16).copy(), lse.numpy().copy()


def rows_of(case, r0, r1):
    return inputs.Case(case.name, case.q8[r0:r1], case.kv8, case.indices[r0:r1],
                       case.counts[r0:r1], case.sm_scale, case.q_scale, case.k_scale,
                       q16=case.q16[r0:r1])


def device_ws(case, dev, grouped=1, bf16=False):
    import torch
    from sparse_mla_decode_gb300 import binding
    if bf16:
        nb = binding.smd_workspace_bytes_bf16q(case.B, case.H, case.W)
    elif grouped > 1:
        nb = binding.smd_workspace_bytes_grouped(case.B, case.H, case.W, grouped)
    else:
        nb = binding.smd_workspace_bytes(case.B, case.H, case.W)
    return torch.zeros(nb, dtype=torch.uint8, device=dev) if nb > 0 else None


def assert_same(a, b, what):
    assert np.array_equal(a[0], b[0]), what
    assert np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32)), what


def test_one_chunk_is_the_device_call(cuda):
    case = inputs.config("latency")
    from sparse_mla_decode_gb300 import binding
    assert binding.smd_plan_host(case.B, case.H, case.W) == 1
    ref = gpu_decode(case, cuda, workspace=device_ws(case, cuda))
    assert_same(host_decode(case, cuda), ref, "latency, one chunk")
    assert_same(host_decode(case, cuda, pinned=False), ref, "latency, pageable host memory")


@pytest.mark.parametrize("chunks", [2, 3, 5])
def test_chunks_are_the_device_calls_on_their_rows(cuda, chunks):
    from sparse_mla_decode_gb300 import binding
    case = inputs.random_case(801 + chunks, B=11, H=32, W=700, N=12000,
                              counts=[700, 1, 0, 513, 699, 64, 300, 2, 700, 128, 45])
    got = host_decode(case, cuda, chunks=chunks)
    n = binding.smd_plan_host(case.B, case.H, case.W, chunks=chunks)
    rows = -(-case.B // chunks)
    assert n == -(-case.B // rows)
    for c in range(n):
        r0, r1 = c * rows, min(case.B, (c + 1) * rows)
        part = rows_of(case, r0, r1)
        ref = gpu_decode(part, cuda)  # the whole batch's plan is not the spread kernel
        assert_same((got[0][r0:r1], got[1][r0:r1]), ref, f"chunk {c} of {n}")
    out_o, lse_o = oracle_decode(case)
    check(got[0], got[1], out_o, lse_o, f"{chunks} chunks vs the oracle")


def test_spread_plan_chunks_use_the_workspace_call(cuda):
    """H = 128 rows longer than a cluster holds: the whole batch runs on the
    spread kernel, so two forced chunks are two workspace calls."""
    from sparse_mla_decode_gb300 import binding
    case = inputs.random_case(811, B=4, H=128, W=2600, N=30000, counts=[2600, 700, 0, 2100])
    assert binding.smd_plan_ws(case.B, case.H, case.W).kernel == binding.SMD_KERNEL_TC_SPREAD
    got = host_decode(case, cuda, chunks=2)
    for r0 in (0, 2):
        part = rows_of(case, r0, r0 + 2)
        ref = gpu_decode(part, cuda, workspace=device_ws(part, cuda))
        assert_same((got[0][r0:r0 + 2], got[1][r0:r0 + 2]), ref, f"rows {r0}..")
    assert_same(host_decode(case, cuda), gpu_decode(case, cuda, workspace=device_ws(case, cuda)),
                "one chunk")


def test_grouped_rows_in_chunks_of_whole_groups(cuda):
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.grouped_case(821, R=6, G=4, H=16, W=1500, N=20000)
    got = host_decode(case, cuda, chunks=2, row_group=4)
    for r0 in (0, 12):
        part = rows_of(case, r0, r0 + 12)
        q, kv, idx, cnt = to_dev(part, cuda)
        status = torch.zeros(1, dtype=torch.int32, device=cuda)
        out, lse = binding.sparse_mla_decode(q, kv, idx, cnt, case.sm_scale, case.q_scale,
                                             case.k_scale, status=status, row_group=4)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ref = (out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy())
        assert_same((got[0][r0:r0 + 12], got[1][r0:r0 + 12]), ref, f"groups from row {r0}")


def test_bf16_query_from_host_memory(cuda):
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.random_case(831, B=5, H=64, W=256, N=20000, counts=[256, 200, 0, 255, 1])
    got = host_decode(case, cuda, bf16=True)
    q16 = torch.from_numpy(case.q16.view(np.int16)).to(cuda).view(torch.bfloat16)
    _, kv, idx, cnt = to_dev(case, cuda)
    ws = device_ws(case, cuda, bf16=True)
    out, lse = binding.sparse_mla_decode_bf16q(q16, kv, idx, cnt, case.sm_scale, case.k_scale,
                                               workspace=ws)
    torch.cuda.synchronize()
    ref = (out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy())
    assert_same(got, ref, "bf16 query")


def test_host_call_is_ordered_on_a_side_stream(cuda):
    """Queued on a side stream behind a long kernel: the results are complete
    when that stream is synchronized, and match the default-stream call."""
    import torch
    case = inputs.random_case(841, B=6, H=16, W=400, N=8000)
    ref = host_decode(case, cuda)
    side = torch.cuda.Stream(cuda)
    with torch.cuda.stream(side):
        big = torch.ones(1 << 26, device=cuda)
        for _ in range(4):
            big.mul_(1.0)  # keeps the side stream busy before the call
    got = host_decode(case, cuda, stream=side)
    assert_same(got, ref, "side stream")


def test_throughput_config_in_wave_chunks_sampled(cuda):
    """The automatic plan cuts the 256 rows at whole waves of the cluster
    kernel (a one-wave chunk, two-wave chunks, the partial wave's rows)."""
    from sparse_mla_decode_gb300 import binding
    case = inputs.config("throughput")
    assert 4 <= binding.smd_plan_host(case.B, case.H, case.W) <= 8
    out_g, lse_g = host_decode(case, cuda)
    rows = [0, 63, 64, 200, 255]
    out_o, lse_o = oracle_decode(case, rows)
    check(out_g[rows], lse_g[rows], out_o, lse_o, "throughput via host buffers")


def test_host_call_replays_in_a_cuda_graph(cuda):
    """Captured with three chunks (the copy streams join the capture and are
    joined back): a replay reads the host inputs as they are at replay time
    and writes the host outputs; both replays give the eager call's bits."""
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.random_case(851, B=12, H=32, W=600, N=9000)
    other = inputs.random_case(852, B=12, H=32, W=600, N=9000)
    other = inputs.Case(other.name, other.q8, case.kv8, other.indices % case.N, other.counts,
                        case.sm_scale, case.q_scale, case.k_scale, q16=other.q16)
    ref = host_decode(case, cuda, chunks=3)
    ref_other = host_decode(other, cuda, chunks=3)
    kv = torch.from_numpy(case.kv8).to(cuda)
    q = torch.from_numpy(case.q8.copy()).pin_memory()
    idx = torch.from_numpy(case.indices.copy()).pin_memory()
    cnt = torch.from_numpy(case.counts.copy()).pin_memory()
    out = torch.zeros((case.B, case.H, 512), dtype=torch.bfloat16).pin_memory()
    lse = torch.zeros((case.B, case.H), dtype=torch.float32).pin_memory()
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    ws = torch.zeros(binding.smd_workspace_bytes_host(case.B, case.H, case.W, chunks=3),
                     dtype=torch.uint8, device=cuda)

    def call():
        binding.sparse_mla_decode_host(q, kv, idx, cnt, case.sm_scale, case.q_scale,
                                       case.k_scale, out=out, lse=lse, status=status,
                                       workspace=ws, chunks=3)

    side = torch.cuda.Stream(cuda)
    side.wait_stream(torch.cuda.current_stream(cuda))
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream(cuda).wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    torch.cuda.synchronize()

    def replay():
        out.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        return out.view(torch.int16).numpy().view(np.uint16).copy(), lse.numpy().copy()

    assert_same(replay(), ref, "first replay")
    q.copy_(torch.from_numpy(other.q8))
    idx.copy_(torch.from_numpy(other.indices))
    cnt.copy_(torch.from_numpy(other.counts))
    assert_same(replay(), ref_other, "replay after the host inputs changed")


@pytest.mark.parametrize("kind", ["mma", "mma_groups", "bf16q", "tc"])
def test_direct_host_access_gives_the_bits_of_the_copies(cuda, kind):
    """One chunk with page-locked buffers: the kernel reads indices and counts
    and writes out and lse in host memory (only q is copied), on the warp-MMA
    kernels and on the tcgen05 cluster kernel. Same bits as copying everything
    (copies = 1) and as the device call."""
    from sparse_mla_decode_gb300 import binding
    if kind == "tc":
        case = inputs.random_case(863, B=4, H=128, W=400, N=9000, counts=[400, 1, 0, 257])
        G, bf16 = 1, False
        assert binding.smd_plan_ws(case.B, case.H, case.W).kernel == binding.SMD_KERNEL_TC
    elif kind == "mma_groups":
        case = inputs.grouped_case(861, R=3, G=2, H=48, W=700, N=9000)
        G, bf16 = 2, False
        assert binding.smd_plan_grouped(case.B, case.H, case.W, 2).kernel == binding.SMD_KERNEL_GROUP
    else:
        case = inputs.random_case(862, B=5, H=64, W=256, N=20000, counts=[256, 200, 0, 255, 1])
        G, bf16 = 1, kind == "bf16q"
    direct = host_decode(case, cuda, row_group=G, bf16=bf16)
    copied = host_decode(case, cuda, row_group=G, bf16=bf16, copies=1)
    assert_same(direct, copied, kind)
    paged = host_decode(case, cuda, row_group=G, bf16=bf16, pinned=False)
    assert_same(paged, copied, kind + ", pageable memory (copies)")
    if kind in ("mma", "tc"):
        assert_same(direct, gpu_decode(case, cuda), "device call")


def test_bf16_query_on_the_spread_plan_read_in_place(cuda):
    """H = 128 rows longer than a cluster holds with a bf16 query: the split
    kernel reads the query from host memory, the spread kernel decodes; same
    bits as copying it (copies = 1) and as the device call with a workspace."""
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.random_case(871, B=3, H=128, W=2600, N=30000, counts=[2600, 0, 1800])
    assert binding.smd_plan_bf16q(case.B, case.H, case.W, 1).kernel == binding.SMD_KERNEL_TC_SPREAD
    direct = host_decode(case, cuda, bf16=True)
    copied = host_decode(case, cuda, bf16=True, copies=1)
    assert_same(direct, copied, "bf16 query, spread plan")
    q16 = torch.from_numpy(case.q16.view(np.int16)).to(cuda).view(torch.bfloat16)
    _, kv, idx, cnt = to_dev(case, cuda)
    ws = device_ws(case, cuda, bf16=True)
    out, lse = binding.sparse_mla_decode_bf16q(q16, kv, idx, cnt, case.sm_scale, case.k_scale,
                                               workspace=ws)
    torch.cuda.synchronize()
    assert_same(direct, (out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy()),
                "device call")


def test_bf16_query_in_chunks(cuda):
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.random_case(881, B=6, H=64, W=300, N=9000, counts=[300, 0, 17, 299, 150, 1])
    got = host_decode(case, cuda, bf16=True, chunks=2)
    for r0 in (0, 3):
        part = rows_of(case, r0, r0 + 3)
        q16 = torch.from_numpy(part.q16.view(np.int16)).to(cuda).view(torch.bfloat16)
        _, kv, idx, cnt = to_dev(part, cuda)
        out, lse = binding.sparse_mla_decode_bf16q(q16, kv, idx, cnt, case.sm_scale, case.k_scale)
        torch.cuda.synchronize()
        ref = (out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy())
        assert_same((got[0][r0:r0 + 3], got[1][r0:r0 + 3]), ref, f"bf16 rows {r0}..")


@pytest.mark.parametrize("copies", [0, 1])
def test_zero_width_rows_from_host_memory(cuda, copies):
    """W = 0 (no index array at all): every row is empty, zeros and -inf."""
    import torch
    from sparse_mla_decode_gb300 import binding
    B, H = 3, 32
    q = torch.from_numpy(inputs.random_case(882, B=B, H=H, W=4, N=100).q8).pin_memory()
    kv = torch.zeros((16, 576), dtype=torch.uint8, device=cuda)
    idx = torch.zeros((B, 0), dtype=torch.int32)
    cnt = torch.tensor([5, 0, -2], dtype=torch.int32).pin_memory()
    out, lse = binding.sparse_mla_decode_host(q, kv, idx, cnt, 0.1, 1.0, 1.0, copies=copies)
    torch.cuda.synchronize()
    assert not torch.any(out.float() != 0)
    assert torch.all(torch.isneginf(lse))
