"""The allocation-free entry point, smd_sparse_mla_decode_noalloc.

Some callers cannot allocate device memory: a plug-in inside a host framework
that owns every device buffer and hands it only inputs and outputs, or a
serving loop whose memory is reserved up front so that no call can fail for
lack of it or stall in the allocator. For them the library exchanges the split
partials of the tcgen05 kernel through scratch it holds itself (a static
device array). This test calls that entry point through the C ABI twice in a
row, on different inputs, and checks each result bit for bit against the
regular entry point's (the split partials are merged by the same tree on both
exchange paths), and a few rows, an empty one among them, against the CPU
oracle within the tolerances of the parity tests.

It lives in a file of its own that pytest collects last, so that a run which
stops at the first failure has run every other test before it.
"""
from __future__ import annotations

import numpy as np
import pytest

from sparse_mla_decode_gb300 import inputs
from test_parity_gpu import check, oracle_decode, to_dev

pytestmark = pytest.mark.gpu


def _call(entry, case, tensors, dev):
    import torch
    from sparse_mla_decode_gb300 import binding
    q, kv, idx, cnt = tensors
    out = torch.empty((case.B, case.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((case.B, case.H), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = entry(q.data_ptr(), kv.data_ptr(), case.N, idx.data_ptr(), case.W, cnt.data_ptr(),
               case.B, case.H, case.sm_scale, case.q_scale, case.k_scale, out.data_ptr(),
               lse.data_ptr(), status.data_ptr(), torch.cuda.current_stream(dev).cuda_stream)
    assert rc == binding.SMD_OK, binding.smd_status_str(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, binding.smd_status_str(int(status.item()))
    return out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy()


def test_noalloc_entry_matches_the_regular_entry_on_two_calls(cuda):
    from sparse_mla_decode_gb300 import binding
    # H = 128 and top-k 2048: the tcgen05 plan splits each row over 4 CTAs,
    # so the partials go through the library's scratch; 64 rows x 4 CTAs
    # exceed the 152 SMs, so its SM slots are reused within each call.
    assert binding.smd_plan(64, 128, 2048).as_dict()["split"] > 1
    for seed, counts in ((401, None), (402, [2048] * 63 + [0])):
        case = inputs.random_case(seed, B=64, H=128, W=2048, N=40000, counts=counts,
                                  heavy_frac=0.01)
        t = to_dev(case, cuda)
        out_n, lse_n = _call(binding.smd_sparse_mla_decode_noalloc, case, t, cuda)
        out_r, lse_r = _call(binding.smd_sparse_mla_decode, case, t, cuda)
        assert np.array_equal(out_n, out_r), f"seed {seed}: out bits"
        assert np.array_equal(lse_n.view(np.uint32), lse_r.view(np.uint32)), f"seed {seed}: lse"
        rows = [0, 31, 62, 63]
        out_o, lse_o = oracle_decode(case, rows)
        check(out_n[rows], lse_n[rows], out_o, lse_o, f"noalloc vs the oracle, seed {seed}")
