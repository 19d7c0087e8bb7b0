"""GPU parity of the top-k select (smd_topk_select) against the oracle
(oracle/topk.py): identical indices and counts, bit for bit, on rows with
many ties, NaNs, row ends, K above the row length, rows longer than the
shared-memory cache, padded row strides, and the full select workload; and
the select feeding the decode."""
from __future__ import annotations

import numpy as np
import pytest

from oracle import topk as ot
from sparse_mla_decode_gb300 import inputs

pytestmark = pytest.mark.gpu


def gpu_select(case, dev, stride=None, ends=True, cluster=0):
    import torch
    from sparse_mla_decode_gb300 import binding
    B, L = case.logits.shape
    if stride is None:
        x = torch.from_numpy(case.logits.view(np.int16)).to(dev).view(torch.bfloat16)
    else:  # a wider buffer with garbage (NaN patterns) in the padding
        buf = np.full((B, stride), 0x7FC1, np.uint16)
        buf[:, :L] = case.logits
        x = torch.from_numpy(buf.view(np.int16)).to(dev).view(torch.bfloat16)[:, :L]
    re = torch.from_numpy(case.row_ends).to(dev) if ends else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    idx, cnt = binding.topk_select(x, case.K, row_ends=re, status=status, cluster=cluster)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return idx.cpu().numpy(), cnt.cpu().numpy()


CASES = [
    # (seed, B, L, K, scale, nan_frac)
    (1, 4, 300, 17, 1.0, 0.0),
    (2, 3, 5000, 2048, 0.01, 0.0),     # many equal values: the tie rule decides
    (3, 5, 4096, 64, 1.0, 0.3),        # NaNs
    (4, 2, 100, 512, 1.0, 0.0),        # K above the row length
    (5, 2, 200000, 2048, 0.1, 0.01),   # parts longer than the shared-memory cache
    (6, 7, 8, 8, 1.0, 0.0),
]


@pytest.mark.parametrize("case_args", CASES, ids=[f"seed{c[0]}L{c[2]}K{c[3]}" for c in CASES])
def test_select_matches_the_oracle(cuda, case_args):
    seed, B, L, K, scale, nan_frac = case_args
    case = inputs.topk_case(seed, B, L, K, scale=scale, nan_frac=nan_frac)
    idx_o, cnt_o = ot.topk_select(case.logits, K, case.row_ends)
    idx_g, cnt_g = gpu_select(case, cuda)
    assert np.array_equal(cnt_g, cnt_o)
    assert np.array_equal(idx_g, idx_o)
    idx_o2, cnt_o2 = ot.topk_select(case.logits, K)  # whole rows
    idx_g2, cnt_g2 = gpu_select(case, cuda, ends=False)
    assert np.array_equal(idx_g2, idx_o2) and np.array_equal(cnt_g2, cnt_o2)
    for cluster in (1, 2, 8):  # the split of a row over CTAs changes nothing
        idx_c, cnt_c = gpu_select(case, cuda, cluster=cluster)
        assert np.array_equal(idx_c, idx_o) and np.array_equal(cnt_c, cnt_o), cluster


def test_select_with_a_padded_row_stride(cuda):
    case = inputs.topk_case(9, 3, 1000, 100, scale=0.05)
    idx_o, cnt_o = ot.topk_select(case.logits, case.K, case.row_ends)
    idx_g, cnt_g = gpu_select(case, cuda, stride=1024)
    assert np.array_equal(idx_g, idx_o) and np.array_equal(cnt_g, cnt_o)


def test_select_workload(cuda):
    """64 rows of up to 65536 logits, top-k 2048: every row, bit for bit."""
    case = inputs.topk_config()
    idx_o, cnt_o = ot.topk_select(case.logits, case.K, case.row_ends)
    idx_g, cnt_g = gpu_select(case, cuda)
    assert np.array_equal(cnt_g, cnt_o)
    assert np.array_equal(idx_g, idx_o)


def test_select_feeds_the_decode(cuda):
    """Indexer logits over a cache pool -> the select -> the decode: the same
    output as the oracle decode on the oracle's selection."""
    import torch
    from sparse_mla_decode_gb300 import binding
    from test_parity_gpu import check, oracle_decode
    N, K = 6000, 700
    dec_case = inputs.random_case(98, B=3, H=64, W=K, N=N, counts=[K, K, K])
    sel = inputs.topk_case(98, 3, N, K, scale=1.0, row_ends=[N, 4000, 650])
    idx_o, cnt_o = ot.topk_select(sel.logits, K, sel.row_ends)
    dec_case.indices = np.where(idx_o >= 0, idx_o, 0).astype(np.int32)
    dec_case.counts = cnt_o
    x = torch.from_numpy(sel.logits.view(np.int16)).to(cuda).view(torch.bfloat16)
    idx_g, cnt_g = binding.topk_select(x, K, row_ends=torch.from_numpy(sel.row_ends).to(cuda))
    q = torch.from_numpy(dec_case.q8).to(cuda)
    kv = torch.from_numpy(dec_case.kv8).to(cuda)
    out, lse = binding.sparse_mla_decode(q, kv, idx_g, cnt_g, dec_case.sm_scale,
                                         dec_case.q_scale, dec_case.k_scale)
    torch.cuda.synchronize()
    out_o, lse_o = oracle_decode(dec_case)
    check(out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy(), out_o, lse_o,
          "select -> decode")


# ---- the select from and to host memory (smd_topk_select_host) ------------------

def host_select(case, dev, stride=None, ends=True, pinned=True, copies=0):
    import torch
    from sparse_mla_decode_gb300 import binding
    B, L = case.logits.shape
    buf = np.full((B, stride or L), 0x7FC1, np.uint16)  # NaN patterns in any padding
    buf[:, :L] = case.logits
    x = torch.from_numpy(buf.view(np.int16)).view(torch.bfloat16)
    re = torch.from_numpy(case.row_ends.copy()) if ends else None
    idx = torch.empty((B, case.K), dtype=torch.int32)
    cnt = torch.empty((B,), dtype=torch.int32)
    if pinned:
        x = x.pin_memory()
        re = re.pin_memory() if re is not None else None
        idx, cnt = idx.pin_memory(), cnt.pin_memory()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    binding.topk_select_host(x[:, :L], case.K, row_ends=re, indices=idx, counts=cnt,
                             status=status, copies=copies, device=dev)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return idx.numpy().copy(), cnt.numpy().copy()


@pytest.mark.parametrize("stride", [None, 1003, 1024])
def test_select_from_host_memory(cuda, stride):
    """In place (page-locked), through copies (copies = 1, and pageable
    memory): the device call's result, which is the oracle's."""
    case = inputs.topk_case(11, 5, 1000, 100, scale=0.05)
    idx_o, cnt_o = ot.topk_select(case.logits, case.K, case.row_ends)
    for kw in (dict(), dict(copies=1), dict(pinned=False)):
        idx_g, cnt_g = host_select(case, cuda, stride=stride, **kw)
        assert np.array_equal(idx_g, idx_o) and np.array_equal(cnt_g, cnt_o), kw
    idx_g, cnt_g = host_select(case, cuda, stride=stride, ends=False)
    idx_o2, cnt_o2 = ot.topk_select(case.logits, case.K)
    assert np.array_equal(idx_g, idx_o2) and np.array_equal(cnt_g, cnt_o2)


def test_select_workload_from_host_memory(cuda):
    case = inputs.topk_config()
    idx_g, cnt_g = host_select(case, cuda)
    idx_o, cnt_o = gpu_select(case, cuda)
    assert np.array_equal(idx_g, idx_o) and np.array_equal(cnt_g, cnt_o)
