"""GPU parity: the CUDA decode (through the C ABI) against the CPU oracle on the
same seeded inputs.

The bar (per row set): max |out_gpu - out_oracle| <= 1e-2 * max |out_oracle|
on the BF16 output, |lse_gpu - lse_oracle| <= 1e-3 where finite, and -inf
exactly where the oracle has -inf. Plans that differ in layout or split (16-head
tiles per CTA, resident-key window, CTAs per row) must agree bit for bit.
"""
from __future__ import annotations

import os

import numpy as np
import pytest

import oracle
from sparse_mla_decode_gb300 import inputs

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2   # relative to max |out|
LSE_TOL = 1e-3   # absolute


def to_dev(case, dev):
    import torch
    return (torch.from_numpy(case.q8).to(dev), torch.from_numpy(case.kv8).to(dev),
            torch.from_numpy(case.indices).to(dev), torch.from_numpy(case.counts).to(dev))


def gpu_decode(case, dev, plan=None, tensors=None, workspace=None):
    import torch
    from sparse_mla_decode_gb300 import binding
    q, kv, idx, cnt = tensors if tensors is not None else to_dev(case, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = binding.sparse_mla_decode(q, kv, idx, cnt, case.sm_scale, case.q_scale,
                                         case.k_scale, status=status, plan=plan,
                                         workspace=workspace)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, binding.smd_status_str(int(status.item()))
    return out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy()


def oracle_decode(case, rows=None):
    if rows is None:
        out, _, lse = oracle.sparse_mla_decode(case.q8, case.kv8, case.indices, case.counts,
                                               case.sm_scale, case.q_scale, case.k_scale)
        return out, lse
    rows = np.asarray(rows)
    out, _, lse = oracle.sparse_mla_decode(case.q8[rows], case.kv8, case.indices[rows],
                                           case.counts[rows], case.sm_scale, case.q_scale,
                                           case.k_scale)
    return out, lse


def check(out_g, lse_g, out_o, lse_o, what=""):
    fg = oracle.bf16_bits_to_f32(out_g).astype(np.float64)
    fo = oracle.bf16_bits_to_f32(out_o).astype(np.float64)
    assert np.all(np.isfinite(fg)), what
    scale = max(np.max(np.abs(fo)), 1e-30)
    err = np.max(np.abs(fg - fo)) if fg.size else 0.0
    assert err <= OUT_TOL * scale, f"{what}: max|err| {err:.3e} vs max|out| {scale:.3e}"
    neg = np.isneginf(lse_o)
    assert np.array_equal(np.isneginf(lse_g), neg), what
    lerr = 0.0
    if np.any(~neg):
        lerr = float(np.max(np.abs(lse_g[~neg] - lse_o[~neg])))
        assert lerr <= LSE_TOL, f"{what}: max|lse err| {lerr:.3e}"
    log = os.environ.get("SMD_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(f"{what}: max|err|/max|out| {err / scale:.3e}  max|lse err| {lerr:.3e}  "
                    f"bf16-equal {np.mean(out_g == out_o):.5f}  n={out_g.size}\n")
    return err / scale


def test_tiny(cuda):
    case = inputs.tiny()
    out_g, lse_g = gpu_decode(case, cuda)
    out_o, lse_o = oracle_decode(case)
    check(out_g, lse_g, out_o, lse_o, "tiny")
    # Same arithmetic up to FP32 summation order: nearly every element agrees.
    assert np.mean(out_g == out_o) > 0.95


def test_latency_config(cuda):
    case = inputs.latency()
    out_g, lse_g = gpu_decode(case, cuda)
    out_o, lse_o = oracle_decode(case)
    check(out_g, lse_g, out_o, lse_o, "latency")
    assert np.all(out_g[case.counts == 0] == 0)


SHAPES = [
    # (B, H, W, N, counts)
    (3, 16, 64, 4096, [64, 1, 0]),
    (4, 32, 100, 3000, [100, 99, 33, 31]),
    (2, 48, 257, 5000, [257, 256]),
    (2, 64, 130, 2000, [65, 63]),
    (1, 128, 40, 500, [40]),
    (5, 16, 7, 64, [7, 3, 0, -4, 1000]),
    (2, 32, 1000, 8000, [1000, 517]),     # several windows per CTA: the re-gather path
    (2, 16, 3000, 9000, [3000, 1999]),
    (6, 16, 33, 700, None),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}H{s[1]}W{s[2]}" for s in SHAPES])
def test_random_shapes(cuda, shape):
    B, H, W, N, counts = shape
    case = inputs.random_case(B * 7 + W, B=B, H=H, W=W, N=N, counts=counts, heavy_frac=0.02)
    out_g, lse_g = gpu_decode(case, cuda)
    out_o, lse_o = oracle_decode(case)
    check(out_g, lse_g, out_o, lse_o, str(shape))


def test_duplicate_indices_count_twice(cuda):
    case = inputs.random_case(44, B=3, H=16, W=50, N=20, counts=[50, 20, 5], dup=True)
    out_g, lse_g = gpu_decode(case, cuda)
    out_o, lse_o = oracle_decode(case)
    check(out_g, lse_g, out_o, lse_o, "dup")


def test_all_rows_empty_and_zero_width(cuda):
    case = inputs.random_case(45, B=4, H=32, W=16, N=100, counts=[0, 0, -1, 0])
    out_g, lse_g = gpu_decode(case, cuda)
    assert np.all(out_g == 0) and np.all(np.isneginf(lse_g))
    z = inputs.random_case(46, B=2, H=16, W=0, N=10, counts=[0, 5])
    out_g, lse_g = gpu_decode(z, cuda)
    assert np.all(out_g == 0) and np.all(np.isneginf(lse_g))


def test_zero_rows_is_a_no_op(cuda):
    import torch
    from sparse_mla_decode_gb300 import binding
    q = torch.zeros((0, 16, 576), dtype=torch.uint8, device=cuda)
    kv = torch.zeros((4, 576), dtype=torch.uint8, device=cuda)
    out, lse = binding.sparse_mla_decode(q, kv, torch.zeros((0, 8), dtype=torch.int32, device=cuda),
                                         torch.zeros(0, dtype=torch.int32, device=cuda), 1., 1., 1.)
    torch.cuda.synchronize()
    assert out.shape == (0, 16, 512) and lse.shape == (0, 16)


@pytest.mark.parametrize("split", [1, 2, 4, 8, 16])
def test_layout_variants_are_bit_identical(cuda, split):
    """tiles and window change only the layout: identical bits (across splits
    as well: the split points are leaf boundaries and the merge is one tree;
    test_split_invariance_gpu covers every variant together)."""
    case = inputs.random_case(50, B=3, H=64, W=600, N=6000, counts=[600, 301, 0],
                              heavy_frac=0.02)
    from sparse_mla_decode_gb300 import binding
    t = to_dev(case, cuda)
    ref = None
    ran = 0
    for tiles in (1, 2):
        for window in (64, 128, 256):
            per = -(-case.W // split)
            if window > max(64, -(-per // 64) * 64):
                continue
            try:
                out_g, lse_g = gpu_decode(case, cuda,
                                          dict(split=split, tiles=tiles, window=window), tensors=t)
            except binding.SmdError as e:  # this layout does not fit in shared memory
                assert e.status == binding.SMD_ERR_PLAN
                continue
            ran += 1
            if ref is None:
                ref = (out_g, lse_g)
                out_o, lse_o = oracle_decode(case)
                check(out_g, lse_g, out_o, lse_o, f"split {split}")
            else:
                assert np.array_equal(out_g, ref[0]), (tiles, window)
                assert np.array_equal(lse_g.view(np.uint32), ref[1].view(np.uint32))
    assert ran >= 2


def test_index_permutation_changes_only_summation_order(cuda):
    case = inputs.random_case(51, B=2, H=32, W=512, N=4000, counts=[512, 300], heavy_frac=0.05)
    out1, lse1 = gpu_decode(case, cuda)
    perm = case.indices.copy()
    rng = np.random.default_rng(3)
    for b, n in enumerate(case.counts):
        perm[b, :n] = perm[b, rng.permutation(n)]
    shuffled = inputs.Case("perm", case.q8, case.kv8, perm, case.counts, case.sm_scale,
                           case.q_scale, case.k_scale)
    out2, lse2 = gpu_decode(shuffled, cuda)
    check(out2, lse2, out1, lse1, "permuted")


def test_timeout_reports_status_and_context_survives(cuda):
    """A barrier armed for 16 bytes that no copy delivers: the bounded wait runs
    out, the call reports SMD_ERR_TIMEOUT in the status word, and the next call
    on the same context is correct."""
    import torch
    from sparse_mla_decode_gb300 import binding
    case = inputs.random_case(60, B=2, H=16, W=64, N=1000, counts=[64, 10])
    q, kv, idx, cnt = to_dev(case, cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    binding.sparse_mla_decode(q, kv, idx, cnt, case.sm_scale, case.q_scale, case.k_scale,
                              status=status, plan=dict(inject_stall=1, wait_budget_us=2000))
    torch.cuda.synchronize()
    assert int(status.item()) == binding.SMD_ERR_TIMEOUT
    out_g, lse_g = gpu_decode(case, cuda, tensors=(q, kv, idx, cnt))
    out_o, lse_o = oracle_decode(case)
    check(out_g, lse_g, out_o, lse_o, "after timeout")


def _full_config(name, cuda, sample_rows):
    case = inputs.config(name)
    out_g, lse_g = gpu_decode(case, cuda)
    rows = np.asarray(sample_rows)
    out_o, lse_o = oracle_decode(case, rows)
    check(out_g[rows], lse_g[rows], out_o, lse_o, name)
    # Every row: finite output, -inf exactly on the empty rows.
    n = case.clamped_counts()
    assert np.all(np.isneginf(lse_g[n == 0])) and np.all(np.isfinite(lse_g[n > 0]))
    return case


@pytest.mark.slow
def test_dsa_config_every_row(cuda):
    """All 64 rows of the DSA workload (its 4 empty rows included)."""
    _full_config("dsa", cuda, np.arange(64))


@pytest.mark.slow
def test_throughput_config_32_rows(cuda):
    """32 of the 256 rows, every 8th: rows in every wave of 36 clusters (all
    four CTAs of a row own columns, so every cluster rank is covered)."""
    _full_config("throughput", cuda, np.arange(0, 256, 8))


@pytest.mark.slow
def test_dense_config_32_rows(cuda):
    """8 whole requests (4 rows each) spread over the 32."""
    _full_config("dense", cuda, np.concatenate([4 * r + np.arange(4) for r in range(0, 32, 4)]))
