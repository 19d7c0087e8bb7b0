"""Host-side checks of the C-ABI library: it builds for sm_103a, loads, exports
every entry point include/smd.h declares, and rejects bad arguments before
any launch. Nothing here launches a kernel or touches device memory."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

from sparse_mla_decode_gb300 import binding as smd
from sparse_mla_decode_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions() -> list[str]:
    text = open(os.path.join(ROOT, "include", "smd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(smd_\w+)\s*\(", text)))


def test_library_builds_and_exports_every_declared_symbol():
    path = build.build()
    assert os.path.exists(path)
    lib = ctypes.CDLL(path)
    names = declared_functions()
    assert "smd_sparse_mla_decode" in names and "smd_plan" in names
    for name in names:
        assert hasattr(lib, name), name


def test_library_is_built_for_sm_103a_only():
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.ARCH)


def test_scale_log2_is_the_rounded_double_product():
    import oracle
    rng = np.random.default_rng(0)
    for _ in range(200):
        sm, qs, ks = (float(np.float32(x)) for x in rng.uniform(1e-4, 2.0, 3))
        assert smd.smd_scale_log2(sm, qs, ks) == oracle.scale_log2(sm, qs, ks)


def test_status_strings():
    for code in range(-10, 1):
        s = smd.smd_status_str(code)
        assert s and s != "unknown status"
    assert smd.smd_status_str(-99) == "unknown status"
    assert smd.smd_version() >= 100


# Fake but well-aligned addresses: every call below must be rejected on the
# host before anything is launched.
A = 1 << 20


def call(q=A, kv=A, N=100, idx=A, W=8, counts=A, B=2, H=16, out=A, lse=A, status=0,
         force=None):
    if force is None:
        return smd.smd_sparse_mla_decode(q, kv, N, idx, W, counts, B, H, 0.1, 0.1, 0.1,
                                         out, lse, status, 0)
    return smd.smd_sparse_mla_decode_ex(q, kv, N, idx, W, counts, B, H, 0.1, 0.1, 0.1,
                                        out, lse, status, 0, 0, 0, force)


@pytest.mark.parametrize("kw,code", [
    (dict(H=0), smd.SMD_ERR_SHAPE),
    (dict(H=17), smd.SMD_ERR_SHAPE),
    (dict(H=-16), smd.SMD_ERR_SHAPE),
    (dict(B=-1), smd.SMD_ERR_SHAPE),
    (dict(W=-1), smd.SMD_ERR_SHAPE),
    (dict(N=-1), smd.SMD_ERR_SHAPE),
    (dict(N=0), smd.SMD_ERR_SHAPE),
    (dict(N=1 << 31), smd.SMD_ERR_SHAPE),
    (dict(q=0), smd.SMD_ERR_NULL),
    (dict(kv=0), smd.SMD_ERR_NULL),
    (dict(idx=0), smd.SMD_ERR_NULL),
    (dict(counts=0), smd.SMD_ERR_NULL),
    (dict(out=0), smd.SMD_ERR_NULL),
    (dict(lse=0), smd.SMD_ERR_NULL),
    (dict(q=A + 8), smd.SMD_ERR_ALIGN),
    (dict(kv=A + 4), smd.SMD_ERR_ALIGN),
    (dict(out=A + 2), smd.SMD_ERR_ALIGN),
    (dict(idx=A + 2), smd.SMD_ERR_ALIGN),
    (dict(counts=A + 1), smd.SMD_ERR_ALIGN),
    (dict(lse=A + 2), smd.SMD_ERR_ALIGN),
    (dict(status=A + 2), smd.SMD_ERR_ALIGN),
    (dict(B=0, q=0, out=0, lse=0, counts=0, idx=0, kv=0), smd.SMD_OK),
])
def test_argument_checks(kw, code):
    assert call(**kw) == code


@pytest.mark.parametrize("force", [
    dict(split=3), dict(split=32), dict(tiles=3), dict(tiles=4), dict(window=65),
    dict(window=4096), dict(kernel=9),
    dict(kernel=2, tiles=2),        # the tcgen05 kernel takes all 16 heads of the row here
])
def test_invalid_forced_plans_are_rejected(force):
    p = smd.SmdPlan()
    for k, v in force.items():
        setattr(p, k, v)
    assert call(force=p) == smd.SMD_ERR_PLAN


@pytest.mark.parametrize("B,H,W", [(2, 16, 64), (5, 64, 256), (64, 128, 2048), (256, 128, 2048),
                                   (128, 16, 8192), (1, 16, 0), (3, 48, 100), (7, 32, 1),
                                   (1, 256, 4096), (4, 16, 16384), (3, 128, 100), (2, 256, 513),
                                   (1, 128, 0), (2, 128, 2049)])
def test_plan_invariants(B, H, W):
    p = smd.smd_plan(B, H, W).as_dict()
    if H % 128 == 0 and 1 <= W <= 2048:
        # tcgen05 kernel: 128 heads per CTA, <= 512 keys per CTA, cluster <= 4
        assert p["kernel"] == smd.SMD_KERNEL_TC
        assert p["split"] in (1, 2, 4) and -(-W // p["split"]) <= 512
        assert p["split"] == 1 or -(-W // (p["split"] // 2)) > 512  # the smallest such split
        assert p["grid_x"] == H // 128 * p["split"] and p["grid_y"] == B
        assert p["threads"] == 512 and p["smem_bytes"] <= 227 * 1024
        return
    assert p["kernel"] == smd.SMD_KERNEL_MMA
    assert p["split"] in (1, 2, 4, 8, 16) and p["cluster_x"] == p["split"]
    assert p["tiles"] in (1, 2) and H % (16 * p["tiles"]) == 0
    assert p["grid_x"] == H // (16 * p["tiles"]) * p["split"] and p["grid_y"] == B
    assert p["key_cap"] >= -(-W // p["split"]) and p["key_cap"] % 64 == 0
    assert p["window"] % 64 == 0 and 64 <= p["window"] <= p["key_cap"]
    assert p["smem_bytes"] <= 227 * 1024 and p["threads"] == 512


def test_plan_rejects_widths_beyond_the_limit():
    with pytest.raises(smd.SmdError) as e:
        smd.smd_plan(1, 16, 1 << 20)
    assert e.value.status == smd.SMD_ERR_SHAPE


def test_cpu_tensors_are_refused():
    import torch
    q = torch.zeros((1, 16, 576), dtype=torch.uint8)
    kv = torch.zeros((8, 576), dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA"):
        smd.sparse_mla_decode(q, kv, torch.zeros((1, 4), dtype=torch.int32),
                              torch.zeros(1, dtype=torch.int32), 0.1, 0.1, 0.1)


@pytest.mark.parametrize("H,W,force", [
    (128, 8, dict(kernel=2, split=8)),     # tcgen05 clusters hold at most 4 CTAs
    (128, 2049, dict(kernel=2)),           # more than 4 x 512 keys
    (128, 2048, dict(kernel=2, split=2)),  # 1024 keys per CTA do not fit in TMEM
    (128, 64, dict(kernel=2, tiles=2)),    # the tcgen05 kernel's layout is fixed
    (144, 64, dict(kernel=2)),             # above 128 heads only whole groups of 128
])
def test_invalid_tc_plans_are_rejected(H, W, force):
    p = smd.SmdPlan()
    for k, v in force.items():
        setattr(p, k, v)
    assert call(H=H, W=W, force=p) == smd.SMD_ERR_PLAN


def test_workspace_size_and_checks():
    # The automatic plan takes a workspace only for the spread kernel: rows
    # of several pieces whose pieces fill at most two waves, or rows longer
    # than a cluster holds; one slot of ~257 KiB per possible piece.
    assert smd.smd_workspace_bytes(64, 128, 2048) >= 64 * 4 * 128 * 512 * 4
    assert smd.smd_workspace_bytes(2, 128, 8192) >= 2 * 16 * 128 * 512 * 4
    assert smd.smd_workspace_bytes(256, 128, 2048) == 0    # four waves: the cluster kernel
    assert smd.smd_workspace_bytes(5, 128, 300) == 0       # one piece per row: no exchange
    assert smd.smd_workspace_bytes(5, 64, 256) == 0        # warp-MMA kernel: on-chip merge
    # a forced cluster plan with a split can exchange through L2: one slot per SM id
    p = smd.SmdPlan()
    p.kernel = smd.SMD_KERNEL_TC
    assert smd.smd_workspace_bytes_ex(256, 128, 2048, p) >= 3 * 128 * 128 * 4 * 152
    need = smd.smd_workspace_bytes(2, 128, 2048)
    assert need > 0
    args = (A, A, 100, A, 2048, A, 2, 128, 0.1, 0.1, 0.1, A, A, 0)
    assert smd.smd_sparse_mla_decode_ws(*args, A, need - 16, 0) == smd.SMD_ERR_WORKSPACE
    assert smd.smd_sparse_mla_decode_ws(*args, A + 8, need, 0) == smd.SMD_ERR_WORKSPACE


def call_grouped(G, B=8, H=16, W=64, q=A, counts=A, force=None):
    if force is None:
        return smd.smd_sparse_mla_decode_grouped(q, A, 100, A, W, counts, B, H, G, 0.1, 0.1, 0.1,
                                                 A, A, 0, 0)
    return smd.smd_sparse_mla_decode_grouped_ex(q, A, 100, A, W, counts, B, H, G, 0.1, 0.1, 0.1,
                                                A, A, 0, 0, 0, 0, force)


@pytest.mark.parametrize("kw,code", [
    (dict(G=3), smd.SMD_ERR_SHAPE),
    (dict(G=8), smd.SMD_ERR_SHAPE),
    (dict(G=0), smd.SMD_ERR_SHAPE),
    (dict(G=4, B=6), smd.SMD_ERR_SHAPE),
    (dict(G=2, H=24), smd.SMD_ERR_SHAPE),
    (dict(G=4, q=0), smd.SMD_ERR_NULL),
    (dict(G=4, q=A + 8), smd.SMD_ERR_ALIGN),
    (dict(G=4, B=0, q=0, counts=0), smd.SMD_OK),
])
def test_grouped_argument_checks(kw, code):
    assert call_grouped(**kw) == code


@pytest.mark.parametrize("force", [dict(split=3), dict(split=32), dict(tiles=2), dict(window=65),
                                   dict(window=1024), dict(kernel=1), dict(kernel=4, split=32),
                                   dict(kernel=4, window=64), dict(kernel=3, split=3)])
def test_invalid_grouped_plans_are_rejected(force):
    p = smd.SmdPlan()
    for k, v in force.items():
        setattr(p, k, v)
    assert call_grouped(4, force=p) == smd.SMD_ERR_PLAN


@pytest.mark.parametrize("B,H,W,G", [(128, 16, 8192, 4), (8, 16, 300, 2), (4, 64, 2048, 4),
                                     (2, 16, 1, 2), (64, 32, 700, 4), (4, 16, 32768, 4),
                                     (6, 32, 9000, 2), (8, 16, 8193, 4)])
def test_grouped_plan_invariants(B, H, W, G):
    p = smd.smd_plan_grouped(B, H, W, G).as_dict()
    assert p["split"] in (1, 2, 4, 8, 16) and p["cluster_x"] == p["split"]
    assert p["threads"] == 512 and 0 < p["smem_bytes"] <= 227 * 1024
    if G * H in (32, 64) and W <= 8192:
        # tcgen05 groups: all G x H lanes in one CTA, <= 512 keys per CTA, smallest split
        assert p["kernel"] == smd.SMD_KERNEL_TC_GROUP and p["tiles"] == G * H // 16
        assert -(-W // p["split"]) <= 512 and (p["split"] == 1 or -(-W // (p["split"] // 2)) > 512)
        assert p["grid_x"] == p["split"] and p["grid_y"] == B // G
    else:
        assert p["kernel"] == smd.SMD_KERNEL_GROUP and p["tiles"] == G
        assert -(-W // p["split"]) <= 2048 and p["key_cap"] >= -(-W // p["split"])
        assert p["grid_x"] == H // 16 * p["split"] and p["grid_y"] == B // G
        assert p["window"] % 64 == 0
    if W <= 16384:  # a group of one is the per-row plan (which takes up to 16 x 1024 keys)
        assert smd.smd_plan_grouped(B, H, W, 1).as_dict() == smd.smd_plan(B, H, W).as_dict()


def test_grouped_plan_rejects_lists_beyond_the_cluster():
    with pytest.raises(smd.SmdError) as e:
        smd.smd_plan_grouped(4, 16, 16 * 2048 + 1, 4)
    assert e.value.status == smd.SMD_ERR_SHAPE


def call_bf16q(q=A, kv=A, N=100, idx=A, W=8, counts=A, B=2, H=16, out=A, lse=A, status=0,
               force=None):
    if force is None:
        return smd.smd_sparse_mla_decode_bf16q(q, kv, N, idx, W, counts, B, H, 0.1, 0.1,
                                               out, lse, status, 0)
    return smd.smd_sparse_mla_decode_bf16q_ex(q, kv, N, idx, W, counts, B, H, 0.1, 0.1,
                                              out, lse, status, 0, 0, 0, force)


@pytest.mark.parametrize("kw,code", [
    (dict(H=17), smd.SMD_ERR_SHAPE),
    (dict(N=0), smd.SMD_ERR_SHAPE),
    (dict(q=0), smd.SMD_ERR_NULL),
    (dict(counts=0), smd.SMD_ERR_NULL),
    (dict(q=A + 8), smd.SMD_ERR_ALIGN),
    (dict(out=A + 2), smd.SMD_ERR_ALIGN),
    (dict(B=0, q=0, out=0, lse=0, counts=0, idx=0, kv=0), smd.SMD_OK),
])
def test_bf16q_argument_checks(kw, code):
    assert call_bf16q(**kw) == code


@pytest.mark.parametrize("force", [dict(kernel=2), dict(kernel=4), dict(split=3), dict(tiles=3),
                                   dict(window=65)])
def test_bf16q_invalid_forced_plans_are_rejected(force):
    p = smd.SmdPlan()
    for k, v in force.items():
        setattr(p, k, v)
    assert call_bf16q(force=p) == smd.SMD_ERR_PLAN


def test_bf16q_workspace_plan():
    """With a workspace the 128-head shapes go to the spread kernel, which
    needs the split query's rows besides its slots; others stay on warp MMA."""
    nb = smd.smd_workspace_bytes_bf16q(64, 128, 2048)
    assert nb >= 64 * 4 * 128 * 512 * 4 + 64 * 128 * (2 * 576 + 4)
    assert smd.smd_plan_bf16q(64, 128, 2048, nb).kernel == smd.SMD_KERNEL_TC_SPREAD
    assert smd.smd_plan_bf16q(64, 128, 2048, 0).kernel == smd.SMD_KERNEL_MMA
    assert smd.smd_workspace_bytes_bf16q(5, 64, 256) == 0
    assert smd.smd_plan_bf16q(5, 64, 256, 1 << 30).kernel == smd.SMD_KERNEL_MMA
    p = smd.SmdPlan()
    p.kernel = smd.SMD_KERNEL_TC_SPREAD
    assert call_bf16q(B=2, H=128, W=64, force=p) == smd.SMD_ERR_WORKSPACE  # no workspace


@pytest.mark.parametrize("B,H,W", [(5, 64, 256), (64, 128, 2048), (2, 16, 8192), (3, 48, 100)])
def test_bf16q_plan_runs_the_warp_mma_kernel_with_both_query_tiles(B, H, W):
    p = smd.smd_plan_bf16q(B, H, W, 0)
    e = smd.smd_plan(B, H, W) if not (H % 128 == 0 and W <= 2048) else None
    assert p.kernel == smd.SMD_KERNEL_MMA
    assert p.split * p.key_cap >= W and p.smem_bytes <= 227 * 1024
    if e is not None and e.split == p.split and e.window == p.window:
        # the second query tile (16 x tiles rows of 592 bytes) is the only growth
        assert p.smem_bytes >= e.smem_bytes + 16 * p.tiles * 592 - 128


@pytest.mark.parametrize("kw,code", [
    (dict(K=0), smd.SMD_ERR_SHAPE),
    (dict(L=-1), smd.SMD_ERR_SHAPE),
    (dict(B=-1), smd.SMD_ERR_SHAPE),
    (dict(stride=8, L=16), smd.SMD_ERR_SHAPE),  # shorter than a row
    (dict(logits=0), smd.SMD_ERR_NULL),
    (dict(indices=0), smd.SMD_ERR_NULL),
    (dict(counts=0), smd.SMD_ERR_NULL),
    (dict(logits=A + 1), smd.SMD_ERR_ALIGN),
    (dict(indices=A + 2), smd.SMD_ERR_ALIGN),
    (dict(row_ends=A + 1), smd.SMD_ERR_ALIGN),
    (dict(B=0, logits=0, indices=0, counts=0), smd.SMD_OK),
])
def test_topk_select_argument_checks(kw, code):
    args = dict(logits=A, stride=64, row_ends=0, B=2, L=64, K=8, indices=A, counts=A)
    args.update(kw)
    assert smd.smd_topk_select(args["logits"], args["stride"], args["row_ends"], args["B"],
                               args["L"], args["K"], args["indices"], args["counts"], 0,
                               0) == code


@pytest.mark.parametrize("cluster", [3, 16, -1])
def test_topk_select_rejects_other_cluster_sizes(cluster):
    assert smd.smd_topk_select_ex(A, 64, 0, 2, 64, 8, A, A, 0, 0, cluster) == smd.SMD_ERR_PLAN


# ---- smd_sparse_mla_decode_host (argument checks before anything is queued) ------

def host_call(q=A, kv=A, N=100, idx=A, W=8, counts=A, B=2, H=16, out=A, lse=A, status=0,
              ws=A, ws_bytes=1 << 40, opts=None):
    return smd.smd_sparse_mla_decode_host(q, kv, N, idx, W, counts, B, H, 0.1, 1.0, 1.0, out,
                                          lse, status, ws, ws_bytes, opts, 0)


@pytest.mark.parametrize("kw,code", [
    (dict(H=15), smd.SMD_ERR_SHAPE),
    (dict(B=-1), smd.SMD_ERR_SHAPE),
    (dict(W=-1), smd.SMD_ERR_SHAPE),
    (dict(N=-1), smd.SMD_ERR_SHAPE),
    (dict(N=0), smd.SMD_ERR_SHAPE),
    (dict(q=0), smd.SMD_ERR_NULL),
    (dict(idx=0), smd.SMD_ERR_NULL),
    (dict(kv=0), smd.SMD_ERR_NULL),
    (dict(counts=0), smd.SMD_ERR_NULL),
    (dict(out=0), smd.SMD_ERR_NULL),
    (dict(lse=0), smd.SMD_ERR_NULL),
    (dict(ws=0), smd.SMD_ERR_NULL),
    (dict(kv=A + 4), smd.SMD_ERR_ALIGN),
    (dict(status=A + 2), smd.SMD_ERR_ALIGN),
    (dict(ws=A + 8), smd.SMD_ERR_WORKSPACE),
    (dict(ws_bytes=1024), smd.SMD_ERR_WORKSPACE),
    (dict(opts=smd.SmdHostOpts(3, 0, 0, 0)), smd.SMD_ERR_SHAPE),
    (dict(opts=smd.SmdHostOpts(4, 0, 0, 0), B=6), smd.SMD_ERR_SHAPE),
    (dict(opts=smd.SmdHostOpts(4, 1, 0, 0), B=4), smd.SMD_ERR_PLAN),
    (dict(opts=smd.SmdHostOpts(1, 2, 0, 0)), smd.SMD_ERR_PLAN),
    (dict(opts=smd.SmdHostOpts(1, 0, 9, 0)), smd.SMD_ERR_PLAN),
    (dict(opts=smd.SmdHostOpts(1, 0, -1, 0)), smd.SMD_ERR_PLAN),
    (dict(opts=smd.SmdHostOpts(1, 0, 0, 2)), smd.SMD_ERR_PLAN),
])
def test_host_call_argument_checks(kw, code):
    assert host_call(**kw) == code


def test_host_call_with_no_rows_is_a_no_op():
    assert host_call(B=0, q=0, idx=0, counts=0, out=0, lse=0, ws=0, ws_bytes=0) == smd.SMD_OK


@pytest.mark.parametrize("B,H,W,G,bf16,chunks", [
    (2, 16, 64, 1, False, 1),       # tiny: one small launch
    (5, 64, 256, 1, False, 1),      # latency
    (64, 128, 2048, 1, False, 1),   # DSA: the spread kernel takes the whole batch
    # throughput: 54 MB of host data over 1024 cluster CTAs, cut at whole waves
    # (here, with no device, a wave is 152 / 4 = 38 rows): 38, 76, 76, 38, then 28
    (256, 128, 2048, 1, False, 5),
    (128, 16, 8192, 4, False, 1),   # dense-as-sparse: 512 CTAs, but only 7.4 MB of host data
    (512, 16, 8192, 4, False, 1),   # four times the requests: the spread kernel takes the batch
    (256, 128, 2048, 1, True, 1),   # bf16 query on the spread kernel
])
def test_host_plan_chunks_large_host_data_where_each_chunk_fills_the_device(B, H, W, G, bf16, chunks):
    # No device here: the plan is made for a 152-SM GB300.
    assert smd.smd_plan_host(B, H, W, G, bf16) == chunks


@pytest.mark.parametrize("B,H,W,G,bf16", [(2, 16, 64, 1, False), (64, 128, 2048, 1, False),
                                          (256, 128, 2048, 1, False), (128, 16, 8192, 4, False),
                                          (12, 64, 300, 1, True)])
def test_host_workspace_holds_the_staging_and_the_chunk_workspace(B, H, W, G, bf16):
    staging = B * H * 576 * (2 if bf16 else 1) + B * W * 4 + B * 4 + B * H * 1024 + B * H * 4
    nb = smd.smd_workspace_bytes_host(B, H, W, G, bf16)
    assert staging <= nb <= staging + 5 * 256 + max(
        0, smd.smd_workspace_bytes_bf16q(B, H, W) if bf16 else
        smd.smd_workspace_bytes_grouped(B, H, W, G) if G > 1 else smd.smd_workspace_bytes(B, H, W))
    for chunks in (1, 2, 3):
        rows = -(-(B // G) // chunks) * G
        assert smd.smd_plan_host(B, H, W, G, bf16, chunks) == -(-B // rows)


@pytest.mark.parametrize("kw,code", [
    (dict(K=0), smd.SMD_ERR_SHAPE),
    (dict(B=-1), smd.SMD_ERR_SHAPE),
    (dict(stride=99), smd.SMD_ERR_SHAPE),
    (dict(copies=2), smd.SMD_ERR_PLAN),
    (dict(idx=0), smd.SMD_ERR_NULL),
    (dict(counts=0), smd.SMD_ERR_NULL),
    (dict(logits=0), smd.SMD_ERR_NULL),
    (dict(logits=A + 1), smd.SMD_ERR_ALIGN),
    (dict(idx=A + 2), smd.SMD_ERR_ALIGN),
    (dict(ends=A + 2), smd.SMD_ERR_ALIGN),
    # no device here, so nothing is mapped: the copies need a workspace
    (dict(), smd.SMD_ERR_WORKSPACE),
    (dict(ws=A, ws_bytes=1024), smd.SMD_ERR_WORKSPACE),
    (dict(ws=A + 8, ws_bytes=1 << 30), smd.SMD_ERR_WORKSPACE),
])
def test_topk_host_argument_checks(kw, code):
    a = dict(logits=A, stride=100, ends=0, B=2, L=100, K=8, idx=A, counts=A, status=0, ws=0,
             ws_bytes=0, copies=0)
    a.update(kw)
    assert smd.smd_topk_select_host(a["logits"], a["stride"], a["ends"], a["B"], a["L"], a["K"],
                                    a["idx"], a["counts"], a["status"], a["ws"], a["ws_bytes"],
                                    a["copies"], 0) == code


def test_topk_host_workspace_pads_rows_to_16_bytes():
    assert smd.smd_workspace_bytes_topk_host(3, 13, 5) >= 3 * 16 * 2 + 3 * 4 + 3 * 5 * 4 + 3 * 4
    assert smd.smd_workspace_bytes_topk_host(0, 13, 5) == 0
    assert smd.smd_workspace_bytes_topk_host(2, 8, 0) == smd.SMD_ERR_SHAPE
    assert smd.smd_topk_select_host(0, 0, 0, 0, 0, 1, 0, 0, 0, 0, 0, 0, 0) == smd.SMD_OK


# ---- smd_validate_indices: argument checks on the host (nothing launched) ----

@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), smd.SMD_ERR_SHAPE),
    (dict(W=-1), smd.SMD_ERR_SHAPE),
    (dict(N=-1), smd.SMD_ERR_SHAPE),
    (dict(status=0), smd.SMD_ERR_NULL),
    (dict(counts=0), smd.SMD_ERR_NULL),
    (dict(idx=0), smd.SMD_ERR_NULL),
    (dict(idx=A + 2), smd.SMD_ERR_ALIGN),
    (dict(counts=A + 1), smd.SMD_ERR_ALIGN),
    (dict(status=A + 2), smd.SMD_ERR_ALIGN),
    (dict(B=0, idx=0, counts=0), smd.SMD_OK),
])
def test_validate_indices_argument_checks(kw, code):
    a = dict(idx=A, W=8, counts=A, B=2, N=100, status=A)
    a.update(kw)
    assert smd.smd_validate_indices(a["idx"], a["W"], a["counts"], a["B"], a["N"], a["status"],
                                    None) == code


def test_trace_calls_in_the_normal_build_report_no_tables():
    """The phase stamps exist only in the tracing build (-DSMD_TRACE); the
    normal library answers every trace call without touching a device."""
    import numpy as np
    assert smd.smd_trace_enabled() == 0
    buf = np.zeros(64, np.uint64)
    for kernel in (smd.SMD_KERNEL_MMA, smd.SMD_KERNEL_TC, smd.SMD_KERNEL_TC_SPREAD,
                   smd.SMD_KERNEL_GROUP, smd.SMD_KERNEL_TC_GROUP):
        assert smd.smd_trace_clear(kernel) == smd.SMD_ERR_PLAN
        assert smd.smd_trace_read(kernel, buf.ctypes.data, buf.size) == smd.SMD_ERR_PLAN
    assert smd.smd_trace_read(smd.SMD_KERNEL_TC, None, 4) == smd.SMD_ERR_NULL
    assert smd.smd_trace_read(smd.SMD_KERNEL_TC, buf.ctypes.data, 8192 * 32 + 1) == smd.SMD_ERR_SHAPE
