"""smd_decode and its options struct, host side: every combination of the
options names the plan and the workspace size of the specialised entry point
it replaces, and invalid combinations are refused before anything is
launched. No GPU is needed (plans are host computations)."""
from __future__ import annotations

import pytest

from sparse_mla_decode_gb300 import binding as smd

SHAPES = [(1, 16, 64), (5, 64, 256), (64, 128, 2048), (256, 128, 2048), (4, 128, 9000),
          (3, 48, 100), (2, 256, 513), (128, 16, 8192)]


def same(a: smd.SmdPlan, b: smd.SmdPlan) -> bool:
    return a.as_dict() == b.as_dict()


@pytest.mark.parametrize("B,H,W", SHAPES)
def test_default_options_are_the_plain_call(B, H, W):
    assert same(smd.smd_decode_plan(B, H, W), smd.smd_plan(B, H, W))
    assert same(smd.smd_decode_plan(B, H, W, smd.smd_options()), smd.smd_plan(B, H, W))
    assert smd.smd_decode_workspace_bytes(B, H, W) == smd.smd_workspace_bytes(B, H, W)


@pytest.mark.parametrize("B,H,W", SHAPES)
def test_a_workspace_gives_the_workspace_plan(B, H, W):
    o = smd.smd_options(workspace_bytes=1)
    assert same(smd.smd_decode_plan(B, H, W, o), smd.smd_plan_ws(B, H, W))


@pytest.mark.parametrize("B,H,W", SHAPES)
@pytest.mark.parametrize("ws", [0, 1])
def test_bf16_query_options_are_the_bf16q_calls(B, H, W, ws):
    o = smd.smd_options(query_type=smd.SMD_QUERY_BF16, workspace_bytes=ws)
    assert same(smd.smd_decode_plan(B, H, W, o), smd.smd_plan_bf16q(B, H, W, ws))
    assert smd.smd_decode_workspace_bytes(B, H, W, o) == smd.smd_workspace_bytes_bf16q(B, H, W)


@pytest.mark.parametrize("B,H,W,G", [(128, 16, 8192, 4), (8, 16, 300, 2), (4, 64, 2048, 4),
                                     (64, 32, 700, 4), (4, 16, 32768, 4), (6, 32, 9000, 2)])
@pytest.mark.parametrize("ws", [0, 1])
def test_row_group_options_are_the_grouped_calls(B, H, W, G, ws):
    o = smd.smd_options(row_group=G, workspace_bytes=ws)
    assert same(smd.smd_decode_plan(B, H, W, o), smd.smd_plan_grouped(B, H, W, G, ws))
    assert smd.smd_decode_workspace_bytes(B, H, W, o) == smd.smd_workspace_bytes_grouped(B, H, W, G)


@pytest.mark.parametrize("force", [dict(kernel=smd.SMD_KERNEL_TC, split=2),
                                   dict(kernel=smd.SMD_KERNEL_MMA, split=8, tiles=1),
                                   dict(kernel=smd.SMD_KERNEL_TC_SPREAD)])
def test_a_forced_plan_is_resolved_and_sized_as_the_ex_call(force):
    B, H, W = 8, 128, 1000
    o = smd.smd_options(force=force, workspace_bytes=1)
    p = smd.smd_decode_plan(B, H, W, o)
    assert p.kernel == force["kernel"]
    if "split" in force:
        assert p.split == force["split"]
    assert smd.smd_decode_workspace_bytes(B, H, W, o) == smd.smd_workspace_bytes_ex(B, H, W, force)


def test_library_scratch_plans_the_plain_call():
    for B, H, W in SHAPES:
        o = smd.smd_options(library_scratch=True)
        assert same(smd.smd_decode_plan(B, H, W, o), smd.smd_plan(B, H, W))


@pytest.mark.parametrize("kw,status", [
    (dict(reserved=1), smd.SMD_ERR_SHAPE),
    (dict(query_type=2), smd.SMD_ERR_SHAPE),
    (dict(query_type=-1), smd.SMD_ERR_SHAPE),
    (dict(row_group=3), smd.SMD_ERR_SHAPE),
    (dict(row_group=8), smd.SMD_ERR_SHAPE),
    (dict(row_group=2, query_type=smd.SMD_QUERY_BF16), smd.SMD_ERR_PLAN),
    (dict(library_scratch=True, workspace=4096), smd.SMD_ERR_PLAN),
    (dict(library_scratch=True, row_group=2), smd.SMD_ERR_PLAN),
    (dict(library_scratch=True, query_type=smd.SMD_QUERY_BF16), smd.SMD_ERR_PLAN),
])
def test_invalid_combinations_are_refused_before_any_launch(kw, status):
    o = smd.smd_options(**kw)
    with pytest.raises(smd.SmdError) as e:
        smd.smd_decode_plan(8, 64, 256, o)
    assert e.value.status == status
    assert smd.smd_decode_workspace_bytes(8, 64, 256, o) == 0
    # The decode itself returns the same status with nothing launched (all
    # pointers null: a valid combination would stop at SMD_ERR_NULL).
    rc = smd.smd_decode(None, None, 1, None, 256, None, 8, 64, 1.0, 1.0, 1.0, None, None, o, None)
    assert rc == status


def test_valid_options_check_pointers_as_the_specialised_calls():
    for kw in (dict(), dict(row_group=2), dict(query_type=smd.SMD_QUERY_BF16),
               dict(library_scratch=True)):
        rc = smd.smd_decode(None, None, 1, None, 256, None, 8, 64, 1.0, 1.0, 1.0, None, None,
                            smd.smd_options(**kw), None)
        assert rc == smd.SMD_ERR_NULL
    # B == 0 is a no-op, as for every decode call.
    assert smd.smd_decode(None, None, 1, None, 256, None, 0, 64, 1.0, 1.0, 1.0, None, None,
                          None, None) == smd.SMD_OK


def test_shape_errors_match_the_plain_call():
    for B, H, W in [(-1, 16, 64), (1, 0, 64), (1, 24, 64), (1, 16, -5)]:
        with pytest.raises(smd.SmdError) as e:
            smd.smd_decode_plan(B, H, W)
        assert e.value.status == smd.SMD_ERR_SHAPE
