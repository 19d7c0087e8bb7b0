"""ctypes binding of libsmd.so (include/smd.h), with the same names.

Argument marshalling only: every step of the decode runs in the library's
CUDA kernels. There is no CPU path; if the library cannot be built or loaded
the import of a decode function raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

SMD_OK = 0
SMD_ERR_NULL = -1
SMD_ERR_SHAPE = -2
SMD_ERR_ALIGN = -3
SMD_ERR_LAUNCH = -4
SMD_ERR_TIMEOUT = -5
SMD_ERR_PLAN = -6
SMD_ERR_DEVICE = -7
SMD_ERR_WORKSPACE = -8
SMD_ERR_GROUP = -9
SMD_ERR_INDEX = -10

SMD_KERNEL_AUTO = 0
SMD_KERNEL_MMA = 1
SMD_KERNEL_TC = 2
SMD_KERNEL_GROUP = 3
SMD_KERNEL_TC_GROUP = 4
SMD_KERNEL_TC_SPREAD = 5

SMD_QUERY_E4M3 = 0
SMD_QUERY_BF16 = 1


class SmdPlan(ctypes.Structure):
    """smd_plan_t."""
    _fields_ = [(name, ctypes.c_int32) for name in (
        "kernel", "split", "tiles", "window", "wait_budget_us", "inject_stall", "key_cap",
        "grid_x", "grid_y", "cluster_x", "threads", "smem_bytes")]

    def as_dict(self) -> dict:
        return {name: int(getattr(self, name)) for name, _ in self._fields_}


class SmdHostOpts(ctypes.Structure):
    """smd_host_opts_t."""
    _fields_ = [(name, ctypes.c_int32) for name in ("row_group", "bf16_query", "chunks",
                                                     "copies")]


class SmdOptions(ctypes.Structure):
    """smd_options_t."""
    _fields_ = [("row_group", ctypes.c_int32), ("query_type", ctypes.c_int32),
                ("library_scratch", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_int64),
                ("status", ctypes.c_void_p), ("force", ctypes.POINTER(SmdPlan))]


class SmdError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        super().__init__(f"{what}: {smd_status_str(status)} ({status})" if what
                         else f"{smd_status_str(status)} ({status})")


_lock = threading.Lock()
_lib = None

_DECODE_ARGS = [
    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,   # q, kv_pool, N
    ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,   # indices, W, counts
    ctypes.c_int32, ctypes.c_int32,                     # B, H
    ctypes.c_float, ctypes.c_float, ctypes.c_float,     # sm_scale, q_scale, k_scale
    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,  # out, lse, status
    ctypes.c_void_p,                                    # stream
]


def lib() -> ctypes.CDLL:
    """The loaded library (built in-tree on first use if missing or stale):
    libsmd.so, or its tracing variant when SMD_TRACE_BUILD=1 (per-phase
    timestamps of the kernels; same results)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build(trace=os.environ.get("SMD_TRACE_BUILD") == "1")
            so = ctypes.CDLL(path)
            so.smd_sparse_mla_decode.restype = ctypes.c_int
            so.smd_sparse_mla_decode.argtypes = _DECODE_ARGS
            ws_args = _DECODE_ARGS[:-1] + [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
            so.smd_sparse_mla_decode_ws.restype = ctypes.c_int
            so.smd_sparse_mla_decode_ws.argtypes = ws_args
            so.smd_sparse_mla_decode_ex.restype = ctypes.c_int
            so.smd_sparse_mla_decode_ex.argtypes = ws_args + [ctypes.POINTER(SmdPlan)]
            so.smd_sparse_mla_decode_noalloc.restype = ctypes.c_int
            so.smd_sparse_mla_decode_noalloc.argtypes = _DECODE_ARGS
            grp_args = _DECODE_ARGS[:8] + [ctypes.c_int32] + _DECODE_ARGS[8:]
            so.smd_sparse_mla_decode_grouped.restype = ctypes.c_int
            so.smd_sparse_mla_decode_grouped.argtypes = grp_args
            grp_ws = grp_args[:-1] + [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
            so.smd_sparse_mla_decode_grouped_ws.restype = ctypes.c_int
            so.smd_sparse_mla_decode_grouped_ws.argtypes = grp_ws
            so.smd_sparse_mla_decode_grouped_ex.restype = ctypes.c_int
            so.smd_sparse_mla_decode_grouped_ex.argtypes = grp_ws + [ctypes.POINTER(SmdPlan)]
            so.smd_workspace_bytes_grouped.restype = ctypes.c_int64
            so.smd_workspace_bytes_grouped.argtypes = [ctypes.c_int32] * 4
            bq_args = ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                        ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                        ctypes.c_float, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                        ctypes.c_void_p, ctypes.c_void_p])
            so.smd_sparse_mla_decode_bf16q.restype = ctypes.c_int
            so.smd_sparse_mla_decode_bf16q.argtypes = bq_args
            bq_ws = bq_args[:-1] + [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
            so.smd_sparse_mla_decode_bf16q_ws.restype = ctypes.c_int
            so.smd_sparse_mla_decode_bf16q_ws.argtypes = bq_ws
            so.smd_sparse_mla_decode_bf16q_ex.restype = ctypes.c_int
            so.smd_sparse_mla_decode_bf16q_ex.argtypes = bq_ws + [ctypes.POINTER(SmdPlan)]
            so.smd_workspace_bytes_bf16q.restype = ctypes.c_int64
            so.smd_workspace_bytes_bf16q.argtypes = [ctypes.c_int32] * 3
            so.smd_plan_bf16q.restype = ctypes.c_int
            so.smd_plan_bf16q.argtypes = [ctypes.c_int32] * 3 + [ctypes.c_int64,
                                                                 ctypes.POINTER(SmdPlan)]
            so.smd_topk_select.restype = ctypes.c_int
            tk_args = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32,
                       ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                       ctypes.c_void_p, ctypes.c_void_p]
            so.smd_topk_select.argtypes = tk_args
            so.smd_topk_select_ex.restype = ctypes.c_int
            so.smd_topk_select_ex.argtypes = tk_args + [ctypes.c_int32]
            so.smd_plan_grouped.restype = ctypes.c_int
            so.smd_plan_grouped.argtypes = [ctypes.c_int32] * 4 + [ctypes.c_int64,
                                                                   ctypes.POINTER(SmdPlan)]
            so.smd_workspace_bytes.restype = ctypes.c_int64
            so.smd_workspace_bytes.argtypes = [ctypes.c_int32] * 3
            so.smd_workspace_bytes_ex.restype = ctypes.c_int64
            so.smd_workspace_bytes_ex.argtypes = [ctypes.c_int32] * 3 + [ctypes.POINTER(SmdPlan)]
            so.smd_plan.restype = ctypes.c_int
            so.smd_plan.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                    ctypes.POINTER(SmdPlan)]
            so.smd_plan_ws.restype = ctypes.c_int
            so.smd_plan_ws.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.POINTER(SmdPlan)]
            so.smd_plan_host.restype = ctypes.c_int
            so.smd_plan_host.argtypes = [ctypes.c_int32] * 3 + [ctypes.POINTER(SmdHostOpts),
                                                                ctypes.POINTER(ctypes.c_int32)]
            so.smd_workspace_bytes_host.restype = ctypes.c_int64
            so.smd_workspace_bytes_host.argtypes = [ctypes.c_int32] * 3 + [
                ctypes.POINTER(SmdHostOpts)]
            so.smd_sparse_mla_decode_host.restype = ctypes.c_int
            so.smd_sparse_mla_decode_host.argtypes = _DECODE_ARGS[:-1] + [
                ctypes.c_void_p, ctypes.c_int64, ctypes.POINTER(SmdHostOpts), ctypes.c_void_p]
            so.smd_workspace_bytes_topk_host.restype = ctypes.c_int64
            so.smd_workspace_bytes_topk_host.argtypes = [ctypes.c_int32] * 3
            so.smd_topk_select_host.restype = ctypes.c_int
            so.smd_topk_select_host.argtypes = tk_args[:-1] + [ctypes.c_void_p, ctypes.c_int64,
                                                               ctypes.c_int32, ctypes.c_void_p]
            so.smd_validate_indices.restype = ctypes.c_int
            so.smd_validate_indices.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                                ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p,
                                                ctypes.c_void_p]
            so.smd_fp8_mma_probe.restype = ctypes.c_int
            so.smd_fp8_mma_probe.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.POINTER(ctypes.c_int32)]
            so.smd_scale_log2.restype = ctypes.c_float
            so.smd_scale_log2.argtypes = [ctypes.c_float] * 3
            so.smd_status_str.restype = ctypes.c_char_p
            so.smd_decode.argtypes = _DECODE_ARGS[:-2] + [ctypes.POINTER(SmdOptions),
                                                           ctypes.c_void_p]
            so.smd_decode.restype = ctypes.c_int
            so.smd_decode_plan.argtypes = [ctypes.c_int32] * 3 + [ctypes.POINTER(SmdOptions),
                                                                  ctypes.POINTER(SmdPlan)]
            so.smd_decode_plan.restype = ctypes.c_int
            so.smd_decode_workspace_bytes.argtypes = [ctypes.c_int32] * 3 + [
                ctypes.POINTER(SmdOptions)]
            so.smd_decode_workspace_bytes.restype = ctypes.c_int64
            so.smd_trace_enabled.argtypes = []
            so.smd_trace_enabled.restype = ctypes.c_int
            so.smd_trace_read.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32]
            so.smd_trace_read.restype = ctypes.c_int
            so.smd_trace_clear.argtypes = [ctypes.c_int32]
            so.smd_trace_clear.restype = ctypes.c_int
            so.smd_status_str.argtypes = [ctypes.c_int]
            so.smd_version.restype = ctypes.c_int
            so.smd_version.argtypes = []
            _lib = so
    return _lib


def library_path() -> str:
    return _build.TRACE_LIB if os.environ.get("SMD_TRACE_BUILD") == "1" else _build.LIB


# ---- raw C-ABI calls (pointers as integers) -----------------------------------

def smd_sparse_mla_decode(q, kv_pool, N, indices, W, counts, B, H, sm_scale, q_scale, k_scale,
                          out, lse, status, stream) -> int:
    return lib().smd_sparse_mla_decode(q, kv_pool, N, indices, W, counts, B, H, sm_scale,
                                       q_scale, k_scale, out, lse, status, stream)


def smd_sparse_mla_decode_ws(q, kv_pool, N, indices, W, counts, B, H, sm_scale, q_scale, k_scale,
                             out, lse, status, workspace, workspace_bytes, stream) -> int:
    return lib().smd_sparse_mla_decode_ws(q, kv_pool, N, indices, W, counts, B, H, sm_scale,
                                          q_scale, k_scale, out, lse, status, workspace,
                                          workspace_bytes, stream)


def smd_sparse_mla_decode_ex(q, kv_pool, N, indices, W, counts, B, H, sm_scale, q_scale, k_scale,
                             out, lse, status, workspace, workspace_bytes, stream,
                             force: SmdPlan | None) -> int:
    ref = ctypes.byref(force) if force is not None else None
    return lib().smd_sparse_mla_decode_ex(q, kv_pool, N, indices, W, counts, B, H, sm_scale,
                                          q_scale, k_scale, out, lse, status, workspace,
                                          workspace_bytes, stream, ref)


def smd_sparse_mla_decode_noalloc(q, kv_pool, N, indices, W, counts, B, H, sm_scale, q_scale,
                                  k_scale, out, lse, status, stream) -> int:
    """The decode for callers that cannot allocate device memory: split
    partials go through the library's own static scratch (see smd.h)."""
    return lib().smd_sparse_mla_decode_noalloc(q, kv_pool, N, indices, W, counts, B, H, sm_scale,
                                               q_scale, k_scale, out, lse, status, stream)


def smd_sparse_mla_decode_grouped(q, kv_pool, N, indices, W, counts, B, H, row_group, sm_scale,
                                  q_scale, k_scale, out, lse, status, stream) -> int:
    return lib().smd_sparse_mla_decode_grouped(q, kv_pool, N, indices, W, counts, B, H,
                                               row_group, sm_scale, q_scale, k_scale, out, lse,
                                               status, stream)


def smd_sparse_mla_decode_grouped_ws(q, kv_pool, N, indices, W, counts, B, H, row_group,
                                     sm_scale, q_scale, k_scale, out, lse, status, workspace,
                                     workspace_bytes, stream) -> int:
    return lib().smd_sparse_mla_decode_grouped_ws(q, kv_pool, N, indices, W, counts, B, H,
                                                  row_group, sm_scale, q_scale, k_scale, out,
                                                  lse, status, workspace, workspace_bytes, stream)


def smd_sparse_mla_decode_grouped_ex(q, kv_pool, N, indices, W, counts, B, H, row_group,
                                     sm_scale, q_scale, k_scale, out, lse, status, workspace,
                                     workspace_bytes, stream, force: SmdPlan | None) -> int:
    ref = ctypes.byref(force) if force is not None else None
    return lib().smd_sparse_mla_decode_grouped_ex(q, kv_pool, N, indices, W, counts, B, H,
                                                  row_group, sm_scale, q_scale, k_scale, out,
                                                  lse, status, workspace, workspace_bytes,
                                                  stream, ref)


def smd_workspace_bytes_grouped(B: int, H: int, W: int, row_group: int) -> int:
    return int(lib().smd_workspace_bytes_grouped(B, H, W, row_group))


def smd_plan_grouped(B: int, H: int, W: int, row_group: int, workspace_bytes: int = 0) -> SmdPlan:
    p = SmdPlan()
    rc = lib().smd_plan_grouped(B, H, W, row_group, int(workspace_bytes), ctypes.byref(p))
    if rc != SMD_OK:
        raise SmdError(rc, "smd_plan_grouped")
    return p


def smd_sparse_mla_decode_bf16q(q, kv_pool, N, indices, W, counts, B, H, sm_scale, k_scale,
                                out, lse, status, stream) -> int:
    return lib().smd_sparse_mla_decode_bf16q(q, kv_pool, N, indices, W, counts, B, H, sm_scale,
                                             k_scale, out, lse, status, stream)


def smd_sparse_mla_decode_bf16q_ws(q, kv_pool, N, indices, W, counts, B, H, sm_scale, k_scale,
                                   out, lse, status, workspace, workspace_bytes, stream) -> int:
    return lib().smd_sparse_mla_decode_bf16q_ws(q, kv_pool, N, indices, W, counts, B, H, sm_scale,
                                                k_scale, out, lse, status, workspace,
                                                workspace_bytes, stream)


def smd_sparse_mla_decode_bf16q_ex(q, kv_pool, N, indices, W, counts, B, H, sm_scale, k_scale,
                                   out, lse, status, workspace, workspace_bytes, stream,
                                   force: SmdPlan | None) -> int:
    ref = ctypes.byref(force) if force is not None else None
    return lib().smd_sparse_mla_decode_bf16q_ex(q, kv_pool, N, indices, W, counts, B, H, sm_scale,
                                                k_scale, out, lse, status, workspace,
                                                workspace_bytes, stream, ref)


def smd_workspace_bytes_bf16q(B: int, H: int, W: int) -> int:
    return int(lib().smd_workspace_bytes_bf16q(B, H, W))


def smd_plan_bf16q(B: int, H: int, W: int, workspace_bytes: int = 0) -> SmdPlan:
    p = SmdPlan()
    rc = lib().smd_plan_bf16q(B, H, W, int(workspace_bytes), ctypes.byref(p))
    if rc != SMD_OK:
        raise SmdError(rc, "smd_plan_bf16q")
    return p


def smd_topk_select(logits, row_stride, row_ends, B, L, K, indices, counts, status,
                    stream) -> int:
    return lib().smd_topk_select(logits, row_stride, row_ends, B, L, K, indices, counts, status,
                                 stream)


def smd_topk_select_ex(logits, row_stride, row_ends, B, L, K, indices, counts, status, stream,
                       cluster) -> int:
    return lib().smd_topk_select_ex(logits, row_stride, row_ends, B, L, K, indices, counts,
                                    status, stream, cluster)


def smd_workspace_bytes(B: int, H: int, W: int) -> int:
    return int(lib().smd_workspace_bytes(B, H, W))


def smd_workspace_bytes_ex(B: int, H: int, W: int, force: SmdPlan | dict | None = None) -> int:
    if isinstance(force, dict):
        p = SmdPlan()
        for k, v in force.items():
            setattr(p, k, int(v))
        force = p
    ref = ctypes.byref(force) if force is not None else None
    return int(lib().smd_workspace_bytes_ex(B, H, W, ref))


def smd_plan(B: int, H: int, W: int) -> SmdPlan:
    p = SmdPlan()
    rc = lib().smd_plan(B, H, W, ctypes.byref(p))
    if rc != SMD_OK:
        raise SmdError(rc, "smd_plan")
    return p


def smd_plan_ws(B: int, H: int, W: int) -> SmdPlan:
    p = SmdPlan()
    rc = lib().smd_plan_ws(B, H, W, ctypes.byref(p))
    if rc != SMD_OK:
        raise SmdError(rc, "smd_plan_ws")
    return p


def _host_opts(row_group: int = 1, bf16_query: bool = False, chunks: int = 0,
               copies: int = 0) -> SmdHostOpts:
    return SmdHostOpts(int(row_group), 1 if bf16_query else 0, int(chunks), int(copies))


def smd_plan_host(B: int, H: int, W: int, row_group: int = 1, bf16_query: bool = False,
                  chunks: int = 0) -> int:
    """The number of row chunks smd_sparse_mla_decode_host pipelines."""
    n = ctypes.c_int32(0)
    o = _host_opts(row_group, bf16_query, chunks)
    rc = lib().smd_plan_host(B, H, W, ctypes.byref(o), ctypes.byref(n))
    if rc != SMD_OK:
        raise SmdError(rc, "smd_plan_host")
    return int(n.value)


def smd_workspace_bytes_host(B: int, H: int, W: int, row_group: int = 1,
                             bf16_query: bool = False, chunks: int = 0) -> int:
    o = _host_opts(row_group, bf16_query, chunks)
    return int(lib().smd_workspace_bytes_host(B, H, W, ctypes.byref(o)))


def smd_sparse_mla_decode_host(q, kv_pool, N, indices, W, counts, B, H, sm_scale, q_scale,
                               k_scale, out, lse, status, workspace, workspace_bytes,
                               opts: SmdHostOpts | None, stream) -> int:
    ref = ctypes.byref(opts) if opts is not None else None
    return lib().smd_sparse_mla_decode_host(q, kv_pool, N, indices, W, counts, B, H, sm_scale,
                                            q_scale, k_scale, out, lse, status, workspace,
                                            workspace_bytes, ref, stream)


def smd_workspace_bytes_topk_host(B: int, L: int, K: int) -> int:
    return int(lib().smd_workspace_bytes_topk_host(B, L, K))


def smd_topk_select_host(logits, row_stride, row_ends, B, L, K, indices, counts, status,
                         workspace, workspace_bytes, copies, stream) -> int:
    return lib().smd_topk_select_host(logits, row_stride, row_ends, B, L, K, indices, counts,
                                      status, workspace, workspace_bytes, copies, stream)


def smd_validate_indices(indices, W, counts, B, N, status, stream) -> int:
    return lib().smd_validate_indices(indices, W, counts, B, N, status, stream)


def smd_fp8_mma_probe(iters: int, status, stream) -> int:
    """Launches the FP8 tensor-pipe rate probe; returns the CTAs launched."""
    n = ctypes.c_int32(0)
    rc = lib().smd_fp8_mma_probe(iters, status, stream, ctypes.byref(n))
    if rc != SMD_OK:
        raise SmdError(rc, "smd_fp8_mma_probe")
    return n.value


def _as_plan(force):
    if isinstance(force, dict):
        p = SmdPlan()
        for k, v in force.items():
            setattr(p, k, int(v))
        return p
    return force


def smd_options(row_group: int = 1, query_type: int = SMD_QUERY_E4M3, library_scratch: bool = False,
                workspace: int = 0, workspace_bytes: int = 0, status: int = 0,
                force: SmdPlan | dict | None = None, reserved: int = 0) -> SmdOptions:
    """An smd_options_t (pointers as integers). The forced plan, if any, is
    kept alive by the returned struct."""
    o = SmdOptions()
    o.row_group, o.query_type, o.library_scratch, o.reserved = (int(row_group), int(query_type),
                                                                int(bool(library_scratch)),
                                                                int(reserved))
    o.workspace, o.workspace_bytes, o.status = int(workspace) or None, int(workspace_bytes), \
        int(status) or None
    force = _as_plan(force)
    if force is not None:
        o._force = force
        o.force = ctypes.pointer(force)
    return o


def smd_decode(q, kv_pool, N, indices, W, counts, B, H, sm_scale, q_scale, k_scale, out, lse,
               options: SmdOptions | None, stream) -> int:
    ref = ctypes.byref(options) if options is not None else None
    return int(lib().smd_decode(q, kv_pool, N, indices, W, counts, B, H, sm_scale, q_scale, k_scale,
                                out, lse, ref, stream))


def smd_decode_plan(B: int, H: int, W: int, options: SmdOptions | None = None) -> SmdPlan:
    p = SmdPlan()
    ref = ctypes.byref(options) if options is not None else None
    rc = lib().smd_decode_plan(B, H, W, ref, ctypes.byref(p))
    if rc != SMD_OK:
        raise SmdError(rc, "smd_decode_plan")
    return p


def smd_decode_workspace_bytes(B: int, H: int, W: int, options: SmdOptions | None = None) -> int:
    ref = ctypes.byref(options) if options is not None else None
    return int(lib().smd_decode_workspace_bytes(B, H, W, ref))


def smd_trace_enabled() -> int:
    return int(lib().smd_trace_enabled())


def smd_trace_read(kernel: int, host, n: int) -> int:
    return int(lib().smd_trace_read(kernel, host, n))


def smd_trace_clear(kernel: int) -> int:
    return int(lib().smd_trace_clear(kernel))


def smd_scale_log2(sm_scale: float, q_scale: float, k_scale: float) -> float:
    return float(lib().smd_scale_log2(sm_scale, q_scale, k_scale))


def smd_status_str(status: int) -> str:
    return lib().smd_status_str(int(status)).decode()


def smd_version() -> int:
    return int(lib().smd_version())


# ---- torch-level marshalling ----------------------------------------------------

def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _bytes_view(t, name: str):
    import torch
    if t.dtype == torch.float8_e4m3fn:
        t = t.view(torch.uint8)
    if t.dtype != torch.uint8:
        raise TypeError(f"{name}: expected uint8 / float8_e4m3fn, got {t.dtype}")
    return t


def sparse_mla_decode(q, kv_pool, indices, counts, sm_scale: float, q_scale: float,
                      k_scale: float, out=None, lse=None, status=None, stream=None,
                      plan: SmdPlan | dict | None = None, workspace=None, row_group: int = 1):
    """Decode on the GPU. q [B,H,576] and kv_pool [N,576] E4M3 (uint8 or
    float8_e4m3fn), indices [B,W] int32, counts [B] int32, all CUDA tensors.
    Returns (out [B,H,512] bfloat16, lse [B,H] float32). ``plan`` forces
    plan fields (smd_sparse_mla_decode_ex); ``status`` is an optional int32
    CUDA tensor that receives device-side errors; ``workspace`` an optional
    CUDA tensor for smd_sparse_mla_decode_ws (at least
    smd_workspace_bytes(B, H, W) bytes: the spread kernel's or the L2
    exchange of split partials); ``row_group`` > 1 calls
    smd_sparse_mla_decode_grouped (rows in groups sharing one index list)."""
    import torch

    q = _bytes_view(q, "q")
    kv_pool = _bytes_view(kv_pool, "kv_pool")
    for name, t in (("q", q), ("kv_pool", kv_pool), ("indices", indices), ("counts", counts)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (the decode has no CPU path)")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if indices.dtype != torch.int32 or counts.dtype != torch.int32:
        raise TypeError("indices and counts must be int32")
    if q.dim() != 3 or q.shape[2] != 576 or kv_pool.dim() != 2 or kv_pool.shape[1] != 576:
        raise ValueError("q must be [B,H,576] and kv_pool [N,576]")
    B, H = int(q.shape[0]), int(q.shape[1])
    W = int(indices.shape[1]) if indices.dim() == 2 else 0
    if indices.dim() != 2 or indices.shape[0] < B or counts.shape[0] < B:
        raise ValueError("indices must be [>=B, W] and counts [>=B]")
    if out is None:
        out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    args = (_ptr(q), _ptr(kv_pool), int(kv_pool.shape[0]), _ptr(indices), W, _ptr(counts), B, H,
            float(sm_scale), float(q_scale), float(k_scale), _ptr(out), _ptr(lse), _ptr(status))
    ws = (_ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size())
    if workspace is not None and not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    if isinstance(plan, dict):
        p = SmdPlan()
        for k, v in plan.items():
            setattr(p, k, int(v))
        plan = p
    if row_group != 1:
        g_args = args[:8] + (int(row_group),) + args[8:]
        if plan is not None:
            rc = smd_sparse_mla_decode_grouped_ex(*g_args, *ws, int(stream), plan)
        elif workspace is not None:
            rc = smd_sparse_mla_decode_grouped_ws(*g_args, *ws, int(stream))
        else:
            rc = smd_sparse_mla_decode_grouped(*g_args, int(stream))
        if rc != SMD_OK:
            raise SmdError(rc, "smd_sparse_mla_decode_grouped")
        return out, lse
    if plan is None and workspace is None:
        rc = smd_sparse_mla_decode(*args, int(stream))
    elif plan is None:
        rc = smd_sparse_mla_decode_ws(*args, *ws, int(stream))
    else:
        rc = smd_sparse_mla_decode_ex(*args, *ws, int(stream), plan)
    if rc != SMD_OK:
        raise SmdError(rc, "smd_sparse_mla_decode")
    return out, lse


def decode(q, kv_pool, indices, counts, sm_scale: float, q_scale: float, k_scale: float,
           out=None, lse=None, status=None, stream=None, plan: SmdPlan | dict | None = None,
           workspace=None, row_group: int = 1, library_scratch: bool = False):
    """Decode on the GPU through smd_decode (one call for every variant).
    q [B,H,576]: E4M3 (uint8 or float8_e4m3fn, with q_scale) or bfloat16 (the
    split query; q_scale is not used); kv_pool [N,576] E4M3, indices [B,W]
    int32, counts [B] int32, all CUDA tensors. ``row_group`` 2 or 4: rows in
    groups sharing one index list; ``workspace``, ``plan``, ``status`` as in
    sparse_mla_decode; ``library_scratch``: the no-alloc exchange. Returns
    (out [B,H,512] bfloat16, lse [B,H] float32)."""
    import torch

    bf16 = q.dtype == torch.bfloat16
    if not bf16:
        q = _bytes_view(q, "q")
    kv_pool = _bytes_view(kv_pool, "kv_pool")
    for name, t in (("q", q), ("kv_pool", kv_pool), ("indices", indices), ("counts", counts)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (the decode has no CPU path)")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if indices.dtype != torch.int32 or counts.dtype != torch.int32:
        raise TypeError("indices and counts must be int32")
    if q.dim() != 3 or q.shape[2] != 576 or kv_pool.dim() != 2 or kv_pool.shape[1] != 576:
        raise ValueError("q must be [B,H,576] and kv_pool [N,576]")
    B, H = int(q.shape[0]), int(q.shape[1])
    if indices.dim() != 2 or indices.shape[0] < B or counts.shape[0] < B:
        raise ValueError("indices must be [>=B, W] and counts [>=B]")
    W = int(indices.shape[1])
    if workspace is not None and not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    if out is None:
        out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    opts = smd_options(row_group=row_group, query_type=SMD_QUERY_BF16 if bf16 else SMD_QUERY_E4M3,
                       library_scratch=library_scratch, workspace=_ptr(workspace),
                       workspace_bytes=0 if workspace is None
                       else workspace.numel() * workspace.element_size(),
                       status=_ptr(status), force=plan)
    rc = smd_decode(_ptr(q), _ptr(kv_pool), int(kv_pool.shape[0]), _ptr(indices), W, _ptr(counts),
                    B, H, float(sm_scale), float(q_scale), float(k_scale), _ptr(out), _ptr(lse),
                    opts, int(stream))
    if rc != SMD_OK:
        raise SmdError(rc, "smd_decode")
    return out, lse


def sparse_mla_decode_bf16q(q, kv_pool, indices, counts, sm_scale: float, k_scale: float,
                            out=None, lse=None, status=None, stream=None,
                            plan: SmdPlan | dict | None = None, workspace=None):
    """Decode with a bfloat16 query q [B,H,576] (split into E4M3 hi + lo per
    (row, head) on the GPU: smd_sparse_mla_decode_bf16q). kv_pool [N,576] E4M3,
    indices [B,W] int32, counts [B] int32, all CUDA tensors. Returns
    (out [B,H,512] bfloat16, lse [B,H] float32)."""
    import torch

    kv_pool = _bytes_view(kv_pool, "kv_pool")
    if q.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"q: expected bfloat16, got {q.dtype}")
    for name, t in (("q", q), ("kv_pool", kv_pool), ("indices", indices), ("counts", counts)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (the decode has no CPU path)")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if indices.dtype != torch.int32 or counts.dtype != torch.int32:
        raise TypeError("indices and counts must be int32")
    if q.dim() != 3 or q.shape[2] != 576 or kv_pool.dim() != 2 or kv_pool.shape[1] != 576:
        raise ValueError("q must be [B,H,576] and kv_pool [N,576]")
    B, H = int(q.shape[0]), int(q.shape[1])
    if indices.dim() != 2 or indices.shape[0] < B or counts.shape[0] < B:
        raise ValueError("indices must be [>=B, W] and counts [>=B]")
    W = int(indices.shape[1])
    if out is None:
        out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    args = (_ptr(q), _ptr(kv_pool), int(kv_pool.shape[0]), _ptr(indices), W, _ptr(counts), B, H,
            float(sm_scale), float(k_scale), _ptr(out), _ptr(lse), _ptr(status))
    ws = (_ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size())
    if isinstance(plan, dict):
        p = SmdPlan()
        for k, v in plan.items():
            setattr(p, k, int(v))
        plan = p
    if plan is not None:
        rc = smd_sparse_mla_decode_bf16q_ex(*args, *ws, int(stream), plan)
    elif workspace is not None:
        rc = smd_sparse_mla_decode_bf16q_ws(*args, *ws, int(stream))
    else:
        rc = smd_sparse_mla_decode_bf16q(*args, int(stream))
    if rc != SMD_OK:
        raise SmdError(rc, "smd_sparse_mla_decode_bf16q")
    return out, lse


def sparse_mla_decode_host(q, kv_pool, indices, counts, sm_scale: float, q_scale: float,
                           k_scale: float, out=None, lse=None, status=None, stream=None,
                           workspace=None, row_group: int = 1, bf16_query: bool = False,
                           chunks: int = 0, copies: int = 0):
    """Decode with q, indices and counts in HOST memory and out / lse returned
    to host memory (smd_sparse_mla_decode_host); kv_pool stays a CUDA tensor.
    q [B,H,576] E4M3 (uint8 or float8_e4m3fn), or bfloat16 with bf16_query;
    indices [B,W] int32; counts [B] int32: contiguous CPU tensors, page-locked
    (``pin_memory()``) for the copies to overlap. ``workspace``: a CUDA tensor
    of at least smd_workspace_bytes_host bytes (allocated here if None).
    Returns (out [B,H,512] bfloat16, lse [B,H] float32) CPU tensors, complete
    once ``stream`` has reached the end of the call (synchronize before
    reading them)."""
    import torch

    if bf16_query:
        if q.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
            raise TypeError(f"q: expected bfloat16, got {q.dtype}")
    else:
        q = _bytes_view(q, "q")
    kv_pool = _bytes_view(kv_pool, "kv_pool")
    if not kv_pool.is_cuda:
        raise ValueError("kv_pool must be a CUDA tensor")
    for name, t in (("q", q), ("indices", indices), ("counts", counts)):
        if t.is_cuda:
            raise ValueError(f"{name} must be a CPU tensor (this call copies it to the GPU)")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if indices.dtype != torch.int32 or counts.dtype != torch.int32:
        raise TypeError("indices and counts must be int32")
    if q.dim() != 3 or q.shape[2] != 576 or kv_pool.dim() != 2 or kv_pool.shape[1] != 576:
        raise ValueError("q must be [B,H,576] and kv_pool [N,576]")
    B, H = int(q.shape[0]), int(q.shape[1])
    if indices.dim() != 2 or indices.shape[0] != B or counts.shape[0] != B:
        raise ValueError("indices must be [B, W] and counts [B]")
    W = int(indices.shape[1])
    if out is None:
        out = torch.empty((B, H, 512), dtype=torch.bfloat16).pin_memory()
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32).pin_memory()
    for name, t in (("out", out), ("lse", lse)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor")
    opts = _host_opts(row_group, bf16_query, chunks, copies)
    if workspace is None:
        nb = smd_workspace_bytes_host(B, H, W, row_group, bf16_query, chunks)
        if nb < 0:
            raise SmdError(nb, "smd_workspace_bytes_host")
        workspace = torch.empty(max(nb, 16), dtype=torch.uint8, device=kv_pool.device)
    if stream is None:
        stream = torch.cuda.current_stream(kv_pool.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    rc = smd_sparse_mla_decode_host(
        _ptr(q), _ptr(kv_pool), int(kv_pool.shape[0]), _ptr(indices), W, _ptr(counts), B, H,
        float(sm_scale), float(q_scale), float(k_scale), _ptr(out), _ptr(lse), _ptr(status),
        _ptr(workspace), workspace.numel() * workspace.element_size(), opts, int(stream))
    if rc != SMD_OK:
        raise SmdError(rc, "smd_sparse_mla_decode_host")
    return out, lse


def topk_select(logits, K: int, row_ends=None, indices=None, counts=None, stream=None,
                status=None, cluster: int = 0):
    """Top-k select on the GPU (smd_topk_select). logits: bfloat16 CUDA tensor
    [B, L] with unit column stride (a column slice of a wider tensor is fine;
    16-byte aligned rows are read fastest); row_ends: optional
    int32 [B]. Returns (indices int32 [B, K], counts int32 [B]), ready to be
    the decode's index list and counts."""
    import torch

    if logits.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"logits: expected bfloat16, got {logits.dtype}")
    if not logits.is_cuda:
        raise ValueError("logits must be a CUDA tensor (the select has no CPU path)")
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be [B, L] with unit column stride")
    B, L = int(logits.shape[0]), int(logits.shape[1])
    stride = int(logits.stride(0)) if B > 1 else L
    if row_ends is not None and (row_ends.dtype != torch.int32 or not row_ends.is_cuda):
        raise TypeError("row_ends must be an int32 CUDA tensor")
    if indices is None:
        indices = torch.empty((B, K), dtype=torch.int32, device=logits.device)
    if counts is None:
        counts = torch.empty((B,), dtype=torch.int32, device=logits.device)
    if stream is None:
        stream = torch.cuda.current_stream(logits.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    rc = smd_topk_select_ex(_ptr(logits), stride, _ptr(row_ends), B, L, int(K), _ptr(indices),
                            _ptr(counts), _ptr(status), int(stream), int(cluster))
    if rc != SMD_OK:
        raise SmdError(rc, "smd_topk_select")
    return indices, counts


def validate_indices(indices, counts, N: int, status=None, stream=None):
    """Range check of an index list on the GPU (smd_validate_indices): every
    valid entry (i < clamp(counts[b], 0, W)) of the int32 CUDA tensor
    indices [B, W] must lie in [0, N). Returns the int32 status tensor (one
    element, zeroed here unless given), which holds SMD_ERR_INDEX after the
    stream reaches the check if an entry lies outside."""
    import torch
    if indices.dim() != 2 or indices.dtype != torch.int32 or counts.dtype != torch.int32:
        raise ValueError("indices [B, W] and counts [B] must be int32")
    if not (indices.is_cuda and counts.is_cuda) or not indices.is_contiguous():
        raise ValueError("indices and counts must be contiguous CUDA tensors")
    B, W = indices.shape
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=indices.device)
    stream = torch.cuda.current_stream(indices.device) if stream is None else stream
    rc = smd_validate_indices(_ptr(indices), W, _ptr(counts), B, int(N), _ptr(status),
                              int(stream.cuda_stream))
    if rc != SMD_OK:
        raise SmdError(rc, "smd_validate_indices")
    return status


def topk_select_host(logits, K: int, row_ends=None, indices=None, counts=None, stream=None,
                     status=None, workspace=None, copies: int = 0, device=None):
    """Top-k select with host buffers (smd_topk_select_host): logits a bfloat16
    CPU tensor [B, L] with unit column stride, row_ends an optional int32 CPU
    tensor [B]; page-locked (``pin_memory()``) for the select to read them in
    place. Returns (indices int32 [B, K], counts int32 [B]) CPU tensors,
    complete once ``stream`` has reached the end of the call."""
    import torch

    if logits.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"logits: expected bfloat16, got {logits.dtype}")
    if logits.is_cuda or logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be a CPU tensor [B, L] with unit column stride")
    B, L = int(logits.shape[0]), int(logits.shape[1])
    stride = int(logits.stride(0)) if B > 1 else L
    if row_ends is not None and (row_ends.dtype != torch.int32 or row_ends.is_cuda):
        raise TypeError("row_ends must be an int32 CPU tensor")
    if indices is None:
        indices = torch.empty((B, K), dtype=torch.int32).pin_memory()
    if counts is None:
        counts = torch.empty((B,), dtype=torch.int32).pin_memory()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    if workspace is None and copies:
        workspace = torch.empty(max(smd_workspace_bytes_topk_host(B, L, int(K)), 16),
                                dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = smd_topk_select_host(_ptr(logits), stride, _ptr(row_ends), B, L, int(K), _ptr(indices),
                              _ptr(counts), _ptr(status), _ptr(workspace), nbytes, int(copies),
                              int(stream))
    if rc == SMD_ERR_WORKSPACE and workspace is None:
        # the buffers could not be read in place: copy through a workspace
        workspace = torch.empty(max(smd_workspace_bytes_topk_host(B, L, int(K)), 16),
                                dtype=torch.uint8, device=dev)
        rc = smd_topk_select_host(_ptr(logits), stride, _ptr(row_ends), B, L, int(K),
                                  _ptr(indices), _ptr(counts), _ptr(status), _ptr(workspace),
                                  workspace.numel(), int(copies), int(stream))
    if rc != SMD_OK:
        raise SmdError(rc, "smd_topk_select_host")
    return indices, counts
