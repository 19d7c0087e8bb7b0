"""CPU oracle for sparse MLA decode (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The decode library never does: it shares no code
with the oracle, and the product path fails loudly when its CUDA library is
missing instead of falling back here.

The arithmetic lives in ``smd_oracle.c`` (plain C, fp64 sums); this module
compiles it with gcc on first use and wraps it with ctypes and numpy.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "smd_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

MODE_RECIPE = 0
MODE_UNQUANT = 1


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u8p = ctypes.POINTER(ctypes.c_uint8)
            i32p = ctypes.POINTER(ctypes.c_int32)
            lib.smo_e4m3_decode.restype = ctypes.c_double
            lib.smo_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.smo_e4m3_encode.restype = ctypes.c_uint8
            lib.smo_e4m3_encode.argtypes = [ctypes.c_double]
            lib.smo_bf16_rne.restype = ctypes.c_uint16
            lib.smo_bf16_rne.argtypes = [ctypes.c_double]
            lib.smo_scale_log2.restype = ctypes.c_float
            lib.smo_scale_log2.argtypes = [ctypes.c_float] * 3
            lib.smo_max_threads.restype = ctypes.c_int
            lib.smo_max_threads.argtypes = []
            lib.smo_sparse_mla_decode.restype = ctypes.c_int
            lib.smo_sparse_mla_decode.argtypes = [
                u8p, u8p, ctypes.c_int64, i32p, ctypes.c_int32, i32p,
                ctypes.c_int32, ctypes.c_int32,
                ctypes.c_float, ctypes.c_float, ctypes.c_float,
                ctypes.c_int, ctypes.c_int,
                ctypes.POINTER(ctypes.c_uint16), ctypes.POINTER(ctypes.c_double),
                ctypes.POINTER(ctypes.c_double)]
            lib.smo_sparse_mla_decode_bf16q.restype = ctypes.c_int
            lib.smo_sparse_mla_decode_bf16q.argtypes = [
                ctypes.POINTER(ctypes.c_uint16), u8p, ctypes.c_int64, i32p, ctypes.c_int32,
                i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_float,
                ctypes.c_int, ctypes.c_int,
                ctypes.POINTER(ctypes.c_uint16), ctypes.POINTER(ctypes.c_double),
                ctypes.POINTER(ctypes.c_double), i32p]
            lib.smo_q_split.restype = ctypes.c_int
            lib.smo_q_split.argtypes = [ctypes.POINTER(ctypes.c_uint16), u8p, u8p]
            lib.smo_q_split_exponent.restype = ctypes.c_int
            lib.smo_q_split_exponent.argtypes = [ctypes.c_double]
            lib.smo_row_head_terms.restype = ctypes.c_int32
            lib.smo_row_head_terms.argtypes = [
                u8p, u8p, ctypes.c_int64, i32p, ctypes.c_int32, i32p,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                ctypes.c_float, ctypes.c_float, ctypes.c_float,
                ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_float),
                ctypes.POINTER(ctypes.c_float), u8p, ctypes.POINTER(ctypes.c_float)]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def e4m3_decode(code: int) -> float:
    return float(_load().smo_e4m3_decode(int(code) & 0xFF))


def e4m3_encode(x: float) -> int:
    return int(_load().smo_e4m3_encode(float(x)))


def bf16_rne(x: float) -> int:
    return int(_load().smo_bf16_rne(float(x)))


def scale_log2(sm_scale: float, q_scale: float, k_scale: float) -> float:
    return float(_load().smo_scale_log2(sm_scale, q_scale, k_scale))


def max_threads() -> int:
    return int(_load().smo_max_threads())


def _inputs(q8, kv8, indices, counts):
    q8 = np.ascontiguousarray(q8, np.uint8)
    kv8 = np.ascontiguousarray(kv8, np.uint8)
    indices = np.ascontiguousarray(indices, np.int32)
    counts = np.ascontiguousarray(counts, np.int32)
    assert q8.ndim == 3 and q8.shape[2] == 576, q8.shape
    assert kv8.ndim == 2 and kv8.shape[1] == 576, kv8.shape
    assert indices.ndim == 2 and indices.shape[0] >= q8.shape[0]
    assert counts.shape[0] >= q8.shape[0]
    return q8, kv8, indices, counts


def sparse_mla_decode(q8, kv8, indices, counts, sm_scale, q_scale, k_scale,
                      mode: int = MODE_RECIPE, threads: int = 0):
    """Returns (out_bf16 uint16 [B,H,512], out_f64 float64 [B,H,512],
    lse float64 [B,H])."""
    q8, kv8, indices, counts = _inputs(q8, kv8, indices, counts)
    B, H = q8.shape[0], q8.shape[1]
    W = indices.shape[1]
    out16 = np.zeros((B, H, 512), np.uint16)
    out64 = np.zeros((B, H, 512), np.float64)
    lse = np.zeros((B, H), np.float64)
    if B * H == 0:
        return out16, out64, lse
    rc = _load().smo_sparse_mla_decode(
        _ptr(q8, ctypes.c_uint8), _ptr(kv8, ctypes.c_uint8), kv8.shape[0],
        _ptr(indices, ctypes.c_int32), W, _ptr(counts, ctypes.c_int32), B, H,
        sm_scale, q_scale, k_scale, int(mode), int(threads),
        _ptr(out16, ctypes.c_uint16), _ptr(out64, ctypes.c_double),
        _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle: an index of a valid entry lies outside the pool")
    return out16, out64, lse


def sparse_mla_decode_bf16q(q16, kv8, indices, counts, sm_scale, k_scale,
                            mode: int = MODE_RECIPE, threads: int = 0):
    """The decode with a BF16 query (q16: bf16 bits, uint16 [B,H,576]), split
    per (row, head) into E4M3 hi + lo (the mla_attn page's q_split). Returns
    (out_bf16, out_f64, lse, k [B,H] the split exponents)."""
    q16 = np.ascontiguousarray(q16, np.uint16)
    _, kv8, indices, counts = _inputs(np.zeros((q16.shape[0], q16.shape[1], 576), np.uint8),
                                      kv8, indices, counts)
    assert q16.ndim == 3 and q16.shape[2] == 576, q16.shape
    B, H = q16.shape[0], q16.shape[1]
    W = indices.shape[1]
    out16 = np.zeros((B, H, 512), np.uint16)
    out64 = np.zeros((B, H, 512), np.float64)
    lse = np.zeros((B, H), np.float64)
    ks = np.zeros((B, H), np.int32)
    if B * H == 0:
        return out16, out64, lse, ks
    rc = _load().smo_sparse_mla_decode_bf16q(
        _ptr(q16, ctypes.c_uint16), _ptr(kv8, ctypes.c_uint8), kv8.shape[0],
        _ptr(indices, ctypes.c_int32), W, _ptr(counts, ctypes.c_int32), B, H,
        sm_scale, k_scale, int(mode), int(threads),
        _ptr(out16, ctypes.c_uint16), _ptr(out64, ctypes.c_double),
        _ptr(lse, ctypes.c_double), _ptr(ks, ctypes.c_int32))
    if rc != 0:
        raise ValueError("oracle: an index of a valid entry lies outside the pool")
    return out16, out64, lse, ks


def q_split(q_row16) -> tuple[np.ndarray, np.ndarray, int]:
    """One 576-column bf16 query row -> (hi codes, lo codes, k)."""
    q_row16 = np.ascontiguousarray(q_row16, np.uint16)
    assert q_row16.shape == (576,)
    hi = np.zeros(576, np.uint8)
    lo = np.zeros(576, np.uint8)
    k = _load().smo_q_split(_ptr(q_row16, ctypes.c_uint16), _ptr(hi, ctypes.c_uint8),
                            _ptr(lo, ctypes.c_uint8))
    return hi, lo, int(k)


def q_split_exponent(amax: float) -> int:
    return int(_load().smo_q_split_exponent(float(amax)))


def row_head_terms(q8, kv8, indices, counts, b, h, sm_scale, q_scale, k_scale):
    """Per-key (S exact, s fp32, P fp32, P8 code) and the anchor m of one
    (row, head)."""
    q8, kv8, indices, counts = _inputs(q8, kv8, indices, counts)
    W = indices.shape[1]
    n_max = max(W, 1)
    S = np.zeros(n_max, np.float64)
    s = np.zeros(n_max, np.float32)
    P = np.zeros(n_max, np.float32)
    P8 = np.zeros(n_max, np.uint8)
    m = ctypes.c_float(0.0)
    n = _load().smo_row_head_terms(
        _ptr(q8, ctypes.c_uint8), _ptr(kv8, ctypes.c_uint8), kv8.shape[0],
        _ptr(indices, ctypes.c_int32), W, _ptr(counts, ctypes.c_int32),
        q8.shape[1], int(b), int(h), sm_scale, q_scale, k_scale,
        _ptr(S, ctypes.c_double), _ptr(s, ctypes.c_float), _ptr(P, ctypes.c_float),
        _ptr(P8, ctypes.c_uint8), ctypes.byref(m))
    if n < 0:
        raise ValueError("oracle: index out of range")
    return S[:n], s[:n], P[:n], P8[:n], float(m.value)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)
