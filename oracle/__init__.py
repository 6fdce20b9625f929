"""FP64 CPU oracle for paged decode attention (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package. The CUDA library never calls it, and it never calls the
CUDA library: the two share nothing but the seeded input generator.

The arithmetic lives in ``paged_attention_oracle.c`` (plain C99, double
precision, OpenMP over query heads). This module builds it with gcc and wraps
it with ctypes; it adds no arithmetic of its own beyond the
``merge_states`` wrapper's argument marshalling.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_attention_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

NHD, HND = 0, 1
BF16, E4M3 = 0, 1

STATUS = {0: "ok", 1: "bad argument", 2: "q_len > seq_len", 3: "page id out of range"}


class OracleError(RuntimeError):
    pass


def build(out_path: str = _LIB_PATH, mutation: int = 0, quiet: bool = True) -> str:
    """Compile the oracle into a shared library (gcc, -O2, OpenMP).

    ``mutation`` > 0 builds a copy with one planted mistake; the pin tests use
    it to show that each plausible mistake fails at least one pin.
    """
    cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
           f"-DORACLE_MUTATION={int(mutation)}", _SRC, "-o", out_path, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise OracleError("oracle build failed:\n" + res.stderr)
    return out_path


def _declare(lib):
    i32, i64, dbl, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
    lib.oracle_paged_decode.restype = i32
    lib.oracle_paged_decode.argtypes = [i32] * 10 + [vp, vp, vp, i64, i64, i64, i64, vp, vp, vp,
                                                     dbl, dbl, dbl, vp, i64, i64, vp, vp, i32]
    lib.oracle_mla_decode.restype = i32
    lib.oracle_mla_decode.argtypes = [i32] * 8 + [dbl, dbl] + [vp, vp, vp, vp, vp, dbl, vp, vp, vp, i32]
    lib.oracle_merge_states.restype = None
    lib.oracle_merge_states.argtypes = [i32, i64, i32, vp, vp, vp, vp]
    lib.oracle_bf16_to_double.restype = dbl
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_e4m3_to_double.restype = dbl
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
    lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
    lib.oracle_paged_append.restype = i32
    lib.oracle_paged_append.argtypes = [i32] * 8 + [vp] * 5 + [ctypes.c_float, ctypes.c_float, vp, vp, i64, i64, i32]
    lib.oracle_max_threads.restype = i32
    lib.oracle_max_threads.argtypes = []
    return lib


def load_library(path: str | None = None):
    """Load (building if needed) the oracle; ``path`` selects another build."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def max_threads(lib=None) -> int:
    return int((lib or load_library()).oracle_max_threads())


def paged_decode(q, k_pool, v_pool, block_tables, seq_lens, q_indptr=None, *,
                 num_q_heads, num_kv_heads, head_dim_qk, head_dim_v, page_size,
                 layout, kv_dtype=BF16, sm_scale, k_scale=1.0, v_scale=1.0,
                 k_page_stride=None, v_page_stride=None, k_row_stride=None,
                 v_row_stride=None, num_pages=None, kv_range=None, sinks=None,
                 num_threads=0, lib=None):
    """Evaluate paged GQA decode in FP64.

    q: uint16 bf16 bits [total_q, Hq, Dqk]; k_pool / v_pool: uint16 (bf16) or
    uint8 (e4m3) arrays whose first axis is the page; block_tables
    [B, max_pages] int32; seq_lens [B] int32; q_indptr [B+1] int32 or None.
    Strides are in elements and default to a compact pool.
    Returns (out [total_q, Hq, Dv] float64, lse [total_q, Hq] float64).
    """
    lib = lib or load_library()
    elem = np.uint16 if kv_dtype == BF16 else np.uint8
    q = _c(q, np.uint16)
    k_pool = _c(k_pool, elem)
    v_pool = _c(v_pool, elem)
    block_tables = _c(block_tables, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    q_indptr = _c(q_indptr, np.int32)
    batch = int(seq_lens.shape[0])
    max_pages = int(block_tables.shape[1]) if block_tables.ndim == 2 else 0
    if num_pages is None:
        num_pages = int(k_pool.shape[0])
    if k_row_stride is None:
        k_row_stride = head_dim_qk
    if v_row_stride is None:
        v_row_stride = head_dim_v
    if k_page_stride is None:
        k_page_stride = int(np.prod(k_pool.shape[1:]))
    if v_page_stride is None:
        v_page_stride = int(np.prod(v_pool.shape[1:]))
    total_q = int(q_indptr[-1]) if q_indptr is not None else batch
    out = np.zeros((total_q, num_q_heads, head_dim_v), np.float64)
    lse = np.zeros((total_q, num_q_heads), np.float64)
    lo, hi = (0, -1) if kv_range is None else kv_range
    st = lib.oracle_paged_decode(
        batch, num_q_heads, num_kv_heads, head_dim_qk, head_dim_v, page_size, num_pages,
        max_pages, layout, kv_dtype, _ptr(q), _ptr(k_pool), _ptr(v_pool), k_page_stride,
        v_page_stride, k_row_stride, v_row_stride, _ptr(block_tables), _ptr(seq_lens),
        _ptr(q_indptr), float(sm_scale), float(k_scale), float(v_scale), _ptr(_c(sinks, np.float64)),
        int(lo), int(hi), _ptr(out), _ptr(lse), int(num_threads))
    if st != 0:
        raise OracleError(f"oracle_paged_decode: {STATUS.get(st, st)}")
    return out, lse


def mla_decode(q, kv_pool, block_tables, seq_lens, q_indptr=None, *, num_heads,
               head_dim_qk=576, head_dim_v=512, page_size, sm_scale, sinks=None, kv_dtype=BF16,
               q_scale=1.0, kv_scale=1.0, num_threads=0, lib=None):
    """Evaluate MLA decode (one shared latent KV head) in FP64.

    q: uint16 [total_q, H, Dqk]; kv_pool: uint16 [num_pages, P, Dqk].
    Returns (out [total_q, H, Dv] float64, lse [total_q, H] float64).
    """
    lib = lib or load_library()
    elem = np.uint16 if kv_dtype == BF16 else np.uint8
    q = _c(q, elem)
    kv_pool = _c(kv_pool, elem)
    block_tables = _c(block_tables, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    q_indptr = _c(q_indptr, np.int32)
    batch = int(seq_lens.shape[0])
    total_q = int(q_indptr[-1]) if q_indptr is not None else batch
    out = np.zeros((total_q, num_heads, head_dim_v), np.float64)
    lse = np.zeros((total_q, num_heads), np.float64)
    st = lib.oracle_mla_decode(batch, num_heads, head_dim_qk, head_dim_v, page_size,
                               int(kv_pool.shape[0]), int(block_tables.shape[1]), int(kv_dtype),
                               float(q_scale), float(kv_scale), _ptr(q),
                               _ptr(kv_pool), _ptr(block_tables), _ptr(seq_lens),
                               _ptr(q_indptr), float(sm_scale), _ptr(_c(sinks, np.float64)),
                               _ptr(out), _ptr(lse), int(num_threads))
    if st != 0:
        raise OracleError(f"oracle_mla_decode: {STATUS.get(st, st)}")
    return out, lse


def merge_states(o_states, lse_states, lib=None):
    """Merge attention states over disjoint key ranges.

    o_states [S, rows, dim], lse_states [S, rows] -> (out [rows, dim], lse [rows]).
    """
    lib = lib or load_library()
    o_states = _c(o_states, np.float64)
    lse_states = _c(lse_states, np.float64)
    S, rows, dim = o_states.shape
    out = np.zeros((rows, dim), np.float64)
    lse = np.zeros((rows,), np.float64)
    lib.oracle_merge_states(S, rows, dim, _ptr(o_states), _ptr(lse_states), _ptr(out), _ptr(lse))
    return out, lse


def bf16_to_double(bits: int, lib=None) -> float:
    return float((lib or load_library()).oracle_bf16_to_double(int(bits)))


def e4m3_to_double(byte: int, lib=None) -> float:
    return float((lib or load_library()).oracle_e4m3_to_double(int(byte)))


def e4m3_from_float(x: float, lib=None) -> int:
    """OCP E4M3FN code of a binary32 value (RN-even, saturating to 448)."""
    return int((lib or load_library()).oracle_e4m3_from_float(float(x)))


def paged_append(k_new, v_new, block_tables, seq_lens, q_indptr, k_pool, v_pool=None, *,
                 num_kv_heads, head_dim, page_size, layout, kv_dtype=BF16, k_scale=1.0,
                 v_scale=1.0, zero_tail=False, lib=None):
    """Write new K/V rows into copies of the pools; returns (k_pool, v_pool, status).

    k_new / v_new: uint16 bf16 bits [total_new, Hkv, D] (v_new may be None);
    pools: uint16 (bf16) or uint8 (e4m3) arrays whose first axis is the page
    (compact). The inputs are not modified.
    """
    lib = lib or load_library()
    elem = np.uint16 if kv_dtype == BF16 else np.uint8
    k_new = _c(k_new, np.uint16)
    v_new = _c(v_new, np.uint16)
    kp = np.array(k_pool, dtype=elem, copy=True, order="C")
    vp = None if v_pool is None else np.array(v_pool, dtype=elem, copy=True, order="C")
    block_tables = _c(block_tables, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    q_indptr = _c(q_indptr, np.int32)
    batch = int(seq_lens.shape[0])
    st = lib.oracle_paged_append(
        batch, num_kv_heads, head_dim, page_size, int(kp.shape[0]), int(block_tables.shape[1]), layout,
        kv_dtype, _ptr(k_new), _ptr(v_new), _ptr(q_indptr), _ptr(seq_lens), _ptr(block_tables),
        float(k_scale), float(v_scale), _ptr(kp), _ptr(vp), int(np.prod(kp.shape[1:])),
        0 if vp is None else int(np.prod(vp.shape[1:])), 1 if zero_tail else 0)
    return kp, vp, int(st)
