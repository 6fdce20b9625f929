"""ctypes binding of libpaged_decode.so (include/paged_decode.h).

Argument marshalling only: every step of the decode path runs in the CUDA
library. The functions keep the C names; ``PagedDecode`` below is a small
convenience that allocates outputs and the workspace with torch (device
memory and streams are all torch is used for) and calls the same entry
points. If the library is missing this module raises instead of falling back
to anything else.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

PD_OK, PD_ERR_INVALID_ARG, PD_ERR_WORKSPACE_TOO_SMALL, PD_ERR_UNSUPPORTED, PD_ERR_CUDA, \
    PD_ERR_DEVICE_FLAG = range(6)
PD_LAYOUT_NHD, PD_LAYOUT_HND = 0, 1
PD_KV_BF16, PD_KV_FP8_E4M3 = 0, 1
PD_ATTN_GQA, PD_ATTN_MLA, PD_ATTN_PREFILL = 0, 1, 2
PD_MERGE_AUTO, PD_MERGE_FUSED, PD_MERGE_KERNEL = 0, 1, 2
PD_SCHED_AUTO, PD_SCHED_STATIC, PD_SCHED_QUEUE = 0, 1, 2
# PD_NO_ALLOC_MAX_WORKSPACE_BYTES: the largest workspace paged_decode_run_no_alloc serves
NO_ALLOC_MAX_WORKSPACE_BYTES = 32 << 20
DEVICE_ERRORS = {0: "ok", 1: "bad page id", 2: "seq_lens differs from the plan",
                 3: "q_indptr differs from the plan", 4: "workspace holds another plan",
                 5: "device wait timed out"}


class pd_problem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "kind", "batch", "num_q_heads", "num_kv_heads", "head_dim_qk", "head_dim_v", "page_size",
        "num_pages", "max_pages_per_seq", "max_kv_len", "layout", "kv_dtype", "max_splits",
        "num_sms", "merge_mode", "schedule")] + [("k_page_stride", ctypes.c_int64),
                                                  ("v_page_stride", ctypes.c_int64)]


class pd_append_problem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "num_kv_heads", "head_dim", "page_size", "num_pages", "max_pages_per_seq", "layout",
        "kv_dtype")] + [("k_page_stride", ctypes.c_int64), ("v_page_stride", ctypes.c_int64)]


class pd_plan_info(ctypes.Structure):
    _fields_ = [("num_units", ctypes.c_int32), ("num_items", ctypes.c_int32),
                ("num_ctas", ctypes.c_int32), ("tile_tokens", ctypes.c_int32),
                ("max_splits_used", ctypes.c_int32), ("rows_per_unit", ctypes.c_int32),
                ("partial_rows", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("plan_id", ctypes.c_uint64), ("merge_mode", ctypes.c_int32),
                ("launches_per_run", ctypes.c_int32)]


class PdError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        detail = ""
        if status == PD_ERR_CUDA:
            try:
                detail = " [" + load().paged_decode_last_cuda_error().decode() + "]"
            except Exception:
                pass
        super().__init__(f"{fn} failed: {status_string(status)} ({status}){detail}")


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(path: Optional[str] = None):
    """Load the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"{p} is missing: build it with paged_kv_cache_199_gb300.build.build()")
    lib = ctypes.CDLL(p)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    PP = ctypes.POINTER(ctypes.c_void_p)
    lib.paged_decode_plan.argtypes = [ctypes.POINTER(pd_problem), vp, vp, PP]
    lib.paged_decode_plan.restype = i32
    lib.paged_decode_workspace_size.argtypes = [vp]
    lib.paged_decode_workspace_size.restype = sz
    lib.paged_decode_plan_get_info.argtypes = [vp, ctypes.POINTER(pd_plan_info)]
    lib.paged_decode_plan_get_info.restype = i32
    lib.paged_decode_plan_get_items.argtypes = [vp, vp]
    lib.paged_decode_plan_get_items.restype = i32
    lib.paged_decode_plan_upload.argtypes = [vp, vp, sz, vp]
    lib.paged_decode_plan_upload.restype = i32
    lib.paged_decode_run.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp,
                                     vp, sz, vp]
    lib.paged_decode_run.restype = i32
    lib.paged_decode_run_no_alloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp]
    lib.paged_decode_run_no_alloc.restype = i32
    lib.mla_decode_run.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, sz, vp]
    lib.mla_decode_run.restype = i32
    lib.paged_decode_run_sinks.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp, vp,
                                           sz, vp]
    lib.paged_decode_run_sinks.restype = i32
    lib.mla_decode_run_sinks.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, sz, vp]
    lib.mla_decode_run_sinks.restype = i32
    lib.mla_decode_run_fp8.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.mla_decode_run_fp8.restype = i32
    lib.paged_prefill_run.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, sz, vp]
    lib.paged_prefill_run.restype = i32
    lib.paged_decode_merge_states.argtypes = [vp, vp, i32, i64, i32, vp, vp, vp]
    lib.paged_decode_merge_states.restype = i32
    lib.paged_decode_read_error.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i32), vp]
    lib.paged_decode_read_error.restype = i32
    lib.paged_kv_append.argtypes = [ctypes.POINTER(pd_append_problem), vp, vp, i32, vp, vp, vp, vp, vp, vp, vp,
                                    i32, vp, vp]
    lib.paged_kv_append.restype = i32
    lib.paged_decode_plan_destroy.argtypes = [vp]
    lib.paged_decode_plan_destroy.restype = None
    lib.pd_status_string.argtypes = [i32]
    lib.pd_status_string.restype = ctypes.c_char_p
    lib.paged_decode_version.argtypes = []
    lib.paged_decode_version.restype = i32
    lib.paged_decode_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.paged_decode_set_wait_limit_ns.restype = i32
    lib.paged_decode_last_cuda_error.argtypes = []
    lib.paged_decode_last_cuda_error.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().pd_status_string(int(status)).decode()
    except ImportError:
        return str(status)


def _check(fn: str, status: int):
    if status != PD_OK:
        raise PdError(fn, status)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ---- C entry points under their own names ------------------------------------------

def paged_decode_plan(problem: pd_problem, seq_lens_host, q_indptr_host=None) -> ctypes.c_void_p:
    """seq_lens_host / q_indptr_host: int32 numpy arrays (host)."""
    import numpy as np
    lib = load()
    sl = np.ascontiguousarray(seq_lens_host, dtype=np.int32)
    qi = None if q_indptr_host is None else np.ascontiguousarray(q_indptr_host, dtype=np.int32)
    plan = ctypes.c_void_p()
    st = lib.paged_decode_plan(ctypes.byref(problem), sl.ctypes.data if sl.size else None,
                               None if qi is None else qi.ctypes.data, ctypes.byref(plan))
    _check("paged_decode_plan", st)
    return plan


def paged_decode_workspace_size(plan) -> int:
    return int(load().paged_decode_workspace_size(plan))


def paged_decode_plan_get_info(plan) -> pd_plan_info:
    info = pd_plan_info()
    _check("paged_decode_plan_get_info", load().paged_decode_plan_get_info(plan, ctypes.byref(info)))
    return info


def paged_decode_plan_get_items(plan):
    import numpy as np
    n = paged_decode_plan_get_info(plan).num_items
    out = np.zeros((max(n, 1), 4), np.int32)
    _check("paged_decode_plan_get_items", load().paged_decode_plan_get_items(plan, out.ctypes.data))
    return out[:n]


def paged_decode_plan_upload(plan, workspace, workspace_bytes=None, stream=None):
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    _check("paged_decode_plan_upload",
           load().paged_decode_plan_upload(plan, _ptr(workspace), nbytes, _stream_ptr(stream)))


def paged_decode_run(plan, q, k_pool, v_pool, block_tables, seq_lens, q_indptr, sm_scale, k_scale,
                     v_scale, out, lse, workspace, workspace_bytes=None, stream=None):
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    _check("paged_decode_run", load().paged_decode_run(
        plan, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(seq_lens),
        _ptr(q_indptr), float(sm_scale), _ptr(k_scale), _ptr(v_scale), _ptr(out), _ptr(lse),
        _ptr(workspace), nbytes, _stream_ptr(stream)))


def paged_decode_run_no_alloc(plan, q, k_pool, v_pool, block_tables, seq_lens, q_indptr, sm_scale, k_scale,
                              v_scale, out, lse, stream=None):
    """paged_decode_run with the library's own fixed workspace (no caller
    workspace, nothing allocated); returns the status instead of raising so
    that callers can test refusals."""
    return int(load().paged_decode_run_no_alloc(
        plan, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(seq_lens), _ptr(q_indptr),
        float(sm_scale), _ptr(k_scale), _ptr(v_scale), _ptr(out), _ptr(lse), _stream_ptr(stream)))


def mla_decode_run(plan, q, kv_pool, block_tables, seq_lens, q_indptr, sm_scale, out, lse,
                   workspace, workspace_bytes=None, stream=None):
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    _check("mla_decode_run", load().mla_decode_run(
        plan, _ptr(q), _ptr(kv_pool), _ptr(block_tables), _ptr(seq_lens), _ptr(q_indptr),
        float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace), nbytes, _stream_ptr(stream)))


def paged_decode_run_sinks(plan, q, k_pool, v_pool, block_tables, seq_lens, q_indptr, sm_scale, k_scale,
                           v_scale, sinks, out, lse, workspace, workspace_bytes=None, stream=None):
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    _check("paged_decode_run_sinks", load().paged_decode_run_sinks(
        plan, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(seq_lens),
        _ptr(q_indptr), float(sm_scale), _ptr(k_scale), _ptr(v_scale), _ptr(sinks), _ptr(out), _ptr(lse),
        _ptr(workspace), nbytes, _stream_ptr(stream)))


def mla_decode_run_sinks(plan, q, kv_pool, block_tables, seq_lens, q_indptr, sm_scale, sinks, out, lse,
                         workspace, workspace_bytes=None, stream=None):
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    _check("mla_decode_run_sinks", load().mla_decode_run_sinks(
        plan, _ptr(q), _ptr(kv_pool), _ptr(block_tables), _ptr(seq_lens), _ptr(q_indptr),
        float(sm_scale), _ptr(sinks), _ptr(out), _ptr(lse), _ptr(workspace), nbytes, _stream_ptr(stream)))


def mla_decode_run_fp8(plan, q, kv_pool, block_tables, seq_lens, q_indptr, sm_scale, q_scale, kv_scale, sinks,
                       out, lse, workspace, workspace_bytes=None, stream=None):
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    _check("mla_decode_run_fp8", load().mla_decode_run_fp8(
        plan, _ptr(q), _ptr(kv_pool), _ptr(block_tables), _ptr(seq_lens), _ptr(q_indptr), float(sm_scale),
        _ptr(q_scale), _ptr(kv_scale), _ptr(sinks), _ptr(out), _ptr(lse), _ptr(workspace), nbytes,
        _stream_ptr(stream)))


def paged_prefill_run(plan, q, k_pool, v_pool, block_tables, seq_lens, q_indptr, sm_scale, sinks, out, lse,
                      workspace, workspace_bytes=None, stream=None):
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    _check("paged_prefill_run", load().paged_prefill_run(
        plan, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(seq_lens), _ptr(q_indptr),
        float(sm_scale), _ptr(sinks), _ptr(out), _ptr(lse), _ptr(workspace), nbytes, _stream_ptr(stream)))


def paged_decode_merge_states(v_states, s_states, out, lse_out=None, stream=None):
    """v_states fp32 [S, rows, dim], s_states fp32 [S, rows] -> out bf16 [rows, dim]."""
    S, rows, dim = v_states.shape
    _check("paged_decode_merge_states", load().paged_decode_merge_states(
        _ptr(v_states), _ptr(s_states), S, rows, dim, _ptr(out), _ptr(lse_out), _stream_ptr(stream)))


def paged_kv_append(k_new, v_new, q_indptr, seq_lens, block_tables, k_pool, v_pool=None, *, num_kv_heads,
                    head_dim, page_size, layout=PD_LAYOUT_NHD, kv_dtype=PD_KV_BF16, k_scale=None, v_scale=None,
                    zero_tail=False, error_word=None, k_page_stride=0, v_page_stride=0, stream=None):
    """Write the new tokens' K/V rows (bf16 [total_new, Hkv, D]) into the pools."""
    prob = pd_append_problem(batch=int(seq_lens.shape[0]), num_kv_heads=num_kv_heads, head_dim=head_dim,
                             page_size=page_size, num_pages=int(k_pool.shape[0]),
                             max_pages_per_seq=int(block_tables.shape[1]), layout=layout, kv_dtype=kv_dtype,
                             k_page_stride=k_page_stride, v_page_stride=v_page_stride)
    total_new = 0 if k_new is None else int(k_new.shape[0])
    _check("paged_kv_append", load().paged_kv_append(
        ctypes.byref(prob), _ptr(k_new), _ptr(v_new), total_new, _ptr(q_indptr), _ptr(seq_lens),
        _ptr(block_tables), _ptr(k_scale), _ptr(v_scale), _ptr(k_pool), _ptr(v_pool), 1 if zero_tail else 0,
        _ptr(error_word), _stream_ptr(stream)))


def paged_decode_read_error(workspace, stream=None):
    """Returns (code, info); code 0 means no device error. Synchronises."""
    code, info = ctypes.c_int32(0), ctypes.c_int32(-1)
    st = load().paged_decode_read_error(_ptr(workspace), ctypes.byref(code), ctypes.byref(info),
                                        _stream_ptr(stream))
    if st not in (PD_OK, PD_ERR_DEVICE_FLAG):
        raise PdError("paged_decode_read_error", st)
    return int(code.value), int(info.value)


def paged_decode_set_wait_limit_ns(limit_ns: int) -> int:
    """Limit of the kernels' pipeline waits for later launches (0: the default)."""
    return int(load().paged_decode_set_wait_limit_ns(int(limit_ns)))


def paged_decode_plan_destroy(plan):
    if plan:
        load().paged_decode_plan_destroy(plan)


# ---- convenience ------------------------------------------------------------------------

def make_problem(inputs, *, max_splits=0, num_sms=0, merge_mode=PD_MERGE_AUTO,
                 schedule=PD_SCHED_AUTO, prefill=False) -> pd_problem:
    """pd_problem for a ``workloads.DecodeInputs`` batch (``prefill``: a GQA
    batch run by the tensor-core prefill kernel)."""
    p = pd_problem()
    p.kind = PD_ATTN_MLA if inputs.kind == "mla" else PD_ATTN_PREFILL if prefill else PD_ATTN_GQA
    p.batch = inputs.batch
    p.num_q_heads = inputs.num_q_heads
    p.num_kv_heads = inputs.num_kv_heads
    p.head_dim_qk = inputs.head_dim_qk
    p.head_dim_v = inputs.head_dim_v
    p.page_size = inputs.page_size
    p.num_pages = inputs.num_pages
    p.max_pages_per_seq = inputs.max_pages_per_seq
    p.max_kv_len = max(inputs.max_kv_len, 0)
    p.layout = PD_LAYOUT_HND if inputs.layout == "HND" else PD_LAYOUT_NHD
    p.kv_dtype = PD_KV_FP8_E4M3 if inputs.kv_dtype == "e4m3" else PD_KV_BF16
    p.max_splits = max_splits
    p.num_sms = num_sms
    p.merge_mode = merge_mode
    p.schedule = schedule
    return p


class PagedDecode:
    """Plan + workspace + run for one batch of ``workloads.DecodeInputs``.

    Owns the plan handle and a torch-allocated workspace on the inputs'
    device. ``run`` enqueues the CUDA kernels on the current stream.
    """

    def __init__(self, inputs, *, max_splits=0, num_sms=0, merge_mode=PD_MERGE_AUTO,
                 schedule=PD_SCHED_AUTO, device=None, upload=True, prefill=False):
        self.inputs = inputs
        self.prefill = prefill
        self.problem = make_problem(inputs, max_splits=max_splits, num_sms=num_sms,
                                    merge_mode=merge_mode, schedule=schedule, prefill=prefill)
        self.plan = paged_decode_plan(self.problem, inputs.seq_lens_host(), inputs.q_indptr_host())
        self.info = paged_decode_plan_get_info(self.plan)
        dev = device if device is not None else inputs.q.device
        self.workspace = torch.empty(max(self.info.workspace_bytes, 256), dtype=torch.uint8, device=dev)
        self.k_scale_t = self.v_scale_t = self.q_scale_t = None
        if inputs.kv_dtype == "e4m3":
            self.k_scale_t = torch.tensor([inputs.k_scale], dtype=torch.float32, device=dev)
            self.v_scale_t = torch.tensor([inputs.v_scale], dtype=torch.float32, device=dev)
            self.q_scale_t = torch.tensor([getattr(inputs, "q_scale", 1.0)], dtype=torch.float32, device=dev)
        if upload:
            self.upload()

    def upload(self, stream=None):
        paged_decode_plan_upload(self.plan, self.workspace, stream=stream)

    def alloc_outputs(self, with_lse=True):
        x = self.inputs
        out = torch.empty((x.total_q, x.num_q_heads, x.head_dim_v), dtype=torch.bfloat16, device=x.q.device)
        lse = torch.empty((x.total_q, x.num_q_heads), dtype=torch.float32, device=x.q.device) if with_lse else None
        return out, lse

    def run(self, out=None, lse=None, with_lse=True, stream=None, q=None, seq_lens=None,
            block_tables=None, q_indptr=None):
        x = self.inputs
        if out is None:
            out, lse = self.alloc_outputs(with_lse)
        q = x.q if q is None else q
        seq_lens = x.seq_lens if seq_lens is None else seq_lens
        block_tables = x.block_tables if block_tables is None else block_tables
        q_indptr = x.q_indptr if q_indptr is None else q_indptr
        sinks = getattr(x, "sinks", None)
        if self.prefill:
            paged_prefill_run(self.plan, q, x.k_pool, x.v_pool, block_tables, seq_lens, q_indptr, x.sm_scale,
                              sinks, out, lse, self.workspace, stream=stream)
        elif x.kind == "mla" and x.kv_dtype == "e4m3":
            mla_decode_run_fp8(self.plan, q, x.k_pool, block_tables, seq_lens, q_indptr, x.sm_scale,
                               self.q_scale_t, self.k_scale_t, sinks, out, lse, self.workspace, stream=stream)
        elif x.kind == "mla" and sinks is None:
            mla_decode_run(self.plan, q, x.k_pool, block_tables, seq_lens, q_indptr, x.sm_scale,
                           out, lse, self.workspace, stream=stream)
        elif x.kind == "mla":
            mla_decode_run_sinks(self.plan, q, x.k_pool, block_tables, seq_lens, q_indptr, x.sm_scale,
                                 sinks, out, lse, self.workspace, stream=stream)
        elif sinks is None:
            paged_decode_run(self.plan, q, x.k_pool, x.v_pool, block_tables, seq_lens, q_indptr,
                             x.sm_scale, self.k_scale_t, self.v_scale_t, out, lse, self.workspace,
                             stream=stream)
        else:
            paged_decode_run_sinks(self.plan, q, x.k_pool, x.v_pool, block_tables, seq_lens, q_indptr,
                                   x.sm_scale, self.k_scale_t, self.v_scale_t, sinks, out, lse,
                                   self.workspace, stream=stream)
        return out, lse

    def read_error(self, stream=None):
        return paged_decode_read_error(self.workspace, stream)

    def close(self):
        if getattr(self, "plan", None):
            paged_decode_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
