"""The allocation-free entry point, paged_decode_run_no_alloc, checked through
the C ABI against paged_decode_run on the same inputs.

It serves callers of this library that may not allocate device memory (a
runtime that reserves all device memory up front, a plugin whose framework
owns the allocator): its workspace is a fixed array inside the library. This
file is collected last so that a stop-at-first-failure run has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_cache_199_gb300 import binding as B
from paged_kv_cache_199_gb300 import build
from paged_kv_cache_199_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_WORKSPACE = 32 << 20  # PD_NO_ALLOC_MAX_WORKSPACE_BYTES in include/paged_decode.h


def _lib():
    build.build()
    lib = B.load()
    vp = ctypes.c_void_p
    fn = lib.paged_decode_run_no_alloc
    fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp]
    fn.restype = ctypes.c_int32
    return lib


def _p(t):
    return None if t is None else t.data_ptr()


def _no_alloc(lib, dec, out, lse):
    x = dec.inputs
    return lib.paged_decode_run_no_alloc(
        dec.plan, _p(x.q), _p(x.k_pool), _p(x.v_pool), _p(x.block_tables), _p(x.seq_lens),
        _p(x.q_indptr), float(x.sm_scale), _p(dec.k_scale_t), _p(dec.v_scale_t), _p(out), _p(lse),
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name", ["gqa8", "ragged", "fp8"])
def test_no_alloc_matches_run(name):
    lib = _lib()
    x = W.workload(name, device="cuda", small=True)
    dec = B.PagedDecode(x, num_sms=300)  # a split plan, so the scratch holds partial states
    assert dec.info.workspace_bytes <= MAX_WORKSPACE
    ref_out, ref_lse = dec.run()
    torch.cuda.synchronize()
    atol = rtol = 1e-2 if x.kv_dtype == "bf16" else 0.1
    for call in range(2):
        out, lse = dec.alloc_outputs(True)
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        assert _no_alloc(lib, dec, out, lse) == B.PD_OK
        torch.cuda.synchronize()
        np.testing.assert_allclose(out.float().cpu().numpy(), ref_out.float().cpu().numpy(),
                                   atol=atol, rtol=rtol, err_msg=f"{name} call {call}")
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), atol=2e-3, rtol=2e-3)


def test_no_alloc_rejects_oversized_plan():
    lib = _lib()
    p = B.pd_problem()
    p.kind = B.PD_ATTN_GQA
    p.batch, p.num_q_heads, p.num_kv_heads = 2048, 64, 8
    p.head_dim_qk = p.head_dim_v = 128
    p.page_size, p.max_pages_per_seq = 64, 256
    p.num_pages, p.max_kv_len = 2048 * 256, 16384
    p.layout, p.num_sms, p.max_splits = B.PD_LAYOUT_HND, 4000, 16
    plan = B.paged_decode_plan(p, np.full(2048, 16384, np.int32))
    try:
        assert B.paged_decode_workspace_size(plan) > MAX_WORKSPACE
        canary = torch.full((4,), 7.0, device="cuda")
        st = lib.paged_decode_run_no_alloc(plan, *([canary.data_ptr()] * 6), 1.0, None, None,
                                           canary.data_ptr(), None,
                                           torch.cuda.current_stream().cuda_stream)
        assert st == B.PD_ERR_WORKSPACE_TOO_SMALL
        torch.cuda.synchronize()
        assert torch.equal(canary, torch.full((4,), 7.0, device="cuda"))
    finally:
        B.paged_decode_plan_destroy(plan)
