"""The allocation-free entry point, paged_decode_run_no_alloc, checked through
the C ABI against paged_decode_run on the same inputs and plan.

It serves callers of this library that may not allocate device memory (a
runtime that reserves all device memory up front and forbids later
cudaMalloc calls, or a plugin whose host framework owns the allocator): its
workspace is a fixed array inside the library. It runs the same kernels on
the same plan as paged_decode_run, so both must give identical bits, on every
call. This file is collected last so that a stop-at-first-failure run has
already run every other test.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_199_gb300 import binding as B
from paged_kv_cache_199_gb300 import build
from paged_kv_cache_199_gb300 import workloads as W
from tests.helpers import assert_close, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    B.load()


def _no_alloc(dec, out, lse):
    x = dec.inputs
    return B.paged_decode_run_no_alloc(dec.plan, x.q, x.k_pool, x.v_pool, x.block_tables, x.seq_lens,
                                       x.q_indptr, x.sm_scale, dec.k_scale_t, dec.v_scale_t, out, lse)


@pytest.mark.parametrize("name", ["gqa8", "ragged", "fp8"])
def test_no_alloc_matches_run(name):
    x = W.workload(name, device="cuda", small=True)
    dec = B.PagedDecode(x, num_sms=300)  # a split plan, so the scratch holds partial states
    assert dec.info.workspace_bytes <= B.NO_ALLOC_MAX_WORKSPACE_BYTES
    assert dec.info.partial_rows > 0
    ref_out, ref_lse = dec.run()
    torch.cuda.synchronize()
    assert dec.read_error()[0] == 0
    for call in range(2):   # the second call finds the first call's contents in the array
        out, lse = dec.alloc_outputs(True)
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        assert _no_alloc(dec, out, lse) == B.PD_OK
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out), f"{name} call {call}: output bits differ from paged_decode_run"
        assert torch.equal(lse, ref_lse), f"{name} call {call}: LSE bits differ from paged_decode_run"
    if name == "ragged":
        o_ref, l_ref, _ = run_oracle(x)
        assert_close(out, lse, o_ref, l_ref, x.kv_dtype, "no-alloc entry point against the oracle")


def test_no_alloc_rejects_oversized_plan():
    p = B.pd_problem()
    p.kind = B.PD_ATTN_GQA
    p.batch, p.num_q_heads, p.num_kv_heads = 2048, 64, 8
    p.head_dim_qk = p.head_dim_v = 128
    p.page_size, p.max_pages_per_seq = 64, 256
    p.num_pages, p.max_kv_len = 2048 * 256, 16384
    p.layout, p.num_sms, p.max_splits = B.PD_LAYOUT_HND, 4000, 16
    plan = B.paged_decode_plan(p, np.full(2048, 16384, np.int32))
    try:
        assert B.paged_decode_workspace_size(plan) > B.NO_ALLOC_MAX_WORKSPACE_BYTES
        canary = torch.full((4,), 7.0, device="cuda")
        ptr = canary.data_ptr()
        st = B.paged_decode_run_no_alloc(plan, ptr, ptr, ptr, ptr, ptr, ptr, 1.0, None, None, ptr, None)
        assert st == B.PD_ERR_WORKSPACE_TOO_SMALL
        torch.cuda.synchronize()
        assert torch.equal(canary, torch.full((4,), 7.0, device="cuda"))
    finally:
        B.paged_decode_plan_destroy(plan)
