"""Error paths of the MLA kernel (BF16 and E4M3): a bad page id or a device
sequence length that differs from the plan is reported through the error
word, the affected request's rows are zero, and every other request still
matches the oracle. The stage that carries the error is skipped by both MMA
issuers and by the softmax warps, so these cases also check that the three
stay in step (no wait runs out: the error word would read "timed out")."""
import numpy as np
import pytest
import torch

from paged_kv_cache_199_gb300 import binding as B
from paged_kv_cache_199_gb300 import workloads as W
from tests.helpers import assert_close, run_oracle

pytestmark = pytest.mark.gpu

MODES = dict(unsplit=dict(max_splits=1), split16=dict(max_splits=16, num_sms=400),
             fused=dict(max_splits=16, num_sms=400, merge_mode=B.PD_MERGE_FUSED),
             static=dict(schedule=B.PD_SCHED_STATIC, num_sms=300))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_199_gb300 import build
    build.build()
    B.load()


def _inputs(kv_dtype):
    # request 1 spans eleven 64-token pages, so page 3 is visible and falls
    # inside an item (not only at its first or last tile)
    return W.make_mla_inputs(seed=31, seq_lens=[300, 700, 150, 520], q_lens=[1, 2, 1, 1], num_heads=16,
                             page_size=64, device="cuda", extra_pages=3, kv_dtype=kv_dtype)


@pytest.mark.parametrize("mode", sorted(MODES))
@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_mla_bad_page_sets_flag_and_zeroes_rows(kv_dtype, mode):
    x = _inputs(kv_dtype)
    bt = x.block_tables.clone()
    bt[1, 3] = x.num_pages + 5
    dec = B.PagedDecode(x, **MODES[mode])
    out, lse = dec.alloc_outputs(True)
    out.fill_(7.0)
    dec.run(out, lse, block_tables=bt)
    torch.cuda.synchronize()
    code, info = dec.read_error()
    assert (code, info) == (1, 1), B.DEVICE_ERRORS.get(code, code)
    qi = x.q_indptr_host()
    assert torch.all(out[qi[1]:qi[2]] == 0)
    keep = [0, 2, 3]
    ref_out, ref_lse, q_rows = run_oracle(x, reqs=keep)
    rows = torch.as_tensor(q_rows, dtype=torch.long, device=out.device)
    assert_close(out[rows], lse[rows], ref_out, ref_lse, kv_dtype, f"MLA {kv_dtype}/{mode} beside a bad page")
    # the next call with a good table is correct again (no state left behind)
    out2, lse2 = dec.run()
    torch.cuda.synchronize()
    assert dec.read_error()[0] == 0
    ref_all, ref_lse_all, _ = run_oracle(x)
    assert_close(out2, lse2, ref_all, ref_lse_all, kv_dtype, f"MLA {kv_dtype}/{mode} after the bad call")


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_mla_seq_len_mismatch_sets_flag(kv_dtype):
    x = _inputs(kv_dtype)
    dec = B.PagedDecode(x, max_splits=16, num_sms=400)
    seq = x.seq_lens.clone()
    seq[2] = 16   # the device copy no longer matches the plan
    out, lse = dec.alloc_outputs(True)
    out.fill_(7.0)
    dec.run(out, lse, seq_lens=seq)
    torch.cuda.synchronize()
    code, info = dec.read_error()
    assert (code, info) == (2, 2), B.DEVICE_ERRORS.get(code, code)
    qi = x.q_indptr_host()
    assert torch.all(out[qi[2]:qi[3]] == 0)
    ref_out, ref_lse, q_rows = run_oracle(x, reqs=[0, 1, 3])
    rows = torch.as_tensor(q_rows, dtype=torch.long, device=out.device)
    assert_close(out[rows], lse[rows], ref_out, ref_lse, kv_dtype, f"MLA {kv_dtype} beside a length mismatch")
