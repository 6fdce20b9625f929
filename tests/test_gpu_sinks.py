"""Attention sinks on the GPU against the oracle: one logit per query head in
the softmax denominator, folded in by the unsplit epilogue or by the split
merge (in-kernel or the separate merge kernel; each asked for explicitly)."""
import numpy as np
import pytest
import torch

from paged_kv_cache_199_gb300 import binding as B
from paged_kv_cache_199_gb300 import workloads as W
from tests.helpers import assert_close, run_oracle

pytestmark = pytest.mark.gpu

MODES = dict(unsplit=dict(max_splits=1), split16=dict(max_splits=16, num_sms=400),
             merge_kernel=dict(max_splits=16, num_sms=400, merge_mode=B.PD_MERGE_KERNEL),
             fused=dict(max_splits=16, num_sms=400, merge_mode=B.PD_MERGE_FUSED))


def _sinks(H, seed):
    g = torch.Generator().manual_seed(seed)
    s = torch.randn(H, generator=g) * 2.0
    s[0] = float("-inf")        # no sink for head 0
    if H > 2:
        s[1] = 10.0             # a sink that dominates every logit
    return s.cuda()


@pytest.mark.parametrize("name", ["tiny", "ragged", "fp8", "mla1", "mla2"])
@pytest.mark.parametrize("mode", sorted(MODES))
def test_sinks_match_oracle(name, mode):
    x = W.workload(name, device="cuda", small=True)
    x.sinks = _sinks(x.num_q_heads, 5)
    dec = B.PagedDecode(x, **MODES[mode])
    out, lse = dec.run()
    torch.cuda.synchronize()
    assert dec.read_error()[0] == 0
    ref_out, ref_lse, _ = run_oracle(x)
    assert_close(out, lse, ref_out, ref_lse, x.kv_dtype, f"{name}/{mode} with sinks")


@pytest.mark.parametrize("name", ["ragged", "mla1"])
def test_minus_inf_sinks_change_nothing(name):
    x = W.workload(name, device="cuda", small=True)
    dec = B.PagedDecode(x, max_splits=16, num_sms=400)
    out0, lse0 = dec.run()
    x.sinks = torch.full((x.num_q_heads,), float("-inf"), device="cuda")
    out1, lse1 = dec.run()
    torch.cuda.synchronize()
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_sinks_pointer_required():
    x = W.workload("tiny", device="cuda", small=True)
    dec = B.PagedDecode(x)
    out, lse = dec.alloc_outputs(True)
    with pytest.raises(B.PdError):
        B.paged_decode_run_sinks(dec.plan, x.q, x.k_pool, x.v_pool, x.block_tables, x.seq_lens, x.q_indptr,
                                 x.sm_scale, None, None, None, out, lse, dec.workspace)
