"""FP8 latent MLA (E4M3 query and pool, kind::f8f6f4 MMAs, E4M3 P) against the
oracle, at the E4M3 tolerance. Besides the default scale (diffuse attention,
small outputs) the cases with sm_scale 0.3 make attention peaked, so outputs
are single value rows of order one and the tolerance is a real check."""
import numpy as np
import pytest
import torch

from paged_kv_cache_199_gb300 import binding as B
from paged_kv_cache_199_gb300 import workloads as W
from tests.helpers import assert_close, run_oracle

pytestmark = pytest.mark.gpu

MODES = dict(auto={}, unsplit=dict(max_splits=1), split16=dict(max_splits=16, num_sms=400),
             merge_kernel=dict(merge_mode=B.PD_MERGE_KERNEL, num_sms=300),
             fused=dict(max_splits=16, num_sms=400, merge_mode=B.PD_MERGE_FUSED),
             queue=dict(schedule=B.PD_SCHED_QUEUE, num_sms=300), static=dict(schedule=B.PD_SCHED_STATIC, num_sms=300))


def _run(x, **kw):
    dec = B.PagedDecode(x, **kw)
    out, lse = dec.run()
    torch.cuda.synchronize()
    assert dec.read_error()[0] == 0
    return out, lse


@pytest.mark.parametrize("mode", sorted(MODES))
def test_mla_fp8_small(mode):
    x = W.workload("mla_fp8", device="cuda", small=True)
    out, lse = _run(x, **MODES[mode])
    ref_out, ref_lse, _ = run_oracle(x)
    assert_close(out, lse, ref_out, ref_lse, "e4m3", f"mla_fp8/{mode}")


@pytest.mark.parametrize("H,P,qmax", [(128, 64, 1), (16, 32, 3), (40, 8, 2), (12, 64, 4), (96, 64, 2)])
@pytest.mark.parametrize("sm_scale", [None, 0.3])
def test_mla_fp8_shapes(H, P, qmax, sm_scale):
    rng = np.random.default_rng(H + P)
    B_ = 4
    ql = rng.integers(1, qmax + 1, B_)
    seq = np.maximum(rng.integers(1, 300, B_), ql)
    x = W.make_mla_inputs(seed=H * P + 1, seq_lens=seq, q_lens=ql, num_heads=H, page_size=P, device="cuda",
                          extra_pages=3, kv_dtype="e4m3", sm_scale=sm_scale)
    ref_out, ref_lse, _ = run_oracle(x)
    if sm_scale is not None:
        assert np.abs(ref_out).max() > 0.5   # peaked: outputs of order one
    for kw in ({}, dict(max_splits=16, num_sms=400)):
        out, lse = _run(x, **kw)
        assert_close(out, lse, ref_out, ref_lse, "e4m3", f"MLA fp8 H={H} P={P} scale={sm_scale} {kw}")


def test_mla_fp8_sinks():
    x = W.make_mla_inputs(seed=3, seq_lens=[200, 90], q_lens=[1, 2], num_heads=16, page_size=64, device="cuda",
                          kv_dtype="e4m3", sm_scale=0.3)
    g = torch.Generator().manual_seed(2)
    x.sinks = (torch.randn(16, generator=g) * 2).cuda()
    ref_out, ref_lse, _ = run_oracle(x)
    for kw in ({}, dict(max_splits=16, num_sms=400)):
        out, lse = _run(x, **kw)
        assert_close(out, lse, ref_out, ref_lse, "e4m3", f"MLA fp8 sinks {kw}")


def test_mla_fp8_requires_scales_and_dtype():
    x = W.workload("mla_fp8", device="cuda", small=True)
    dec = B.PagedDecode(x)
    out, lse = dec.alloc_outputs()
    with pytest.raises(B.PdError):   # scales missing
        B.mla_decode_run_fp8(dec.plan, x.q, x.k_pool, x.block_tables, x.seq_lens, x.q_indptr, x.sm_scale,
                             None, None, None, out, lse, dec.workspace)
    with pytest.raises(B.PdError):   # an E4M3 plan through the BF16 entry point
        B.mla_decode_run(dec.plan, x.q, x.k_pool, x.block_tables, x.seq_lens, x.q_indptr, x.sm_scale,
                         out, lse, dec.workspace)
