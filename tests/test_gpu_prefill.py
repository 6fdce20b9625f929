"""The tensor-core prefill kernel (paged_prefill_run) against the FP64 oracle:
many new tokens per request with the inclusive causal bound, units of up to
256 packed (token, head) rows in two 128-row query tiles, 128 keys per tile,
split units merged by the LSE-merge kernel."""
import numpy as np
import pytest
import torch

from paged_kv_cache_199_gb300 import binding as B
from paged_kv_cache_199_gb300 import workloads as W
from tests.helpers import assert_close, gather_requests, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_199_gb300 import build
    build.build()
    B.load()


def run_prefill(x, **kw):
    dec = B.PagedDecode(x, prefill=True, **kw)
    out, lse = dec.run()
    torch.cuda.synchronize()
    code, info = dec.read_error()
    assert code == 0, f"device error {B.DEVICE_ERRORS.get(code, code)} (request {info})"
    return dec, out, lse


MODES = dict(auto={}, unsplit=dict(max_splits=1), split16=dict(max_splits=16, num_sms=400),
             queue=dict(schedule=B.PD_SCHED_QUEUE, num_sms=300), static=dict(schedule=B.PD_SCHED_STATIC, num_sms=300))


@pytest.mark.parametrize("mode", sorted(MODES))
def test_small_prefill_workload(mode):
    x = W.workload("prefill", device="cuda", small=True)
    dec, out, lse = run_prefill(x, **MODES[mode])
    assert dec.info.rows_per_unit == 256 and dec.info.tile_tokens == 128
    ref_out, ref_lse, _ = run_oracle(x)
    assert_close(out, lse, ref_out, ref_lse, "bf16", f"prefill/{mode}")


@pytest.mark.parametrize("merge", ["auto", "fused_request"])
def test_prefill_split_long_context(merge):
    """Few units over long caches: the planner splits them and the LSE-merge
    kernel combines the split states (a fused-merge request is served by the
    merge kernel too)."""
    x = W.make_paged_inputs(seed=21, seq_lens=[5000, 3100], q_lens=[48, 20], num_q_heads=32, num_kv_heads=4,
                            head_dim=128, page_size=64, layout="HND", device="cuda", extra_pages=2)
    kw = dict(max_splits=16, num_sms=400)
    if merge == "fused_request":
        kw["merge_mode"] = B.PD_MERGE_FUSED
    dec, out, lse = run_prefill(x, **kw)
    assert dec.info.max_splits_used > 1 and dec.info.partial_rows > 0
    ref_out, ref_lse, _ = run_oracle(x)
    assert_close(out, lse, ref_out, ref_lse, "bf16", f"prefill split/{merge}")


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("Hq,Hkv,P", [(8, 8, 16), (32, 8, 32), (64, 8, 8), (32, 2, 64), (16, 1, 128), (128, 1, 24)])
def test_prefill_shapes(layout, Hq, Hkv, P):
    """Groups 1..128, page sizes that are and are not powers of two, q_len
    that is and is not a multiple of 128 / G, requests whose every token is
    new, single-token requests and a ragged batch."""
    rng = np.random.default_rng(Hq * 31 + Hkv * 7 + P)
    G = Hq // Hkv
    ql = np.array([1, 128 // G + 3, 257, 40, 128 // G], dtype=np.int64)
    seq = ql + rng.integers(0, 600, ql.size)
    seq[2] = ql[2]            # prompt only: every key is a new token
    x = W.make_paged_inputs(seed=int(Hq + P), seq_lens=seq, q_lens=ql, num_q_heads=Hq, num_kv_heads=Hkv,
                            head_dim=128, page_size=P, layout=layout, device="cuda", extra_pages=3)
    for kw in ({}, dict(max_splits=16, num_sms=600)):
        _, out, lse = run_prefill(x, **kw)
        ref_out, ref_lse, _ = run_oracle(x)
        assert_close(out, lse, ref_out, ref_lse, "bf16", f"prefill {layout} Hq={Hq} Hkv={Hkv} P={P} {kw}")


def test_prefill_matches_decode_kernel():
    """The two kernels compute the same function: outputs agree within the
    BF16 tolerance on the small prefill workload."""
    x = W.workload("prefill", device="cuda", small=True)
    _, out_p, lse_p = run_prefill(x)
    dec = B.PagedDecode(x)
    out_d, lse_d = dec.run()
    torch.cuda.synchronize()
    assert torch.allclose(out_p.float(), out_d.float(), atol=1e-2, rtol=1e-2)
    assert torch.allclose(lse_p, lse_d, atol=2e-3, rtol=2e-3)


@pytest.mark.parametrize("mode", ["unsplit", "split16"])
def test_prefill_sinks(mode):
    x = W.workload("prefill", device="cuda", small=True)
    g = torch.Generator().manual_seed(9)
    s = torch.randn(x.num_q_heads, generator=g) * 2.0
    s[0] = float("-inf")
    s[1] = 10.0
    x.sinks = s.cuda()
    _, out, lse = run_prefill(x, **MODES[mode])
    ref_out, ref_lse, _ = run_oracle(x)
    assert_close(out, lse, ref_out, ref_lse, "bf16", f"prefill sinks/{mode}")


def test_prefill_bad_page_sets_flag_and_zeroes_rows():
    x = W.workload("prefill", device="cuda", small=True)
    bt = x.block_tables.clone()
    bt[1, 2] = x.num_pages + 5
    dec = B.PagedDecode(x, prefill=True)
    out, lse = dec.alloc_outputs(True)
    out.fill_(7.0)
    dec.run(out, lse, block_tables=bt)
    torch.cuda.synchronize()
    code, info = dec.read_error()
    assert code == 1 and info == 1   # PD_DEV_BAD_PAGE, request 1
    qi = x.q_indptr_host()
    assert torch.all(out[qi[1]:qi[2]] == 0)
    ref_out, ref_lse, q_rows = run_oracle(x, reqs=[0])
    assert_close(out[q_rows], lse[q_rows], ref_out, ref_lse, "bf16", "prefill request 0 beside a bad page")


def test_prefill_full_size_sampled():
    """The benchmark's workload (4 x 511 new tokens over 2047) in the
    benchmark's launch configuration: the last request element by element."""
    x = W.workload("prefill", device="cuda")
    _, out, lse = run_prefill(x)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    arrays = gather_requests(x, [x.batch - 1])
    ref_out, ref_lse, q_rows = run_oracle(x, arrays=arrays)
    rows = torch.as_tensor(q_rows, dtype=torch.long, device=out.device)
    assert_close(out[rows], lse[rows], ref_out, ref_lse, "bf16", "prefill full size")


def test_prefill_rejects_non_positive_scale():
    x = W.workload("prefill", device="cuda", small=True)
    dec = B.PagedDecode(x, prefill=True)
    out, lse = dec.alloc_outputs(True)
    for bad in (0.0, -0.1, float("inf"), float("nan")):
        with pytest.raises(B.PdError):
            B.paged_prefill_run(dec.plan, x.q, x.k_pool, x.v_pool, x.block_tables, x.seq_lens, x.q_indptr, bad,
                                None, out, lse, dec.workspace)


def test_prefill_is_deterministic():
    """The same call gives the same bits every time (each unit's tiles are
    processed in one order by one CTA, whatever the queue order): a check
    against races between the pipeline's stages."""
    x = W.workload("prefill", device="cuda")
    dec = B.PagedDecode(x, prefill=True)
    out0, lse0 = dec.run()
    torch.cuda.synchronize()
    for _ in range(4):
        out, lse = dec.run()
        torch.cuda.synchronize()
        assert torch.equal(out, out0) and torch.equal(lse, lse0)
