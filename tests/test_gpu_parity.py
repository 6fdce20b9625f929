"""GPU parity: the CUDA library (through its C ABI) against the FP64 oracle
on the same seeded bytes."""
import numpy as np
import pytest
import torch

from paged_kv_cache_199_gb300 import binding as B
from paged_kv_cache_199_gb300 import workloads as W
from tests.helpers import assert_close, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_199_gb300 import build
    build.build()
    B.load()


def run_gpu(x, **kw):
    dec = B.PagedDecode(x, **kw)
    out, lse = dec.run()
    torch.cuda.synchronize()
    code, info = dec.read_error()
    assert code == 0, f"device error {B.DEVICE_ERRORS.get(code, code)} (request {info})"
    return dec, out, lse


@pytest.mark.parametrize("name", ["tiny", "gqa8", "ragged", "fp8", "prefill"])
@pytest.mark.parametrize("mode", ["auto", "unsplit", "split16", "merge_kernel", "fused", "queue", "static",
                                  "static_cap2"])
def test_small_workloads(name, mode):
    x = W.workload(name, device="cuda", small=True)
    kw = dict(auto={}, unsplit=dict(max_splits=1), split16=dict(max_splits=16, num_sms=400),
              merge_kernel=dict(merge_mode=B.PD_MERGE_KERNEL, num_sms=300),
              fused=dict(max_splits=16, num_sms=400, merge_mode=B.PD_MERGE_FUSED),
              queue=dict(schedule=B.PD_SCHED_QUEUE, num_sms=300),
              static=dict(schedule=B.PD_SCHED_STATIC, num_sms=300),
              # few wide static ranges under a split cap of 2 (each unit meets at most two)
              static_cap2=dict(schedule=B.PD_SCHED_STATIC, num_sms=7, max_splits=2))[mode]
    dec, out, lse = run_gpu(x, **kw)
    ref_out, ref_lse, _ = run_oracle(x)
    assert_close(out, lse, ref_out, ref_lse, x.kv_dtype, f"{name}/{mode}")
    if mode in ("split16", "fused") and name not in ("tiny", "prefill"):   # prefill: more units than slots
        assert dec.info.max_splits_used > 1
    if mode == "static_cap2":
        assert dec.info.max_splits_used <= 2


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("P", [1, 3, 16, 48, 64, 128])
@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_page_sizes_and_layouts(layout, P, kv_dtype):
    rng = np.random.default_rng(P)
    seq = rng.integers(1, 300, 5)
    seq[0] = 1
    x = W.make_paged_inputs(seed=10 + P, seq_lens=seq, q_lens=[1] * 5, num_q_heads=16,
                            num_kv_heads=2, head_dim=128, page_size=P, layout=layout,
                            kv_dtype=kv_dtype, device="cuda", extra_pages=3)
    for kw in ({}, dict(max_splits=16, num_sms=600)):
        _, out, lse = run_gpu(x, **kw)
        ref_out, ref_lse, _ = run_oracle(x)
        assert_close(out, lse, ref_out, ref_lse, kv_dtype, f"P={P} {layout} {kv_dtype} {kw}")


@pytest.mark.parametrize("Hq,Hkv,qmax", [(8, 8, 3), (32, 1, 2), (12, 4, 4), (64, 8, 2), (8, 1, 5)])
def test_group_shapes_and_multirow_queries(Hq, Hkv, qmax):
    rng = np.random.default_rng(Hq * 7 + Hkv)
    B_ = 6
    ql = rng.integers(1, qmax + 1, B_)
    seq = np.maximum(rng.integers(1, 700, B_), ql)
    seq[1] = ql[1]  # every token is a new one
    x = W.make_paged_inputs(seed=Hq + Hkv, seq_lens=seq, q_lens=ql, num_q_heads=Hq,
                            num_kv_heads=Hkv, head_dim=128, page_size=16, layout="HND",
                            device="cuda", extra_pages=2)
    for kw in ({}, dict(max_splits=16, num_sms=500), dict(merge_mode=B.PD_MERGE_KERNEL, num_sms=500),
               dict(schedule=B.PD_SCHED_QUEUE, num_sms=500), dict(schedule=B.PD_SCHED_STATIC, num_sms=500)):
        _, out, lse = run_gpu(x, **kw)
        ref_out, ref_lse, _ = run_oracle(x)
        assert_close(out, lse, ref_out, ref_lse, "bf16", f"Hq={Hq} Hkv={Hkv} {kw}")


def test_no_lse_and_empty_batch():
    x = W.workload("tiny", device="cuda")
    dec = B.PagedDecode(x)
    out, _ = dec.run(with_lse=False)
    torch.cuda.synchronize()
    ref_out, ref_lse, _ = run_oracle(x)
    assert_close(out, None, ref_out, ref_lse, "bf16", "no lse")
    e = W.make_paged_inputs(seed=1, seq_lens=[], q_lens=[], num_q_heads=8, num_kv_heads=1,
                            head_dim=128, page_size=16, device="cuda", extra_pages=1,
                            max_pages_per_seq=1)
    dec = B.PagedDecode(e)
    assert dec.info.num_items == 0
    out, lse = dec.run()
    torch.cuda.synchronize()
    assert out.shape[0] == 0


@pytest.mark.parametrize("name", ["mla1", "mla2"])
@pytest.mark.parametrize("mode", ["auto", "unsplit", "split16", "merge_kernel", "fused", "queue", "static"])
def test_mla_small(name, mode):
    x = W.workload(name, device="cuda", small=True)
    kw = dict(auto={}, unsplit=dict(max_splits=1), split16=dict(max_splits=16, num_sms=400),
              merge_kernel=dict(merge_mode=B.PD_MERGE_KERNEL, num_sms=300),
              fused=dict(max_splits=16, num_sms=400, merge_mode=B.PD_MERGE_FUSED),
              queue=dict(schedule=B.PD_SCHED_QUEUE, num_sms=300),
              static=dict(schedule=B.PD_SCHED_STATIC, num_sms=300))[mode]
    dec, out, lse = run_gpu(x, **kw)
    ref_out, ref_lse, _ = run_oracle(x)
    assert_close(out, lse, ref_out, ref_lse, "bf16", f"{name}/{mode}")
    if mode == "fused":
        assert dec.info.max_splits_used > 1


@pytest.mark.parametrize("H,P,qmax", [(128, 64, 1), (16, 32, 3), (6, 8, 2), (40, 64, 4)])
def test_mla_shapes(H, P, qmax):
    rng = np.random.default_rng(H + P)
    B_ = 5
    ql = rng.integers(1, qmax + 1, B_)
    seq = np.maximum(rng.integers(1, 400, B_), ql)
    seq[0] = ql[0]
    x = W.make_mla_inputs(seed=H * P, seq_lens=seq, q_lens=ql, num_heads=H, page_size=P,
                          device="cuda", extra_pages=3)
    for kw in ({}, dict(max_splits=16, num_sms=400), dict(schedule=B.PD_SCHED_QUEUE, num_sms=200)):
        _, out, lse = run_gpu(x, **kw)
        ref_out, ref_lse, _ = run_oracle(x)
        assert_close(out, lse, ref_out, ref_lse, "bf16", f"MLA H={H} P={P} {kw}")
