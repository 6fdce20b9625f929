"""GPU: the bounded device waits run out on their own and end the kernel
cleanly. With the pipeline wait limit set to 1 ns (in effect the ~20 us of
one suspended try_wait), a full-size call has waits that last longer than
that (a scheduler waiting for a slot while a 4096-token item streams), so its
CTAs give up, drain their own copies and tensor-core work, and flag
PD_DEV_TIMEOUT in the workspace error word. The context must stay usable:
after the limit is restored and the plan uploaded again, the next call on the
same workspace matches the oracle. No GPU fault is involved: the waits end
because their limit passes, not because anything is broken."""
import numpy as np
import pytest
import torch

from paged_kv_cache_199_gb300 import binding as B
from paged_kv_cache_199_gb300 import workloads as W
from tests.helpers import assert_close, gather_requests, run_oracle

pytestmark = pytest.mark.gpu

PD_DEV_TIMEOUT = 5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_199_gb300 import build
    build.build()
    B.load()
    yield
    B.paged_decode_set_wait_limit_ns(0)


def _set_limit(ns):
    assert B.paged_decode_set_wait_limit_ns(ns) == B.PD_OK


# small grids give every CTA several items, so a scheduler waits for a slot
# while one item streams (tens of microseconds), past the limit
@pytest.mark.parametrize("name,kw", [("gqa8", dict(max_splits=1, num_sms=8)), ("fp8", dict(num_sms=8)),
                                     ("mla1", {}), ("mla_fp8", {}), ("prefill", dict(prefill=True, num_sms=4))])
def test_wait_limit_runs_out_then_next_call_is_correct(name, kw):
    x = W.workload(name, device="cuda")
    dec = B.PagedDecode(x, **kw)
    out, lse = dec.alloc_outputs(True)
    try:
        _set_limit(1)
        dec.run(out, lse)
        torch.cuda.synchronize()
    finally:
        _set_limit(0)
    code, _ = dec.read_error()
    assert code == PD_DEV_TIMEOUT, f"{name}: expected a timeout flag, got {code}"
    # the context is usable and the workspace, uploaded again, serves the next call
    assert float(torch.ones(4, device="cuda").sum().item()) == 4.0
    dec.upload()
    out.zero_()
    dec.run(out, lse)
    torch.cuda.synchronize()
    assert dec.read_error()[0] == 0
    reqs = [0, x.batch - 1]
    ref_out, ref_lse, q_rows = run_oracle(x, arrays=gather_requests(x, reqs))
    rows = torch.as_tensor(q_rows, dtype=torch.long, device=out.device)
    assert_close(out[rows], lse[rows], ref_out, ref_lse, x.kv_dtype, f"{name} after a timed-out call")
    del dec, out, lse, x
    torch.cuda.empty_cache()


def test_default_limit_restored():
    """After the limit is reset to 0 (the default), a split plan with the fused
    merge runs without a flag and matches the oracle."""
    x = W.workload("ragged", device="cuda", small=True)
    dec = B.PagedDecode(x, max_splits=16, num_sms=300, merge_mode=B.PD_MERGE_FUSED)
    out, lse = dec.run()
    torch.cuda.synchronize()
    assert dec.read_error()[0] == 0
    ref_out, ref_lse, _ = run_oracle(x)
    assert_close(out, lse, ref_out, ref_lse, "bf16", "default wait limit")
    assert np.isfinite(lse.cpu().numpy()).all()
