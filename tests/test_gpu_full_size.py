"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (the default plan): sampled requests are checked element by
element against the FP64 oracle, and every output row of the batch against
properties that hold at any size (finite outputs, finite LSE, each output
inside the convex hull bound max|v| of the values it averages)."""
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


def _sampled_requests(x, name):
    seq = x.seq_lens_host()
    ql = np.diff(x.q_indptr_host())
    rng = np.random.default_rng(11)
    picks = {0, x.batch - 1, int(rng.integers(0, x.batch))}
    if name == "ragged":
        # the longest request (split the most), the shortest, and a 4-row one
        picks |= {int(np.argmax(seq)), int(np.argmin(seq))}
        four = np.flatnonzero(ql == 4)
        if four.size:
            picks.add(int(four[0]))
    if name == "prefill":
        picks = {x.batch - 1}
    return sorted(picks)


@pytest.mark.parametrize("name", ["gqa8", "ragged", "fp8", "mla1", "mla2", "mla_fp8", "prefill"])
def test_full_size_sampled(name):
    x = W.workload(name, device="cuda")
    dec = B.PagedDecode(x)
    out, lse = dec.run()
    torch.cuda.synchronize()
    code, info = dec.read_error()
    assert code == 0, f"device error {B.DEVICE_ERRORS.get(code, code)} (request {info})"

    assert torch.isfinite(out.float()).all(), f"{name}: non-finite output"
    assert torch.isfinite(lse).all(), f"{name}: non-finite LSE"

    reqs = _sampled_requests(x, name)
    arrays = gather_requests(x, reqs)
    ref_out, ref_lse, q_rows = run_oracle(x, arrays=arrays)
    rows = torch.as_tensor(q_rows, dtype=torch.long, device=out.device)
    assert_close(out[rows], lse[rows], ref_out, ref_lse, x.kv_dtype, f"{name} full size, requests {reqs}")
    del dec, out, lse, x
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["gqa8", "ragged", "fp8", "mla1", "mla_fp8"])
def test_full_size_deterministic(name):
    """Repeated calls give the same bits: every unit's tiles are reduced in
    one order and split states are merged in split order, whichever CTA
    runs them, so a difference between calls would mean a race between
    pipeline stages."""
    x = W.workload(name, device="cuda")
    dec = B.PagedDecode(x)
    out0, lse0 = dec.run()
    torch.cuda.synchronize()
    for _ in range(3):
        out, lse = dec.run()
        torch.cuda.synchronize()
        assert torch.equal(out, out0), f"{name}: output differs between calls"
        assert torch.equal(lse, lse0), f"{name}: LSE differs between calls"
    del dec, out0, lse0, x
    torch.cuda.empty_cache()
