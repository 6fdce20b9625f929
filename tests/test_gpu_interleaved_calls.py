"""GPU: many calls of different kernels, interleaved on one stream, all finish
without a device error flag and give the same bits on every call.

The FP8 latent MLA kernel keeps two P buffers, so its softmax warps may write
the P tiles of two consecutive key tiles before the O issuer looks. With one
shared P-full barrier, those two arrivals could complete two phases before
the issuer's parity wait saw the first, and the CTA then waited until the
bounded wait gave up (a timeout flag on a fraction of a percent of calls, and
only when other kernels ran between them). Each P buffer now has its own
barrier. This test runs a few hundred interleaved calls and checks every one.
"""
import pytest
import torch

from paged_kv_cache_199_gb300 import binding as B
from paged_kv_cache_199_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ROUNDS = 150


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_199_gb300 import build
    build.build()
    B.load()


def test_interleaved_calls_never_flag_and_repeat_bit_for_bit():
    flush = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    runs = []
    for name, small in (("mla_fp8", False), ("mla1", True), ("fp8", False), ("ragged", True), ("prefill", True)):
        x = W.workload(name, device="cuda", small=small)
        dec = B.PagedDecode(x, prefill=(name == "prefill"))
        out, lse = dec.alloc_outputs(True)
        dec.run(out, lse)
        torch.cuda.synchronize()
        assert dec.read_error()[0] == 0, name
        runs.append((name, dec, out, lse, out.clone(), lse.clone()))
    for r in range(ROUNDS):
        for name, dec, out, lse, _, _ in runs:
            flush.add_(1)   # other work between calls, as in a serving loop
            dec.run(out, lse)
        torch.cuda.synchronize()
        for name, dec, out, lse, out0, lse0 in runs:
            code, info = dec.read_error()
            assert code == 0, f"{name}: device error {code} (info {info}) in round {r}"
    for name, dec, out, lse, out0, lse0 in runs:
        assert torch.equal(out, out0), f"{name}: output bits changed between calls"
        assert torch.equal(lse, lse0), f"{name}: LSE bits changed between calls"
