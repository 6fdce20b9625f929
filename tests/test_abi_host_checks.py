"""Host-side argument checks of the run entry points (no GPU needed): every
call below breaks one rule of the C ABI's contract, so it must return its
status before any CUDA call is made. Pointers are fake addresses that the
library never dereferences when validation fails first."""
import numpy as np
import pytest

from paged_kv_cache_199_gb300 import binding as B
from paged_kv_cache_199_gb300 import build
from tests.test_abi_cpu import gqa_problem

FAKE = 1 << 20          # 16-byte aligned; never dereferenced
NAN = float("nan")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.load()


def _mla_problem(fp8=False):
    p = B.pd_problem()
    p.kind = B.PD_ATTN_MLA
    p.batch, p.num_q_heads, p.num_kv_heads = 2, 16, 1
    p.head_dim_qk, p.head_dim_v, p.page_size = 576, 512, 64
    p.max_pages_per_seq, p.num_pages, p.max_kv_len, p.num_sms = 8, 16, 512, 8
    p.kv_dtype = B.PD_KV_FP8_E4M3 if fp8 else B.PD_KV_BF16
    return p


class Plan:
    def __init__(self, lib, p, seq, qi):
        self.h = B.paged_decode_plan(p, np.asarray(seq, np.int32), np.asarray(qi, np.int32))
        self.ws = int(lib.paged_decode_workspace_size(self.h))
        assert self.ws > 0

    def close(self):
        B.paged_decode_plan_destroy(self.h)


@pytest.fixture(scope="module")
def plans(lib):
    made = {
        "gqa": Plan(lib, gqa_problem(2, Hq=16, Hkv=2, P=16, max_len=512, num_sms=8), [300, 40], [0, 1, 2]),
        "gqa_fp8": Plan(lib, gqa_problem(2, Hq=16, Hkv=2, P=16, max_len=512, num_sms=8, kv_dtype=B.PD_KV_FP8_E4M3),
                        [300, 40], [0, 1, 2]),
        "mla": Plan(lib, _mla_problem(), [300, 40], [0, 1, 2]),
        "mla_fp8": Plan(lib, _mla_problem(fp8=True), [300, 40], [0, 1, 2]),
        "prefill": Plan(lib, gqa_problem(2, Hq=16, Hkv=2, P=16, max_len=512, num_sms=8, kind=B.PD_ATTN_PREFILL),
                        [300, 40], [0, 100, 120]),
    }
    yield made
    for pl in made.values():
        pl.close()


def gqa_call(lib, plan, *, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, sl=FAKE, out=FAKE, scale=0.1, ks=None, vs=None,
             sinks=None, ws=FAKE, ws_bytes=None, entry="run"):
    wsb = plan.ws if ws_bytes is None else ws_bytes
    if entry == "sinks":
        return lib.paged_decode_run_sinks(plan.h, q, k, v, bt, sl, None, scale, ks, vs, sinks, out, None, ws, wsb,
                                          None)
    return lib.paged_decode_run(plan.h, q, k, v, bt, sl, None, scale, ks, vs, out, None, ws, wsb, None)


def mla_call(lib, plan, *, fp8, q=FAKE, kv=FAKE, bt=FAKE, sl=FAKE, out=FAKE, scale=0.1, qs=FAKE, kvs=FAKE,
             ws=FAKE, sinks_entry=False, sinks=None):
    if fp8:
        return lib.mla_decode_run_fp8(plan.h, q, kv, bt, sl, None, scale, qs, kvs, None, out, None, ws, plan.ws,
                                      None)
    if sinks_entry:
        return lib.mla_decode_run_sinks(plan.h, q, kv, bt, sl, None, scale, sinks, out, None, ws, plan.ws, None)
    return lib.mla_decode_run(plan.h, q, kv, bt, sl, None, scale, out, None, ws, plan.ws, None)


def prefill_call(lib, plan, *, q=FAKE, k=FAKE, v=FAKE, out=FAKE, scale=0.1, ws=FAKE):
    return lib.paged_prefill_run(plan.h, q, k, v, FAKE, FAKE, FAKE, scale, None, out, None, ws, plan.ws, None)


def test_gqa_run_rejects_bad_arguments(lib, plans):
    g, f8, mla = plans["gqa"], plans["gqa_fp8"], plans["mla"]
    bad = B.PD_ERR_INVALID_ARG
    assert gqa_call(lib, mla) == bad                      # an MLA plan
    assert lib.paged_decode_run(None, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0.1, None, None, FAKE, None, FAKE,
                                g.ws, None) == bad        # no plan
    assert gqa_call(lib, g, ws=None) == bad
    assert gqa_call(lib, g, ws=FAKE + 8) == bad           # workspace not 16-byte aligned
    assert gqa_call(lib, g, ws_bytes=g.ws - 1) == B.PD_ERR_WORKSPACE_TOO_SMALL
    for arg in ("q", "k", "v", "bt", "sl", "out"):
        assert gqa_call(lib, g, **{arg: None}) == bad, arg
    for arg in ("q", "k", "v", "out"):
        assert gqa_call(lib, g, **{arg: FAKE + 2}) == bad, arg
    assert gqa_call(lib, g, scale=NAN) == bad
    assert gqa_call(lib, f8, ks=None, vs=FAKE) == bad     # E4M3 needs both scales
    assert gqa_call(lib, f8, ks=FAKE, vs=None) == bad
    assert gqa_call(lib, g, entry="sinks", sinks=None) == bad


def test_mla_run_rejects_bad_arguments(lib, plans):
    m, m8, g = plans["mla"], plans["mla_fp8"], plans["gqa"]
    bad = B.PD_ERR_INVALID_ARG
    assert mla_call(lib, g, fp8=False) == bad             # a GQA plan
    assert mla_call(lib, m8, fp8=False) == bad            # BF16 entry, E4M3 plan
    assert mla_call(lib, m, fp8=True) == bad              # E4M3 entry, BF16 plan
    assert mla_call(lib, m8, fp8=True, qs=None) == bad
    assert mla_call(lib, m8, fp8=True, kvs=None) == bad
    for arg in ("q", "kv", "bt", "sl", "out"):
        assert mla_call(lib, m, fp8=False, **{arg: None}) == bad, arg
        assert mla_call(lib, m8, fp8=True, **{arg: None}) == bad, arg
    for arg in ("q", "kv", "out"):
        assert mla_call(lib, m, fp8=False, **{arg: FAKE + 4}) == bad, arg
    assert mla_call(lib, m, fp8=False, scale=NAN) == bad
    assert mla_call(lib, m, fp8=False, ws=None) == bad
    assert mla_call(lib, m, fp8=False, sinks_entry=True, sinks=None) == bad


def test_prefill_run_rejects_bad_arguments(lib, plans):
    pf, g = plans["prefill"], plans["gqa"]
    bad = B.PD_ERR_INVALID_ARG
    assert prefill_call(lib, g) == bad                    # a decode plan
    for scale in (0.0, -0.5, float("inf"), NAN):          # the kernel needs a positive, finite scale
        assert prefill_call(lib, pf, scale=scale) == bad, scale
    for arg in ("q", "k", "v", "out"):
        assert prefill_call(lib, pf, **{arg: None}) == bad, arg
        assert prefill_call(lib, pf, **{arg: FAKE + 2}) == bad, arg
    assert prefill_call(lib, pf, ws=None) == bad


def test_merge_states_rejects_bad_arguments(lib):
    bad = B.PD_ERR_INVALID_ARG

    def call(S=4, rows=8, dim=128, v=FAKE, s=FAKE, out=FAKE):
        return lib.paged_decode_merge_states(v, s, S, rows, dim, out, None, None)

    for kw in (dict(S=0), dict(S=65), dict(rows=-1), dict(dim=4), dict(dim=12), dict(dim=2048),
               dict(v=None), dict(s=None), dict(out=None), dict(v=FAKE + 4), dict(out=FAKE + 2)):
        assert call(**kw) == bad, kw
    assert call(rows=0) == B.PD_OK                        # nothing to merge: no launch


def test_no_alloc_entry_point_refuses_before_any_cuda_call(lib, plans):
    """paged_decode_run_no_alloc checks its plan and arguments before it looks
    up its array or copies the plan (on this GPU-less host any CUDA call would
    return PD_ERR_CUDA instead)."""
    na = B.paged_decode_run_no_alloc
    args = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, sl=FAKE, qi=None, scale=0.1, ks=None, vs=None, out=FAKE, lse=None)

    def call(plan, **kw):
        a = dict(args, **kw)
        return na(plan, a["q"], a["k"], a["v"], a["bt"], a["sl"], a["qi"], a["scale"], a["ks"], a["vs"],
                  a["out"], a["lse"], stream=0)

    assert call(None) == B.PD_ERR_INVALID_ARG
    assert call(plans["mla"].h) == B.PD_ERR_INVALID_ARG          # not a GQA plan
    assert call(plans["prefill"].h) == B.PD_ERR_INVALID_ARG
    g = plans["gqa"].h
    assert call(g, q=None) == B.PD_ERR_INVALID_ARG
    assert call(g, out=FAKE + 8) == B.PD_ERR_INVALID_ARG          # misaligned
    assert call(g, scale=NAN) == B.PD_ERR_INVALID_ARG
    assert call(plans["gqa_fp8"].h) == B.PD_ERR_INVALID_ARG      # E4M3 pools need both scales
