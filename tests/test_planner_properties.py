"""Randomised properties of the host split planner (CPU only).

Whatever the shape, lengths, query counts, SM count, schedule and split cap,
a plan must cover every key tile that a unit's last row can see exactly once,
number each unit's splits 0 .. n - 1 in key order, stay within the split cap,
and size its partial-state rows to the split units it made. Units are rebuilt
here from the problem alone: GQA decode units are blocks of 8 or 16 packed
(token, head) rows of one KV head, MLA units 64-row blocks of all heads, and
prefill units 256-row blocks of one KV head."""
import numpy as np
import pytest

from paged_kv_cache_199_gb300 import binding as B
from paged_kv_cache_199_gb300 import build

try:
    from hypothesis import HealthCheck, given, settings
    from hypothesis import strategies as st
except ImportError:   # not installed everywhere; the test is then collected as skipped
    st = None


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.load()


def make_problem(c):
    p = B.pd_problem()
    p.kind = {"gqa": B.PD_ATTN_GQA, "mla": B.PD_ATTN_MLA, "prefill": B.PD_ATTN_PREFILL}[c["kind"]]
    p.batch = c["batch"]
    p.num_kv_heads = c["hkv"]
    p.num_q_heads = c["hkv"] * c["group"]
    if c["kind"] == "mla":
        p.head_dim_qk, p.head_dim_v = 576, 512
    else:
        p.head_dim_qk = p.head_dim_v = 128
    p.page_size = c["page"]
    p.max_pages_per_seq = (c["max_len"] + c["page"] - 1) // c["page"]
    p.num_pages = c["batch"] * p.max_pages_per_seq
    p.max_kv_len = c["max_len"]
    p.layout = B.PD_LAYOUT_HND
    p.kv_dtype = B.PD_KV_FP8_E4M3 if c["fp8"] else B.PD_KV_BF16
    p.num_sms = c["num_sms"]
    p.schedule = c["schedule"]
    p.max_splits = c["max_splits"]
    return p


def expected_units(c, rows_per_unit, T):
    """(tiles, rows) of every unit, in the planner's order."""
    units = []
    G = c["group"]
    for b in range(c["batch"]):
        L, q = int(c["seq"][b]), int(c["ql"][b])
        rows = q * G
        heads = [0] if c["kind"] == "mla" else range(c["hkv"])
        for _ in heads:
            for r0 in range(0, rows, rows_per_unit):
                n = min(rows_per_unit, rows - r0)
                visible = L - q + (r0 + n - 1) // G + 1
                units.append(((visible + T - 1) // T, n))
    return units


if st is not None:
    SCHEDULES = [B.PD_SCHED_QUEUE, B.PD_SCHED_STATIC, B.PD_SCHED_AUTO]

    @st.composite
    def problems(draw):
        kind = draw(st.sampled_from(["gqa", "mla", "prefill"]))
        batch = draw(st.one_of(st.integers(1, 40), st.integers(41, 300)))
        if kind == "gqa":
            hkv = draw(st.sampled_from([1, 2, 4, 8]))
            group = draw(st.sampled_from([1, 2, 4, 5, 8, 16]))
            page = draw(st.sampled_from([1, 3, 8, 16, 32, 64]))
            qmax = 4
        elif kind == "mla":
            hkv, group = 1, draw(st.sampled_from([16, 40, 64, 128]))
            page = draw(st.sampled_from([8, 32, 64]))
            qmax = 3
        else:
            hkv = draw(st.sampled_from([1, 2, 8]))
            group = draw(st.sampled_from([1, 2, 4, 8, 16]))
            page = draw(st.sampled_from([8, 32]))
            qmax = 600
        max_len = draw(st.sampled_from([64, 1000, 4096, 9000, 131072]))
        seq = np.asarray(draw(st.lists(st.integers(0, max_len), min_size=batch, max_size=batch)), np.int64)
        ql = np.asarray([draw(st.integers(0, min(int(s), qmax))) for s in seq], np.int64)
        return dict(kind=kind, batch=batch, hkv=hkv, group=group, page=page, max_len=max_len, seq=seq, ql=ql,
                    num_sms=draw(st.sampled_from([1, 7, 152])), schedule=draw(st.sampled_from(SCHEDULES)),
                    max_splits=draw(st.sampled_from([0, 1, 2, 5, 16])),
                    fp8=draw(st.booleans()) and kind != "prefill")

    @settings(max_examples=300, deadline=None, suppress_health_check=[HealthCheck.function_scoped_fixture])
    @given(c=problems())
    def test_plan_properties(lib, c):
        qi = np.concatenate([[0], np.cumsum(c["ql"])]).astype(np.int32)
        plan = B.paged_decode_plan(make_problem(c), c["seq"].astype(np.int32), qi)
        try:
            info = B.paged_decode_plan_get_info(plan)
            items = np.asarray(B.paged_decode_plan_get_items(plan)).reshape(-1, 4)
            ws = B.paged_decode_workspace_size(plan)
        finally:
            B.paged_decode_plan_destroy(plan)
        G = c["group"]
        if c["kind"] == "gqa":
            want_rows = 8 if int((c["ql"] * G).max(initial=0)) <= 8 else 16
        else:
            want_rows = {"mla": 64, "prefill": 256}[c["kind"]]
        if info.num_units:
            assert info.rows_per_unit == want_rows
        units = expected_units(c, want_rows, info.tile_tokens)
        assert info.num_units == len(units)
        assert info.num_items == len(items)
        assert ws == info.workspace_bytes

        cap = c["max_splits"] or 16
        assert info.max_splits_used <= cap
        pieces = {}
        for u, t0, t1, s in items:
            assert 0 <= u < len(units)
            assert 0 <= t0 < t1 <= units[u][0]
            pieces.setdefault(int(u), []).append((int(t0), int(t1), int(s)))
        partial_rows = 0
        for u, (tiles, nrows) in enumerate(units):
            got = sorted(pieces.get(u, []))
            # the pieces tile [0, tiles) exactly, split k being the k-th in key order
            assert got and got[0][0] == 0 and got[-1][1] == tiles, (u, got, tiles)
            assert all(a[1] == b[0] for a, b in zip(got, got[1:])), (u, got)
            assert [s for _, _, s in got] == list(range(len(got))), (u, got)
            assert len(got) <= cap
            if len(got) > 1:
                partial_rows += len(got) * nrows
        assert info.partial_rows == partial_rows
        # the split states fit in the workspace: an fp32 LSE and row per partial row
        assert info.workspace_bytes >= partial_rows * 4 * (1 + (512 if c["kind"] == "mla" else 128))
        # CTA slots: two per SM for GQA decode, one for MLA and prefill
        slots = c["num_sms"] * (2 if c["kind"] == "gqa" else 1)
        assert 1 <= info.num_ctas <= slots
        if c["schedule"] == B.PD_SCHED_QUEUE or c["max_splits"] == 1:
            # the shared queue: as many CTAs as items (up to the slots), longest first,
            # ties by (unit, split)
            assert info.num_ctas == max(1, min(slots, len(items)))
            lengths = items[:, 2] - items[:, 1]
            keys = list(zip(-lengths, items[:, 0], items[:, 3]))
            assert keys == sorted(keys)
else:
    @pytest.mark.skip(reason="hypothesis is not installed")
    def test_plan_properties():
        pass
