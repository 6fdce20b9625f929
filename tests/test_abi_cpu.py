"""CPU checks of the C-ABI library: it loads, exports every declared entry
point, and its host planner obeys its contract (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

from paged_kv_cache_199_gb300 import binding as B
from paged_kv_cache_199_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.load()


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(inc, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M):
            name = m.group(1)
            if name not in ("if", "typedef", "sizeof"):
                names.append(name)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "paged_decode_run" in names and "mla_decode_run" in names and "paged_decode_plan" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert lib.paged_decode_version() == 0x000100


def gqa_problem(batch, Hq=64, Hkv=8, P=32, max_len=4096, layout=B.PD_LAYOUT_HND, **kw):
    p = B.pd_problem()
    p.kind = B.PD_ATTN_GQA
    p.batch = batch
    p.num_q_heads, p.num_kv_heads = Hq, Hkv
    p.head_dim_qk = p.head_dim_v = 128
    p.page_size = P
    p.max_pages_per_seq = (max_len + P - 1) // P
    p.num_pages = max(1, batch * p.max_pages_per_seq)
    p.max_kv_len = max_len
    p.layout = layout
    p.kv_dtype = B.PD_KV_BF16
    p.num_sms = kw.pop("num_sms", 152)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def plan_items(p, seq, qi=None):
    plan = B.paged_decode_plan(p, np.asarray(seq, np.int32), None if qi is None else np.asarray(qi, np.int32))
    try:
        info = B.paged_decode_plan_get_info(plan)
        items = B.paged_decode_plan_get_items(plan)
        return info, items
    finally:
        B.paged_decode_plan_destroy(plan)


@pytest.mark.parametrize("schedule", [B.PD_SCHED_QUEUE, B.PD_SCHED_STATIC, B.PD_SCHED_AUTO])
@pytest.mark.parametrize("num_sms", [148, 152, 7])
@pytest.mark.parametrize("case", ["uniform", "ragged", "mqa"])
def test_planner_covers_every_tile_once(lib, case, num_sms, schedule):
    rng = np.random.default_rng(3)
    if case == "uniform":
        B_, Hq, Hkv = 32, 64, 8
        seq = np.full(B_, 4096)
        ql = np.ones(B_, int)
    elif case == "ragged":
        B_, Hq, Hkv = 128, 32, 8
        ql = rng.choice([1, 2, 4], B_)
        seq = np.clip(np.floor(np.exp(rng.uniform(0, np.log(16385), B_))).astype(int), ql, 16384)
    else:
        B_, Hq, Hkv = 9, 40, 1   # 40 rows per unit -> three row blocks
        ql = rng.choice([1, 2], B_)
        seq = rng.integers(2, 3000, B_)
    qi = np.concatenate([[0], np.cumsum(ql)])
    p = gqa_problem(B_, Hq=Hq, Hkv=Hkv, P=64, max_len=16384, num_sms=num_sms, schedule=schedule)
    info, items = plan_items(p, seq, qi)
    assert info.max_splits_used <= 16
    T = info.tile_tokens
    # rebuild the unit list the plan must cover
    G = Hq // Hkv
    units = []
    R = info.rows_per_unit
    assert R == (8 if (ql * G).max() <= 8 else 16)
    for b in range(B_):
        rows = ql[b] * G
        for g in range(Hkv):
            for r0 in range(0, rows, R):
                n = min(R, rows - r0)
                i_last = (r0 + n - 1) // G
                visible = seq[b] - ql[b] + i_last + 1
                units.append((visible + T - 1) // T)
    assert info.num_units == len(units)
    cover = [np.zeros(t, int) for t in units]
    splits = {}
    for u, t0, t1, s in items:
        assert 0 <= t0 < t1 <= units[u]
        cover[u][t0:t1] += 1
        splits.setdefault(u, set()).add(s)
    for u, c in enumerate(cover):
        assert (c == 1).all(), f"unit {u} tiles covered {c}"
        assert splits[u] == set(range(len(splits[u])))
    lengths = items[:, 2] - items[:, 1]
    if schedule == B.PD_SCHED_QUEUE:
        # longest first; ties by (unit, split)
        keys = list(zip(-lengths, items[:, 0], items[:, 3]))
        assert keys == sorted(keys)
        assert info.num_ctas == min(2 * num_sms, len(items))
    if schedule == B.PD_SCHED_STATIC:
        # every CTA range holds (nearly) the same number of tiles
        assert info.num_ctas <= 2 * num_sms
        assert lengths.sum() == sum(units)
    assert info.workspace_bytes >= 256 + 48 * info.num_units + 16 * info.num_items


def test_max_splits_one_means_unsplit(lib):
    p = gqa_problem(4, max_splits=1)
    info, items = plan_items(p, [4096, 100, 3000, 1])
    assert info.max_splits_used == 1 and info.partial_rows == 0
    assert (items[:, 3] == 0).all()


def test_planner_splits_small_batches(lib):
    # 8 units of 64 tiles on 152 SMs: the planner should split to fill the GPU
    p = gqa_problem(1)
    info, _ = plan_items(p, [4096])
    assert info.max_splits_used > 1 and info.partial_rows > 0


@pytest.mark.parametrize("bad", ["qlen_gt_len", "len_gt_max", "neg_len", "bad_heads", "page0",
                                 "splits17", "bad_dim", "bad_indptr0", "stride"])
def test_planner_rejects(lib, bad):
    p = gqa_problem(2, max_len=100, P=16)
    seq, qi = [50, 60], [0, 1, 2]
    want = B.PD_ERR_INVALID_ARG
    if bad == "qlen_gt_len":
        seq, qi = [1, 60], [0, 3, 4]
    elif bad == "len_gt_max":
        seq = [50, 101]
    elif bad == "neg_len":
        seq = [-1, 3]
    elif bad == "bad_heads":
        p.num_q_heads = 10
    elif bad == "page0":
        p.page_size = 0
    elif bad == "splits17":
        p.max_splits = 17
    elif bad == "bad_dim":
        p.head_dim_qk = p.head_dim_v = 64
        want = B.PD_ERR_UNSUPPORTED
    elif bad == "bad_indptr0":
        qi = [1, 2, 3]
    elif bad == "stride":
        p.k_page_stride = 7
    with pytest.raises(B.PdError) as e:
        B.paged_decode_plan(p, np.asarray(seq, np.int32), np.asarray(qi, np.int32))
    assert e.value.status == want


def test_empty_batch_plan(lib):
    p = gqa_problem(0)
    info, items = plan_items(p, [])
    assert info.num_items == 0 and items.shape == (0, 4)


def test_plan_id_depends_on_lengths(lib):
    p = gqa_problem(2, max_len=200, P=16)
    plans = [B.paged_decode_plan(p, np.asarray(s, np.int32)) for s in ([100, 50], [100, 51], [100, 50])]
    ids = [B.paged_decode_plan_get_info(x).plan_id for x in plans]
    for x in plans:
        B.paged_decode_plan_destroy(x)
    assert ids[0] != ids[1] and ids[0] == ids[2]


def test_mla_plan(lib):
    p = B.pd_problem()
    p.kind = B.PD_ATTN_MLA
    p.batch, p.num_q_heads, p.num_kv_heads = 4, 128, 1
    p.head_dim_qk, p.head_dim_v, p.page_size = 576, 512, 64
    p.max_pages_per_seq, p.num_pages, p.max_kv_len, p.num_sms = 64, 256, 4096, 152
    info, items = plan_items(p, [4096, 10, 4096, 2], [0, 2, 4, 6, 8])
    assert info.rows_per_unit == 64
    assert info.num_units == 4 * 4   # 2 x 128 rows -> four 64-row blocks per request


@pytest.mark.parametrize("schedule", [B.PD_SCHED_QUEUE, B.PD_SCHED_STATIC, B.PD_SCHED_AUTO])
def test_mla_plan_covers_every_tile_once(lib, schedule):
    """MLA units are 64-row blocks of (token, head) rows; each covers the keys
    visible to its last row in 64-key tiles, every tile exactly once."""
    rng = np.random.default_rng(5)
    B_, H, P = 24, 40, 32
    ql = rng.choice([1, 2, 3], B_)
    seq = np.maximum(rng.integers(1, 3000, B_), ql)
    p = B.pd_problem()
    p.kind = B.PD_ATTN_MLA
    p.batch, p.num_q_heads, p.num_kv_heads = B_, H, 1
    p.head_dim_qk, p.head_dim_v, p.page_size = 576, 512, P
    p.max_pages_per_seq, p.max_kv_len = 3072 // P, 3072
    p.num_pages, p.num_sms, p.schedule = B_ * p.max_pages_per_seq, 19, schedule
    qi = np.concatenate([[0], np.cumsum(ql)])
    info, items = plan_items(p, seq, qi)
    assert info.rows_per_unit == 64
    T = info.tile_tokens
    units = []
    for b in range(B_):
        rows = ql[b] * H
        for r0 in range(0, rows, 64):
            last = min(r0 + 64, rows) - 1
            units.append((seq[b] - ql[b] + last // H + 1 + T - 1) // T)
    assert info.num_units == len(units)
    cover = [np.zeros(t, int) for t in units]
    for u, t0, t1, _ in items:
        assert 0 <= t0 < t1 <= units[u]
        cover[u][t0:t1] += 1
    for u, c in enumerate(cover):
        assert (c == 1).all(), f"unit {u} tiles covered {c}"


def test_mla_page_size_must_be_multiple_of_8(lib):
    p = B.pd_problem()
    p.kind = B.PD_ATTN_MLA
    p.batch, p.num_q_heads, p.num_kv_heads = 1, 16, 1
    p.head_dim_qk, p.head_dim_v = 576, 512
    p.max_kv_len, p.num_sms = 48, 8
    for P, ok in ((12, False), (4, False), (16, True), (24, True)):
        p.page_size = P
        p.max_pages_per_seq = (48 + P - 1) // P
        p.num_pages = 4 * p.max_pages_per_seq
        if ok:
            info, _ = plan_items(p, [48], [0, 1])
            assert info.num_units == 1
        else:
            with pytest.raises(B.PdError) as e:
                B.paged_decode_plan(p, np.asarray([48], np.int32), np.asarray([0, 1], np.int32))
            assert e.value.status == B.PD_ERR_UNSUPPORTED, P


def test_prefill_plan(lib):
    """Prefill units are up to 256 packed rows (two 128-row query tiles) of
    whole groups with 128-key tiles;
    every visible tile of every unit is covered once; splits are merged by
    the merge kernel."""
    p = gqa_problem(3, Hq=32, Hkv=8, P=32, max_len=2048, kind=B.PD_ATTN_PREFILL, num_sms=16)
    seq, ql = [2047, 300, 129], [511, 300, 1]
    qi = np.concatenate([[0], np.cumsum(ql)])
    info, items = plan_items(p, seq, qi)
    assert info.rows_per_unit == 256 and info.tile_tokens == 128
    G = 4
    n_units = sum(8 * ((q * G + 255) // 256) for q in ql)
    assert info.num_units == n_units
    # tiles of a unit: keys visible to its last row, in 128-key tiles
    want = {}
    u = 0
    for L, q in zip(seq, ql):
        for g in range(8):
            for r0 in range(0, q * G, 256):
                last = min(r0 + 256, q * G) - 1
                want[u] = (L - q + last // G + 1 + 127) // 128
                u += 1
    got = {}
    for unit, t0, t1, _ in items.reshape(-1, 4):
        got.setdefault(int(unit), []).append((int(t0), int(t1)))
    for unit, n in want.items():
        ranges = sorted(got[unit])
        assert ranges[0][0] == 0 and ranges[-1][1] == n
        assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))


@pytest.mark.parametrize("what", ["fp8", "page_size", "group"])
def test_prefill_plan_rejects_unsupported(lib, what):
    kw = dict(kind=B.PD_ATTN_PREFILL, num_sms=16)
    if what == "fp8":
        p = gqa_problem(1, kv_dtype=B.PD_KV_FP8_E4M3, **kw)
    elif what == "page_size":
        p = gqa_problem(1, P=12, **kw)
    else:
        p = gqa_problem(1, Hq=24, Hkv=8, **kw)   # group 3 does not divide 128
    with pytest.raises(B.PdError) as e:
        B.paged_decode_plan(p, np.asarray([100], np.int32), np.asarray([0, 10], np.int32))
    assert e.value.status == B.PD_ERR_UNSUPPORTED


def test_append_host_validation(lib):
    """paged_kv_append rejects bad host arguments before touching the GPU."""
    import ctypes
    p = B.pd_append_problem(batch=2, num_kv_heads=2, head_dim=128, page_size=16, num_pages=8,
                            max_pages_per_seq=4, layout=B.PD_LAYOUT_NHD, kv_dtype=B.PD_KV_BF16)
    fake = 1 << 20  # never dereferenced: every call below fails validation first

    def call(prob, k_new=fake, v_new=fake, total=4, k_pool=fake, v_pool=fake, ks=None, vs=None, zero_tail=0):
        return lib.paged_kv_append(ctypes.byref(prob), k_new, v_new, total, fake, fake, fake, ks, vs,
                                   k_pool, v_pool, zero_tail, None, None)

    for field, value in (("head_dim", 100), ("head_dim", 2048), ("page_size", 0), ("num_kv_heads", 0),
                         ("layout", 7), ("kv_dtype", 5), ("batch", -1), ("k_page_stride", 3)):
        q = B.pd_append_problem.from_buffer_copy(p)
        setattr(q, field, value)
        assert call(q) == B.PD_ERR_INVALID_ARG, field
    assert call(p, v_pool=None) == B.PD_ERR_INVALID_ARG          # v_new without v_pool
    assert call(p, k_new=fake + 4) == B.PD_ERR_INVALID_ARG       # misaligned rows
    q = B.pd_append_problem.from_buffer_copy(p)
    q.kv_dtype = B.PD_KV_FP8_E4M3
    assert call(q) == B.PD_ERR_INVALID_ARG                       # E4M3 needs scales
    q.batch = 0
    assert call(q) == B.PD_OK                                    # empty batch: no-op
    assert call(p, total=0) == B.PD_OK                           # nothing to write


def test_resolved_merge_mode_and_launch_count(lib):
    """The plan summary reports the merge the plan runs and the kernels one
    run call enqueues: AUTO resolves to the merge kernel, FUSED is kept for
    decode (one launch), prefill always uses the merge kernel, and an
    unsplit plan is one launch whatever the mode."""
    seq = [4096, 100, 3000, 1]
    info, _ = plan_items(gqa_problem(4, max_splits=16, num_sms=300), seq)
    assert info.merge_mode == B.PD_MERGE_KERNEL and info.partial_rows > 0 and info.launches_per_run == 2
    info, _ = plan_items(gqa_problem(4, max_splits=16, num_sms=300, merge_mode=B.PD_MERGE_FUSED), seq)
    assert info.merge_mode == B.PD_MERGE_FUSED and info.partial_rows > 0 and info.launches_per_run == 1
    info, _ = plan_items(gqa_problem(4, max_splits=1), seq)
    assert info.merge_mode == B.PD_MERGE_KERNEL and info.partial_rows == 0 and info.launches_per_run == 1
    p = gqa_problem(1, Hq=32, Hkv=8, P=32, max_len=2048, kind=B.PD_ATTN_PREFILL, num_sms=4,
                    merge_mode=B.PD_MERGE_FUSED)
    info, _ = plan_items(p, [2047], [0, 511])
    assert info.merge_mode == B.PD_MERGE_KERNEL
    assert info.launches_per_run == (2 if info.partial_rows > 0 else 1)
    m = B.pd_problem()
    m.kind = B.PD_ATTN_MLA
    m.batch, m.num_q_heads, m.num_kv_heads = 2, 128, 1
    m.head_dim_qk, m.head_dim_v, m.page_size = 576, 512, 64
    m.max_pages_per_seq, m.num_pages, m.max_kv_len, m.num_sms = 64, 128, 4096, 152
    info, _ = plan_items(m, [4096, 4096], [0, 1, 2])
    assert info.merge_mode == B.PD_MERGE_KERNEL
    assert info.launches_per_run == (2 if info.partial_rows > 0 else 1)


def test_sm_count_query(lib):
    """num_sms = 0 asks the planner to query the current device: with none,
    the plan fails with PD_ERR_CUDA and the CUDA error text is recorded for
    paged_decode_last_cuda_error; with one, the plan uses its SM count."""
    import torch
    p = gqa_problem(2, Hq=8, Hkv=1, P=16, max_len=128, num_sms=0)
    if torch.cuda.is_available():
        info, _ = plan_items(p, [100, 5])
        sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        assert 1 <= info.num_ctas <= 2 * sms
    else:
        with pytest.raises(B.PdError) as e:
            B.paged_decode_plan(p, np.asarray([100, 5], np.int32))
        assert e.value.status == B.PD_ERR_CUDA
        assert lib.paged_decode_last_cuda_error().decode().startswith("SM count query")
