"""GPU: bit-exact index probes, device error paths, metadata lifetime, CUDA
graph replay with a changed block table, the merge-states entry point."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_199_gb300 import binding as B
from paged_kv_cache_199_gb300 import workloads as W
from tests.helpers import assert_close, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_199_gb300 import build
    build.build()
    B.load()


# ---------------------------------------------------------------------------
# Index probes: every query row's output must be exactly the value row of
# one chosen key. Values encode (page, slot, kv head) in exact small
# integers, keys are zero except one large logit per query row at its target
# key, and a decoy with an even larger logit sits one position past the
# row's causal bound (visible only to later rows).
# ---------------------------------------------------------------------------

def _probe_gqa(layout, P, kv_dtype, G=4, Hkv=2, seed=0):
    rng = np.random.default_rng(seed)
    B_ = 6
    ql = rng.integers(1, 4, B_)
    seq = np.maximum(rng.integers(5, 300, B_), ql + 2)
    x = W.make_paged_inputs(seed=seed, seq_lens=seq, q_lens=ql, num_q_heads=G * Hkv, num_kv_heads=Hkv,
                            head_dim=128, page_size=P, layout=layout, kv_dtype=kv_dtype,
                            device="cpu", extra_pages=4, poison=False)
    # a logit margin of 4096 makes every other weight exactly 0 in fp32
    bigk = 16.0 if kv_dtype == "e4m3" else 64.0   # exact in E4M3 / bf16 (decoy: 2x)
    bigq = 4096.0 / bigk
    kf = torch.zeros(x.k_pool.shape, dtype=torch.float32)
    vf = torch.zeros(x.v_pool.shape, dtype=torch.float32)
    table = x.block_tables.numpy()
    mod = 16 if kv_dtype == "e4m3" else 256

    def rowview(pool, page, slot, g):
        return pool[page, slot, g] if layout == "NHD" else pool[page, g, slot]

    # value rows: (page % mod, page // mod % mod, slot % mod, g) in channels 0..3
    for page in range(x.num_pages):
        for slot in range(P):
            for g in range(Hkv):
                v = rowview(vf, page, slot, g)
                v[0], v[1], v[2], v[3] = page % mod, (page // mod) % mod, slot % mod, g
    q = torch.zeros(x.q.shape, dtype=torch.float32)
    expected = {}
    qi = x.q_indptr.numpy()
    for b in range(B_):
        L, n = int(seq[b]), int(ql[b])
        for g in range(Hkv):
            for i in range(n):
                pos = L - n + i
                t = int(rng.integers(0, pos + 1))
                if i == 0 and b % 2 == 0:
                    t = pos  # the newest visible key
                page, slot = int(table[b, t // P]), t % P
                rowview(kf, page, slot, g)[4 + i] = bigk
                if pos + 1 < L:  # decoy for this row, visible to row i + 1 only
                    dp, ds = int(table[b, (pos + 1) // P]), (pos + 1) % P
                    rowview(kf, dp, ds, g)[4 + i] = 2 * bigk
                for hh in range(G):
                    q[qi[b] + i, g * G + hh, 4 + i] = bigq
                    expected[(qi[b] + i, g * G + hh)] = (page, slot, g)
    if kv_dtype == "e4m3":
        x.k_pool = kf.to(torch.float8_e4m3fn).view(torch.uint8)
        x.v_pool = vf.to(torch.float8_e4m3fn).view(torch.uint8)
    else:
        x.k_pool = kf.to(torch.bfloat16)
        x.v_pool = vf.to(torch.bfloat16)
    x.q = q.to(torch.bfloat16)
    x.sm_scale = 1.0
    x.k_scale = x.v_scale = 1.0  # codes are the values themselves
    return x.to("cuda"), expected, mod


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("P", [1, 16, 64])
@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_index_probe_bit_exact(layout, P, kv_dtype):
    x, expected, mod = _probe_gqa(layout, P, kv_dtype, seed=P + (layout == "HND"))
    for kw in ({}, dict(max_splits=16, num_sms=300), dict(schedule=B.PD_SCHED_QUEUE, num_sms=300)):
        dec = B.PagedDecode(x, **kw)
        out, _ = dec.run()
        torch.cuda.synchronize()
        assert dec.read_error()[0] == 0
        o = out.float().cpu().numpy()
        # the oracle on the same bytes picks the same rows (decoys included)
        ref, _, _ = run_oracle(x)
        np.testing.assert_array_equal(o[:, :, :4], np.round(ref[:, :, :4], 6))
        hits = 0
        for (row, head), (page, slot, g) in expected.items():
            want = [page % mod, (page // mod) % mod, slot % mod, g]
            if np.array_equal(np.round(ref[row, head, :4], 6), want):
                assert o[row, head, :4].tolist() == want, (row, head, o[row, head, :4], want)
                hits += 1
        assert hits > len(expected) // 2


def test_mla_index_probe_bit_exact():
    rng = np.random.default_rng(7)
    B_, H, P = 4, 16, 16
    ql = np.array([1, 2, 3, 1])
    seq = np.array([40, 9, 77, 3])
    x = W.make_mla_inputs(seed=7, seq_lens=seq, q_lens=ql, num_heads=H, page_size=P, device="cpu",
                          extra_pages=2, poison=False)
    kv = torch.zeros(x.k_pool.shape, dtype=torch.float32)
    table = x.block_tables.numpy()
    for page in range(x.num_pages):
        for slot in range(P):
            kv[page, slot, 0], kv[page, slot, 1], kv[page, slot, 2] = page % 256, page // 256, slot
    q = torch.zeros(x.q.shape, dtype=torch.float32)
    qi = x.q_indptr.numpy()
    for b in range(B_):
        L, n = int(seq[b]), int(ql[b])
        for i in range(n):
            pos = L - n + i
            t = int(rng.integers(0, pos + 1)) if b % 2 else pos
            kv[int(table[b, t // P]), t % P, 512 + i] = 64.0   # rope channels: key only
            if pos + 1 < L:
                kv[int(table[b, (pos + 1) // P]), (pos + 1) % P, 512 + i] = 128.0
            q[qi[b] + i, :, 512 + i] = 64.0
    x.k_pool = x.v_pool = kv.to(torch.bfloat16)
    x.q = q.to(torch.bfloat16)
    x.sm_scale = 1.0
    x = x.to("cuda")
    for kw in ({}, dict(max_splits=16, num_sms=200)):
        dec = B.PagedDecode(x, **kw)
        out, _ = dec.run()
        torch.cuda.synchronize()
        ref, _, _ = run_oracle(x)
        np.testing.assert_array_equal(out.float().cpu().numpy()[:, :, :3], np.round(ref[:, :, :3], 6))


# ---------------------------------------------------------------------------
# Device error paths: no fault, an error word, zeros for the affected rows
# ---------------------------------------------------------------------------

def _small(device="cuda", **kw):
    return W.make_paged_inputs(seed=3, seq_lens=[90, 130, 17, 64], q_lens=[1, 2, 1, 1], num_q_heads=16,
                               num_kv_heads=2, head_dim=128, page_size=16, layout="HND", device=device,
                               extra_pages=3, **kw)


@pytest.mark.parametrize("sched", [B.PD_SCHED_STATIC, B.PD_SCHED_QUEUE])
def test_bad_page_id_sets_flag(sched):
    x = _small()
    ref, ref_lse, _ = run_oracle(x)
    x.block_tables[1, 3] = x.num_pages + 5  # a visible page of request 1
    dec = B.PagedDecode(x, schedule=sched, num_sms=64)
    out, lse = dec.run()
    torch.cuda.synchronize()
    code, info = dec.read_error()
    assert code == 1 and info == 1
    o = out.float().cpu().numpy()
    qi = x.q_indptr.cpu().numpy()
    assert np.all(o[qi[1]:qi[2]] == 0)
    keep = np.r_[qi[0]:qi[1], qi[2]:qi[4]]
    assert_close(o[keep], None, ref[keep], None, "bf16", "other requests")


def test_seq_len_mismatch_sets_flag():
    x = _small()
    dec = B.PagedDecode(x)
    x.seq_lens[2] = 16  # the device copy no longer matches the plan
    out, _ = dec.run()
    torch.cuda.synchronize()
    code, info = dec.read_error()
    assert code == 2 and info == 2
    qi = x.q_indptr.cpu().numpy()
    assert torch.all(out[qi[2]:qi[3]] == 0)


@pytest.mark.parametrize("merge_mode", [B.PD_MERGE_FUSED, B.PD_MERGE_KERNEL])
def test_workspace_of_another_plan_is_refused(merge_mode):
    # the other plan has split units, so the merge (in-kernel or the separate
    # merge kernel) would run if the workspace check let it
    x = _small()
    dec = B.PagedDecode(x)
    y = W.make_paged_inputs(seed=4, seq_lens=[100, 200, 300, 400], q_lens=[1, 1, 1, 1], num_q_heads=16,
                            num_kv_heads=2, head_dim=128, page_size=16, layout="HND", device="cuda")
    other = B.PagedDecode(y, upload=False, max_splits=16, num_sms=400, merge_mode=merge_mode)
    assert other.info.partial_rows > 0
    nbytes = max(other.info.workspace_bytes, dec.info.workspace_bytes)
    other.workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    B.paged_decode_plan_upload(dec.plan, other.workspace)  # the workspace now holds x's plan
    out, lse = other.alloc_outputs()
    out.fill_(3.0)
    other.run(out, lse)
    torch.cuda.synchronize()
    code, _ = other.read_error()
    assert code == 4
    assert torch.all(out == 3.0)


def test_metadata_lifetime_reuses_buffers():
    """A new plan for new lengths in the same workspace and tensors gives the
    new results (no stale host or device metadata)."""
    x = _small()
    dec = B.PagedDecode(x)
    ws = dec.workspace
    dec.run()
    for new_lens in ([91, 131, 18, 65], [3, 2, 1, 64]):
        y = W.make_paged_inputs(seed=3, seq_lens=new_lens, q_lens=[1, 2, 1, 1], num_q_heads=16,
                                num_kv_heads=2, head_dim=128, page_size=16, layout="HND", device="cuda",
                                extra_pages=3)
        d2 = B.PagedDecode(y, upload=False)
        if d2.info.workspace_bytes <= ws.numel():
            d2.workspace = ws
        d2.upload()
        out, lse = d2.run()
        torch.cuda.synchronize()
        assert d2.read_error()[0] == 0
        ref, ref_lse, _ = run_oracle(y)
        assert_close(out, lse, ref, ref_lse, "bf16", f"lens {new_lens}")


def test_cuda_graph_replay_with_changed_block_table():
    x = _small()
    dec = B.PagedDecode(x, num_sms=64)
    out, lse = dec.alloc_outputs()
    dec.run(out, lse)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dec.run(out, lse)
    # move every referenced page to another physical page (same lengths)
    table = x.block_tables.cpu().numpy()
    used = sorted(set(int(p) for p in table.ravel() if p >= 0))
    free = [p for p in range(x.num_pages) if p not in used]
    rng = np.random.default_rng(9)
    perm = rng.permutation(used + free)
    remap = {p: int(perm[k]) for k, p in enumerate(used)}
    new_k = x.k_pool.clone()
    new_v = x.v_pool.clone()
    for p_old, p_new in remap.items():
        new_k[p_new] = x.k_pool[p_old]
        new_v[p_new] = x.v_pool[p_old]
    new_table = np.where(table >= 0, np.vectorize(lambda p: remap.get(int(p), -1))(table), -1)
    x.k_pool.copy_(new_k)
    x.v_pool.copy_(new_v)
    x.block_tables.copy_(torch.from_numpy(new_table.astype(np.int32)))
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        ref, ref_lse, _ = run_oracle(x)
        assert_close(out, lse, ref, ref_lse, "bf16", "graph replay")


def test_untouched_output_rows():
    x = _small()
    dec = B.PagedDecode(x)
    big = torch.full((x.total_q + 3, x.num_q_heads, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    dec.run(big[: x.total_q], None)
    torch.cuda.synchronize()
    assert torch.all(big[x.total_q:] == 5.0)


@pytest.mark.parametrize("S,rows,dim", [(1, 7, 128), (5, 33, 128), (16, 100, 512), (3, 1, 8)])
def test_merge_states_entry_point(S, rows, dim):
    rng = np.random.default_rng(S * rows)
    v = rng.normal(0, 1, (S, rows, dim)).astype(np.float32)
    s = rng.normal(0, 3, (S, rows)).astype(np.float32)
    s[0, 0] = -np.inf  # an empty state
    if rows > 1:
        s[:, 1] = -np.inf  # a row with no state at all
    ref, ref_lse = oracle.merge_states(v.astype(np.float64), s.astype(np.float64))
    out = torch.empty((rows, dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((rows,), dtype=torch.float32, device="cuda")
    B.paged_decode_merge_states(torch.from_numpy(v).cuda(), torch.from_numpy(s).cuda(), out, lse)
    torch.cuda.synchronize()
    np.testing.assert_allclose(out.float().cpu().numpy(), ref, atol=1e-2, rtol=1e-2)
    got = lse.cpu().numpy()
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(got[fin], ref_lse[fin], atol=1e-4, rtol=1e-5)
    assert np.all(np.isneginf(got[~fin]))
