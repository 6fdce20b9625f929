"""Pins for the FP64 oracle: checks against facts that do not come from the
oracle itself (library routines, closed forms, invariants, a spec table).

Each ``pin_*`` takes the loaded oracle library (so that the mutation test can
run the same pins against a copy of the oracle with a planted mistake) and
raises AssertionError when the oracle disagrees.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# Input helpers (test-side; independent of the oracle's address arithmetic)
# ---------------------------------------------------------------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


class Dense:
    """A batch held as dense per-request K/V ([L_b, Hkv, D]) plus the paged
    pool the same tokens are scattered into."""

    def __init__(self, seed, seq_lens, q_lens, Hq, Hkv, D, Dv=None, P=4, layout=oracle.NHD,
                 extra_pages=3, std=1.0):
        rng = np.random.default_rng(seed)
        Dv = D if Dv is None else Dv
        self.Hq, self.Hkv, self.D, self.Dv, self.P, self.layout = Hq, Hkv, D, Dv, P, layout
        self.seq_lens = np.asarray(seq_lens, np.int32)
        self.q_lens = np.asarray(q_lens, np.int32)
        self.q_indptr = np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)
        B = len(seq_lens)
        self.k = [bf16_bits(rng.normal(0, std, (L, Hkv, D))) for L in seq_lens]
        self.v = [bf16_bits(rng.normal(0, std, (L, Hkv, Dv))) for L in seq_lens]
        self.q = bf16_bits(rng.normal(0, std, (int(self.q_indptr[-1]), Hq, D)))
        self.npages = [(int(L) + P - 1) // P for L in seq_lens]
        self.num_pages = sum(self.npages) + extra_pages
        self.perm = rng.permutation(self.num_pages)
        self.repage(P, layout, self.perm)

    def repage(self, P, layout, perm):
        """Scatter the dense tokens into a fresh pool (NaN in unused slots)."""
        self.P, self.layout = P, layout
        B = len(self.seq_lens)
        npages = [(int(L) + P - 1) // P for L in self.seq_lens]
        num_pages = max(sum(npages), len(perm))
        maxp = max(npages + [1])
        table = np.full((B, maxp), -1, np.int32)
        c = 0
        for b in range(B):
            table[b, :npages[b]] = perm[c:c + npages[b]]
            c += npages[b]
        nan = np.uint16(0x7FC0)
        if layout == oracle.NHD:
            kp = np.full((num_pages, P, self.Hkv, self.D), nan, np.uint16)
            vp = np.full((num_pages, P, self.Hkv, self.Dv), nan, np.uint16)
        else:
            kp = np.full((num_pages, self.Hkv, P, self.D), nan, np.uint16)
            vp = np.full((num_pages, self.Hkv, P, self.Dv), nan, np.uint16)
        for b in range(B):
            for t in range(int(self.seq_lens[b])):
                page, slot = table[b, t // P], t % P
                if layout == oracle.NHD:
                    kp[page, slot] = self.k[b][t]
                    vp[page, slot] = self.v[b][t]
                else:
                    kp[page, :, slot] = self.k[b][t]
                    vp[page, :, slot] = self.v[b][t]
        self.k_pool, self.v_pool, self.table = kp, vp, table
        return self

    def run(self, lib, sm_scale, kv_range=None):
        return oracle.paged_decode(
            self.q, self.k_pool, self.v_pool, self.table, self.seq_lens, self.q_indptr,
            num_q_heads=self.Hq, num_kv_heads=self.Hkv, head_dim_qk=self.D, head_dim_v=self.Dv,
            page_size=self.P, layout=self.layout, sm_scale=sm_scale, kv_range=kv_range, lib=lib)

    def sdpa(self, sm_scale):
        """torch's scaled_dot_product_attention in float64 on the dense
        tokens, GQA by enable_gqa, bottom-right causal mask (row i of a
        request with q_len rows sees keys 0 .. L - q_len + i)."""
        outs, lses = [], []
        for b in range(len(self.seq_lens)):
            L, ql = int(self.seq_lens[b]), int(self.q_lens[b])
            q = torch.from_numpy(bits_to_f64(self.q[self.q_indptr[b]:self.q_indptr[b + 1]]))
            k = torch.from_numpy(bits_to_f64(self.k[b]))
            v = torch.from_numpy(bits_to_f64(self.v[b]))
            q4 = q.permute(1, 0, 2)[None]          # [1, Hq, ql, D]
            k4 = k.permute(1, 0, 2)[None]          # [1, Hkv, L, D]
            v4 = v.permute(1, 0, 2)[None]
            mask = torch.ones(ql, L, dtype=torch.bool).tril(diagonal=L - ql)
            o = torch.nn.functional.scaled_dot_product_attention(
                q4, k4, v4, attn_mask=mask, scale=sm_scale, enable_gqa=True)
            outs.append(o[0].permute(1, 0, 2).numpy())
            kk = k4.repeat_interleave(self.Hq // self.Hkv, dim=1)
            logits = (q4 @ kk.transpose(-1, -2)) * sm_scale
            logits = logits.masked_fill(~mask, float("-inf"))
            lses.append(torch.logsumexp(logits, dim=-1)[0].permute(1, 0).numpy())
        return np.concatenate(outs), np.concatenate(lses)


# ---------------------------------------------------------------------------
# Pins
# ---------------------------------------------------------------------------

def pin_library_sdpa(lib):
    """Paged oracle == torch SDPA (float64) on the dense tokens, for both
    layouts, several page sizes, GQA groups and multi-row (causal) queries."""
    cases = [
        dict(seq_lens=[5, 17, 1], q_lens=[1, 3, 1], Hq=4, Hkv=1, D=8, P=4, layout=oracle.NHD),
        dict(seq_lens=[9, 23], q_lens=[2, 4], Hq=8, Hkv=2, D=12, P=3, layout=oracle.HND),
        dict(seq_lens=[31, 6, 12], q_lens=[1, 2, 1], Hq=6, Hkv=6, D=16, P=16, layout=oracle.NHD),
        dict(seq_lens=[14], q_lens=[3], Hq=4, Hkv=2, D=8, Dv=6, P=1, layout=oracle.HND),
    ]
    for i, c in enumerate(cases):
        d = Dense(100 + i, **c)
        scale = 1.0 / math.sqrt(c["D"]) * (1.5 if i % 2 else 1.0)
        out, lse = d.run(lib, scale)
        ref_out, ref_lse = d.sdpa(scale)
        np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def pin_single_key(lib):
    """One visible key: the output is that value row exactly and the LSE is
    the key's logit."""
    d = Dense(7, seq_lens=[1, 1], q_lens=[1, 1], Hq=4, Hkv=2, D=16, P=2)
    scale = 0.25
    out, lse = d.run(lib, scale)
    for b in range(2):
        for h in range(4):
            g = h // 2
            np.testing.assert_array_equal(out[b, h], bits_to_f64(d.v[b][0, g]))
            qf = bits_to_f64(d.q[b, h])
            kf = bits_to_f64(d.k[b][0, g])
            assert abs(lse[b, h] - scale * float(np.dot(qf, kf))) < 1e-12


def pin_constant_v(lib):
    """Every value row equal to c (a power of two): the output is c exactly."""
    d = Dense(8, seq_lens=[13, 40], q_lens=[1, 2], Hq=4, Hkv=1, D=8, P=4)
    c = -0.5
    for b in range(2):
        d.v[b][:] = bf16_bits(np.full(d.v[b].shape, c))
    d.repage(d.P, d.layout, d.perm)
    out, _ = d.run(lib, 0.3)
    np.testing.assert_array_equal(out, np.full(out.shape, c))


def pin_zero_query(lib):
    """q = 0: uniform weights, output = mean of the visible values,
    LSE = ln(number of visible keys)."""
    d = Dense(9, seq_lens=[11, 7], q_lens=[3, 1], Hq=2, Hkv=1, D=8, P=4)
    d.q[:] = 0
    out, lse = d.run(lib, 0.7)
    row = 0
    for b in range(2):
        L, ql = int(d.seq_lens[b]), int(d.q_lens[b])
        for i in range(ql):
            n = L - ql + i + 1
            mean = bits_to_f64(d.v[b][:n, 0]).mean(axis=0)
            for h in range(2):
                np.testing.assert_allclose(out[row, h], mean, rtol=1e-13, atol=1e-14)
                assert abs(lse[row, h] - math.log(n)) < 1e-13
            row += 1


def pin_two_keys(lib):
    """Two keys: out = sigmoid(s0 - s1) v0 + sigmoid(s1 - s0) v1."""
    d = Dense(10, seq_lens=[2], q_lens=[1], Hq=1, Hkv=1, D=8, P=1)
    scale = 0.4
    out, lse = d.run(lib, scale)
    q = bits_to_f64(d.q[0, 0])
    s = [scale * float(np.dot(q, bits_to_f64(d.k[0][t, 0]))) for t in range(2)]
    sig = lambda x: 1.0 / (1.0 + math.exp(-x))
    ref = sig(s[0] - s[1]) * bits_to_f64(d.v[0][0, 0]) + sig(s[1] - s[0]) * bits_to_f64(d.v[0][1, 0])
    np.testing.assert_allclose(out[0, 0], ref, rtol=1e-13, atol=1e-14)
    assert abs(lse[0, 0] - (max(s) + math.log1p(math.exp(-abs(s[0] - s[1]))))) < 1e-13


def pin_causal_one_hot(lib):
    """q_len = 2 at L = 3 with K = 0 and one-hot values: query row 0 sees keys
    {0, 1}, row 1 sees {0, 1, 2} (inclusive bound)."""
    d = Dense(11, seq_lens=[3], q_lens=[2], Hq=1, Hkv=1, D=4, P=2)
    d.k[0][:] = 0
    eye = np.zeros((3, 1, 4), np.float32)
    for t in range(3):
        eye[t, 0, t] = 1.0
    d.v[0] = bf16_bits(eye)
    d.repage(d.P, d.layout, d.perm)
    out, lse = d.run(lib, 1.0)
    np.testing.assert_allclose(out[0, 0], [0.5, 0.5, 0.0, 0.0], atol=1e-15)
    np.testing.assert_allclose(out[1, 0], [1 / 3, 1 / 3, 1 / 3, 0.0], atol=1e-15)
    assert abs(lse[0, 0] - math.log(2)) < 1e-15 and abs(lse[1, 0] - math.log(3)) < 1e-15


def pin_invariances(lib):
    """Bit-identical results under a physical page permutation, a different
    page size and the NHD <-> HND relayout (same tokens, same order)."""
    d = Dense(12, seq_lens=[37, 64, 5], q_lens=[1, 2, 1], Hq=8, Hkv=2, D=16, P=16)
    base, base_lse = d.run(lib, 0.2)
    rng = np.random.default_rng(5)
    for P, layout in [(16, oracle.HND), (1, oracle.NHD), (64, oracle.HND), (3, oracle.NHD)]:
        n = sum((int(L) + P - 1) // P for L in d.seq_lens) + 4
        d.repage(P, layout, rng.permutation(n))
        out, lse = d.run(lib, 0.2)
        np.testing.assert_array_equal(out, base)
        np.testing.assert_array_equal(lse, base_lse)


def pin_split_merge(lib):
    """States over disjoint key ranges merged by log-sum-exp equal the
    unsplit result (the split-KV reduction)."""
    d = Dense(13, seq_lens=[50, 29], q_lens=[2, 1], Hq=4, Hkv=2, D=8, P=4)
    full, full_lse = d.run(lib, 0.35)
    cuts = [0, 7, 20, 33, 1 << 30]
    states = [d.run(lib, 0.35, kv_range=(cuts[i], cuts[i + 1])) for i in range(len(cuts) - 1)]
    rows = full.shape[0] * full.shape[1]
    o = np.stack([s[0].reshape(rows, -1) for s in states])
    l = np.stack([s[1].reshape(rows) for s in states])
    out, lse = oracle.merge_states(o, l, lib=lib)
    np.testing.assert_allclose(out.reshape(full.shape), full, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse.reshape(full_lse.shape), full_lse, rtol=1e-12, atol=1e-13)
    # an empty state is neutral; two equal states keep out and add ln 2
    e_o, e_l = oracle.merge_states(np.stack([o[0], np.zeros_like(o[0])]),
                                   np.stack([l[0], np.full_like(l[0], -np.inf)]), lib=lib)
    np.testing.assert_array_equal(e_o, o[0])
    np.testing.assert_array_equal(e_l, l[0])
    t_o, t_l = oracle.merge_states(np.stack([o[1], o[1]]), np.stack([l[1], l[1]]), lib=lib)
    np.testing.assert_allclose(t_o, o[1], rtol=1e-15)
    np.testing.assert_allclose(t_l, l[1] + math.log(2), rtol=1e-15)


def pin_shift(lib):
    """An extra channel with k = 1 on every key and q = c / sm_scale adds c to
    every logit: the output is unchanged and the LSE moves by exactly c."""
    d = Dense(14, seq_lens=[21, 9], q_lens=[1, 2], Hq=2, Hkv=1, D=8, P=4)
    scale, c = 0.125, 2.0
    base, base_lse = d.run(lib, scale)
    for b in range(2):
        d.k[b] = np.concatenate([d.k[b], bf16_bits(np.ones(d.k[b].shape[:2] + (1,)))], axis=2)
    d.q = np.concatenate([d.q, bf16_bits(np.full(d.q.shape[:2] + (1,), c / scale))], axis=2)
    d.D += 1
    d.repage(d.P, d.layout, d.perm)
    out, lse = d.run(lib, scale)
    np.testing.assert_allclose(out, base, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, base_lse + c, rtol=1e-13, atol=1e-13)


def pin_mla_is_gqa(lib):
    """MLA = GQA with one KV head, K = the whole cached row and V its first
    d_v channels (same pool, value row stride = d_qk); and MLA == torch SDPA
    on the gathered rows."""
    rng = np.random.default_rng(15)
    P, dqk, dv, H = 4, 12, 8, 6
    seq_lens = np.array([9, 14], np.int32)
    q_lens = np.array([1, 2], np.int32)
    qi = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    npg = [(int(L) + P - 1) // P for L in seq_lens]
    perm = rng.permutation(sum(npg) + 2)
    table = np.full((2, max(npg)), -1, np.int32)
    table[0, :npg[0]] = perm[:npg[0]]
    table[1, :npg[1]] = perm[npg[0]:npg[0] + npg[1]]
    pool = bf16_bits(rng.normal(0, 0.5, (len(perm), P, dqk)))
    q = bf16_bits(rng.normal(0, 0.5, (int(qi[-1]), H, dqk)))
    scale = 1.0 / math.sqrt(dqk)
    out, lse = oracle.mla_decode(q, pool, table, seq_lens, qi, num_heads=H, head_dim_qk=dqk,
                                 head_dim_v=dv, page_size=P, sm_scale=scale, lib=lib)
    g_out, g_lse = oracle.paged_decode(
        q, pool.reshape(len(perm), P, 1, dqk), pool.reshape(len(perm), P, 1, dqk), table,
        seq_lens, qi, num_q_heads=H, num_kv_heads=1, head_dim_qk=dqk, head_dim_v=dv,
        page_size=P, layout=oracle.NHD, sm_scale=scale, k_row_stride=dqk, v_row_stride=dqk,
        k_page_stride=P * dqk, v_page_stride=P * dqk, lib=lib)
    np.testing.assert_allclose(out, g_out, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(lse, g_lse, rtol=1e-14, atol=1e-15)
    # the same through the library routine, rows gathered with numpy indexing
    for b in range(2):
        L = int(seq_lens[b])
        rows = bits_to_f64(pool[table[b, :npg[b]]].reshape(-1, dqk)[:L])
        qq = torch.from_numpy(bits_to_f64(q[qi[b]:qi[b + 1]])).permute(1, 0, 2)[None]
        kk = torch.from_numpy(rows)[None, None]
        vv = torch.from_numpy(rows[:, :dv])[None, None]
        mask = torch.ones(int(q_lens[b]), L, dtype=torch.bool).tril(diagonal=L - int(q_lens[b]))
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask,
                                                               scale=scale, enable_gqa=True)
        np.testing.assert_allclose(out[qi[b]:qi[b + 1]], ref[0].permute(1, 0, 2).numpy(),
                                   rtol=1e-12, atol=1e-12)


def pin_e4m3_table(lib):
    """All 256 E4M3 codes decode like torch's float8_e4m3fn, and the OCP
    spec's special values are met exactly."""
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(b, lib=lib) for b in range(256)])
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    np.testing.assert_array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)])
    with open(os.path.join(GOLDEN, "e4m3_ocp_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            byte, val = line.split()[:2]
            v = oracle.e4m3_to_double(int(byte, 16), lib=lib)
            if val == "nan":
                assert math.isnan(v), byte
            else:
                assert v == float(val) and math.copysign(1, v) == math.copysign(1, float(val)), byte


def pin_fp8_path(lib):
    """E4M3 pools with scalar scales == SDPA on the values dequantised by
    torch (x = code * scale)."""
    rng = np.random.default_rng(16)
    P, Hkv, Hq, D = 8, 2, 8, 16
    seq_lens, q_lens = [19, 8], [1, 1]
    k32 = rng.normal(0, 1, (4, Hkv, P, D)).astype(np.float32)
    v32 = rng.normal(0, 1, (4, Hkv, P, D)).astype(np.float32)
    ks, vs = float(np.abs(k32).max() / 448), float(np.abs(v32).max() / 448)
    kb = torch.from_numpy(k32 / ks).clamp(-448, 448).to(torch.float8_e4m3fn)
    vb = torch.from_numpy(v32 / vs).clamp(-448, 448).to(torch.float8_e4m3fn)
    table = np.array([[2, 0, 3], [1, -1, -1]], np.int32)
    q = bf16_bits(rng.normal(0, 1, (2, Hq, D)))
    scale = 1 / math.sqrt(D)
    out, lse = oracle.paged_decode(
        q, kb.view(torch.uint8).numpy(), vb.view(torch.uint8).numpy(), table,
        np.array(seq_lens, np.int32), np.array([0, 1, 2], np.int32), num_q_heads=Hq,
        num_kv_heads=Hkv, head_dim_qk=D, head_dim_v=D, page_size=P, layout=oracle.HND,
        kv_dtype=oracle.E4M3, sm_scale=scale, k_scale=ks, v_scale=vs, lib=lib)
    kd = kb.to(torch.float64) * ks
    vd = vb.to(torch.float64) * vs
    for b, L in enumerate(seq_lens):
        pages = table[b, :(L + P - 1) // P]
        kk = kd[pages].permute(1, 0, 2, 3).reshape(Hkv, -1, D)[:, :L][None]
        vv = vd[pages].permute(1, 0, 2, 3).reshape(Hkv, -1, D)[:, :L][None]
        qq = torch.from_numpy(bits_to_f64(q[b:b + 1])).permute(1, 0, 2)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=scale, enable_gqa=True)
        np.testing.assert_allclose(out[b], ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-12)


def pin_e4m3_encode(lib):
    """The E4M3 encoder: every finite code round-trips; every midpoint between
    neighbouring codes goes to the even code; values beyond 448 saturate; NaN
    stays NaN; random binary32 values within range encode like torch's
    float8_e4m3fn cast (round to nearest even)."""
    finite = [c for c in range(256) if (c & 0x7F) != 0x7F]
    for c in finite:
        assert oracle.e4m3_from_float(oracle.e4m3_to_double(c, lib=lib), lib=lib) == c, hex(c)
    for sign in (0x00, 0x80):
        for c in range(0, 0x7E):
            lo = oracle.e4m3_to_double(sign | c, lib=lib)
            hi = oracle.e4m3_to_double(sign | (c + 1), lib=lib)
            want = sign | (c if c % 2 == 0 else c + 1)
            assert oracle.e4m3_from_float((lo + hi) / 2, lib=lib) == want, hex(sign | c)
    for v, code in ((449.0, 0x7E), (464.0, 0x7E), (1e30, 0x7E), (-1e30, 0xFE), (float("inf"), 0x7E)):
        assert oracle.e4m3_from_float(v, lib=lib) == code, v
    assert oracle.e4m3_from_float(float("nan"), lib=lib) & 0x7F == 0x7F
    rng = np.random.default_rng(21)
    xs = np.concatenate([rng.normal(0, 1, 2000), rng.normal(0, 100, 2000), rng.normal(0, 0.01, 2000),
                         rng.uniform(-448, 448, 2000)]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_float(float(x), lib=lib) for x in xs], np.uint8)
    np.testing.assert_array_equal(got, ref)


def _pool_rows(pool, layout, page, slot, Hkv):
    """[Hkv, D] rows of (page, slot) in an NHD [pages, P, Hkv, D] or HND
    [pages, Hkv, P, D] pool (test-side indexing)."""
    return pool[page, slot] if layout == oracle.NHD else pool[page, :, slot]


def pin_append(lib):
    """Appending new tokens: each new row lands at position L - n + i of its
    request (read back through the table with numpy indexing), BF16 bits are
    copied and E4M3 bytes are torch's RN-even encoding of x / scale; the tail
    slots of the last page are zeroed on request; no other byte changes."""
    rng = np.random.default_rng(22)
    for layout in (oracle.NHD, oracle.HND):
        for kv_dtype in (oracle.BF16, oracle.E4M3):
            for zero_tail in (False, True):
                P, Hkv, D = 4, 2, 8
                seq_lens = np.array([7, 4, 13, 9], np.int32)
                q_lens = np.array([2, 4, 1, 3], np.int32)
                qi = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
                npg = (seq_lens + P - 1) // P
                num_pages = int(npg.sum()) + 3
                perm = rng.permutation(num_pages)
                table = np.full((4, int(npg.max())), -1, np.int32)
                k = 0
                for b in range(4):
                    table[b, :npg[b]] = perm[k:k + npg[b]]
                    k += npg[b]
                shape = (num_pages, P, Hkv, D) if layout == oracle.NHD else (num_pages, Hkv, P, D)
                if kv_dtype == oracle.BF16:
                    k_pool = bf16_bits(rng.normal(0, 1, shape))
                    v_pool = bf16_bits(rng.normal(0, 1, shape))
                else:
                    k_pool = rng.integers(0, 0x7E, shape).astype(np.uint8)
                    v_pool = rng.integers(0, 0x7E, shape).astype(np.uint8)
                kx = rng.normal(0, 3, (int(qi[-1]), Hkv, D))
                kx[0, 0, 0] = 5000.0  # saturates with the scale below
                k_new = bf16_bits(kx)
                v_new = bf16_bits(rng.normal(0, 3, (int(qi[-1]), Hkv, D)))
                ks, vs = 0.5, 0.25
                kp, vp, st = oracle.paged_append(k_new, v_new, table, seq_lens, qi, k_pool, v_pool,
                                                 num_kv_heads=Hkv, head_dim=D, page_size=P, layout=layout,
                                                 kv_dtype=kv_dtype, k_scale=ks, v_scale=vs,
                                                 zero_tail=zero_tail, lib=lib)
                assert st == 0
                if kv_dtype == oracle.BF16:
                    want_k, want_v = k_new, v_new
                else:
                    def enc(bits, sc):
                        x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float() / sc
                        return x.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                    want_k, want_v = enc(k_new, ks), enc(v_new, vs)
                touched = np.zeros(shape, bool)
                for b in range(4):
                    L, n = int(seq_lens[b]), int(q_lens[b])
                    for i in range(n):
                        pos = L - n + i
                        page, slot = int(table[b, pos // P]), pos % P
                        np.testing.assert_array_equal(_pool_rows(kp, layout, page, slot, Hkv), want_k[qi[b] + i])
                        np.testing.assert_array_equal(_pool_rows(vp, layout, page, slot, Hkv), want_v[qi[b] + i])
                        _pool_rows(touched, layout, page, slot, Hkv)[...] = True
                    if zero_tail and L % P:
                        page = int(table[b, (L - 1) // P])
                        for slot in range(L % P, P):
                            assert not _pool_rows(kp, layout, page, slot, Hkv).any()
                            assert not _pool_rows(vp, layout, page, slot, Hkv).any()
                            _pool_rows(touched, layout, page, slot, Hkv)[...] = True
                np.testing.assert_array_equal(kp[~touched], k_pool[~touched])
                np.testing.assert_array_equal(vp[~touched], v_pool[~touched])


def pin_sinks(lib):
    """Attention sinks: one visible key gives sigma(s0 - sink) v0 and
    lse = log(e^s0 + e^sink); a sink of -inf changes nothing; and a sink
    equals one extra key, visible to every row, whose logit is the sink and
    whose value is zero (evaluated by torch SDPA on dense tensors with an
    added channel); MLA with sinks equals GQA with one KV head."""
    d = Dense(31, seq_lens=[1, 1], q_lens=[1, 1], Hq=4, Hkv=2, D=16, P=2)
    scale = 0.25
    sinks = np.array([0.3, -1.2, 2.0, -30.0])
    out, lse = oracle.paged_decode(d.q, d.k_pool, d.v_pool, d.table, d.seq_lens, d.q_indptr, num_q_heads=4,
                                   num_kv_heads=2, head_dim_qk=16, head_dim_v=16, page_size=2,
                                   layout=d.layout, sm_scale=scale, sinks=sinks, lib=lib)
    for b in range(2):
        for h in range(4):
            g = h // 2
            s0 = scale * float(np.dot(bits_to_f64(d.q[b, h]), bits_to_f64(d.k[b][0, g])))
            w = 1.0 / (1.0 + math.exp(sinks[h] - s0))
            np.testing.assert_allclose(out[b, h], w * bits_to_f64(d.v[b][0, g]), rtol=1e-13, atol=1e-15)
            assert abs(lse[b, h] - np.logaddexp(s0, sinks[h])) < 1e-12
    d = Dense(32, seq_lens=[9, 5, 12], q_lens=[1, 3, 2], Hq=6, Hkv=2, D=8, P=4)
    kw = dict(num_q_heads=6, num_kv_heads=2, head_dim_qk=8, head_dim_v=8, page_size=4, layout=d.layout,
              sm_scale=0.5, lib=lib)
    base = oracle.paged_decode(d.q, d.k_pool, d.v_pool, d.table, d.seq_lens, d.q_indptr, **kw)
    none = oracle.paged_decode(d.q, d.k_pool, d.v_pool, d.table, d.seq_lens, d.q_indptr,
                               sinks=np.full(6, -np.inf), **kw)
    np.testing.assert_array_equal(base[0], none[0])
    np.testing.assert_array_equal(base[1], none[1])
    sinks = np.array([0.5, -2.0, 1.5, 0.0, 3.0, -0.7])
    out, lse = oracle.paged_decode(d.q, d.k_pool, d.v_pool, d.table, d.seq_lens, d.q_indptr, sinks=sinks, **kw)
    for b in range(3):
        L, ql = int(d.seq_lens[b]), int(d.q_lens[b])
        q = torch.from_numpy(bits_to_f64(d.q[d.q_indptr[b]:d.q_indptr[b + 1]])).permute(1, 0, 2)  # [Hq, ql, D]
        k = torch.from_numpy(bits_to_f64(d.k[b])).permute(1, 0, 2).repeat_interleave(3, dim=0)    # [Hq, L, D]
        v = torch.from_numpy(bits_to_f64(d.v[b])).permute(1, 0, 2).repeat_interleave(3, dim=0)
        # channel D carries the sink: q' = [q, 1], k'_t = [k_t, 0], k* = [0, sink / scale], v* = 0
        q2 = torch.cat([q, torch.ones(6, ql, 1, dtype=torch.float64)], -1)
        k2 = torch.cat([torch.zeros(6, 1, 8, dtype=torch.float64), k], 1)
        k2 = torch.cat([k2, torch.zeros(6, L + 1, 1, dtype=torch.float64)], -1)
        k2[:, 0, 8] = torch.from_numpy(sinks) / 0.5
        v2 = torch.cat([torch.zeros(6, 1, 8, dtype=torch.float64), v], 1)
        mask = torch.ones(ql, L + 1, dtype=torch.bool).tril(diagonal=L + 1 - ql)
        ref = torch.nn.functional.scaled_dot_product_attention(q2[None], k2[None], v2[None], attn_mask=mask,
                                                               scale=0.5)
        logits = (q2 @ k2.transpose(-1, -2)) * 0.5
        ref_lse = torch.logsumexp(logits.masked_fill(~mask, float("-inf")), dim=-1)       # [Hq, ql]
        np.testing.assert_allclose(out[d.q_indptr[b]:d.q_indptr[b + 1]], ref[0].permute(1, 0, 2).numpy(),
                                   rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[d.q_indptr[b]:d.q_indptr[b + 1]], ref_lse.permute(1, 0).numpy(),
                                   rtol=1e-12, atol=1e-12)
    # MLA with sinks == GQA with one KV head and the same sinks
    rng = np.random.default_rng(33)
    P, dqk, dv, H = 4, 12, 8, 3
    seq_lens = np.array([7, 10], np.int32)
    qi = np.array([0, 1, 3], np.int32)
    table = np.array([[0, 3, -1], [1, 2, 4]], np.int32)
    pool = bf16_bits(rng.normal(0, 0.5, (5, P, dqk)))
    q = bf16_bits(rng.normal(0, 0.5, (3, H, dqk)))
    sinks = np.array([0.2, -1.0, 1.1])
    out, lse = oracle.mla_decode(q, pool, table, seq_lens, qi, num_heads=H, head_dim_qk=dqk, head_dim_v=dv,
                                 page_size=P, sm_scale=0.3, sinks=sinks, lib=lib)
    g_out, g_lse = oracle.paged_decode(
        q, pool.reshape(5, P, 1, dqk), pool.reshape(5, P, 1, dqk), table, seq_lens, qi, num_q_heads=H,
        num_kv_heads=1, head_dim_qk=dqk, head_dim_v=dv, page_size=P, layout=oracle.NHD, sm_scale=0.3,
        k_row_stride=dqk, v_row_stride=dqk, k_page_stride=P * dqk, v_page_stride=P * dqk, sinks=sinks, lib=lib)
    np.testing.assert_allclose(out, g_out, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(lse, g_lse, rtol=1e-14, atol=1e-15)


def pin_mla_fp8(lib):
    """FP8 latent MLA (E4M3 query and pool with scalar scales) == torch SDPA in
    float64 on the values torch dequantises (code * scale)."""
    rng = np.random.default_rng(41)
    P, dqk, dv, H = 4, 12, 8, 3
    seq_lens = np.array([7, 10], np.int32)
    qi = np.array([0, 1, 3], np.int32)
    table = np.array([[0, 3, -1], [1, 2, 4]], np.int32)
    qs, ks = 0.02, 0.005
    qf = rng.normal(0, 1, (3, H, dqk))
    kvf = rng.normal(0, 1, (5, P, dqk))
    qb = torch.from_numpy(qf / qs).clamp(-448, 448).to(torch.float8_e4m3fn)
    kvb = torch.from_numpy(kvf / ks).clamp(-448, 448).to(torch.float8_e4m3fn)
    out, lse = oracle.mla_decode(qb.view(torch.uint8).numpy(), kvb.view(torch.uint8).numpy(), table, seq_lens, qi,
                                 num_heads=H, head_dim_qk=dqk, head_dim_v=dv, page_size=P, sm_scale=0.3,
                                 kv_dtype=oracle.E4M3, q_scale=qs, kv_scale=ks, lib=lib)
    qd = qb.to(torch.float64) * qs
    kvd = kvb.to(torch.float64) * ks
    for b in range(2):
        L, ql = int(seq_lens[b]), int(qi[b + 1] - qi[b])
        rows = kvd[table[b, :(L + P - 1) // P]].reshape(-1, dqk)[:L]
        qq = qd[qi[b]:qi[b + 1]].permute(1, 0, 2)[None]
        mask = torch.ones(ql, L, dtype=torch.bool).tril(diagonal=L - ql)
        ref = torch.nn.functional.scaled_dot_product_attention(qq, rows[None, None], rows[:, :dv][None, None],
                                                               attn_mask=mask, scale=0.3, enable_gqa=True)
        np.testing.assert_allclose(out[qi[b]:qi[b + 1]], ref[0].permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13)


ALL_PINS = [pin_library_sdpa, pin_single_key, pin_constant_v, pin_zero_query, pin_two_keys,
            pin_causal_one_hot, pin_invariances, pin_split_merge, pin_shift, pin_mla_is_gqa,
            pin_e4m3_table, pin_fp8_path, pin_e4m3_encode, pin_append, pin_sinks, pin_mla_fp8]
