"""GPU: bit-exact index probes for the page walks of the tensor-core prefill
kernel (128-key tiles, 3-D query boxes, many new tokens per request) and of
the FP8 latent MLA kernel (five 128-byte E4M3 slabs per 576-channel row, the
last one zero-filled past the row).

Every query row's output must be exactly the value row of one chosen key.
Value rows encode (page, slot[, kv head]) as small integers that are exact in
the pool's element type; keys are zero except one large logit per query row
at its target key, and a decoy with twice that logit sits one position past
the row's inclusive causal bound (visible to later rows only, which query
another channel). The oracle on the same bytes must agree bit for bit."""
import numpy as np
import pytest
import torch

from paged_kv_cache_199_gb300 import binding as B
from paged_kv_cache_199_gb300 import workloads as W
from tests.helpers import run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_199_gb300 import build
    build.build()
    B.load()


def _encode_values(vf, layout, Hkv, mod):
    """Value row (page, slot, g): channels 0..3 = page % mod, page // mod % mod,
    slot % mod, g."""
    pages, P = vf.shape[0], (vf.shape[1] if layout == "NHD" else vf.shape[2])
    pg = torch.arange(pages, dtype=torch.float32)
    sl = torch.arange(P, dtype=torch.float32)
    gg = torch.arange(Hkv, dtype=torch.float32)
    if layout == "NHD":   # [pages][P][Hkv][D]
        vf[..., 0] = (pg % mod)[:, None, None]
        vf[..., 1] = ((pg // mod) % mod)[:, None, None]
        vf[..., 2] = (sl % mod)[None, :, None]
        vf[..., 3] = gg[None, None, :]
    else:                 # [pages][Hkv][P][D]
        vf[..., 0] = (pg % mod)[:, None, None]
        vf[..., 1] = ((pg // mod) % mod)[:, None, None]
        vf[..., 2] = (sl % mod)[None, None, :]
        vf[..., 3] = gg[None, :, None]


def _prefill_probe(layout, P, G, Hkv, seed):
    rng = np.random.default_rng(seed)
    ql = np.array([120, 37, 1, 90], dtype=np.int64)      # <= 124 rows: channel 4 + i per row
    seq = ql + rng.integers(0, 400, ql.size)
    seq[1] = ql[1]                                        # every key a new token
    x = W.make_paged_inputs(seed=seed, seq_lens=seq, q_lens=ql, num_q_heads=G * Hkv, num_kv_heads=Hkv,
                            head_dim=128, page_size=P, layout=layout, device="cpu", extra_pages=3,
                            poison=False)
    bigk, bigq = 64.0, 64.0           # logit 4096: every other weight is exactly 0 in fp32
    kf = torch.zeros(x.k_pool.shape, dtype=torch.float32)
    vf = torch.zeros(x.v_pool.shape, dtype=torch.float32)
    _encode_values(vf, layout, Hkv, 256)
    table = x.block_tables.numpy()
    q = torch.zeros(x.q.shape, dtype=torch.float32)
    qi = x.q_indptr.numpy()

    def rowview(pool, page, slot, g):
        return pool[page, slot, g] if layout == "NHD" else pool[page, g, slot]

    for b in range(len(seq)):
        L, n = int(seq[b]), int(ql[b])
        for g in range(Hkv):
            for i in range(n):
                pos = L - n + i
                t = pos if (i + g) % 3 == 0 else int(rng.integers(0, pos + 1))
                rowview(kf, int(table[b, t // P]), t % P, g)[4 + i] = bigk
                if pos + 1 < L:
                    rowview(kf, int(table[b, (pos + 1) // P]), (pos + 1) % P, g)[4 + i] = 2 * bigk
                q[qi[b] + i, g * G:(g + 1) * G, 4 + i] = bigq
    x.k_pool = kf.to(torch.bfloat16)
    x.v_pool = vf.to(torch.bfloat16)
    x.q = q.to(torch.bfloat16)
    x.sm_scale = 1.0
    return x.to("cuda")


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("P", [8, 24, 64])
@pytest.mark.parametrize("G,Hkv", [(4, 2), (16, 1)])
def test_prefill_index_probe_bit_exact(layout, P, G, Hkv):
    x = _prefill_probe(layout, P, G, Hkv, seed=P * 3 + G + (layout == "HND"))
    ref, _, _ = run_oracle(x)
    want = np.round(ref[:, :, :4], 6)
    # every row found its target: the encoded (slot, kv head) channels hold
    # integers, and the kv-head channel equals the head's group
    assert np.array_equal(want, np.round(want))
    assert np.array_equal(want[:, :, 3], np.broadcast_to(np.arange(G * Hkv) // G, want[:, :, 3].shape))
    for kw in ({}, dict(max_splits=16, num_sms=400), dict(schedule=B.PD_SCHED_STATIC, num_sms=300)):
        dec = B.PagedDecode(x, prefill=True, **kw)
        out, _ = dec.run()
        torch.cuda.synchronize()
        assert dec.read_error()[0] == 0
        np.testing.assert_array_equal(out.float().cpu().numpy()[:, :, :4], want, err_msg=f"{layout} P={P} {kw}")


@pytest.mark.parametrize("P", [16, 64])
def test_mla_fp8_index_probe_bit_exact(P):
    rng = np.random.default_rng(P + 1)
    H = 16
    ql = np.array([1, 2, 3, 1, 2])
    seq = np.array([40, 9, 300, 3, 130])
    x = W.make_mla_inputs(seed=P, seq_lens=seq, q_lens=ql, num_heads=H, page_size=P, device="cpu",
                          extra_pages=2, poison=False, kv_dtype="e4m3")
    kv = torch.zeros(x.k_pool.shape, dtype=torch.float32)
    table = x.block_tables.numpy()
    pg = torch.arange(x.num_pages, dtype=torch.float32)
    sl = torch.arange(P, dtype=torch.float32)
    # integers below 16 are exact E4M3 codes
    kv[:, :, 0] = (pg % 16)[:, None]
    kv[:, :, 1] = ((pg // 16) % 16)[:, None]
    kv[:, :, 2] = (sl % 16)[None, :]
    q = torch.zeros(x.q.shape, dtype=torch.float32)
    qi = x.q_indptr.numpy()
    for b in range(len(seq)):
        L, n = int(seq[b]), int(ql[b])
        for i in range(n):
            pos = L - n + i
            t = int(rng.integers(0, pos + 1)) if b % 2 else pos
            kv[int(table[b, t // P]), t % P, 512 + i] = 16.0        # rope channels: key only
            if pos + 1 < L:
                kv[int(table[b, (pos + 1) // P]), (pos + 1) % P, 512 + i] = 32.0
            q[qi[b] + i, :, 512 + i] = 16.0                          # logit 256, decoy 512
    x.k_pool = x.v_pool = kv.to(torch.float8_e4m3fn).view(torch.uint8)
    x.q = q.to(torch.float8_e4m3fn).view(torch.uint8)
    x.q_scale = x.k_scale = x.v_scale = 1.0
    x.sm_scale = 1.0
    x = x.to("cuda")
    ref, _, _ = run_oracle(x)
    want = np.round(ref[:, :, :3], 6)
    assert np.array_equal(want, np.round(want))
    for kw in ({}, dict(max_splits=16, num_sms=200), dict(schedule=B.PD_SCHED_QUEUE, num_sms=100)):
        dec = B.PagedDecode(x, **kw)
        out, _ = dec.run()
        torch.cuda.synchronize()
        assert dec.read_error()[0] == 0
        np.testing.assert_array_equal(out.float().cpu().numpy()[:, :, :3], want, err_msg=f"P={P} {kw}")
