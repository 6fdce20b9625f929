"""Paged KV append on the GPU against the oracle: every byte of both pools
is compared (the append is integer/byte work, so parity is bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_199_gb300 import binding as B
from tests.helpers import run_oracle, assert_close
from paged_kv_cache_199_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _case(seed, P, layout, kv_dtype, Hkv=2, D=128, seq_lens=(37, 64, 5, 130, 1), q_lens=(3, 64, 5, 1, 1)):
    rng = np.random.default_rng(seed)
    seq_lens = np.array(seq_lens, np.int32)
    q_lens = np.array(q_lens, np.int32)
    qi = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    npg = (seq_lens + P - 1) // P
    num_pages = int(npg.sum()) + 4
    perm = rng.permutation(num_pages)
    table = np.full((len(seq_lens), int(npg.max()) + 1), -1, np.int32)
    k = 0
    for b in range(len(seq_lens)):
        table[b, :npg[b]] = perm[k:k + npg[b]]
        k += npg[b]
    shape = (num_pages, P, Hkv, D) if layout == B.PD_LAYOUT_NHD else (num_pages, Hkv, P, D)
    if kv_dtype == B.PD_KV_BF16:
        k_pool = torch.randn(shape, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
        v_pool = torch.randn(shape, generator=torch.Generator().manual_seed(seed + 1)).to(torch.bfloat16)
    else:
        k_pool = torch.from_numpy(rng.integers(0, 256, shape).astype(np.uint8) & 0xFE)
        v_pool = torch.from_numpy(rng.integers(0, 256, shape).astype(np.uint8) & 0xFE)
    g = torch.Generator().manual_seed(seed + 2)
    k_new = (torch.randn((int(qi[-1]), Hkv, D), generator=g) * 3)
    k_new[0, 0, :8] = torch.tensor([5000., -5000., 1e-3, -1e-3, 2e-4, 0., -0., 447.])  # saturation, subnormals
    v_new = torch.randn((int(qi[-1]), Hkv, D), generator=g) * 0.5
    return dict(seq_lens=seq_lens, qi=qi, table=table, k_pool=k_pool, v_pool=v_pool,
                k_new=k_new.to(torch.bfloat16), v_new=v_new.to(torch.bfloat16), Hkv=Hkv, D=D, P=P)


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def _at_offset(t, dev, elems):
    """t on the device, starting `elems` bf16 values into a larger buffer (an
    offset of 4 values makes it 8-byte but not 16-byte aligned)."""
    if elems == 0:
        return t.to(dev)
    buf = torch.zeros(t.numel() + elems, dtype=t.dtype, device=dev)
    buf[elems:].copy_(t.reshape(-1).to(dev))
    return buf[elems:].view(t.shape)


def _run_both(c, layout, kv_dtype, zero_tail, with_v=True, k_scale=0.75, v_scale=0.125, k_off=0, v_off=0):
    dev = "cuda"
    kp, vp = c["k_pool"].to(dev), (c["v_pool"].to(dev) if with_v else None)
    ks = torch.tensor([k_scale], dtype=torch.float32, device=dev)
    vs = torch.tensor([v_scale], dtype=torch.float32, device=dev)
    err = torch.zeros(2, dtype=torch.int32, device=dev)
    B.paged_kv_append(_at_offset(c["k_new"], dev, k_off), _at_offset(c["v_new"], dev, v_off) if with_v else None,
                      torch.from_numpy(c["qi"]).to(dev), torch.from_numpy(c["seq_lens"]).to(dev),
                      torch.from_numpy(c["table"]).to(dev), kp, vp, num_kv_heads=c["Hkv"], head_dim=c["D"],
                      page_size=c["P"], layout=layout, kv_dtype=kv_dtype, k_scale=ks, v_scale=vs,
                      zero_tail=zero_tail, error_word=err)
    torch.cuda.synchronize()
    okp, ovp, st = oracle.paged_append(
        _bits(c["k_new"]), _bits(c["v_new"]) if with_v else None, c["table"], c["seq_lens"], c["qi"],
        _bits(c["k_pool"]), _bits(c["v_pool"]) if with_v else None, num_kv_heads=c["Hkv"], head_dim=c["D"],
        page_size=c["P"], layout=oracle.NHD if layout == B.PD_LAYOUT_NHD else oracle.HND,
        kv_dtype=oracle.BF16 if kv_dtype == B.PD_KV_BF16 else oracle.E4M3, k_scale=k_scale, v_scale=v_scale,
        zero_tail=zero_tail)
    return kp.cpu(), (vp.cpu() if with_v else None), err.cpu().tolist(), okp, ovp, st


@pytest.mark.parametrize("kv_dtype", [B.PD_KV_BF16, B.PD_KV_FP8_E4M3])
@pytest.mark.parametrize("layout", [B.PD_LAYOUT_NHD, B.PD_LAYOUT_HND])
@pytest.mark.parametrize("P", [1, 16, 64])
@pytest.mark.parametrize("zero_tail", [False, True])
def test_append_bit_exact(kv_dtype, layout, P, zero_tail):
    c = _case(100 + P, P, layout, kv_dtype)
    kp, vp, err, okp, ovp, st = _run_both(c, layout, kv_dtype, zero_tail)
    assert st == 0 and err == [0, 0]
    np.testing.assert_array_equal(_bits(kp), okp)
    np.testing.assert_array_equal(_bits(vp), ovp)


@pytest.mark.parametrize("kv_dtype", [B.PD_KV_BF16, B.PD_KV_FP8_E4M3])
@pytest.mark.parametrize("k_off,v_off", [(4, 4), (0, 4), (4, 0)])
def test_append_inputs_8_byte_aligned(kv_dtype, k_off, v_off):
    """Inputs that are 8-byte but not 16-byte aligned take the 4-channel
    chunks; every byte still matches the oracle."""
    for layout in (B.PD_LAYOUT_NHD, B.PD_LAYOUT_HND):
        c = _case(300 + k_off + v_off, 16, layout, kv_dtype, Hkv=3, D=72)
        kp, vp, err, okp, ovp, st = _run_both(c, layout, kv_dtype, True, k_off=k_off, v_off=v_off)
        assert st == 0 and err == [0, 0]
        np.testing.assert_array_equal(_bits(kp), okp)
        np.testing.assert_array_equal(_bits(vp), ovp)


def test_append_mla_latent_rows():
    """A K-only pool: one 576-wide latent row per token (the MLA cache)."""
    c = _case(7, 64, B.PD_LAYOUT_NHD, B.PD_KV_BF16, Hkv=1, D=576)
    kp, _, err, okp, _, st = _run_both(c, B.PD_LAYOUT_NHD, B.PD_KV_BF16, True, with_v=False)
    assert st == 0 and err == [0, 0]
    np.testing.assert_array_equal(_bits(kp), okp)


def test_append_bad_metadata_skips_rows_and_flags():
    c = _case(9, 16, B.PD_LAYOUT_HND, B.PD_KV_BF16)
    c["table"][1, 2] = c["k_pool"].shape[0] + 5   # a page that request 1 writes into
    kp, vp, err, okp, ovp, st = _run_both(c, B.PD_LAYOUT_HND, B.PD_KV_BF16, True)
    assert st == 3 and err[0] == 1 and err[1] == 1
    np.testing.assert_array_equal(_bits(kp), okp)
    np.testing.assert_array_equal(_bits(vp), ovp)
    c = _case(9, 16, B.PD_LAYOUT_HND, B.PD_KV_BF16)
    c["seq_lens"][2] = 3                            # q_len 5 > seq_len 3
    kp, vp, err, okp, ovp, st = _run_both(c, B.PD_LAYOUT_HND, B.PD_KV_BF16, True)
    assert st == 2 and err == [2, 2]
    np.testing.assert_array_equal(_bits(kp), okp)
    np.testing.assert_array_equal(_bits(vp), ovp)


def test_append_then_decode():
    """Append the last q_len tokens of every request through the library, then
    decode: the result equals the oracle's decode of the dense cache."""
    x = W.workload("ragged", device="cpu", small=True)
    dec_inputs = x.to("cuda")
    qi = x.q_indptr.numpy()
    P = x.page_size
    # the new tokens' rows, read from the full pool, then erased from a copy
    k_pool = x.k_pool.clone()
    v_pool = x.v_pool.clone()
    table = x.block_tables.numpy()
    Hkv, D = x.num_kv_heads, x.head_dim_qk
    rows_k, rows_v = [], []
    for b in range(x.batch):
        L, n = int(x.seq_lens[b]), int(qi[b + 1] - qi[b])
        for i in range(n):
            pos = L - n + i
            page, slot = int(table[b, pos // P]), pos % P
            sel = (page, slot) if x.layout == "NHD" else (page, slice(None), slot)
            rows_k.append(x.k_pool[sel].clone())
            rows_v.append(x.v_pool[sel].clone())
            k_pool[sel] = 0
            v_pool[sel] = 0
    k_new = torch.stack(rows_k).cuda()
    v_new = torch.stack(rows_v).cuda()
    kp, vp = k_pool.cuda(), v_pool.cuda()
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    layout = B.PD_LAYOUT_NHD if x.layout == "NHD" else B.PD_LAYOUT_HND
    B.paged_kv_append(k_new, v_new, dec_inputs.q_indptr, dec_inputs.seq_lens, dec_inputs.block_tables, kp, vp,
                      num_kv_heads=Hkv, head_dim=D, page_size=P, layout=layout, error_word=err)
    torch.cuda.synchronize()
    assert err.tolist() == [0, 0]
    dec_inputs.k_pool, dec_inputs.v_pool = kp, vp
    dec = B.PagedDecode(dec_inputs)
    out, lse = dec.run()
    torch.cuda.synchronize()
    ref_out, ref_lse, _ = run_oracle(x)
    assert_close(out, lse, ref_out, ref_lse, "bf16", "append then decode")


@pytest.mark.parametrize("scale", [0.75, 0.1, 1.0 / 3.0, 7.3e-3, 2.5])
def test_append_e4m3_rounding_ties(scale):
    """New values placed at and one binary32 ulp around every E4M3 rounding
    midpoint (times the scale): the codes equal the oracle's, whose quotient
    is a true binary32 division."""
    codes = [c for c in range(0x7E)]
    mids = []
    for c in codes:
        lo, hi = oracle.e4m3_to_double(c), oracle.e4m3_to_double(c + 1)
        mids.append((lo + hi) / 2)
    mids = np.array(mids + [448.0, 464.0, 480.0, 2.0 ** -10], np.float64)
    x = (mids * scale).astype(np.float32)
    xs = np.concatenate([x, np.nextafter(x, np.float32(np.inf)), np.nextafter(x, np.float32(0)), -x])
    bits = torch.from_numpy(xs).to(torch.bfloat16)         # the append reads bf16 rows
    Hkv, D, P = 1, 8, 8
    n = (bits.numel() + D - 1) // D
    k_new = torch.zeros(n * D, dtype=torch.bfloat16)
    k_new[:bits.numel()] = bits
    k_new = k_new.view(n, Hkv, D)
    table = np.arange((n + P - 1) // P, dtype=np.int32)[None]
    c = dict(seq_lens=np.array([n], np.int32), qi=np.array([0, n], np.int32), table=table,
             k_pool=torch.zeros((table.shape[1], P, Hkv, D), dtype=torch.uint8),
             v_pool=torch.zeros((table.shape[1], P, Hkv, D), dtype=torch.uint8),
             k_new=k_new, v_new=k_new.clone(), Hkv=Hkv, D=D, P=P)
    kp, vp, err, okp, ovp, st = _run_both(c, B.PD_LAYOUT_NHD, B.PD_KV_FP8_E4M3, False, k_scale=scale,
                                          v_scale=scale)
    assert st == 0 and err == [0, 0]
    np.testing.assert_array_equal(_bits(kp), okp)
