"""Shared test helpers: run the oracle on a DecodeInputs batch (or a subset
of its requests) and compare a GPU result against it."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances the pages state for the public decode rows (PR #4557 validation
# paragraph): BF16 atol = rtol = 1e-2, FP8 e4m3 atol = rtol = 0.1.
TOL = {"bf16": (1e-2, 1e-2), "e4m3": (0.1, 0.1)}
# LSE is produced in fp32 from fp32 row statistics.
LSE_TOL = {"bf16": (2e-3, 2e-3), "e4m3": (2e-2, 2e-2)}


def subset(inputs, reqs):
    """numpy arrays of the given requests (pools shared), for the oracle."""
    a = inputs.oracle_arrays()
    reqs = np.asarray(reqs)
    qi = a["q_indptr"]
    q_rows = np.concatenate([np.arange(qi[b], qi[b + 1]) for b in reqs]) if len(reqs) else np.zeros(0, int)
    q_lens = qi[reqs + 1] - qi[reqs]
    new_qi = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    return dict(q=a["q"][q_rows], k_pool=a["k_pool"], v_pool=a["v_pool"],
                block_tables=a["block_tables"][reqs], seq_lens=a["seq_lens"][reqs],
                q_indptr=new_qi), q_rows


def gather_requests(inputs, reqs):
    """Like `subset`, but copies to the host only the pages the given requests
    reference (renumbered 0..n-1 in table order), so that requests of a
    multi-GB device pool can be checked one by one."""
    reqs = np.asarray(reqs)
    table = inputs.block_tables.cpu().numpy()
    seq = inputs.seq_lens_host()
    qi = inputs.q_indptr_host()
    P = inputs.page_size
    pages, new_table = [], np.full((len(reqs), table.shape[1]), -1, np.int32)
    for r, b in enumerate(reqs):
        n = (int(seq[b]) + P - 1) // P
        new_table[r, :n] = np.arange(len(pages), len(pages) + n)
        pages.extend(int(p) for p in table[b, :n])
    idx = torch.as_tensor(pages, dtype=torch.long, device=inputs.k_pool.device)

    def host(t):
        t = t.index_select(0, idx).cpu().contiguous()
        return t.numpy() if t.dtype == torch.uint8 else t.view(torch.int16).numpy().view(np.uint16)

    k = host(inputs.k_pool)
    v = k if inputs.kind == "mla" else host(inputs.v_pool)
    q_rows = np.concatenate([np.arange(qi[b], qi[b + 1]) for b in reqs]) if len(reqs) else np.zeros(0, int)
    qt = inputs.q[torch.as_tensor(q_rows, dtype=torch.long, device=inputs.q.device)].cpu().contiguous()
    q = qt.numpy() if qt.dtype == torch.uint8 else qt.view(torch.int16).numpy().view(np.uint16)
    q_lens = qi[reqs + 1] - qi[reqs]
    new_qi = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    return dict(q=q, k_pool=k, v_pool=v, block_tables=new_table, seq_lens=seq[reqs].astype(np.int32),
                q_indptr=new_qi), q_rows


def _sinks(inputs):
    s = getattr(inputs, "sinks", None)
    return None if s is None else s.detach().cpu().double().numpy()


def run_oracle(inputs, reqs=None, arrays=None, num_threads=0):
    """FP64 oracle over `reqs` (default: all). Returns (out, lse, q_rows)."""
    if reqs is None:
        reqs = np.arange(inputs.batch)
    a, q_rows = subset(inputs, reqs) if arrays is None else arrays
    if inputs.kind == "mla":
        out, lse = oracle.mla_decode(a["q"], a["k_pool"], a["block_tables"], a["seq_lens"],
                                     a["q_indptr"], num_heads=inputs.num_q_heads,
                                     head_dim_qk=inputs.head_dim_qk, head_dim_v=inputs.head_dim_v,
                                     page_size=inputs.page_size, sm_scale=inputs.sm_scale,
                                     sinks=_sinks(inputs),
                                     kv_dtype=oracle.BF16 if inputs.kv_dtype == "bf16" else oracle.E4M3,
                                     q_scale=getattr(inputs, "q_scale", 1.0), kv_scale=inputs.k_scale,
                                     num_threads=num_threads)
    else:
        out, lse = oracle.paged_decode(
            a["q"], a["k_pool"], a["v_pool"], a["block_tables"], a["seq_lens"], a["q_indptr"],
            num_q_heads=inputs.num_q_heads, num_kv_heads=inputs.num_kv_heads,
            head_dim_qk=inputs.head_dim_qk, head_dim_v=inputs.head_dim_v,
            page_size=inputs.page_size, layout=oracle.NHD if inputs.layout == "NHD" else oracle.HND,
            kv_dtype=oracle.BF16 if inputs.kv_dtype == "bf16" else oracle.E4M3,
            sm_scale=inputs.sm_scale, k_scale=inputs.k_scale, v_scale=inputs.v_scale,
            sinks=_sinks(inputs), num_threads=num_threads)
    return out, lse, q_rows


def assert_close(gpu_out, gpu_lse, ref_out, ref_lse, kv_dtype, what=""):
    atol, rtol = TOL[kv_dtype]
    g = gpu_out.float().cpu().numpy().astype(np.float64) if isinstance(gpu_out, torch.Tensor) else gpu_out
    bad = ~(np.abs(g - ref_out) <= atol + rtol * np.abs(ref_out))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} outputs outside atol={atol} rtol={rtol}; "
            f"max abs err {np.nanmax(np.abs(g - ref_out)):.4g}; first {idx.tolist()} "
            f"gpu {[float(g[tuple(i)]) for i in idx]} ref {[float(ref_out[tuple(i)]) for i in idx]}")
    if gpu_lse is not None:
        la, lr = LSE_TOL[kv_dtype]
        gl = gpu_lse.float().cpu().numpy().astype(np.float64) if isinstance(gpu_lse, torch.Tensor) else gpu_lse
        bad = ~(np.abs(gl - ref_lse) <= la + lr * np.abs(ref_lse))
        if bad.any():
            idx = np.argwhere(bad)[:5]
            raise AssertionError(f"{what}: {int(bad.sum())} LSE values off; first {idx.tolist()} "
                                 f"gpu {[float(gl[tuple(i)]) for i in idx]} "
                                 f"ref {[float(ref_lse[tuple(i)]) for i in idx]}")


def max_err(gpu_out, ref_out):
    g = gpu_out.float().cpu().numpy().astype(np.float64)
    return float(np.max(np.abs(g - ref_out))) if g.size else 0.0
