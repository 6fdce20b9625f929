"""Seeded synthetic inputs for paged decode attention.

This module only draws numbers and lays them out; it holds none of the
attention arithmetic. Both the CUDA library's tests/benchmark and the FP64
oracle consume what it makes, so the two sides always see the same bytes.

Structure (lengths, query counts, page permutation, block tables) comes from
numpy's PCG64 seeded with ``seed`` and does not depend on the device. Values
come from a torch generator seeded from ``seed`` on the device the tensors
are made on; the bytes therefore differ between a CPU and a CUDA draw of the
same seed, and every consumer reads the bytes that were actually made.

Layouts (names as on the FlashInfer cake_fmha API page and PR #5952):
  NHD pool  [num_pages, page_size, Hkv, D]
  HND pool  [num_pages, Hkv, page_size, D]
  MLA pool  [num_pages, page_size, 576]   (512 latent + 64 rope channels)
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

NHD, HND = "NHD", "HND"
BF16, E4M3 = "bf16", "e4m3"

# Poison values: NaN in pages no request references, large finite garbage
# in the unused tail of a request's last page.
_BF16_NAN_BITS = 0x7FC0
_E4M3_NAN_BYTE = 0x7F
_TAIL_GARBAGE_BF16 = 1.0e4
_TAIL_GARBAGE_E4M3 = 448.0


@dataclasses.dataclass
class DecodeInputs:
    """One batch of decode inputs. Tensors live on ``device``."""

    kind: str                      # "gqa" or "mla"
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim_qk: int
    head_dim_v: int
    page_size: int
    num_pages: int
    layout: str                    # NHD / HND ("NHD" for MLA's single head)
    kv_dtype: str                  # bf16 / e4m3
    q: torch.Tensor                # bf16 [total_q, Hq, Dqk]
    k_pool: torch.Tensor           # bf16 or uint8 (e4m3 bytes); MLA: the latent pool
    v_pool: torch.Tensor           # same tensor as k_pool for MLA
    block_tables: torch.Tensor     # int32 [B, max_pages]
    seq_lens: torch.Tensor         # int32 [B]   total length incl. new tokens
    q_indptr: torch.Tensor         # int32 [B+1]
    sm_scale: float
    k_scale: float = 1.0
    v_scale: float = 1.0
    name: str = ""
    sinks: Optional[torch.Tensor] = None   # fp32 [Hq] attention-sink logits, or None
    q_scale: float = 1.0                   # E4M3 MLA query: value = code * q_scale

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_kv_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.batch else 0

    @property
    def max_q_len(self) -> int:
        qi = self.q_indptr.cpu().numpy()
        return int((qi[1:] - qi[:-1]).max()) if self.batch else 0

    def seq_lens_host(self) -> np.ndarray:
        return self.seq_lens.cpu().numpy().astype(np.int32)

    def q_indptr_host(self) -> np.ndarray:
        return self.q_indptr.cpu().numpy().astype(np.int32)

    def kv_bytes(self) -> int:
        """K/V bytes of every visible token row (the algorithmic traffic)."""
        elem = 1 if self.kv_dtype == E4M3 else 2
        total_tokens = int(self.seq_lens.to(torch.int64).sum().item())
        if self.kind == "mla":
            return total_tokens * self.head_dim_qk * elem
        return total_tokens * self.num_kv_heads * (self.head_dim_qk + self.head_dim_v) * elem

    def to(self, device) -> "DecodeInputs":
        fields = {f.name: getattr(self, f.name) for f in dataclasses.fields(self)}
        for k, v in fields.items():
            if isinstance(v, torch.Tensor):
                fields[k] = v.to(device)
        if self.kind == "mla":
            fields["v_pool"] = fields["k_pool"]
        return DecodeInputs(**fields)

    # Host views for the oracle -------------------------------------------
    def oracle_arrays(self):
        """numpy views: q bits (uint16, or uint8 E4M3 codes for FP8 MLA), pools
        (uint16 bf16 bits or uint8)."""
        if self.q.dtype == torch.uint8:
            q = self.q.cpu().contiguous().numpy()
        else:
            q = self.q.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        if self.kv_dtype == BF16:
            k = self.k_pool.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
            v = self.v_pool.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        else:
            k = self.k_pool.cpu().contiguous().numpy()
            v = self.v_pool.cpu().contiguous().numpy()
        return dict(q=q, k_pool=k, v_pool=v,
                    block_tables=self.block_tables.cpu().numpy().astype(np.int32),
                    seq_lens=self.seq_lens_host(), q_indptr=self.q_indptr_host())


def _torch_gen(seed: int, device) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev.type if dev.type != "cuda" else dev)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def _normal(shape, std, gen, device, chunk_elems=1 << 28):
    """float32 N(0, std^2) drawn in chunks (bounded temporary memory)."""
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=torch.float32, device=device)
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        out[s:e].normal_(0.0, std, generator=gen)
    return out.view(shape)


def _to_e4m3_bytes(x: torch.Tensor) -> torch.Tensor:
    """float32 -> OCP E4M3FN bytes, round to nearest even, saturated at 448."""
    return x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def make_paged_inputs(*, seed: int, seq_lens: Sequence[int], q_lens: Sequence[int],
                      num_q_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                      layout: str = HND, kv_dtype: str = BF16, device="cpu",
                      extra_pages: int = 0, max_pages_per_seq: Optional[int] = None,
                      value_std: float = 1.0, k_outlier_prob: float = 0.0,
                      k_outlier_mult: float = 8.0, poison: bool = True,
                      sm_scale: Optional[float] = None, name: str = "",
                      v_channel_mean: float = 0.0) -> DecodeInputs:
    """Paged GQA decode inputs with a shuffled page pool.

    Every request's logical page j is stored at a physical page drawn from a
    seeded permutation of the pool; ``extra_pages`` unreferenced pages are
    mixed in and (with ``poison``) filled with NaN, and the unused tail slots
    of each request's last page hold large finite garbage.

    ``v_channel_mean`` > 0 shifts every (kv head, channel) of V by its own
    offset of magnitude U(m, 2m) and random sign (drawn from the structure
    generator), so that outputs, which are convex combinations of value
    rows, are of order m instead of near zero.
    """
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    B = int(seq_lens.shape[0])
    assert q_lens.shape == (B,)
    n_pages_req = [(int(L) + page_size - 1) // page_size for L in seq_lens]
    n_ref = int(sum(n_pages_req))
    num_pages = n_ref + int(extra_pages)
    if max_pages_per_seq is None:
        max_pages_per_seq = max([1] + n_pages_req)
    perm = rng.permutation(num_pages)
    table = np.full((B, max_pages_per_seq), -1, dtype=np.int32)
    cursor = 0
    for b in range(B):
        table[b, : n_pages_req[b]] = perm[cursor: cursor + n_pages_req[b]]
        cursor += n_pages_req[b]
    referenced = np.zeros(num_pages, dtype=bool)
    referenced[perm[:n_ref]] = True

    gen = _torch_gen(seed * 7919 + 17, device)
    D = head_dim
    if layout == NHD:
        pool_shape = (num_pages, page_size, num_kv_heads, D)
    elif layout == HND:
        pool_shape = (num_pages, num_kv_heads, page_size, D)
    else:
        raise ValueError(layout)
    total_q = int(q_lens.sum())
    q = _normal((total_q, num_q_heads, D), value_std, gen, device).to(torch.bfloat16)
    k32 = _normal(pool_shape, value_std, gen, device)
    if k_outlier_prob > 0:
        mask = torch.rand(pool_shape, generator=gen, device=device) < k_outlier_prob
        k32 = torch.where(mask, k32 * k_outlier_mult, k32)
    v32 = _normal(pool_shape, value_std, gen, device)
    if v_channel_mean > 0:
        mag = rng.uniform(v_channel_mean, 2 * v_channel_mean, (num_kv_heads, D))
        sign = np.where(rng.integers(0, 2, (num_kv_heads, D)) == 1, 1.0, -1.0)
        mean = torch.from_numpy((mag * sign).astype(np.float32)).to(device)
        v32 = v32 + (mean if layout == NHD else mean[:, None, :])

    k_scale = v_scale = 1.0
    if kv_dtype == E4M3:
        # per-tensor scale: the largest magnitude maps to E4M3's 448
        k_scale = float(k32.abs().max().item()) / 448.0
        v_scale = float(v32.abs().max().item()) / 448.0
        k_pool = _to_e4m3_bytes(k32 / k_scale)
        v_pool = _to_e4m3_bytes(v32 / v_scale)
    elif kv_dtype == BF16:
        k_pool = k32.to(torch.bfloat16)
        v_pool = v32.to(torch.bfloat16)
    else:
        raise ValueError(kv_dtype)
    del k32, v32

    if poison:
        _poison(k_pool, v_pool, referenced, table, seq_lens, page_size, layout, kv_dtype, rng)

    q_indptr = np.zeros(B + 1, dtype=np.int32)
    q_indptr[1:] = np.cumsum(q_lens)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    return DecodeInputs(
        kind="gqa", batch=B, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
        head_dim_qk=D, head_dim_v=D, page_size=page_size, num_pages=num_pages, layout=layout,
        kv_dtype=kv_dtype, q=q, k_pool=k_pool, v_pool=v_pool,
        block_tables=torch.from_numpy(table).to(device),
        seq_lens=torch.from_numpy(seq_lens.astype(np.int32)).to(device),
        q_indptr=torch.from_numpy(q_indptr).to(device), sm_scale=float(sm_scale),
        k_scale=k_scale, v_scale=v_scale, name=name)


def _poison(k_pool, v_pool, referenced, table, seq_lens, P, layout, kv_dtype, rng):
    unref = np.nonzero(~referenced)[0]
    if kv_dtype == BF16:
        nan_val = torch.tensor(_BF16_NAN_BITS, dtype=torch.int16).view(torch.bfloat16).item()
        for pool in (k_pool, v_pool):
            if unref.size:
                pool[torch.from_numpy(unref).to(pool.device)] = nan_val
    else:
        for pool in (k_pool, v_pool):
            if unref.size:
                pool[torch.from_numpy(unref).to(pool.device)] = _E4M3_NAN_BYTE
    garbage = _TAIL_GARBAGE_BF16 if kv_dtype == BF16 else _TAIL_GARBAGE_E4M3
    for b, L in enumerate(seq_lens):
        L = int(L)
        if L == 0 or L % P == 0:
            continue
        page = int(table[b, (L - 1) // P])
        tail = slice(L % P, P)
        sign = 1.0 if rng.integers(0, 2) else -1.0
        for pool in (k_pool, v_pool):
            if kv_dtype == BF16:
                val = sign * garbage
                if layout == NHD:
                    pool[page, tail] = val
                else:
                    pool[page, :, tail] = val
            else:
                byte = 0x7E if sign > 0 else 0xFE  # +-448
                if layout == NHD:
                    pool[page, tail] = byte
                else:
                    pool[page, :, tail] = byte


def make_mla_inputs(*, seed: int, seq_lens: Sequence[int], q_lens: Sequence[int],
                    num_heads: int = 128, head_dim_qk: int = 576, head_dim_v: int = 512,
                    page_size: int = 64, device="cpu", extra_pages: int = 0,
                    value_std: float = 0.5, poison: bool = True,
                    sm_scale: Optional[float] = None, name: str = "",
                    kv_dtype: str = BF16) -> DecodeInputs:
    """MLA decode inputs: one latent KV head shared by every query head.
    kv_dtype E4M3: query and latent pool are E4M3 codes of x / scale with
    per-tensor scales amax / 448 (query: q_scale; pool: k_scale = v_scale)."""
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    B = int(seq_lens.shape[0])
    n_pages_req = [(int(L) + page_size - 1) // page_size for L in seq_lens]
    n_ref = int(sum(n_pages_req))
    num_pages = n_ref + int(extra_pages)
    max_pages = max([1] + n_pages_req)
    perm = rng.permutation(num_pages)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    cursor = 0
    for b in range(B):
        table[b, : n_pages_req[b]] = perm[cursor: cursor + n_pages_req[b]]
        cursor += n_pages_req[b]
    referenced = np.zeros(num_pages, dtype=bool)
    referenced[perm[:n_ref]] = True
    gen = _torch_gen(seed * 7919 + 29, device)
    total_q = int(q_lens.sum())
    qf = _normal((total_q, num_heads, head_dim_qk), value_std, gen, device)
    kvf = _normal((num_pages, page_size, head_dim_qk), value_std, gen, device)
    q_scale = kv_scale = 1.0
    if kv_dtype == E4M3:
        q_scale = float(qf.abs().max().item()) / 448.0 if total_q else 1.0
        kv_scale = float(kvf.abs().max().item()) / 448.0
        q = _to_e4m3_bytes(qf / q_scale)
        kv = _to_e4m3_bytes(kvf / kv_scale)
    else:
        q = qf.to(torch.bfloat16)
        kv = kvf.to(torch.bfloat16)
    if poison:
        unref = np.nonzero(~referenced)[0]
        if unref.size:
            if kv_dtype == E4M3:
                nan_val = 0x7F
            else:
                nan_val = torch.tensor(_BF16_NAN_BITS, dtype=torch.int16).view(torch.bfloat16).item()
            kv[torch.from_numpy(unref).to(kv.device)] = nan_val
        for b, L in enumerate(seq_lens):
            L = int(L)
            if L and L % page_size:
                page = int(table[b, (L - 1) // page_size])
                if kv_dtype == E4M3:
                    kv[page, L % page_size:] = 0x7E if rng.integers(0, 2) else 0xFE   # +-448
                else:
                    kv[page, L % page_size:] = _TAIL_GARBAGE_BF16 * (1 if rng.integers(0, 2) else -1)
    q_indptr = np.zeros(B + 1, dtype=np.int32)
    q_indptr[1:] = np.cumsum(q_lens)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(head_dim_qk)
    return DecodeInputs(
        kind="mla", batch=B, num_q_heads=num_heads, num_kv_heads=1, head_dim_qk=head_dim_qk,
        head_dim_v=head_dim_v, page_size=page_size, num_pages=num_pages, layout=NHD,
        kv_dtype=kv_dtype, q=q, k_pool=kv, v_pool=kv,
        block_tables=torch.from_numpy(table).to(device),
        seq_lens=torch.from_numpy(seq_lens.astype(np.int32)).to(device),
        q_indptr=torch.from_numpy(q_indptr).to(device), sm_scale=float(sm_scale), name=name,
        k_scale=kv_scale, v_scale=kv_scale, q_scale=q_scale)


# ---------------------------------------------------------------------------
# The five workloads (and scaled-down variants of the same structure).
# ---------------------------------------------------------------------------

def ragged_lengths(seed: int, batch: int, max_len: int = 16384, q_choices=(1, 2, 4)):
    """q_len uniform over ``q_choices``; seq_len log-uniform in [1, max_len],
    floor(exp(U(0, ln(max_len + 1)))) clamped to [q_len, max_len]."""
    rng = np.random.default_rng(seed + 1000003)
    q_lens = rng.choice(np.asarray(q_choices), size=batch)
    u = rng.uniform(0.0, math.log(max_len + 1), size=batch)
    L = np.floor(np.exp(u)).astype(np.int64)
    L = np.clip(L, q_lens, max_len)
    return L, q_lens


def workload(name: str, device="cpu", small: bool = False, seed: Optional[int] = None,
             batch: Optional[int] = None, v_channel_mean: float = 0.0) -> DecodeInputs:
    """Named workloads.

    tiny      B=2, Hq=8, Hkv=1, D=128, P=16, NHD, pool of 16 pages, L={37,64}
    gqa8      B=32, Hq=64, Hkv=8, D=128, P=32, HND, L=4096
    ragged    B=128, q_len in {1,2,4}, Hq=32, Hkv=8, D=128, P=64, HND, L log-uniform
              in [1,16384], 1% of K elements x8, 5% extra NaN pages
    fp8       B=16, Hq=64, Hkv=8, D=128, P=64, HND, L=4096, e4m3 K/V, scalar scales
    mla1/mla2 B=512, q_len 1 / 2, 128 heads, 576/512, P=64, L=4096, N(0, 0.5^2)
    mla_fp8   B=128, q_len 1, 128 heads, E4M3 query and latent pool (per-tensor
              scales), P=64, L=4096
    prefill   B=4, q_len=511 new tokens over L=2047 cached, HND, P=32, one
              shared K/V table (a BF16 context profile of the cake_fmha API
              page), heads of the GQA-8 decode shape (Hq=64, Hkv=8, D=128)
    ``small`` keeps the structure and shrinks batch and lengths so that the
    oracle finishes in seconds; ``batch`` overrides the batch size alone (for
    profiling a smaller case of the same shape); ``v_channel_mean`` (fp8 only)
    gives V per-channel offsets so that outputs are of order one (a test
    variant, not the workload's statement).
    """
    if name == "tiny":
        s = 1 if seed is None else seed
        return make_paged_inputs(seed=s, seq_lens=[37, 64], q_lens=[1, 1], num_q_heads=8,
                                 num_kv_heads=1, head_dim=128, page_size=16, layout=NHD,
                                 device=device, extra_pages=9, max_pages_per_seq=4, name=name)
    if name == "gqa8":
        s = 2 if seed is None else seed
        B, L = (4, 1000) if small else (32, 4096)
        B = batch or B
        return make_paged_inputs(seed=s, seq_lens=[L] * B, q_lens=[1] * B, num_q_heads=64,
                                 num_kv_heads=8, head_dim=128, page_size=32, layout=HND,
                                 device=device, name=name)
    if name == "ragged":
        s = 3 if seed is None else seed
        B, maxL = (12, 1500) if small else (128, 16384)
        B = batch or B
        L, ql = ragged_lengths(s, B, maxL)
        n_ref = int(sum((int(x) + 63) // 64 for x in L))
        return make_paged_inputs(seed=s, seq_lens=L, q_lens=ql, num_q_heads=32, num_kv_heads=8,
                                 head_dim=128, page_size=64, layout=HND, device=device,
                                 extra_pages=max(1, int(round(0.05 * n_ref))),
                                 k_outlier_prob=0.01, name=name)
    if name == "fp8":
        s = 4 if seed is None else seed
        B, L = (2, 1100) if small else (16, 4096)
        B = batch or B
        return make_paged_inputs(seed=s, seq_lens=[L] * B, q_lens=[1] * B, num_q_heads=64,
                                 num_kv_heads=8, head_dim=128, page_size=64, layout=HND,
                                 kv_dtype=E4M3, device=device, name=name,
                                 v_channel_mean=v_channel_mean)
    if name in ("mla1", "mla2"):
        s = 5 if seed is None else seed
        ql = 1 if name == "mla1" else 2
        B, L = (2, 700) if small else (512, 4096)
        B = batch or B
        return make_mla_inputs(seed=s, seq_lens=[L] * B, q_lens=[ql] * B, device=device,
                               name=name)
    if name == "mla_fp8":
        s = 6 if seed is None else seed
        B, L = (2, 700) if small else (128, 4096)
        B = batch or B
        return make_mla_inputs(seed=s, seq_lens=[L] * B, q_lens=[1] * B, device=device, name=name,
                               kv_dtype=E4M3)
    if name == "prefill":
        s = 7 if seed is None else seed
        B, ql, L = (2, 100, 300) if small else (4, 511, 2047)
        B = batch or B
        return make_paged_inputs(seed=s, seq_lens=[L] * B, q_lens=[ql] * B, num_q_heads=64,
                                 num_kv_heads=8, head_dim=128, page_size=32, layout=HND,
                                 device=device, name=name)
    raise KeyError(name)


WORKLOADS = ("tiny", "gqa8", "ragged", "fp8", "mla1", "mla2", "mla_fp8", "prefill")
