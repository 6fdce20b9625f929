// Paged KV append: the new tokens' K and V rows written into the paged
// pools, the step just before decode.
//
// What it computes: PR #5952 ("feat(cake_fused_qk_rope_append): fused BF16 QK
// RMSNorm + NeoX RoPE + paged KV append"), commit #5956 "Contract": seq_lens
// is the total length after the append, so token i of a request with n new
// tokens sits at position seq_lens[b] - n + i, in page block_tables[b][pos / P]
// and slot pos % P; E4M3 pools store x / k_scale and x / v_scale rounded to
// nearest even and saturated to the largest finite value; the last page's
// slots past the sequence end are zeroed. (The pages' fused RMSNorm and RoPE
// steps are not part of this call: it appends the rows it is given.)
//
// Design: one warp per new token (every kv head, K and V), four channels per
// lane and chunk (8-byte loads, 8-byte BF16 or 4-byte E4M3 stores), with a
// group of loads in flight before the stores; warps past the tokens zero the
// tail slots of one request. A warp finds its request with a ballot search
// of q_indptr (32 entries per round). Invalid metadata skips the affected rows and
// records the first error in the caller's error word; nothing is read or
// written outside the pools and the new rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "paged_decode.h"

namespace pd {
namespace {

struct AppendParams {
  const uint16_t* k_new;      // bf16 bits [total_new][Hkv][D]
  const uint16_t* v_new;      // or nullptr (a K-only pool)
  const int32_t* q_indptr;
  const int32_t* seq_lens;
  const int32_t* block_tables;
  const float* k_scale;       // E4M3 pools
  const float* v_scale;
  uint8_t* k_pool;
  uint8_t* v_pool;
  int64_t k_page_stride;      // elements
  int64_t v_page_stride;
  int32_t* error;             // [code, info] or nullptr
  int64_t row_tasks;          // total_new (a warp per new token)
  int64_t tasks;              // + batch tail tasks when zeroing tails
  int32_t batch, num_kv_heads, head_dim, page_size, num_pages, max_pages_per_seq, layout, fp8;
};

__device__ __forceinline__ void flag(const AppendParams& p, int code, int info) {
  if (p.error != nullptr && atomicCAS(&p.error[0], 0, code) == 0) atomicExch(&p.error[1], info);
}

// Element offset of (page, slot, kv head, channel 0).
__device__ __forceinline__ int64_t row_off(const AppendParams& p, int64_t page, int slot, int g, int64_t stride) {
  return p.layout == PD_LAYOUT_NHD ? page * stride + ((int64_t)slot * p.num_kv_heads + g) * p.head_dim
                                   : page * stride + ((int64_t)g * p.page_size + slot) * p.head_dim;
}

// Two binary32 values to two E4M3 codes, round to nearest even, saturating
// (the first value in the low byte).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits) { return __uint_as_float(bits << 16); }

// x / s rounded to nearest, from the correctly rounded reciprocal ys = RN(1/s)
// and one FMA residual step (Markstein's correction: with ys within half an
// ulp of 1/s and q within one ulp of x / s, RN(q + (x - q s) ys) = RN(x / s);
// P. Markstein, IBM J. Res. Dev. 34(1), 1990). r is exact; r == 0 means q is
// already exact (this also keeps the sign of zero); a non-finite q (overflow,
// infinite x) saturates in the E4M3 conversion either way. Quotients that
// underflow binary32 encode to (signed) zero in E4M3 whatever their last bit.
__device__ __forceinline__ float div_rn(float x, float s, float ys) {
  const float q = x * ys;
  const float r = fmaf(-q, s, x);
  return (r == 0.f || !isfinite(q)) ? q : fmaf(r, ys, q);
}

// Last request b with q_indptr[b] <= r, by the whole warp: each round reads
// 32 evenly spaced entries at once and keeps the interval the ballot picks
// (one round for up to 32 requests, two up to 1024).
__device__ __forceinline__ int find_request(const int32_t* q_indptr, int batch, int64_t r, int lane) {
  int lo = 0, hi = batch;   // q_indptr[lo] <= r, and r < q_indptr[hi] when hi < batch
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) / 32;
    const int idx = lo + lane * step;
    const bool le = idx < hi && __ldg(&q_indptr[idx]) <= r;
    const unsigned m = __ballot_sync(0xffffffffu, le);
    const int k = 31 - __clz(m);          // m has bit 0 set: q_indptr[lo] <= r
    lo += k * step;
    hi = min(hi, lo + step);
  }
  return lo;
}

constexpr int kChunksPerLane = 8;   // 8-byte chunks a lane holds in flight per tensor

__global__ void __launch_bounds__(256) paged_append_kernel(const AppendParams p) {
  const int64_t task = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (task >= p.tasks) return;
  const int H = p.num_kv_heads, D = p.head_dim, P = p.page_size;
  const int row_chunks = D / 4;                 // 4-element chunks of one head's row
  const int chunks = H * row_chunks;            // of one token (all heads)
  if (task < p.row_tasks) {
    // ---- one new token, all kv heads, K and V
    const int64_t r = task;
    const int b = find_request(p.q_indptr, p.batch, r, lane);
    const int q0 = __ldg(&p.q_indptr[b]);
    const int n = __ldg(&p.q_indptr[b + 1]) - q0;
    const int L = __ldg(&p.seq_lens[b]);
    const int64_t i = r - q0;
    if (i < 0 || i >= n) {
      if (lane == 0) flag(p, PD_DEV_Q_INDPTR_MISMATCH, b);
      return;
    }
    if (n > L) {
      if (lane == 0 && i == 0) flag(p, PD_DEV_SEQ_LEN_MISMATCH, b);
      return;
    }
    const int64_t pos = (int64_t)L - n + i;
    const int page = __ldg(&p.block_tables[(int64_t)b * p.max_pages_per_seq + pos / P]);
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) flag(p, PD_DEV_BAD_PAGE, b);
      return;
    }
    const int slot = (int)(pos % P);
    const float ks = p.fp8 ? __ldg(p.k_scale) : 1.f;
    const float vs = (p.fp8 && p.v_new != nullptr) ? __ldg(p.v_scale) : 1.f;
    const float kr = __frcp_rn(ks), vr = __frcp_rn(vs);
    const uint2* kin = reinterpret_cast<const uint2*>(p.k_new + r * H * D);
    const uint2* vin = p.v_new ? reinterpret_cast<const uint2*>(p.v_new + r * H * D) : nullptr;
    for (int c0 = lane; c0 < chunks; c0 += 32 * kChunksPerLane) {
      // every load of the group in flight before the first store
      uint2 kw[kChunksPerLane], vw[kChunksPerLane];
#pragma unroll
      for (int j = 0; j < kChunksPerLane; ++j) {
        const int c = c0 + 32 * j;
        kw[j] = c < chunks ? __ldg(kin + c) : make_uint2(0u, 0u);
        vw[j] = (vin && c < chunks) ? __ldg(vin + c) : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < kChunksPerLane; ++j) {
        const int c = c0 + 32 * j;
        if (c >= chunks) break;
        const int g = c / row_chunks, cc = c - g * row_chunks;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          uint8_t* pool = t == 0 ? p.k_pool : p.v_pool;
          if (t == 1 && vin == nullptr) continue;
          const uint2 w = t == 0 ? kw[j] : vw[j];
          const int64_t dst = row_off(p, page, slot, g, t == 0 ? p.k_page_stride : p.v_page_stride) + 4 * cc;
          if (!p.fp8) {
            *reinterpret_cast<uint2*>(pool + dst * 2) = w;
          } else {
            const float scale = t == 0 ? ks : vs, rs = t == 0 ? kr : vr;
            const float x0 = div_rn(bf16_bits_to_float(w.x & 0xffffu), scale, rs);
            const float x1 = div_rn(bf16_bits_to_float(w.x >> 16), scale, rs);
            const float x2 = div_rn(bf16_bits_to_float(w.y & 0xffffu), scale, rs);
            const float x3 = div_rn(bf16_bits_to_float(w.y >> 16), scale, rs);
            *reinterpret_cast<uint32_t*>(pool + dst) = e4m3x2(x0, x1) | (e4m3x2(x2, x3) << 16);
          }
        }
      }
    }
  } else {
    // ---- the last page's slots past the sequence end of one request
    const int b = (int)(task - p.row_tasks);
    const int L = __ldg(&p.seq_lens[b]);
    const int n = __ldg(&p.q_indptr[b + 1]) - __ldg(&p.q_indptr[b]);
    if (n > L || L <= 0 || L % P == 0) return;   // a bad length is reported by the row tasks
    const int page = __ldg(&p.block_tables[(int64_t)b * p.max_pages_per_seq + (L - 1) / P]);
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) flag(p, PD_DEV_BAD_PAGE, b);
      return;
    }
    const int elem = p.fp8 ? 1 : 2;
    const int words = D * elem / 4;             // 4-byte words of one row
    for (int slot = L % P; slot < P; ++slot)
      for (int g = 0; g < H; ++g)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          uint8_t* pool = k == 0 ? p.k_pool : p.v_pool;
          if (k == 1 && p.v_new == nullptr) continue;
          const int64_t dst = row_off(p, page, slot, g, k == 0 ? p.k_page_stride : p.v_page_stride) * elem;
          for (int c = lane; c < words; c += 32) *reinterpret_cast<uint32_t*>(pool + dst + 4 * c) = 0u;
        }
  }
}

}  // namespace
}  // namespace pd

extern "C" pd_status paged_kv_append(const pd_append_problem* prob, const void* k_new, const void* v_new,
                                     int32_t total_new, const int32_t* q_indptr, const int32_t* seq_lens,
                                     const int32_t* block_tables, const float* k_scale, const float* v_scale,
                                     void* k_pool, void* v_pool, int32_t zero_tail, int32_t* error_word,
                                     pd_stream_t stream) {
  if (!prob) return PD_ERR_INVALID_ARG;
  const pd_append_problem& q = *prob;
  if (q.batch < 0 || total_new < 0 || q.num_kv_heads < 1 || q.page_size < 1 || q.num_pages < 0 ||
      q.max_pages_per_seq < 0 || q.k_page_stride < 0 || q.v_page_stride < 0)
    return PD_ERR_INVALID_ARG;
  if (q.head_dim < 8 || q.head_dim > 1024 || q.head_dim % 8 != 0) return PD_ERR_INVALID_ARG;
  if (q.layout != PD_LAYOUT_NHD && q.layout != PD_LAYOUT_HND) return PD_ERR_INVALID_ARG;
  if (q.kv_dtype != PD_KV_BF16 && q.kv_dtype != PD_KV_FP8_E4M3) return PD_ERR_INVALID_ARG;
  const bool fp8 = q.kv_dtype == PD_KV_FP8_E4M3;
  const int64_t elem = fp8 ? 1 : 2;
  const int64_t compact = (int64_t)q.page_size * q.num_kv_heads * q.head_dim;
  const int64_t ks = q.k_page_stride ? q.k_page_stride : compact;
  const int64_t vs = q.v_page_stride ? q.v_page_stride : compact;
  if (ks < compact || vs < compact || (ks * elem) % 16 != 0 || (vs * elem) % 16 != 0) return PD_ERR_INVALID_ARG;
  if (q.batch == 0 || (total_new == 0 && !zero_tail)) return PD_OK;
  if (!q_indptr || !seq_lens || !block_tables || !k_pool || q.num_pages < 1 || q.max_pages_per_seq < 1)
    return PD_ERR_INVALID_ARG;
  if (total_new > 0 && !k_new) return PD_ERR_INVALID_ARG;
  if ((v_new == nullptr) != (v_pool == nullptr)) return PD_ERR_INVALID_ARG;
  if (fp8 && (!k_scale || (v_new && !v_scale))) return PD_ERR_INVALID_ARG;
  auto misaligned = [](const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0; };
  if (misaligned(k_new, 8) || misaligned(v_new, 8) || misaligned(k_pool, 16) || misaligned(v_pool, 16) ||
      misaligned(error_word, 4))
    return PD_ERR_INVALID_ARG;
  pd::AppendParams p{};
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.q_indptr = q_indptr;
  p.seq_lens = seq_lens;
  p.block_tables = block_tables;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.k_pool = static_cast<uint8_t*>(k_pool);
  p.v_pool = static_cast<uint8_t*>(v_pool);
  p.k_page_stride = ks;
  p.v_page_stride = vs;
  p.error = error_word;
  p.row_tasks = total_new;                              // one warp per new token
  p.tasks = p.row_tasks + (zero_tail ? q.batch : 0);    // and one per request's tail
  p.batch = q.batch;
  p.num_kv_heads = q.num_kv_heads;
  p.head_dim = q.head_dim;
  p.page_size = q.page_size;
  p.num_pages = q.num_pages;
  p.max_pages_per_seq = q.max_pages_per_seq;
  p.layout = q.layout;
  p.fp8 = fp8 ? 1 : 0;
  const int64_t blocks = (p.tasks + 7) / 8;
  if (blocks > 0x7fffffffLL) return PD_ERR_INVALID_ARG;
  pd::paged_append_kernel<<<(unsigned)blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PD_OK : pd::cuda_fail(e, "paged KV append launch");
}
