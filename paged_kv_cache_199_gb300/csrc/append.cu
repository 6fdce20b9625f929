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
// group of loads in flight before the stores (the first group issued before
// the token's metadata look-ups, which it does not depend on); warps past the tokens zero the
// tail slots of one request. A warp finds its request with a ballot search
// of q_indptr (32 entries per round). Invalid metadata skips the affected rows and
// records the first error in the caller's error word; nothing is read or
// written outside the pools and the new rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <type_traits>

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

// Packed binary32 pairs (.f32x2 arithmetic, element 0 in the low word): each
// element gets exactly the IEEE operation of its scalar form.
__device__ __forceinline__ uint64_t f2(uint32_t lo_bits, uint32_t hi_bits) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo_bits), "r"(hi_bits));
  return r;
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint32_t e4m3x2_packed(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return e4m3x2(lo, hi);
}

// Scale constants of one E4M3 tensor: s, RN(1/s), and the bf16 magnitude
// (bits without the sign) below which x / s is finite with room to spare and
// the packed path applies; 0 turns the packed path off (s not positive, or
// 1/s not finite).
struct QuantConsts {
  float s, ys;
  uint32_t fast_limit;
};
__device__ __forceinline__ QuantConsts quant_consts(float s) {
  QuantConsts c{s, __frcp_rn(s), 0u};
  if (s > 0.f && isfinite(s) && isfinite(c.ys)) {
    // |x| < 2^127 s keeps x RN(1/s), the residual and the corrected quotient
    // finite; truncating the bound's bits rounds it toward zero
    const float lim = 1.7014118e38f * s;
    c.fast_limit = isfinite(lim) ? min(__float_as_uint(lim) >> 16, 0x7f80u) : 0x7f80u;
  }
  return c;
}

// Largest bf16 magnitude (bits without the sign) of N chunks of 4 (uint2) or
// 8 (uint4) values.
__device__ __forceinline__ uint32_t mag2(uint32_t w) { return w & 0x7fff7fffu; }
template <int N>
__device__ __forceinline__ uint32_t max_mag(const uint2 (&w)[N]) {
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < N; ++j) m = __vmaxu2(m, __vmaxu2(mag2(w[j].x), mag2(w[j].y)));
  return max(m & 0xffffu, m >> 16);
}
template <int N>
__device__ __forceinline__ uint32_t max_mag(const uint4 (&w)[N]) {
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < N; ++j)
    m = __vmaxu2(m, __vmaxu2(__vmaxu2(mag2(w[j].x), mag2(w[j].y)), __vmaxu2(mag2(w[j].z), mag2(w[j].w))));
  return max(m & 0xffffu, m >> 16);
}

// Four bf16 values (two words, first value in the low half) divided by s and
// encoded as E4M3 (first value in the low byte), scalar path: div_rn per
// value. Any input.
__device__ __forceinline__ uint32_t quant4_scalar(uint2 w, const QuantConsts& c) {
  const float x0 = div_rn(bf16_bits_to_float(w.x & 0xffffu), c.s, c.ys);
  const float x1 = div_rn(bf16_bits_to_float(w.x >> 16), c.s, c.ys);
  const float x2 = div_rn(bf16_bits_to_float(w.y & 0xffffu), c.s, c.ys);
  const float x3 = div_rn(bf16_bits_to_float(w.y >> 16), c.s, c.ys);
  return e4m3x2(x0, x1) | (e4m3x2(x2, x3) << 16);
}

// The same for magnitudes below c.fast_limit (finite quotients, s > 0), two
// values per packed operation, on the negated quotient: n = RN(x (-ys)) = -q,
// r = RN(x + n s) = x - q s exactly as div_rn's residual, then
// RN(n + r (-ys)) = -RN(q + r ys). Negation commutes with RN, and with r = 0
// the sum keeps n as it is (for n = -0, r = +0: -0 + -0 = -0; for n = +0,
// r = +0: +0 + -0 = +0), so the codes equal div_rn's, sign of zero included,
// once their sign bits are flipped back.
__device__ __forceinline__ uint32_t quant4_fast(uint2 w, uint64_t s2, uint64_t nys2) {
  uint32_t out = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t word = h == 0 ? w.x : w.y;
    const uint64_t x = f2(word << 16, word & 0xffff0000u);
    const uint64_t n = f2mul(x, nys2);
    const uint64_t r = f2fma(n, s2, x);
    out |= e4m3x2_packed(f2fma(r, nys2, n)) << (16 * h);
  }
  return out ^ 0x80808080u;
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

constexpr int kWarpsPerBlock = 8;

// Input chunks of CE bf16 values: 8-byte (CE = 4) or, when both inputs are
// 16-byte aligned, 16-byte (CE = 8) loads; a lane holds 64 bytes of each
// tensor in flight either way.
template <int CE>
struct Chunk {
  using T = typename std::conditional<CE == 4, uint2, uint4>::type;
  static constexpr int kPerLane = 32 / CE;   // chunks a lane holds per tensor
  __device__ static T zero() {
    if constexpr (CE == 4)
      return make_uint2(0u, 0u);
    else
      return make_uint4(0u, 0u, 0u, 0u);
  }
};

// One group of a token's input chunks (every kv head, K and V), by lane:
// chunk c0 + 32 j of the token's H x D/CE chunks.
template <int CE>
struct RowGroup {
  typename Chunk<CE>::T k[Chunk<CE>::kPerLane], v[Chunk<CE>::kPerLane];
};

template <int CE>
__device__ __forceinline__ void load_group(const AppendParams& p, int64_t r, int c0, int chunks, RowGroup<CE>& d) {
  using T = typename Chunk<CE>::T;
  const int64_t row = r * p.num_kv_heads * p.head_dim;
  const T* kin = reinterpret_cast<const T*>(p.k_new + row);
  const T* vin = p.v_new ? reinterpret_cast<const T*>(p.v_new + row) : nullptr;
#pragma unroll
  for (int j = 0; j < Chunk<CE>::kPerLane; ++j) {
    const int c = c0 + 32 * j;
    d.k[j] = c < chunks ? __ldg(kin + c) : Chunk<CE>::zero();
    d.v[j] = (vin && c < chunks) ? __ldg(vin + c) : Chunk<CE>::zero();
  }
}

// E4M3 codes of one chunk: four codes in a word (CE = 4) or eight in two.
__device__ __forceinline__ uint32_t quant_chunk(uint2 w, bool fast, uint64_t s2, uint64_t nys2, const QuantConsts& q) {
  return fast ? quant4_fast(w, s2, nys2) : quant4_scalar(w, q);
}
__device__ __forceinline__ uint2 quant_chunk(uint4 w, bool fast, uint64_t s2, uint64_t nys2, const QuantConsts& q) {
  return make_uint2(quant_chunk(make_uint2(w.x, w.y), fast, s2, nys2, q),
                    quant_chunk(make_uint2(w.z, w.w), fast, s2, nys2, q));
}

// Where a token's rows go: element offsets of its (page, slot) row of kv
// head 0 in each pool, and the step between kv heads.
struct RowDst {
  int64_t kbase, vbase, hstep;
};

// Stores one group of chunks (group c0) of a token.
template <int CE>
__device__ __forceinline__ void store_group(const AppendParams& p, const RowDst& dst, const RowGroup<CE>& w, int c0,
                                            int chunks, int row_chunks, const QuantConsts& kq,
                                            const QuantConsts& vq) {
  using T = typename Chunk<CE>::T;
  using Q = typename std::conditional<CE == 4, uint32_t, uint2>::type;   // E4M3 codes of one chunk
  // E4M3: one magnitude test per tensor and group picks the packed path
  bool kfast = false, vfast = false;
  uint64_t ks2 = 0, knys2 = 0, vs2 = 0, vnys2 = 0;
  if (p.fp8) {
    kfast = max_mag(w.k) < kq.fast_limit;
    vfast = max_mag(w.v) < vq.fast_limit;
    ks2 = f2(__float_as_uint(kq.s), __float_as_uint(kq.s));
    knys2 = f2(__float_as_uint(-kq.ys), __float_as_uint(-kq.ys));
    vs2 = f2(__float_as_uint(vq.s), __float_as_uint(vq.s));
    vnys2 = f2(__float_as_uint(-vq.ys), __float_as_uint(-vq.ys));
  }
  // chunk c0 + 32 j is channel CE cc of head g: when a head's row has a
  // divisor of 32 chunks (128-channel heads) each step moves 32 / row_chunks
  // heads; otherwise one division per group, then steps of 32 chunks
  int g = c0 / row_chunks, cc = c0 - g * row_chunks;
  const bool whole = 32 % row_chunks == 0;
#pragma unroll
  for (int j = 0; j < Chunk<CE>::kPerLane; ++j) {
    const int c = c0 + 32 * j;
    if (c >= chunks) break;
    const int64_t off = (int64_t)g * dst.hstep + CE * cc;
    if (!p.fp8) {
      *reinterpret_cast<T*>(p.k_pool + (dst.kbase + off) * 2) = w.k[j];
      if (p.v_new) *reinterpret_cast<T*>(p.v_pool + (dst.vbase + off) * 2) = w.v[j];
    } else {
      *reinterpret_cast<Q*>(p.k_pool + dst.kbase + off) = quant_chunk(w.k[j], kfast, ks2, knys2, kq);
      if (p.v_new) *reinterpret_cast<Q*>(p.v_pool + dst.vbase + off) = quant_chunk(w.v[j], vfast, vs2, vnys2, vq);
    }
    if (whole) {
      g += 32 / row_chunks;
    } else {
      cc += 32;
      while (cc >= row_chunks) {
        cc -= row_chunks;
        ++g;
      }
    }
  }
}

// Persistent warps. Each appends a contiguous run of new tokens: the
// request's metadata and the current page id are looked up once and reused
// by the run's following tokens, and the next token's first group of input
// chunks is in flight while the current one is encoded and stored. Then the
// warps share out the requests' tail zeroing.
template <int CE>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) paged_append_kernel(const AppendParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t nw = (int64_t)gridDim.x * kWarpsPerBlock;
  const int64_t gw = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int H = p.num_kv_heads, D = p.head_dim, P = p.page_size;
  const int row_chunks = D / CE;                // CE-element chunks of one head's row
  const int chunks = H * row_chunks;            // of one token (all heads)
  const int64_t hstep = p.layout == PD_LAYOUT_NHD ? (int64_t)D : (int64_t)P * D;
  const int64_t slot_step = p.layout == PD_LAYOUT_NHD ? (int64_t)H * D : (int64_t)D;

  // ---- new tokens [r_begin, r_end) of this warp, every kv head, K and V
  const int64_t per = (p.row_tasks + nw - 1) / nw;
  const int64_t r_begin = min(p.row_tasks, gw * per), r_end = min(p.row_tasks, r_begin + per);
  if (r_begin < r_end) {
    const QuantConsts kq = quant_consts(p.fp8 ? __ldg(p.k_scale) : 1.f);
    const QuantConsts vq = quant_consts((p.fp8 && p.v_new != nullptr) ? __ldg(p.v_scale) : 1.f);
    RowGroup<CE> cur, nxt;
    load_group(p, r_begin, lane, chunks, cur);
    int b = -1, q0 = 0, n = 0, L = 0;            // request of the latest token
    int64_t pi_cached = -1;                      // its page index, and the page id
    int page = 0;
    for (int64_t r = r_begin; r < r_end; ++r) {
      if (r + 1 < r_end) load_group(p, r + 1, lane, chunks, nxt);
      if (b < 0 || r < q0 || r >= (int64_t)q0 + n) {
        b = find_request(p.q_indptr, p.batch, r, lane);
        q0 = __ldg(&p.q_indptr[b]);
        n = __ldg(&p.q_indptr[b + 1]) - q0;
        L = __ldg(&p.seq_lens[b]);
        pi_cached = -1;
      }
      const int64_t i = r - q0;
      if (i < 0 || i >= n) {
        if (lane == 0) flag(p, PD_DEV_Q_INDPTR_MISMATCH, b);
      } else if (n > L) {
        if (lane == 0 && i == 0) flag(p, PD_DEV_SEQ_LEN_MISMATCH, b);
      } else {
        const int64_t pos = (int64_t)L - n + i;
        const int64_t pi = pos / P;
        if (pi != pi_cached) {
          page = __ldg(&p.block_tables[(int64_t)b * p.max_pages_per_seq + pi]);
          pi_cached = pi;
        }
        if (page < 0 || page >= p.num_pages) {
          if (lane == 0) flag(p, PD_DEV_BAD_PAGE, b);
        } else {
          const int64_t sterm = (pos - pi * P) * slot_step;
          const RowDst dst{(int64_t)page * p.k_page_stride + sterm, (int64_t)page * p.v_page_stride + sterm, hstep};
          store_group(p, dst, cur, lane, chunks, row_chunks, kq, vq);
          for (int c0 = lane + 32 * Chunk<CE>::kPerLane; c0 < chunks; c0 += 32 * Chunk<CE>::kPerLane) {
            RowGroup<CE> w;   // wide rows: later groups are read here
            load_group(p, r, c0, chunks, w);
            store_group(p, dst, w, c0, chunks, row_chunks, kq, vq);
          }
        }
      }
      cur = nxt;
    }
  }

  // ---- the last page's slots past the sequence end, one request per warp
  const int64_t tails = p.tasks - p.row_tasks;
  for (int64_t t = gw; t < tails; t += nw) {
    const int b = (int)t;
    const int L = __ldg(&p.seq_lens[b]);
    const int n = __ldg(&p.q_indptr[b + 1]) - __ldg(&p.q_indptr[b]);
    if (n > L || L <= 0 || L % P == 0) continue;   // a bad length is reported by the row tasks
    const int page = __ldg(&p.block_tables[(int64_t)b * p.max_pages_per_seq + (L - 1) / P]);
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) flag(p, PD_DEV_BAD_PAGE, b);
      continue;
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

// Blocks of one launch: every task's warp, up to the blocks that fit on the
// device at once (the warps then loop). Found once per device (for the first
// 64 device ordinals; others query at every launch). 0 when a query fails.
int append_grid_cap() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const bool cached = dev >= 0 && dev < 64;
  if (cached) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, paged_append_kernel<8>, kWarpsPerBlock * 32, 0) !=
          cudaSuccess)
    return 0;
  const int c = std::max(1, sms * std::max(1, per_sm));
  if (cached) cache[dev].store(c, std::memory_order_relaxed);
  return c;
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
  const int cap = pd::append_grid_cap();
  if (cap <= 0) return pd::cuda_fail(cudaGetLastError(), "paged KV append: device query");
  const int64_t blocks = std::min<int64_t>((p.tasks + pd::kWarpsPerBlock - 1) / pd::kWarpsPerBlock, cap);
  // 16-byte input chunks when both inputs allow them (rows are multiples of
  // 16 bytes: head_dim is a multiple of 8)
  const bool wide = !misaligned(k_new, 16) && !misaligned(v_new, 16);
  if (wide)
    pd::paged_append_kernel<8><<<(unsigned)blocks, pd::kWarpsPerBlock * 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  else
    pd::paged_append_kernel<4><<<(unsigned)blocks, pd::kWarpsPerBlock * 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PD_OK : pd::cuda_fail(e, "paged KV append launch");
}
