// Paged GQA decode attention for sm_103a.
//
// What it computes: the paged decode contract of the FlashInfer
// "flashinfer.cake_fmha" API page (trtllm_batch_decode_with_kv_cache):
// each request's query rows of one KV-head group read that request's K/V
// pages through the block table and form softmax(q K^T * scale) V, with the
// inclusive causal bound of PR #4557's review ("Exclusive causal bound drops
// the newest key") for multi-row (speculative) queries, and the E4M3 storage
// convention of PR #5956 ("Contract": K/V hold x / scale).
//
// Design (GB300-first, not the pages' 15-stage tcgen05 MLA design):
//  * persistent CTAs, one per SM, pull work items (unit, tile range) from an
//    atomic queue the host ordered longest first;
//  * warp 4 is the producer: per 64-token tile it translates tokens to pages
//    through the block table (prefetched one tile ahead, bounds-checked
//    against num_pages) and issues 4-D TMA tensor copies of the K and V rows
//    into a multi-stage shared-memory ring (128-byte swizzle, mbarrier
//    completion, L2 evict-first hint);
//  * warps 0-3 are consumers, each owning 16 tokens of a tile: Q K^T and P V
//    on mma.sync m16n8k16 (the <= 16 packed query rows of a GQA group fill
//    one M=16 tile), row max/sum with warp shuffles, online softmax in the
//    exp2 domain. The E4M3 variant loads 16-byte rows with ld.shared.v4,
//    transposes V bytes with prmt and converts pairs with
//    cvt.rn.f16x2.e4m3x2 (exact) for f16 MMAs; the token and channel order
//    inside the contraction is permuted consistently for P and V (and for Q
//    and K) so every shared-memory read is a conflict-free 16-byte load;
//  * epilogue: the four warps' partial states are merged in shared memory;
//    an unsplit unit writes bf16 output (+ LSE) directly, a split writes an
//    fp32 partial state, and the last split to arrive (atomic counter that
//    resets itself) merges all partial states by log-sum-exp (PR #5591
//    "last-arriver split merge").
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "device_common.cuh"
#include "kernels.h"
#include "paged_decode.h"
#include "ws_layout.h"

namespace pd {
namespace {

constexpr int kTile = 64;           // tokens per stage
constexpr int kD = 128;             // head dim
constexpr int kNCW = 4;             // consumer warps
constexpr int kThreads = (kNCW + 1) * 32;
constexpr int kRows = 16;           // packed query rows per unit (MMA M)
constexpr int kObufStride = 136;    // floats per row of the merge buffer (bank-conflict padding)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum : int { F_FIRST = 1, F_LAST = 2, F_BAD = 4, F_INVALID = 8, F_END = 16 };

struct StageInfo {
  int32_t item;
  int32_t tile;
  int32_t flags;
  int32_t pad;
};

template <bool FP8>
struct Cfg {
  static constexpr int kRowBytes = FP8 ? 128 : 256;          // one token's K (or V) row
  static constexpr int kHalfBytes = kTile * 128;             // one 128-byte-wide slab of a tile
  static constexpr int kKBytes = kTile * kRowBytes;
  static constexpr int kStageBytes = 2 * kKBytes;            // K + V
  static constexpr int kStages = FP8 ? 10 : 5;
  static constexpr int kQSlotBytes = kRows * kD * 2;         // bf16 query rows
  static constexpr int kOffQ = kStages * kStageBytes;
  static constexpr int kOffObuf = kOffQ + 2 * kQSlotBytes;
  static constexpr int kOffRed = kOffObuf + kNCW * kRows * kObufStride * 4;
  static constexpr int kOffInfo = kOffRed + 2 * kNCW * kRows * 4 + 64;
  static constexpr int kOffBars = kOffInfo + kStages * (int)sizeof(StageInfo);
  static constexpr int kSmemBytes = kOffBars + (2 * kStages + 4) * 8 + 1024;  // + alignment slack
};

__device__ __forceinline__ float warp_max4(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
  return v;
}

template <bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    gqa_decode_kernel(const __grid_constant__ CUtensorMap k_map,
                      const __grid_constant__ CUtensorMap v_map, const GqaParams p) {
  using C = Cfg<FP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* qbuf = smem + C::kOffQ;
  float* obuf = reinterpret_cast<float*>(smem + C::kOffObuf);
  float* red_m = reinterpret_cast<float*>(smem + C::kOffRed);
  float* red_l = red_m + kNCW * kRows;
  int* s_flag = reinterpret_cast<int*>(red_l + kNCW * kRows);
  StageInfo* sinfo = reinterpret_cast<StageInfo*>(smem + C::kOffInfo);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* empty = full + C::kStages;
  uint64_t* qfull = empty + C::kStages;
  uint64_t* qempty = qfull + 2;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  WsHeader* hdr = p.hdr;

  if (threadIdx.x == 0) {
    int ok = (hdr->magic == kWsMagic && hdr->plan_id == p.plan_id) ? 1 : 0;
    if (!ok) set_error(hdr, PD_DEV_PLAN_MISMATCH, -1);
    s_flag[1] = ok;
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kNCW);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&qfull[s], 1);
      mbar_init(&qempty[s], kNCW);
    }
    fence_barrier_init();
    fence_proxy_async();
  }
  __syncthreads();
  if (!s_flag[1]) return;  // this workspace holds another plan: touch nothing

  const int G = p.group;
  const int P = p.page_size;
  const int BR = p.box_rows;

  if (warp == kNCW) {
    // ============================== producer ==============================
    prefetch_tensormap(&k_map);
    prefetch_tensormap(&v_map);
    const uint64_t pol = l2_evict_first_policy();
    uint32_t stage = 0, phase = 0;
    int qslot = 0;
    uint32_t qphase = 0;
    uint32_t armed = 0, armed_par = 0;  // stages with a copy in flight, and its phase parity
    bool dead = false;
    uint32_t next = 0;
    if (lane == 0) next = atomicAdd(&hdr->queue_counter, 1u);
    next = __shfl_sync(0xffffffffu, next, 0);
    while (next < (uint32_t)p.num_items) {
      const uint32_t cur = next;
      if (lane == 0) next = atomicAdd(&hdr->queue_counter, 1u);
      next = __shfl_sync(0xffffffffu, next, 0);
      const ItemDesc it = p.items[cur];
      const UnitDesc u = p.units[it.unit];
      int err = 0;
      if (lane == 0) {
        if (__ldg(&p.seq_lens[u.b]) != u.kv_len) {
          err = PD_DEV_SEQ_LEN_MISMATCH;
        } else if (p.q_indptr != nullptr && (__ldg(&p.q_indptr[u.b]) != u.q_start ||
                                             __ldg(&p.q_indptr[u.b + 1]) != u.q_start + u.q_len)) {
          err = PD_DEV_Q_INDPTR_MISMATCH;
        }
        if (err) set_error(hdr, err, u.b);
      }
      err = __shfl_sync(0xffffffffu, err, 0);

      // ---- query rows of this unit -> Q slot
      if (!mbar_wait(&qempty[qslot], qphase ^ 1)) { dead = true; break; }
      if (lane == 0) {
        uint8_t* dst = qbuf + qslot * C::kQSlotBytes;
        if (err) {
          mbar_arrive(&qfull[qslot]);
        } else {
          mbar_arrive_expect_tx(&qfull[qslot], (uint32_t)u.nrows * kD * 2);
          int r = 0;
          while (r < u.nrows) {
            const int pr = u.row0 + r;
            const int i = pr / G, hh = pr - (pr / G) * G;
            const int cnt = min(G - hh, u.nrows - r);
            const __nv_bfloat16* src = p.q + ((size_t)(u.q_start + i) * p.num_q_heads + (size_t)u.g * G + hh) * kD;
            bulk_load(dst + r * kD * 2, src, (uint32_t)cnt * kD * 2, &qfull[qslot]);
            r += cnt;
          }
        }
      }
      qslot ^= 1;
      if (qslot == 0) qphase ^= 1;

      if (err) {
        if (!mbar_wait(&empty[stage], phase ^ 1)) { dead = true; break; }
        if (lane == 0) {
          sinfo[stage] = StageInfo{(int32_t)cur, it.tile_begin, F_FIRST | F_LAST | F_INVALID, 0};
          mbar_arrive(&full[stage]);
        }
        if (++stage == (uint32_t)C::kStages) { stage = 0; phase ^= 1; }
        continue;
      }

      // ---- K/V tiles
      const int L = u.kv_len;
      const int32_t* trow = p.block_tables + (size_t)u.b * p.max_pages_per_seq;
      // page ids of boxes `lane` and `lane + 32` of a tile
      auto load_pages = [&](int t, int& pg0, int& pg1) {
        const int tok0 = t * kTile;
        const int nvalid = min(kTile, L - tok0);
        const int nbox = (nvalid + BR - 1) / BR;
        pg0 = lane < nbox ? __ldg(trow + (tok0 + lane * BR) / P) : 0;
        pg1 = lane + 32 < nbox ? __ldg(trow + (tok0 + (lane + 32) * BR) / P) : 0;
      };
      int pg0, pg1;
      load_pages(it.tile_begin, pg0, pg1);
      for (int t = it.tile_begin; t < it.tile_end; ++t) {
        int npg0 = 0, npg1 = 0;
        if (t + 1 < it.tile_end) load_pages(t + 1, npg0, npg1);
        const int tok0 = t * kTile;
        const int nvalid = min(kTile, L - tok0);
        const int nbox = (nvalid + BR - 1) / BR;
        const bool bad0 = lane < nbox && (pg0 < 0 || pg0 >= p.num_pages);
        const bool bad1 = lane + 32 < nbox && (pg1 < 0 || pg1 >= p.num_pages);
        const bool bad = __any_sync(0xffffffffu, bad0 || bad1);
        if (!mbar_wait(&empty[stage], phase ^ 1)) { dead = true; break; }
        int flags = (t == it.tile_begin ? F_FIRST : 0) | (t == it.tile_end - 1 ? F_LAST : 0);
        if (bad) {
          if (lane == 0) {
            set_error(hdr, PD_DEV_BAD_PAGE, u.b);
            sinfo[stage] = StageInfo{(int32_t)cur, t, flags | F_BAD, 0};
            mbar_arrive(&full[stage]);
          }
        } else {
          if (lane == 0) {
            sinfo[stage] = StageInfo{(int32_t)cur, t, flags, 0};
            mbar_arrive_expect_tx(&full[stage], (uint32_t)nbox * BR * 128 * (FP8 ? 2 : 4));
          }
          uint8_t* kdst = stages + stage * C::kStageBytes;
          uint8_t* vdst = kdst + C::kKBytes;
          for (int j = 0; j < nbox; ++j) {
            const int page = __shfl_sync(0xffffffffu, j < 32 ? pg0 : pg1, j & 31);
            if (lane == 0) {
              const int slot = (tok0 + j * BR) % P;
              const int c1 = p.layout == PD_LAYOUT_HND ? slot : u.g;
              const int c2 = p.layout == PD_LAYOUT_HND ? u.g : slot;
              const int row_off = j * BR * 128;
              if (FP8) {
                tma_load_4d(kdst + row_off, &k_map, 0, c1, c2, page, &full[stage], pol);
                tma_load_4d(vdst + row_off, &v_map, 0, c1, c2, page, &full[stage], pol);
              } else {
                tma_load_4d(kdst + row_off, &k_map, 0, c1, c2, page, &full[stage], pol);
                tma_load_4d(kdst + C::kHalfBytes + row_off, &k_map, 64, c1, c2, page, &full[stage], pol);
                tma_load_4d(vdst + row_off, &v_map, 0, c1, c2, page, &full[stage], pol);
                tma_load_4d(vdst + C::kHalfBytes + row_off, &v_map, 64, c1, c2, page, &full[stage], pol);
              }
            }
          }
        }
        armed |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        if (++stage == (uint32_t)C::kStages) { stage = 0; phase ^= 1; }
        pg0 = npg0;
        pg1 = npg1;
      }
      if (dead) break;
    }
    // ---- end marker for the consumers
    if (!dead && mbar_wait(&empty[stage], phase ^ 1)) {
      if (lane == 0) {
        sinfo[stage] = StageInfo{-1, 0, F_END, 0};
        mbar_arrive(&full[stage]);
      }
    } else {
      dead = true;
    }
    if (dead) {
      // drain: wait (bounded) for every copy this warp put in flight
      if (lane == 0) set_error(hdr, PD_DEV_TIMEOUT, -1);
      for (int s = 0; s < C::kStages; ++s)
        if (armed & (1u << s)) mbar_wait(&full[s], (armed_par >> s) & 1u, 100000000ull);
    }
  } else {
    // ============================== consumers ==============================
    const int g8 = lane >> 2;   // row group (rows g8 and g8 + 8)
    const int j4 = lane & 3;
    const int tokw = warp * 16; // this warp's tokens within a tile
    const uint32_t swz = p.swizzle ? 7u : 0u;
    const float kscale = (FP8 && p.k_scale) ? __ldg(p.k_scale) : 1.0f;
    const float vscale = (FP8 && p.v_scale) ? __ldg(p.v_scale) : 1.0f;
    const float scale2 = p.sm_scale * kscale * kLog2e;

    uint32_t stage = 0, phase = 0;
    int qslot = 0;
    uint32_t qphase = 0;
    float m[2], l[2], o[16][4];
    uint32_t qa[8][4];
    UnitDesc u{};
    int errored = 0;
    int pos_r[2] = {0, 0};  // last visible token of rows g8, g8 + 8
    int cur_unit = -1;

    while (true) {
      if (!mbar_wait(&full[stage], phase)) {
        if (lane == 0) set_error(hdr, PD_DEV_TIMEOUT, -1);
        break;
      }
      const StageInfo info = sinfo[stage];
      if (info.flags & F_END) break;
      if (info.flags & F_FIRST) {
        cur_unit = p.items[info.item].unit;
        u = p.units[cur_unit];
        errored = (info.flags & F_INVALID) ? 1 : 0;
        if (!mbar_wait(&qfull[qslot], qphase)) {
          if (lane == 0) set_error(hdr, PD_DEV_TIMEOUT, -1);
          break;
        }
        const uint32_t qb = smem_u32(qbuf + qslot * C::kQSlotBytes);
        if (!FP8) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const int row = (lane & 7) + (((lane >> 3) & 1) << 3);
            const int chunk = 2 * kk + (lane >> 4);
            ldsm_x4(qb + row * 256 + chunk * 16, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
          }
        } else {
          // f16 fragments, channels permuted: k16 step (h, s) covers channels
          // 16 (j4 + 4h) + 4 s + {0,1 | 2,3} for k slots {2j4, 2j4+1 | 2j4+8, 2j4+9}
          const uint8_t* qrow0 = qbuf + qslot * C::kQSlotBytes + g8 * 256;
          const uint8_t* qrow1 = qrow0 + 8 * 256;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              const int d = 16 * (j4 + 4 * h) + 4 * s;
              const uint2 x0 = *reinterpret_cast<const uint2*>(qrow0 + d * 2);
              const uint2 x1 = *reinterpret_cast<const uint2*>(qrow1 + d * 2);
              uint32_t* a = qa[h * 4 + s];
              a[0] = pack_f16_sat(bf16lo(x0.x), bf16hi(x0.x));
              a[1] = pack_f16_sat(bf16lo(x1.x), bf16hi(x1.x));
              a[2] = pack_f16_sat(bf16lo(x0.y), bf16hi(x0.y));
              a[3] = pack_f16_sat(bf16lo(x1.y), bf16hi(x1.y));
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&qempty[qslot]);
        qslot ^= 1;
        if (qslot == 0) qphase ^= 1;
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
#pragma unroll
        for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        pos_r[0] = u.kv_len - u.q_len + (u.row0 + g8) / G;
        pos_r[1] = u.kv_len - u.q_len + (u.row0 + g8 + 8) / G;
      }

      if (info.flags & (F_BAD | F_INVALID)) {
        errored = 1;
      } else {
        const int tok0 = info.tile * kTile;
        const uint32_t sb = smem_u32(stages + stage * C::kStageBytes);
        const uint32_t vb = sb + C::kKBytes;
        const int first_tok = tok0 + tokw;
        // zero V rows past the sequence end (tail slots / rows never loaded)
        if (first_tok + 15 >= u.kv_len) {
          uint8_t* vrows = stages + stage * C::kStageBytes + C::kKBytes;
          constexpr int kChunksPerRow = FP8 ? 8 : 16;
#pragma unroll
          for (int k = 0; k < kChunksPerRow / 2; ++k) {
            const int q = lane + 32 * k;
            const int r = q / kChunksPerRow;
            const int c = q % kChunksPerRow;
            if (first_tok + r >= u.kv_len) {
              const int tok = tokw + r;
              uint8_t* dst = FP8 ? vrows + tok * 128 + c * 16
                                 : vrows + (c >> 3) * C::kHalfBytes + tok * 128 + (c & 7) * 16;
              *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
            }
          }
          fence_proxy_async();  // these generic writes precede later TMA writes to the stage
          __syncwarp();
        }

        // ---- S = Q K^T (16 rows x 16 tokens)
        float s[2][4];
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
        if (!FP8) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const int half = kk >> 2;
            const int tok = tokw + (lane & 7) + ((lane >> 4) << 3);
            const uint32_t chunk = (uint32_t)((kk & 3) * 2 + ((lane >> 3) & 1));
            const uint32_t addr = sb + half * C::kHalfBytes + tok * 128 + ((chunk ^ (tok & swz)) << 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(addr, b0, b1, b2, b3);
            mma_bf16(s[0], qa[kk], b0, b1);
            mma_bf16(s[1], qa[kk], b2, b3);
          }
        } else {
#pragma unroll
          for (int nb = 0; nb < 2; ++nb) {
            const int tok = tokw + (g8 >> 1) + 4 * (2 * nb + (g8 & 1));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t chunk = (uint32_t)(j4 + 4 * h);
              uint32_t w[4];
              lds128(sb + tok * 128 + ((chunk ^ (tok & swz)) << 4), w[0], w[1], w[2], w[3]);
#pragma unroll
              for (int sidx = 0; sidx < 4; ++sidx) {
                const uint32_t b0 = e4m3x2_to_f16x2(w[sidx] & 0xffffu);
                const uint32_t b1 = e4m3x2_to_f16x2(w[sidx] >> 16);
                mma_f16(s[nb], qa[h * 4 + sidx], b0, b1);
              }
            }
          }
        }

        // ---- mask + online softmax (exp2 domain)
        const bool need_mask = first_tok + 15 > min(pos_r[0], pos_r[1]);
        float pr[2][4];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          float v[4];
#pragma unroll
          for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float x = s[nb][2 * rr + e] * scale2;
              if (need_mask) {
                const int tok = FP8 ? first_tok + j4 + 8 * nb + 4 * e : first_tok + 8 * nb + 2 * j4 + e;
                if (tok > pos_r[rr]) x = -INFINITY;
              }
              v[nb * 2 + e] = x;
            }
          }
          float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
          mx = warp_max4(mx);
          const float m_new = fmaxf(m[rr], mx);
          const float m_use = m_new == -INFINITY ? 0.f : m_new;
          const float alpha = fast_exp2(m[rr] - m_use);
          float sum = 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            pr[rr][k] = fast_exp2(v[k] - m_use);
            sum += pr[rr][k];
          }
          l[rr] = l[rr] * alpha + sum;
          m[rr] = m_new;
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            o[n][2 * rr] *= alpha;
            o[n][2 * rr + 1] *= alpha;
          }
        }

        // ---- O += P V
        uint32_t pa[4];
        if (!FP8) {
          pa[0] = pack_bf16(pr[0][0], pr[0][1]);
          pa[1] = pack_bf16(pr[1][0], pr[1][1]);
          pa[2] = pack_bf16(pr[0][2], pr[0][3]);
          pa[3] = pack_bf16(pr[1][2], pr[1][3]);
#pragma unroll
          for (int np = 0; np < 8; ++np) {
            const int tok = tokw + (lane & 7) + (((lane >> 3) & 1) << 3);
            const int c = 2 * np + (lane >> 4);
            const uint32_t addr = vb + (c >> 3) * C::kHalfBytes + tok * 128 + ((((uint32_t)c & 7u) ^ (tok & swz)) << 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(addr, b0, b1, b2, b3);
            mma_bf16(o[2 * np], pa, b0, b1);
            mma_bf16(o[2 * np + 1], pa, b2, b3);
          }
        } else {
          pa[0] = pack_f16(pr[0][0], pr[0][1]);
          pa[1] = pack_f16(pr[1][0], pr[1][1]);
          pa[2] = pack_f16(pr[0][2], pr[0][3]);
          pa[3] = pack_f16(pr[1][2], pr[1][3]);
          // rows j4, j4+4, j4+8, j4+12 of this warp's tokens; 16 channels
          // 16 cv .. 16 cv + 15 with cv = ((g8 & 1) << 2) | (g8 >> 1)
          const uint32_t cv = (uint32_t)(((g8 & 1) << 2) | (g8 >> 1));
          uint32_t w[4][4];
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            const int tok = tokw + j4 + 4 * rr;
            lds128(vb + tok * 128 + ((cv ^ (tok & swz)) << 4), w[rr][0], w[rr][1], w[rr][2], w[rr][3]);
          }
#pragma unroll
          for (int qd = 0; qd < 4; ++qd) {
            const uint32_t t0 = prmt(w[0][qd], w[1][qd], 0x5140);
            const uint32_t t1 = prmt(w[0][qd], w[1][qd], 0x7362);
            const uint32_t t2 = prmt(w[2][qd], w[3][qd], 0x5140);
            const uint32_t t3 = prmt(w[2][qd], w[3][qd], 0x7362);
            uint32_t col[4];
            col[0] = prmt(t0, t2, 0x5410);
            col[1] = prmt(t0, t2, 0x7632);
            col[2] = prmt(t1, t3, 0x5410);
            col[3] = prmt(t1, t3, 0x7632);
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
              const uint32_t b0 = e4m3x2_to_f16x2(col[bb] & 0xffffu);
              const uint32_t b1 = e4m3x2_to_f16x2(col[bb] >> 16);
              mma_f16(o[4 * qd + bb], pa, b0, b1);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == (uint32_t)C::kStages) { stage = 0; phase ^= 1; }

      if (!(info.flags & F_LAST)) continue;

      // ============================ epilogue ============================
      const ItemDesc it = p.items[info.item];
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], 1);
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], 2);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], 1);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], 2);
      if (j4 == 0) {
        red_m[warp * kRows + g8] = m[0];
        red_m[warp * kRows + g8 + 8] = m[1];
        red_l[warp * kRows + g8] = l[0];
        red_l[warp * kRows + g8 + 8] = l[1];
      }
      named_barrier(1, kNCW * 32);
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int row = g8 + 8 * rr;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kNCW; ++w) M = fmaxf(M, red_m[w * kRows + row]);
        const float sc = (m[rr] == -INFINITY) ? 0.f : fast_exp2(m[rr] - M);
        float* orow = obuf + (warp * kRows + row) * kObufStride;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          if (!FP8) {
            *reinterpret_cast<float2*>(orow + 8 * n + 2 * j4) = make_float2(o[n][2 * rr] * sc, o[n][2 * rr + 1] * sc);
          } else {
            orow[16 * j4 + n] = o[n][2 * rr] * sc;
            orow[16 * (j4 + 4) + n] = o[n][2 * rr + 1] * sc;
          }
        }
      }
      named_barrier(1, kNCW * 32);

      const int t = threadIdx.x;         // 0..127
      const int row = t >> 3;            // 0..15
      const int c0 = (t & 7) * 16;       // 16 channels per thread
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kNCW; ++w) M = fmaxf(M, red_m[w * kRows + row]);
      float Ls = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kNCW; ++w) {
          const float mw = red_m[w * kRows + row];
          if (mw != -INFINITY) Ls += red_l[w * kRows + row] * fast_exp2(mw - M);
        }
      }
      float acc[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[k] = 0.f;
#pragma unroll
      for (int w = 0; w < kNCW; ++w) {
        const float* src = obuf + (w * kRows + row) * kObufStride + c0;
#pragma unroll
        for (int k = 0; k < 16; k += 4) {
          const float4 x = *reinterpret_cast<const float4*>(src + k);
          acc[k] += x.x;
          acc[k + 1] += x.y;
          acc[k + 2] += x.z;
          acc[k + 3] += x.w;
        }
      }
      const float inv = Ls > 0.f ? vscale / Ls : 0.f;
      const bool valid_row = row < u.nrows;
      const int pr_ = u.row0 + row;
      const int qi = pr_ / G;
      const int head = u.g * G + (pr_ - qi * G);
      const size_t out_row = (size_t)(u.q_start + qi) * p.num_q_heads + head;

      if (u.n_splits == 1) {
        if (valid_row) {
          uint32_t packed[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            packed[k] = errored ? 0u : pack_bf16(acc[2 * k] * inv, acc[2 * k + 1] * inv);
          uint4* dst = reinterpret_cast<uint4*>(p.out + out_row * kD + c0);
          dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
          dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
          if (p.lse != nullptr && (t & 7) == 0)
            p.lse[out_row] = errored ? NAN : (Ls > 0.f ? (M + __log2f(Ls)) * kLn2 : -INFINITY);
        }
        named_barrier(1, kNCW * 32);  // obuf / red reuse by the next item
      } else {
        const size_t prow = (size_t)u.partial_base + (size_t)it.split * u.nrows + row;
        if (valid_row) {
          float* dst = p.po + prow * kD + c0;
#pragma unroll
          for (int k = 0; k < 16; k += 4)
            *reinterpret_cast<float4*>(dst + k) = make_float4(acc[k] * inv, acc[k + 1] * inv, acc[k + 2] * inv, acc[k + 3] * inv);
          if ((t & 7) == 0) p.plse[prow] = errored ? NAN : (Ls > 0.f ? M + __log2f(Ls) : -INFINITY);
        }
        if (p.fused_merge) {
          __threadfence();
          named_barrier(1, kNCW * 32);
          if (t == 0) {
            const uint32_t old = atomicAdd(&p.counters[cur_unit], 1u);
            const int last = old == (uint32_t)(u.n_splits - 1);
            if (last) p.counters[cur_unit] = 0u;
            s_flag[0] = last;
          }
          named_barrier(1, kNCW * 32);
          if (s_flag[0]) {
            __threadfence();
            if (valid_row) {
              const size_t base = (size_t)u.partial_base + row;
              float Mx = -INFINITY;
              bool bad = false;
              for (int s = 0; s < u.n_splits; ++s) {
                const float x = ld_cg(p.plse + base + (size_t)s * u.nrows);
                bad |= isnan(x);
                Mx = fmaxf(Mx, x);
              }
              float W = 0.f;
              float mo[16];
#pragma unroll
              for (int k = 0; k < 16; ++k) mo[k] = 0.f;
              if (!bad && Mx != -INFINITY) {
                for (int s = 0; s < u.n_splits; ++s) {
                  const size_t r = base + (size_t)s * u.nrows;
                  const float x = ld_cg(p.plse + r);
                  if (x == -INFINITY) continue;
                  const float w = fast_exp2(x - Mx);
                  W += w;
                  const float* src = p.po + r * kD + c0;
#pragma unroll
                  for (int k = 0; k < 16; k += 4) {
                    const float4 v = ld_cg4(src + k);
                    mo[k] += w * v.x;
                    mo[k + 1] += w * v.y;
                    mo[k + 2] += w * v.z;
                    mo[k + 3] += w * v.w;
                  }
                }
              }
              const float winv = W > 0.f ? 1.f / W : 0.f;
              uint32_t packed[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) packed[k] = bad ? 0u : pack_bf16(mo[2 * k] * winv, mo[2 * k + 1] * winv);
              uint4* dst = reinterpret_cast<uint4*>(p.out + out_row * kD + c0);
              dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
              dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
              if (p.lse != nullptr && (t & 7) == 0)
                p.lse[out_row] = bad ? NAN : (W > 0.f ? (Mx + __log2f(W)) * kLn2 : -INFINITY);
            }
          }
        }
        named_barrier(1, kNCW * 32);
      }
    }
  }

  // ---- leave the queue; the last CTA out resets it for the next launch
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&hdr->done_counter, 1u) == gridDim.x - 1) {
      hdr->queue_counter = 0u;
      hdr->done_counter = 0u;
      __threadfence();
    }
  }
}

}  // namespace

template <bool FP8>
static cudaError_t launch_impl(const CUtensorMap& kmap, const CUtensorMap& vmap, const GqaParams& p,
                               int grid, cudaStream_t stream) {
  using C = Cfg<FP8>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(gqa_decode_kernel<FP8>), C::kSmemBytes);
  if (e != cudaSuccess) return e;
  gqa_decode_kernel<FP8><<<grid, kThreads, C::kSmemBytes, stream>>>(kmap, vmap, p);
  return cudaGetLastError();
}

cudaError_t launch_gqa_decode(const CUtensorMap& kmap, const CUtensorMap& vmap, const GqaParams& p,
                              bool fp8, int grid, cudaStream_t stream) {
  return fp8 ? launch_impl<true>(kmap, vmap, p, grid, stream) : launch_impl<false>(kmap, vmap, p, grid, stream);
}

int gqa_smem_bytes(bool fp8) { return fp8 ? Cfg<true>::kSmemBytes : Cfg<false>::kSmemBytes; }

}  // namespace pd
