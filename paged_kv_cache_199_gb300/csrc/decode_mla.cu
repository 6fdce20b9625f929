// Paged MLA decode attention for sm_103a: every query head attends over one
// shared latent KV head.
//
// What it computes: PR #4557 ("feat(cake_mla): add generated Blackwell
// TRT-LLM MLA decode backend") calls trtllm_batch_decode_with_kv_cache_mla
// over a paged latent cache whose row is 512 latent + 64 rope channels
// (PR #5552, "Kimi-K3 FP8 latent MLA"): the key is the whole 576-channel row
// and the value its first 512 channels; query rows are packed (token, head)
// pairs; the causal bound is inclusive (PR #4557 review "Exclusive causal
// bound drops the newest key").
//
// Design (mma.sync, not the pages' tcgen05 15-stage pipeline):
//  * one persistent CTA per SM; a unit is 64 packed query rows of one
//    request, its keys are cut into 64-token tiles;
//  * scheduler warp 9 pops items (or walks the CTA's static range), checks
//    the device metadata, prefetches page ids and TMA-loads the unit's
//    64 x 576 query block (nine 128-byte swizzled slabs); it also counts
//    split arrivals and queues the unit merge on the last one;
//  * producer warp 8 TMA-loads each 64 x 576 key tile (nine swizzled slabs,
//    two stages of 72 KB); values are the first eight slabs of the same tile;
//  * eight consumer warps: warp w computes S = Q K^T for rows 16 (w & 3) ..
//    +16 and keys 32 (w >> 2) .. +32 (144 mma.sync per tile), the two warps
//    of a row block exchange their row maxima through shared memory, write P
//    (bf16, swizzled) to shared memory, and warp w then accumulates
//    O += P V for its 16 rows and latent channels 256 (w >> 2) .. +256 over
//    all 64 keys (128 mma.sync per tile); the two warps' row sums are
//    combined once per item.
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

constexpr int kTile = 64;            // tokens per stage
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kSlabs = kDqk / 64;    // 128-byte wide slabs of a 576-channel row
constexpr int kRows = 64;            // packed query rows per unit
constexpr int kNCW = 8;              // consumer warps
constexpr int kProducerWarp = kNCW;
constexpr int kSchedulerWarp = kNCW + 1;
// Three warpgroups: two of consumers, one holding the producer, the
// scheduler and two idle warps. Launched at 168 registers per thread
// (384 x 168 <= 64K); the consumer warpgroups raise their limit to 232 and
// the third lowers its to 40: 256 x 232 + 128 x 40 = 64512 <= 65536.
constexpr int kThreads = (kNCW + 4) * 32;
constexpr int kConsumerRegs = 232;
constexpr int kOtherRegs = 40;
constexpr int kStages = 2;
constexpr int kSlots = 2;
constexpr int kWin = 64;             // page ids prefetched per item
constexpr int kSlabBytes = kTile * 128;                 // 8 KB
constexpr int kStageBytes = kSlabs * kSlabBytes;        // 72 KB
constexpr int kQBytes = kSlabs * kRows * 128;           // 72 KB
constexpr int kPBytes = kRows * kTile * 2;              // 8 KB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum : int { F_FIRST = 1, F_LAST = 2, F_BAD = 4, F_INVALID = 8, F_END = 16, F_MERGE = 32, F_NOP = 64 };
enum : int { T_ITEM = 0, T_MERGE = 1, T_NOP = 2, T_END = 3 };

struct StageInfo {
  int32_t slot;
  int32_t tile;
  int32_t flags;
  int32_t pad;
};

struct SlotMeta {
  ItemDesc it;
  int32_t item;
  int32_t err;
  int32_t kind;
  int32_t win0;
  int32_t nwin;
  int32_t pad[3];
  int32_t pages[kWin];
};
static_assert(sizeof(SlotMeta) % 16 == 0, "slot size");

constexpr int kOffStages = 0;
constexpr int kOffQ = kOffStages + kStages * kStageBytes;
constexpr int kOffP = kOffQ + kQBytes;
constexpr int kOffMeta = kOffP + kPBytes;
constexpr int kOffRed = kOffMeta + kSlots * (int)sizeof(SlotMeta);
constexpr int kOffInfo = kOffRed + 4 * kRows * 4 + 64;
constexpr int kOffBars = kOffInfo + kStages * (int)sizeof(StageInfo);
constexpr int kNumBars = 2 * kStages + 2 * kSlots + 2;
constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ uint32_t swz(int row, int chunk) { return (uint32_t)((chunk ^ (row & 7)) << 4); }

// MERGE task: combine the split states of one 64-row unit (256 threads).
__device__ __noinline__ void mla_merge_unit(const MlaParams& p, const UnitDesc u) {
  const int t = threadIdx.x;   // 0..255
  const int row = t >> 2;      // 64 rows, four threads each
  const int cbase = (t & 3) * 128;
  if (row >= u.nrows) return;
  const size_t base = (size_t)u.partial_base + row;
  const int ns = u.n_splits;
  float ls[kMaxSplits];
#pragma unroll
  for (int k = 0; k < kMaxSplits; ++k) ls[k] = k < ns ? ld_cg(p.plse + base + (size_t)k * u.nrows) : -INFINITY;
  float Mx = -INFINITY;
  bool bad = false;
#pragma unroll
  for (int k = 0; k < kMaxSplits; ++k) {
    bad |= isnan(ls[k]);
    Mx = fmaxf(Mx, ls[k]);
  }
  float w[kMaxSplits];
  float W = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxSplits; ++k) {
    w[k] = (bad || ls[k] == -INFINITY || Mx == -INFINITY) ? 0.f : fast_exp2(ls[k] - Mx);
    W += w[k];
  }
  const float winv = W > 0.f ? 1.f / W : 0.f;
  const int pr = u.row0 + row;
  const int qi = pr / p.num_heads;
  const size_t out_row = (size_t)(u.q_start + qi) * p.num_heads + (pr - qi * p.num_heads);
  for (int c = cbase; c < cbase + 128; c += 8) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int k = 0; k < ns; ++k) {
      const float* src = p.po + (base + (size_t)k * u.nrows) * kDv + c;
      const float4 a = ld_cg4(src), b = ld_cg4(src + 4);
      acc[0] += w[k] * a.x; acc[1] += w[k] * a.y; acc[2] += w[k] * a.z; acc[3] += w[k] * a.w;
      acc[4] += w[k] * b.x; acc[5] += w[k] * b.y; acc[6] += w[k] * b.z; acc[7] += w[k] * b.w;
    }
    uint4 v;
    v.x = bad ? 0u : pack_bf16(acc[0] * winv, acc[1] * winv);
    v.y = bad ? 0u : pack_bf16(acc[2] * winv, acc[3] * winv);
    v.z = bad ? 0u : pack_bf16(acc[4] * winv, acc[5] * winv);
    v.w = bad ? 0u : pack_bf16(acc[6] * winv, acc[7] * winv);
    *reinterpret_cast<uint4*>(p.out + out_row * kDv + c) = v;
  }
  if (p.lse != nullptr && (t & 3) == 0)
    p.lse[out_row] = bad ? NAN : (W > 0.f ? (Mx + __log2f(W)) * kLn2 : -INFINITY);
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
                      const MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem + kOffStages;
  uint8_t* qbuf = smem + kOffQ;
  uint8_t* pbuf = smem + kOffP;
  SlotMeta* meta = reinterpret_cast<SlotMeta*>(smem + kOffMeta);
  float* red_m = reinterpret_cast<float*>(smem + kOffRed);   // [2][64] half maxima
  float* red_l = red_m + 2 * kRows;                           // [2][64] half sums
  int* s_flag = reinterpret_cast<int*>(red_l + 2 * kRows);
  StageInfo* sinfo = reinterpret_cast<StageInfo*>(smem + kOffInfo);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* empty = full + kStages;
  uint64_t* slot_full = empty + kStages;
  uint64_t* slot_empty = slot_full + kSlots;
  uint64_t* q_full = slot_empty + kSlots;   // the query block landed
  uint64_t* q_empty = q_full + 1;           // the consumers are done with it

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  WsHeader* hdr = p.hdr;
  const int H = p.num_heads;

  if (threadIdx.x == 0) {
    int ok = (hdr->magic == kWsMagic && hdr->plan_id == p.plan_id) ? 1 : 0;
    if (!ok) set_error(hdr, PD_DEV_PLAN_MISMATCH, -1);
    s_flag[1] = ok;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kNCW);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&slot_full[s], 1);
      mbar_init(&slot_empty[s], kNCW);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, kNCW);
    fence_barrier_init();
    fence_proxy_async();
  }
  __syncthreads();
  if (!s_flag[1]) return;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int P = p.page_size;
  const int BR = p.box_rows;

  if (warp >= kNCW) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
  if (warp == kSchedulerWarp) {
    // ============================== scheduler ==============================
    uint32_t s = 0, sph = 0;
    uint32_t qph = 0;       // q_empty phase (one per work item)
    bool dead = false, exhausted = false, first_pop = true;
    int k_next = 0, k_end = 0;
    if (p.cta_items != nullptr) {
      k_next = __ldg(&p.cta_items[blockIdx.x]);
      k_end = __ldg(&p.cta_items[blockIdx.x + 1]);
    }
    int used[kSlots], split_unit[kSlots], split_n[kSlots];
#pragma unroll
    for (int k = 0; k < kSlots; ++k) used[k] = 0, split_unit[k] = -1, split_n[k] = 0;
    while (true) {
      int merge_unit = -1;
      if (!mbar_wait(&slot_empty[s], sph ^ 1)) { dead = true; break; }
      if (used[s] && split_unit[s] >= 0) {
        int last = 0;
        if (lane == 0) {
          __threadfence();
          const uint32_t old = atomicAdd(&p.counters[split_unit[s]], 1u);
          last = old == (uint32_t)(split_n[s] - 1);
          if (last) {
            p.counters[split_unit[s]] = 0u;
            __threadfence();
          }
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) merge_unit = split_unit[s];
      }
      SlotMeta& m = meta[s];
      split_unit[s] = -1;
      if (merge_unit >= 0) {
        if (lane == 0) {
          m.kind = T_MERGE;
          m.item = merge_unit;
          m.it.unit = merge_unit;
          m.it.u = p.units[merge_unit];
          m.err = 0;
          mbar_arrive(&slot_full[s]);
        }
        used[s] = 1;
        if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
        continue;
      }
      uint32_t idx = (uint32_t)p.num_items;
      if (!exhausted && p.cta_items != nullptr) {
        if (k_next < k_end) idx = (uint32_t)k_next++;
        exhausted = idx >= (uint32_t)p.num_items;
      } else if (!exhausted) {
        if (first_pop) {
          idx = blockIdx.x;
          first_pop = false;
        } else {
          if (lane == 0) idx = gridDim.x + atomicAdd(&hdr->queue_counter, 1u);
          idx = __shfl_sync(0xffffffffu, idx, 0);
        }
        if (idx >= (uint32_t)p.num_items) exhausted = true;
      }
      if (exhausted) {
        bool pending = false;
#pragma unroll
        for (int k = 0; k < kSlots; ++k) pending |= (k != (int)s) && split_unit[k] >= 0;
        if (lane == 0) {
          m.kind = pending ? T_NOP : T_END;
          m.err = 0;
          mbar_arrive(&slot_full[s]);
        }
        if (!pending) break;
        used[s] = 1;
        if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
        continue;
      }
      const ItemDesc it = p.items[idx];
      const UnitDesc& u = it.u;
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
      const int tok_first = it.tile_begin * kTile;
      const int tok_end = min(it.tile_end * kTile, u.kv_len);
      const int pg_first = tok_first / P;
      const int nwin = err ? 0 : min(kWin, (tok_end - 1) / P - pg_first + 1);
      const int32_t* trow = p.block_tables + (size_t)u.b * p.max_pages_per_seq + pg_first;
      for (int k = lane; k < nwin; k += 32) m.pages[k] = __ldg(trow + k);
      if (lane == 0) {
        m.it = it;
        m.item = (int32_t)idx;
        m.err = err;
        m.kind = T_ITEM;
        m.win0 = pg_first;
        m.nwin = nwin;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&slot_full[s]);
      // the query block has one buffer: wait until the previous item is done with it
      if (!mbar_wait(q_empty, qph ^ 1)) { dead = true; break; }
      qph ^= 1;
      if (lane == 0) {
        if (err) {
          mbar_arrive(q_full);
        } else {
          mbar_arrive_expect_tx(q_full, (uint32_t)kQBytes);
          const int grow = u.q_start * H + u.row0;   // packed (token, head) rows are contiguous
          for (int c = 0; c < kSlabs; ++c)
            tma_load_4d(qbuf + c * kRows * 128, &q_map, 64 * c, grow, 0, 0, q_full, l2_evict_last_policy());
        }
      }
      used[s] = 1;
      if (u.n_splits > 1 && p.fused_merge) {
        split_unit[s] = it.unit;
        split_n[s] = u.n_splits;
      }
      if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
    }
    if (dead && lane == 0) set_error(hdr, PD_DEV_TIMEOUT, -1);
  } else if (warp == kProducerWarp) {
    // ============================== producer ==============================
    prefetch_tensormap(&kv_map);
    const uint64_t pol = l2_evict_first_policy();
    uint32_t stage = 0, phase = 0;
    uint32_t s = 0, sph = 0;
    uint32_t armed = 0, armed_par = 0;
    bool dead = false;
    while (true) {
      if (!mbar_wait(&slot_full[s], sph)) { dead = true; break; }
      const SlotMeta& m = meta[s];
      const int kind = m.kind;
      if (kind == T_END) break;
      const ItemDesc it = m.it;
      const UnitDesc& u = it.u;
      if (kind != T_ITEM || m.err) {
        const int f = kind == T_MERGE ? F_MERGE : kind == T_NOP ? F_NOP : F_INVALID;
        if (!mbar_wait(&empty[stage], phase ^ 1)) { dead = true; break; }
        if (lane == 0) {
          sinfo[stage] = StageInfo{(int32_t)s, it.tile_begin, F_FIRST | F_LAST | f, 0};
          mbar_arrive(&full[stage]);
        }
        if (++stage == (uint32_t)kStages) { stage = 0; phase ^= 1; }
        if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
        continue;
      }
      const int L = u.kv_len;
      const int win0 = m.win0, nwin = m.nwin;
      const int32_t* trow = p.block_tables + (size_t)u.b * p.max_pages_per_seq;
      for (int t = it.tile_begin; t < it.tile_end; ++t) {
        const int tok0 = t * kTile;
        const int nvalid = min(kTile, L - tok0);
        const int nbox = (nvalid + BR - 1) / BR;
        int pg0 = 0, pg1 = 0;
        if (lane < nbox) {
          const int pi = (tok0 + lane * BR) / P - win0;
          pg0 = pi < nwin ? m.pages[pi] : __ldg(trow + win0 + pi);
        }
        if (lane + 32 < nbox) {
          const int pi = (tok0 + (lane + 32) * BR) / P - win0;
          pg1 = pi < nwin ? m.pages[pi] : __ldg(trow + win0 + pi);
        }
        const bool bad0 = lane < nbox && (pg0 < 0 || pg0 >= p.num_pages);
        const bool bad1 = lane + 32 < nbox && (pg1 < 0 || pg1 >= p.num_pages);
        const bool bad = __any_sync(0xffffffffu, bad0 || bad1);
        if (!mbar_wait(&empty[stage], phase ^ 1)) { dead = true; break; }
        const int flags = (t == it.tile_begin ? F_FIRST : 0) | (t == it.tile_end - 1 ? F_LAST : 0);
        if (bad) {
          if (lane == 0) {
            set_error(hdr, PD_DEV_BAD_PAGE, u.b);
            sinfo[stage] = StageInfo{(int32_t)s, t, flags | F_BAD, 0};
            mbar_arrive(&full[stage]);
          }
        } else {
          if (lane == 0) {
            sinfo[stage] = StageInfo{(int32_t)s, t, flags, 0};
            mbar_arrive_expect_tx(&full[stage], (uint32_t)nbox * BR * 128 * kSlabs);
          }
          uint8_t* dst = stages + stage * kStageBytes;
          for (int j = 0; j < nbox; ++j) {
            const int page = __shfl_sync(0xffffffffu, j < 32 ? pg0 : pg1, j & 31);
            if (lane == 0) {
              const int slot = (tok0 + j * BR) % P;
              for (int c = 0; c < kSlabs; ++c)
                tma_load_4d(dst + c * kSlabBytes + j * BR * 128, &kv_map, 64 * c, 0, slot, page, &full[stage], pol);
            }
          }
        }
        armed |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        if (++stage == (uint32_t)kStages) { stage = 0; phase ^= 1; }
      }
      if (dead) break;
      if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
    }
    if (!dead && mbar_wait(&empty[stage], phase ^ 1)) {
      if (lane == 0) {
        sinfo[stage] = StageInfo{-1, 0, F_END, 0};
        mbar_arrive(&full[stage]);
      }
    } else {
      dead = true;
    }
    if (dead) {
      if (lane == 0) set_error(hdr, PD_DEV_TIMEOUT, -1);
      for (int k = 0; k < kStages; ++k)
        if (armed & (1u << k)) mbar_wait(&full[k], (armed_par >> k) & 1u, 100000000ull);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsumerRegs));
    // ============================== consumers ==============================
    const int g8 = lane >> 2, j4 = lane & 3;
    const int rw = warp & 3;     // row block of 16 within the unit's 64 rows
    const int th = warp >> 2;    // key half of each tile for S; channel half of O
    const int row_a = 16 * rw + g8, row_b = row_a + 8;
    const float scale2 = p.sm_scale * kLog2e;
    const uint32_t qb = smem_u32(qbuf), pb = smem_u32(pbuf);

    uint32_t stage = 0, phase = 0, s = 0, sph = 0, qph = 0;
    float m[2], l[2], o[32][4];
    int errored = 0, kv_len = 0;
    int pos[2] = {0, 0};

    while (true) {
      if (!mbar_wait(&full[stage], phase)) {
        if (lane == 0) set_error(hdr, PD_DEV_TIMEOUT, -1);
        break;
      }
      const StageInfo info = sinfo[stage];
      if (info.flags & F_END) break;
      if (info.flags & (F_MERGE | F_NOP)) {
        if (!mbar_wait(&slot_full[s], sph)) {
          if (lane == 0) set_error(hdr, PD_DEV_TIMEOUT, -1);
          break;
        }
        if (info.flags & F_MERGE) mla_merge_unit(p, meta[s].it.u);
        named_barrier(1, kNCW * 32);
        if (lane == 0) {
          mbar_arrive(&empty[stage]);
          mbar_arrive(&slot_empty[s]);
        }
        if (++stage == (uint32_t)kStages) { stage = 0; phase ^= 1; }
        if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
        continue;
      }
      if (info.flags & F_FIRST) {
        if (!mbar_wait(&slot_full[s], sph) || !mbar_wait(q_full, qph)) {
          if (lane == 0) set_error(hdr, PD_DEV_TIMEOUT, -1);
          break;
        }
        qph ^= 1;
        const UnitDesc& fu = meta[s].it.u;
        kv_len = fu.kv_len;
        errored = (info.flags & F_INVALID) ? 1 : 0;
        pos[0] = fu.kv_len - fu.q_len + (fu.row0 + row_a) / H;
        pos[1] = fu.kv_len - fu.q_len + (fu.row0 + row_b) / H;
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
#pragma unroll
        for (int n = 0; n < 32; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
      }
      const bool last = (info.flags & F_LAST) != 0;

      if (info.flags & (F_BAD | F_INVALID)) {
        errored = 1;
      } else {
        const int tok0 = info.tile * kTile;
        uint8_t* st = stages + stage * kStageBytes;
        const uint32_t sb = smem_u32(st);
        // zero value rows past the sequence end (slabs 0..7 of those keys)
        if (tok0 + kTile > kv_len) {
          const int t = threadIdx.x;  // 0..255: key row t / 4, slab pair
          const int r = t >> 2;
          if (tok0 + r >= kv_len) {
#pragma unroll
            for (int c = 2 * (t & 3); c < 2 * (t & 3) + 2; ++c)
#pragma unroll
              for (int k = 0; k < 8; ++k)
                *reinterpret_cast<uint4*>(st + c * kSlabBytes + r * 128 + k * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async();
        }

        // ---- S = Q K^T: rows 16 rw .. +16, keys 32 th .. +32
        float sacc[4][4];
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) sacc[nb][0] = sacc[nb][1] = sacc[nb][2] = sacc[nb][3] = 0.f;
#pragma unroll 4
        for (int kk = 0; kk < 36; ++kk) {
          const int c = kk >> 2, cc = kk & 3;
          uint32_t a[4];
          {
            const int row = 16 * rw + (lane & 7) + (((lane >> 3) & 1) << 3);
            const int chunk = 2 * cc + (lane >> 4);
            ldsm_x4(qb + c * (kRows * 128) + row * 128 + swz(row, chunk), a[0], a[1], a[2], a[3]);
          }
#pragma unroll
          for (int pq = 0; pq < 2; ++pq) {
            const int tok = 32 * th + 16 * pq + (lane & 7) + ((lane >> 4) << 3);
            const int chunk = 2 * cc + ((lane >> 3) & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(sb + c * kSlabBytes + tok * 128 + swz(tok, chunk), b0, b1, b2, b3);
            mma_bf16(sacc[2 * pq], a, b0, b1);
            mma_bf16(sacc[2 * pq + 1], a, b2, b3);
          }
        }

        // ---- row maxima of this key half, exchanged with the partner warp
        const int first = tok0 + 32 * th;
        const bool need_mask = first + 31 > min(pos[0], pos[1]);
        float x[2][8];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          float mx = -INFINITY;
#pragma unroll
          for (int nb = 0; nb < 4; ++nb)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float v = sacc[nb][2 * rr + e] * scale2;
              if (need_mask && first + 8 * nb + 2 * j4 + e > pos[rr]) v = -INFINITY;
              x[rr][2 * nb + e] = v;
              mx = fmaxf(mx, v);
            }
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          if (j4 == 0) red_m[th * kRows + (rr ? row_b : row_a)] = mx;
        }
        named_barrier(1, kNCW * 32);
        bool rescale = false;
        float alpha[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int row = rr ? row_b : row_a;
          const float mt = fmaxf(red_m[row], red_m[kRows + row]);
          const float m_new = fmaxf(m[rr], mt);
          const float m_use = m_new == -INFINITY ? 0.f : m_new;
          alpha[rr] = fast_exp2(m[rr] - m_use);
          rescale |= alpha[rr] != 1.f;
          float sum = 0.f;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            x[rr][k] = fast_exp2(x[rr][k] - m_use);
            sum += x[rr][k];
          }
          l[rr] = l[rr] * alpha[rr] + sum;
          m[rr] = m_new;
          // P (bf16) rows of this warp, keys 32 th + 8 nb + 2 j4 + {0,1}
#pragma unroll
          for (int nb = 0; nb < 4; ++nb) {
            const int key = 32 * th + 8 * nb + 2 * j4;
            *reinterpret_cast<uint32_t*>(pbuf + row * 128 + swz(row, key >> 3) + (key & 7) * 2) =
                pack_bf16(x[rr][2 * nb], x[rr][2 * nb + 1]);
          }
        }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int n = 0; n < 32; ++n) {
            o[n][0] *= alpha[0];
            o[n][1] *= alpha[0];
            o[n][2] *= alpha[1];
            o[n][3] *= alpha[1];
          }
        }
        named_barrier(1, kNCW * 32);  // P of both key halves written

        // ---- O += P V: rows 16 rw .. +16, channels 256 th .. +256, all 64 keys
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          uint32_t a[4];
          {
            const int row = 16 * rw + (lane & 7) + (((lane >> 3) & 1) << 3);
            const int chunk = 2 * ks + (lane >> 4);
            ldsm_x4(pb + row * 128 + swz(row, chunk), a[0], a[1], a[2], a[3]);
          }
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int tok = 16 * ks + (lane & 7) + (((lane >> 3) & 1) << 3);
            const int cg = 32 * th + 2 * q + (lane >> 4);   // 8-channel group of the latent row
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(sb + (cg >> 3) * kSlabBytes + tok * 128 + swz(tok, cg & 7), b0, b1, b2, b3);
            mma_bf16(o[2 * q], a, b0, b1);
            mma_bf16(o[2 * q + 1], a, b2, b3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&empty[stage]);
        if (last) mbar_arrive(q_empty);  // the query block may be replaced
      }
      if (++stage == (uint32_t)kStages) { stage = 0; phase ^= 1; }
      if (!last) continue;

      // ============================ epilogue ============================
      const ItemDesc& it = meta[s].it;
      const UnitDesc& u = it.u;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 1);
        l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 2);
        if (j4 == 0) red_l[th * kRows + (rr ? row_b : row_a)] = l[rr];
      }
      named_barrier(1, kNCW * 32);
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int row = rr ? row_b : row_a;
        const float Ls = red_l[row] + red_l[kRows + row];
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        const bool valid = row < u.nrows;
        const int pr = u.row0 + row;
        const int qi = pr / H;
        const size_t out_row = (size_t)(u.q_start + qi) * H + (pr - qi * H);
        const float lse2 = Ls > 0.f ? m[rr] + __log2f(Ls) : -INFINITY;
        if (!valid) continue;
        if (u.n_splits == 1) {
          __nv_bfloat16* dst = p.out + out_row * kDv + 256 * th + 2 * j4;
#pragma unroll
          for (int n = 0; n < 32; ++n)
            *reinterpret_cast<uint32_t*>(dst + 8 * n) =
                errored ? 0u : pack_bf16(o[n][2 * rr] * inv, o[n][2 * rr + 1] * inv);
          if (p.lse != nullptr && th == 0 && j4 == 0) p.lse[out_row] = errored ? NAN : lse2 * kLn2;
        } else {
          const size_t prow = (size_t)u.partial_base + (size_t)it.split * u.nrows + row;
          float* dst = p.po + prow * kDv + 256 * th + 2 * j4;
#pragma unroll
          for (int n = 0; n < 32; ++n)
            *reinterpret_cast<float2*>(dst + 8 * n) = make_float2(o[n][2 * rr] * inv, o[n][2 * rr + 1] * inv);
          if (th == 0 && j4 == 0) p.plse[prow] = errored ? NAN : lse2;
        }
      }
      named_barrier(1, kNCW * 32);  // red arrays and the slot may be reused
      if (lane == 0) mbar_arrive(&slot_empty[s]);
      if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
    }
  }

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

cudaError_t launch_mla_decode(const CUtensorMap& kvmap, const CUtensorMap& qmap, const MlaParams& p,
                              int grid, cudaStream_t stream) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(mla_decode_kernel), kSmemBytes);
  if (e != cudaSuccess) return e;
  mla_decode_kernel<<<grid, kThreads, kSmemBytes, stream>>>(kvmap, qmap, p);
  return cudaGetLastError();
}

}  // namespace pd
