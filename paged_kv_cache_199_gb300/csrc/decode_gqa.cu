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
//  * warp 5 is the scheduler: it pops items up to four ahead, checks the
//    device seq_lens / q_indptr against the plan, prefetches the item's page
//    ids into shared memory and TMA-loads its query rows, so no global-memory
//    round trip sits on the copy path;
//  * warp 4 is the producer: per 64-token tile it translates tokens to pages
//    (ids bounds-checked against num_pages) and issues 4-D TMA tensor copies
//    of the K and V rows into a multi-stage shared-memory ring (128-byte
//    swizzle, mbarrier completion, L2 evict-first hint);
//  * two such CTAs share an SM, so one CTA's epilogue overlaps the other's
//    streaming;
//  * warps 0-3 are consumers, each owning 16 keys of a tile: S^T = K Q^T and
//    O^T += V^T P^T on mma.sync m16n8k16 with the keys as M and the <= 8 or
//    <= 16 packed query rows of a GQA group as N (movmatrix moves P^T into
//    B-fragment order), row max/sum with warp shuffles, online softmax in the
//    exp2 domain. The E4M3 variant loads 16-byte rows with ld.shared.v4,
//    transposes V bytes with prmt and converts pairs with
//    cvt.rn.f16x2.e4m3x2 (exact) for f16 MMAs; the token and channel order
//    inside the contraction is permuted consistently for P and V (and for Q
//    and K) so every shared-memory read is a conflict-free 16-byte load;
//  * epilogue: the four warps' partial states are merged in shared memory;
//    an unsplit unit writes bf16 output (+ LSE) directly, a split writes an
//    fp32 partial state; with the fused merge the last split to arrive
//    (atomic counter that resets itself) merges all partial states by
//    log-sum-exp (PR #5591 "last-arriver split merge"), otherwise the
//    LSE-merge kernel launched after this one does.
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

constexpr int kD = 128;             // head dim
constexpr int kNCW = 4;             // consumer warps
constexpr int kProducerWarp = kNCW;
constexpr int kSchedulerWarp = kNCW + 1;
constexpr int kThreads = (kNCW + 2) * 32;
constexpr int kSlots = 2;           // work items the scheduler may run ahead
constexpr int kWin = 256;           // page ids prefetched per item
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum : int { F_FIRST = 1, F_LAST = 2, F_BAD = 4, F_INVALID = 8, F_END = 16, F_MERGE = 32, F_NOP = 64 };
// What an item slot holds.
enum : int { T_ITEM = 0, T_MERGE = 1, T_NOP = 2, T_END = 3 };

struct StageInfo {
  int32_t slot;
  int32_t tile;
  int32_t flags;
  int32_t pad;
};

// One work item as the scheduler warp hands it to the producer and consumers.
struct SlotMeta {
  ItemDesc it;
  int32_t item;    // queue position
  int32_t err;     // pd_device_error found while validating, 0 if none
  int32_t kind;    // T_ITEM / T_MERGE (merge a unit's split states) / T_NOP / T_END
  int32_t win0;    // page index of pages[0]
  int32_t nwin;    // page ids held in pages[]
  int32_t pad[3];
  int32_t pages[kWin];
};
static_assert(sizeof(SlotMeta) % 16 == 0, "slot size");

// NB = number of 8-row n-blocks of packed query rows (1: <= 8 rows, 2: <= 16).
template <bool FP8, int NB>
struct Cfg {
  static constexpr int kRows = 8 * NB;
  // tokens per stage: E4M3 stages hold 128 tokens (32 KB, like a 64-token
  // BF16 stage), so each consumer warp owns 32 keys (two 16-key m-blocks)
  static constexpr int kTile = FP8 ? 128 : 64;
  static constexpr int kMB = kTile / (kNCW * 16);             // 16-key m-blocks per warp
  static constexpr int kRowBytes = FP8 ? 128 : 256;          // one token's K (or V) row
  static constexpr int kHalfBytes = kTile * 128;             // one 128-byte-wide slab of a tile
  static constexpr int kKBytes = kTile * kRowBytes;
  static constexpr int kStageBytes = 2 * kKBytes;            // K + V
  static constexpr int kStages = 3;
  static constexpr int kCtasPerSm = 2;   // resident CTAs per SM (the planner's assumption)
  static constexpr int kQSlotBytes = kRows * kD * 2;         // bf16 query rows
  static constexpr int kOffQ = kStages * kStageBytes;
  static constexpr int kOffMeta = kOffQ + kSlots * kQSlotBytes;
  static constexpr int kOffRed = kOffMeta + kSlots * (int)sizeof(SlotMeta);
  static constexpr int kOffInfo = kOffRed + 2 * kNCW * 16 * 4 + 64;
  static constexpr int kOffBars = kOffInfo + kStages * (int)sizeof(StageInfo);
  static constexpr int kSmemBytes = kOffBars + (2 * kStages + 3 * kSlots) * 8 + 1024;  // + alignment slack
  static_assert(2 * kRows * kD * 4 <= kStageBytes, "merge buffers must fit in one stage");
};

// Max over the 8 lanes that share lane & 3 (the 16 keys of one query row).
__device__ __forceinline__ float rowmax8(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
  return v;
}
__device__ __forceinline__ float rowsum8(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  return v;
}

// Merge the split states of one unit into its output rows (a MERGE task,
// run by the 128 consumer threads of the CTA whose split arrived last):
// lse = log2-sum of the split LSEs, out = sum_s 2^(lse_s - lse) out_s.
template <int kRows>
__device__ __noinline__ void merge_unit_states(const GqaParams& p, const UnitDesc u, int G) {
  constexpr int kTpr = 128 / kRows;  // threads per row
  constexpr int kCpt = kD / kTpr;    // channels per thread
  constexpr int kBatch = kCpt == 8 ? 8 : 4;  // splits whose partial rows are loaded together
  const int t = threadIdx.x;
  const int row = t / kTpr;
  const int c0 = (t % kTpr) * kCpt;
  // Ordering: every split's writes precede its arrival count (release fence
  // in its scheduler), this CTA's scheduler fenced after seeing the last
  // count, and the slot barrier orders these reads after that fence. The
  // loads bypass L1.
  if (row >= u.nrows) return;
  const size_t base = (size_t)u.partial_base + row;
  const int ns = u.n_splits;
  float ls[kMaxSplits];
#pragma unroll
  for (int k = 0; k < kMaxSplits; ++k) ls[k] = k < ns ? ld_cg(p.plse + base + (size_t)k * u.nrows) : -INFINITY;
  const int pr = u.row0 + row;
  const int qi = pr / G;
  const int head = u.g * G + (pr - qi * G);
  const float s2 = sink_log2(p.sinks, head);
  float Mx = s2;
  bool bad = false;
#pragma unroll
  for (int k = 0; k < kMaxSplits; ++k) {
    bad |= isnan(ls[k]);
    Mx = fmaxf(Mx, ls[k]);
  }
  float W = (bad || s2 == -INFINITY) ? 0.f : fast_exp2(s2 - Mx);
  float acc[kCpt];
#pragma unroll
  for (int k = 0; k < kCpt; ++k) acc[k] = 0.f;
  if (!bad && Mx != -INFINITY) {
#pragma unroll
    for (int b0 = 0; b0 < kMaxSplits; b0 += kBatch) {
      if (b0 >= ns) break;
      float4 v[kBatch][kCpt / 4];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const float* src = p.po + (base + (size_t)(b0 + k) * u.nrows) * kD + c0;
#pragma unroll
        for (int q = 0; q < kCpt / 4; ++q) v[k][q] = b0 + k < ns ? ld_cg4(src + 4 * q) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const float x = ls[b0 + k];
        const float w = x == -INFINITY ? 0.f : fast_exp2(x - Mx);
        W += w;
#pragma unroll
        for (int q = 0; q < kCpt / 4; ++q) {
          acc[4 * q] += w * v[k][q].x;
          acc[4 * q + 1] += w * v[k][q].y;
          acc[4 * q + 2] += w * v[k][q].z;
          acc[4 * q + 3] += w * v[k][q].w;
        }
      }
    }
  }
  const float winv = W > 0.f ? 1.f / W : 0.f;
  const size_t out_row = (size_t)(u.q_start + qi) * p.num_q_heads + head;
  uint32_t packed[kCpt / 2];
#pragma unroll
  for (int k = 0; k < kCpt / 2; ++k) packed[k] = bad ? 0u : pack_bf16(acc[2 * k] * winv, acc[2 * k + 1] * winv);
  uint4* dst = reinterpret_cast<uint4*>(p.out + out_row * kD + c0);
#pragma unroll
  for (int k = 0; k < kCpt / 8; ++k)
    dst[k] = make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]);
  if (p.lse != nullptr && (t % kTpr) == 0)
    p.lse[out_row] = bad ? NAN : (W > 0.f ? (Mx + __log2f(W)) * kLn2 : -INFINITY);
}

template <bool FP8, int NB>
__global__ void __launch_bounds__(kThreads, Cfg<FP8, NB>::kCtasPerSm)
    gqa_decode_kernel(const __grid_constant__ CUtensorMap k_map,
                      const __grid_constant__ CUtensorMap v_map, const GqaParams p) {
  using C = Cfg<FP8, NB>;
  constexpr int kRows = C::kRows;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* qbuf = smem + C::kOffQ;
  SlotMeta* meta = reinterpret_cast<SlotMeta*>(smem + C::kOffMeta);
  float* red_m = reinterpret_cast<float*>(smem + C::kOffRed);
  float* red_l = red_m + kNCW * 16;
  int* s_flag = reinterpret_cast<int*>(red_l + kNCW * 16);
  StageInfo* sinfo = reinterpret_cast<StageInfo*>(smem + C::kOffInfo);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* empty = full + C::kStages;
  uint64_t* slot_full = empty + C::kStages;
  uint64_t* slot_empty = slot_full + kSlots;
  uint64_t* q_full = slot_empty + kSlots;     // query rows of the slot landed

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  WsHeader* hdr = p.hdr;

  if (threadIdx.x == 0) {
    s_flag[1] = 1;  // cleared by the scheduler if the workspace holds another plan
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kNCW);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&slot_full[s], 1);
      mbar_init(&slot_empty[s], kNCW);
      mbar_init(&q_full[s], 1);
    }
    fence_barrier_init();
    fence_proxy_async();
  }
  __syncthreads();
  // a dependent LSE-merge grid may be scheduled now; it waits for this grid
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int G = p.group;
  const int P = p.page_size;
  const int BR = p.box_rows;

  if (warp == kSchedulerWarp) {
    // ============================== scheduler ==============================
    // Fills the item slots in order. For a work item it pops the queue,
    // validates the item's metadata against the device copies and prefetches
    // its page ids and query rows. When a slot comes back after a split item
    // it counts the split's arrival for the unit (release fence + atomic, off
    // the consumers' path); the CTA whose split arrives last gets a MERGE task
    // in that slot, which its consumer warps execute. After the queue runs
    // dry, NOP tasks keep the slots turning until no split arrival is pending.
    uint32_t s = 0, sph = 0;
    bool dead = false;
    bool exhausted = false;
    bool first_pop = true;
    // per slot: its latest q_full phase carries query copies of this warp
    // (parity q_par); they must land before the CTA exits
    uint32_t q_loaded = 0, q_par = 0;
    int k_next = 0, k_end = 0;
    if (p.cta_items != nullptr) {
      k_next = __ldg(&p.cta_items[blockIdx.x]);
      k_end = __ldg(&p.cta_items[blockIdx.x + 1]);
    }
    // The workspace must hold this plan. The check runs here, with the read of
    // the CTA's first item descriptor in flight beside it, rather than ahead
    // of every warp; on a mismatch no item is started and nothing is written.
    uint32_t ws_magic = 0;
    uint64_t ws_plan = 0;
    if (lane == 0) {
      ws_magic = hdr->magic;
      ws_plan = hdr->plan_id;
    }
    const bool first_from_queue = p.cta_items == nullptr && blockIdx.x < (uint32_t)p.num_items;
    ItemDesc first_it{};
    if (first_from_queue) first_it = p.items[blockIdx.x];
    int plan_ok = 1;
    if (lane == 0 && (ws_magic != kWsMagic || ws_plan != p.plan_id)) {
      plan_ok = 0;
      set_error(hdr, PD_DEV_PLAN_MISMATCH, -1);
      s_flag[1] = 0;
      meta[0].kind = T_END;
      meta[0].err = 0;
      mbar_arrive(&slot_full[0]);
      mbar_arrive(&q_full[0]);
    }
    plan_ok = __shfl_sync(0xffffffffu, plan_ok, 0);
    int used[kSlots];
    int split_unit[kSlots];   // unit of the split item a slot holds, or -1
    int split_n[kSlots];
#pragma unroll
    for (int k = 0; k < kSlots; ++k) {
      used[k] = 0;
      split_unit[k] = -1;
      split_n[k] = 0;
    }
    bool took_first = false;
    while (plan_ok) {
      int merge_unit = -1;
      if (used[s]) {
        if (!mbar_wait(&slot_empty[s], sph ^ 1, p.wait_ns)) { dead = true; break; }
        if (split_unit[s] >= 0) {
          int last = 0;
          if (lane == 0) {
            __threadfence();  // this CTA's partial writes (seen through the slot barrier) first
            const uint32_t old = atomicAdd(&p.counters[split_unit[s]], 1u);
            last = old == (uint32_t)(split_n[s] - 1);
            if (last) {
              p.counters[split_unit[s]] = 0u;  // ready for the next launch
              __threadfence();                 // every split's writes before the merge reads
            }
          }
          last = __shfl_sync(0xffffffffu, last, 0);
          if (last) merge_unit = split_unit[s];
        }
      } else {
        // first use of this slot: pass the phase-0 wait of a fresh barrier
        if (!mbar_wait(&slot_empty[s], sph ^ 1, p.wait_ns)) { dead = true; break; }
      }
      SlotMeta& m = meta[s];
      split_unit[s] = -1;
      q_loaded &= ~(1u << s);   // set again below if this fill copies query rows
      if (merge_unit >= 0) {
        if (lane == 0) {
          m.kind = T_MERGE;
          m.item = merge_unit;
          m.it.unit = merge_unit;
          m.it.u = p.units[merge_unit];
          m.err = 0;
          mbar_arrive(&slot_full[s]);
          mbar_arrive(&q_full[s]);  // every slot fill completes one q_full phase
        }
        used[s] = 1;
        if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
        continue;
      }
      uint32_t idx = (uint32_t)p.num_items;
      if (!exhausted && p.cta_items != nullptr) {
        // static schedule: this CTA's own item range
        if (k_next < k_end) idx = (uint32_t)k_next++;
        exhausted = idx >= (uint32_t)p.num_items;
      } else if (!exhausted) {
        // item blockIdx.x is this CTA's first; the queue hands out the rest
        if (first_pop) {
          idx = blockIdx.x;
          first_pop = false;
          took_first = true;
        } else {
          if (lane == 0) idx = gridDim.x + atomicAdd(&hdr->queue_counter, 1u);
          idx = __shfl_sync(0xffffffffu, idx, 0);
        }
        if (idx >= (uint32_t)p.num_items) exhausted = true;
      }
      if (exhausted) {
        // done once no other slot still owes a split arrival
        bool pending = false;
#pragma unroll
        for (int k = 0; k < kSlots; ++k) pending |= (k != (int)s) && split_unit[k] >= 0;
        if (lane == 0) {
          m.kind = pending ? T_NOP : T_END;
          m.err = 0;
          mbar_arrive(&slot_full[s]);
          mbar_arrive(&q_full[s]);
        }
        if (!pending) break;
        used[s] = 2;  // a NOP in flight
        if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
        continue;
      }
      const ItemDesc it = took_first ? first_it : p.items[idx];
      took_first = false;
      const UnitDesc& u = it.u;
      // the metadata check and the page-id reads are independent: issue them
      // together (page ids within the planned length stay inside the table row)
      int32_t sl = 0, qi0 = 0, qi1 = 0;
      if (lane == 0) {
        sl = __ldg(&p.seq_lens[u.b]);
        if (p.q_indptr != nullptr) {
          qi0 = __ldg(&p.q_indptr[u.b]);
          qi1 = __ldg(&p.q_indptr[u.b + 1]);
        }
      }
      const int tok_first = it.tile_begin * C::kTile;
      const int tok_end = min(it.tile_end * C::kTile, u.kv_len);
      const int pg_first = tok_first / P;
      const int nwin = min(kWin, (tok_end - 1) / P - pg_first + 1);
      const int32_t* trow = p.block_tables + (size_t)u.b * p.max_pages_per_seq + pg_first;
      int32_t pw[(kWin + 31) / 32];
#pragma unroll
      for (int k = 0; k < (kWin + 31) / 32; ++k) pw[k] = lane + 32 * k < nwin ? __ldg(trow + lane + 32 * k) : 0;
      int err = 0;
      if (lane == 0) {
        if (sl != u.kv_len)
          err = PD_DEV_SEQ_LEN_MISMATCH;
        else if (p.q_indptr != nullptr && (qi0 != u.q_start || qi1 != u.q_start + u.q_len))
          err = PD_DEV_Q_INDPTR_MISMATCH;
        if (err) set_error(hdr, err, u.b);
      }
      err = __shfl_sync(0xffffffffu, err, 0);
#pragma unroll
      for (int k = 0; k < (kWin + 31) / 32; ++k)
        if (lane + 32 * k < nwin) m.pages[lane + 32 * k] = pw[k];
      if (lane == 0) {
        m.it = it;
        m.item = (int32_t)idx;
        m.err = err;
        m.kind = T_ITEM;
        m.win0 = pg_first;
        m.nwin = err ? 0 : nwin;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&slot_full[s]);  // fields and page ids: the producer may start
        if (err) {
          mbar_arrive(&q_full[s]);
        } else {
          q_loaded |= 1u << s;
          q_par = (q_par & ~(1u << s)) | (sph << s);
          uint8_t* dst = qbuf + s * C::kQSlotBytes;
          mbar_arrive_expect_tx(&q_full[s], (uint32_t)u.nrows * kD * 2);
          int r = 0;
          while (r < u.nrows) {
            const int pr = u.row0 + r;
            const int i = pr / G, hh = pr - (pr / G) * G;
            const int cnt = min(G - hh, u.nrows - r);
            const __nv_bfloat16* src = p.q + ((size_t)(u.q_start + i) * p.num_q_heads + (size_t)u.g * G + hh) * kD;
            bulk_load(dst + r * kD * 2, src, (uint32_t)cnt * kD * 2, &q_full[s]);
            r += cnt;
          }
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
    if (lane == 0)
      for (int k = 0; k < kSlots; ++k)
        if (q_loaded & (1u << k)) mbar_wait(&q_full[k], (q_par >> k) & 1u, kDrainLimitNs);
  } else if (warp == kProducerWarp) {
    // ============================== producer ==============================
    prefetch_tensormap(&k_map);
    prefetch_tensormap(&v_map);
    const uint64_t pol = l2_evict_first_policy();
    uint32_t stage = 0, phase = 0;
    uint32_t s = 0, sph = 0;
    bool dead = false;
    while (true) {
      if (!mbar_wait(&slot_full[s], sph, p.wait_ns)) { dead = true; break; }
      const SlotMeta& m = meta[s];
      const int kind = m.kind;
      if (kind == T_END) break;
      const ItemDesc it = m.it;
      const UnitDesc& u = it.u;
      if (kind != T_ITEM || m.err) {
        // no copies: an invalid item, a merge task or a NOP is one bare stage
        const int f = kind == T_MERGE ? F_MERGE : kind == T_NOP ? F_NOP : F_INVALID;
        if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns)) { dead = true; break; }
        if (lane == 0) {
          sinfo[stage] = StageInfo{(int32_t)s, it.tile_begin, F_FIRST | F_LAST | f, 0};
          mbar_arrive(&full[stage]);
        }
        if (++stage == (uint32_t)C::kStages) { stage = 0; phase ^= 1; }
        if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
        continue;
      }
      const int L = u.kv_len;
      const int win0 = m.win0, nwin = m.nwin;
      const int32_t* trow = p.block_tables + (size_t)u.b * p.max_pages_per_seq;
      for (int t = it.tile_begin; t < it.tile_end; ++t) {
        const int tok0 = t * C::kTile;
        const int nvalid = min(C::kTile, L - tok0);
        const int nbox = (nvalid + BR - 1) / BR;
        constexpr int kBoxWords = C::kTile / 32;   // boxes per lane at one token per box
        int pg[kBoxWords];
        bool badl = false;
#pragma unroll
        for (int k = 0; k < kBoxWords; ++k) {
          pg[k] = 0;
          const int j = lane + 32 * k;
          if (j < nbox) {
            const int pi = (tok0 + j * BR) / P - win0;
            pg[k] = pi < nwin ? m.pages[pi] : __ldg(trow + win0 + pi);
            badl |= pg[k] < 0 || pg[k] >= p.num_pages;
          }
        }
        const bool bad = __any_sync(0xffffffffu, badl);
        if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns)) { dead = true; break; }
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
            mbar_arrive_expect_tx(&full[stage], (uint32_t)nbox * BR * 128 * (FP8 ? 2 : 4));
          }
          uint8_t* kdst = stages + stage * C::kStageBytes;
          uint8_t* vdst = kdst + C::kKBytes;
          for (int j = 0; j < nbox; ++j) {
            int sel = pg[0];
#pragma unroll
            for (int k = 1; k < kBoxWords; ++k)
              if ((j >> 5) == k) sel = pg[k];
            const int page = __shfl_sync(0xffffffffu, sel, j & 31);
            if (lane == 0) {
              const int slot = (tok0 + j * BR) % P;
              const int c1 = p.layout == PD_LAYOUT_HND ? slot : u.g;
              const int c2 = p.layout == PD_LAYOUT_HND ? u.g : slot;
              const int row_off = j * BR * 128;
              tma_load_4d(kdst + row_off, &k_map, 0, c1, c2, page, &full[stage], pol);
              tma_load_4d(vdst + row_off, &v_map, 0, c1, c2, page, &full[stage], pol);
              if (!FP8) {
                tma_load_4d(kdst + C::kHalfBytes + row_off, &k_map, 64, c1, c2, page, &full[stage], pol);
                tma_load_4d(vdst + C::kHalfBytes + row_off, &v_map, 64, c1, c2, page, &full[stage], pol);
              }
            }
          }
        }
        if (++stage == (uint32_t)C::kStages) { stage = 0; phase ^= 1; }
      }
      if (dead) break;
      if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
    }
    // ---- end marker for the consumers
    if (!dead && mbar_wait(&empty[stage], phase ^ 1, p.wait_ns)) {
      if (lane == 0) {
        sinfo[stage] = StageInfo{-1, 0, F_END, 0};
        mbar_arrive(&full[stage]);
      }
      if (++stage == (uint32_t)C::kStages) { stage = 0; phase ^= 1; }
    } else {
      dead = true;
    }
    if (dead && lane == 0) set_error(hdr, PD_DEV_TIMEOUT, -1);
    // the copies this warp put in flight land before the CTA exits (on the
    // normal path they have, and these waits return at once)
    drain_ring(full, C::kStages, stage, phase);
  } else {
    // ============================== consumers ==============================
    // Keys are the M side of the MMAs (16 per warp per tile), packed query
    // rows the N side (8 per n-block): S^T = K Q^T, then O^T += V^T P^T with
    // P^T moved into B-fragment order by movmatrix.
    const int g8 = lane >> 2;
    const int j4 = lane & 3;
    constexpr int MB = C::kMB;
    const int tokw = warp * 16 * MB;  // this warp's tokens within a tile
    // E4M3 token order inside a 16-key slice (keeps 16-byte reads conflict-free)
    const int tau0 = FP8 ? ((g8 >> 1) + 4 * (g8 & 1)) : g8;
    const int tau1 = 8 + tau0;
    const uint32_t cv = (uint32_t)(((g8 & 1) << 2) | (g8 >> 1));  // E4M3 V channel block
    const uint32_t swz = p.swizzle ? 7u : 0u;
    const float kscale = (FP8 && p.k_scale) ? __ldg(p.k_scale) : 1.0f;
    const float vscale = (FP8 && p.v_scale) ? __ldg(p.v_scale) : 1.0f;
    const float scale2 = p.sm_scale * kscale * kLog2e;
    // E4M3: the query is scaled per item by a power of two 2^qexp before its
    // f16 conversion (folded back into the logit scale), so that its largest
    // element sits in [2^14, 2^15): no bf16 query saturates or flushes in f16
    float scale2_item = scale2;

    uint32_t stage = 0, phase = 0;
    uint32_t s = 0, sph = 0;
    float m[NB][2], l[NB][2], o[8][NB][4];
    uint32_t qb[NB][8][2];
    int errored = 0;
    int kv_len = 0;
    int pos_r[NB][2];
    int pos_min = 0;

    while (true) {
      if (!mbar_wait(&full[stage], phase, p.wait_ns)) {
        if (lane == 0) set_error(hdr, PD_DEV_TIMEOUT, -1);
        break;
      }
      const StageInfo info = sinfo[stage];
      if (info.flags & F_END) break;
      if (info.flags & (F_MERGE | F_NOP)) {
        if (!mbar_wait(&slot_full[s], sph, p.wait_ns)) {
          if (lane == 0) set_error(hdr, PD_DEV_TIMEOUT, -1);
          break;
        }
        if (info.flags & F_MERGE) merge_unit_states<kRows>(p, meta[s].it.u, G);
        named_barrier(1, kNCW * 32);
        if (lane == 0) {
          mbar_arrive(&empty[stage]);
          mbar_arrive(&slot_empty[s]);
        }
        if (++stage == (uint32_t)C::kStages) { stage = 0; phase ^= 1; }
        if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
        continue;
      }
      if (info.flags & F_FIRST) {
        // acquire the slot's fields, then its query rows
        if (!mbar_wait(&slot_full[s], sph, p.wait_ns) || !mbar_wait(&q_full[s], sph, p.wait_ns)) {
          if (lane == 0) set_error(hdr, PD_DEV_TIMEOUT, -1);
          break;
        }
        const UnitDesc& fu = meta[s].it.u;
        kv_len = fu.kv_len;
        errored = (info.flags & F_INVALID) ? 1 : 0;
        if (!FP8) {
          const uint32_t qs = smem_u32(qbuf + s * C::kQSlotBytes);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int kq = 0; kq < 4; ++kq)
              ldsm_x4(qs + (8 * nb + (lane & 7)) * 256 + (4 * kq + (lane >> 3)) * 16, qb[nb][2 * kq][0],
                      qb[nb][2 * kq][1], qb[nb][2 * kq + 1][0], qb[nb][2 * kq + 1][1]);
        } else {
          // f16 B fragments, channels permuted: k16 step (h, s) covers channels
          // 16 (j4 + 4h) + 4 s + {0,1 | 2,3} for k slots {2j4, 2j4+1 | 2j4+8, 2j4+9}.
          // The warp's fragments cover every query element of the item, so a
          // warp-wide maximum gives the item's power-of-two query scale. Rows
          // past the unit's last hold another item's (or no) data: they take
          // no part in the maximum, and their logits are never used.
          uint2 qraw[NB][8];
          float qmax = 0.f;
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            const bool row_used = 8 * nb + g8 < fu.nrows;
            const uint8_t* qrow = qbuf + s * C::kQSlotBytes + (8 * nb + g8) * 256;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int ss = 0; ss < 4; ++ss) {
                const int d = 16 * (j4 + 4 * h) + 4 * ss;
                const uint2 x = *reinterpret_cast<const uint2*>(qrow + d * 2);
                qraw[nb][4 * h + ss] = x;
                if (row_used)
                  qmax = fmaxf(qmax, fmaxf(fmaxf(fabsf(bf16lo(x.x)), fabsf(bf16hi(x.x))),
                                           fmaxf(fabsf(bf16lo(x.y)), fabsf(bf16hi(x.y)))));
              }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, o));
          int qexp = 0;
          if (qmax > 0.f && qmax <= 3.0e38f) {
            int e2;
            frexpf(qmax, &e2);                      // qmax = f 2^e2, f in [0.5, 1)
            qexp = max(-100, min(100, 15 - e2));    // qmax 2^qexp in [2^14, 2^15)
          }
          scale2_item = scale2 * ldexpf(1.f, -qexp);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint2 x = qraw[nb][k];
              qb[nb][k][0] = pack_f16_sat(ldexpf(bf16lo(x.x), qexp), ldexpf(bf16hi(x.x), qexp));
              qb[nb][k][1] = pack_f16_sat(ldexpf(bf16lo(x.y), qexp), ldexpf(bf16hi(x.y), qexp));
            }
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          m[nb][0] = m[nb][1] = -INFINITY;
          l[nb][0] = l[nb][1] = 0.f;
          pos_r[nb][0] = fu.kv_len - fu.q_len + (fu.row0 + 8 * nb + 2 * j4) / G;
          pos_r[nb][1] = fu.kv_len - fu.q_len + (fu.row0 + 8 * nb + 2 * j4 + 1) / G;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) o[mt][nb][0] = o[mt][nb][1] = o[mt][nb][2] = o[mt][nb][3] = 0.f;
        }
        pos_min = fu.kv_len - fu.q_len + fu.row0 / G;
      }
      const bool last = (info.flags & F_LAST) != 0;

      if (info.flags & (F_BAD | F_INVALID)) {
        errored = 1;
      } else {
        const int tok0 = info.tile * C::kTile;
        const uint32_t sb = smem_u32(stages + stage * C::kStageBytes);
        const uint32_t vb = sb + C::kKBytes;
        const int first_tok = tok0 + tokw;
        // zero V rows past the sequence end (tail slots / rows never loaded)
        if (first_tok + 16 * MB - 1 >= kv_len) {
          uint8_t* vrows = stages + stage * C::kStageBytes + C::kKBytes;
          constexpr int kChunksPerRow = FP8 ? 8 : 16;
#pragma unroll
          for (int k = 0; k < 16 * MB * kChunksPerRow / 32; ++k) {
            const int q = lane + 32 * k;
            const int r = q / kChunksPerRow;
            const int c = q % kChunksPerRow;
            if (first_tok + r >= kv_len) {
              const int tok = tokw + r;
              uint8_t* dst = FP8 ? vrows + tok * 128 + c * 16
                                 : vrows + (c >> 3) * C::kHalfBytes + tok * 128 + (c & 7) * 16;
              *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
            }
          }
          fence_proxy_async();  // these generic writes precede later TMA writes to the stage
          __syncwarp();
        }

        // V fragments for this warp's keys, loaded ahead of the Q K^T chain so
        // that their latency overlaps it
        uint32_t vfrag[8][4];
        uint32_t vraw[MB][4][4];
        if (!FP8) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const int tok = tokw + (lane & 7) + ((lane >> 4) << 3);
            const int c = 2 * mt + ((lane >> 3) & 1);
            const uint32_t addr = vb + (c >> 3) * C::kHalfBytes + tok * 128 + ((((uint32_t)c & 7u) ^ (tok & swz)) << 4);
            ldsm_x4_t(addr, vfrag[mt][0], vfrag[mt][1], vfrag[mt][2], vfrag[mt][3]);
          }
        } else {
#pragma unroll
          for (int mb = 0; mb < MB; ++mb)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              const int tok = tokw + 16 * mb + j4 + 4 * rr;
              lds128(vb + tok * 128 + ((cv ^ (tok & swz)) << 4), vraw[mb][rr][0], vraw[mb][rr][1], vraw[mb][rr][2],
                     vraw[mb][rr][3]);
            }
        }

        // ---- S^T = K Q^T: 16 keys x 8*NB rows; with one n-block the k steps
        // alternate between two accumulators so two MMA chains are in flight
        constexpr int CH = NB == 1 ? 2 : 1;
        float sa[MB][NB][CH][4];
#pragma unroll
        for (int mb = 0; mb < MB; ++mb)
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int c = 0; c < CH; ++c)
#pragma unroll
              for (int k = 0; k < 4; ++k) sa[mb][nb][c][k] = 0.f;
        if (!FP8) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const int tok = tokw + (lane & 7) + (((lane >> 3) & 1) << 3);
            const uint32_t chunk = (uint32_t)(2 * (kk & 3) + (lane >> 4));
            const uint32_t addr = sb + (kk >> 2) * C::kHalfBytes + tok * 128 + ((chunk ^ (tok & swz)) << 4);
            uint32_t a[4];
            ldsm_x4(addr, a[0], a[1], a[2], a[3]);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_bf16(sa[0][nb][(kk & 1) % CH], a, qb[nb][kk][0], qb[nb][kk][1]);
          }
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t chunk = (uint32_t)(j4 + 4 * h);
            uint32_t w0[MB][4], w1[MB][4];
#pragma unroll
            for (int mb = 0; mb < MB; ++mb) {
              const int r0 = tokw + 16 * mb + tau0, r1 = tokw + 16 * mb + tau1;
              lds128(sb + r0 * 128 + ((chunk ^ (r0 & swz)) << 4), w0[mb][0], w0[mb][1], w0[mb][2], w0[mb][3]);
              lds128(sb + r1 * 128 + ((chunk ^ (r1 & swz)) << 4), w1[mb][0], w1[mb][1], w1[mb][2], w1[mb][3]);
            }
#pragma unroll
            for (int ss = 0; ss < 4; ++ss)
#pragma unroll
              for (int mb = 0; mb < MB; ++mb) {
                uint32_t a[4];
                e4m3x4_to_f16x2x2(w0[mb][ss], a[0], a[2]);
                e4m3x4_to_f16x2x2(w1[mb][ss], a[1], a[3]);
#pragma unroll
                for (int nb = 0; nb < NB; ++nb)
                  mma_f16(sa[mb][nb][h % CH], a, qb[nb][4 * h + ss][0], qb[nb][4 * h + ss][1]);
              }
          }
        }

        // ---- mask + online softmax (exp2 domain); rows are columns of S^T
        const bool need_mask = first_tok + 16 * MB - 1 > pos_min;
        float pv[MB][NB][2][2];
        float alpha[NB][2];
        bool rescale = false;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float mx = -INFINITY;
#pragma unroll
            for (int mb = 0; mb < MB; ++mb) {
              float x0 = (CH == 2 ? sa[mb][nb][0][e] + sa[mb][nb][CH - 1][e] : sa[mb][nb][0][e]) * scale2_item;
              float x1 = (CH == 2 ? sa[mb][nb][0][2 + e] + sa[mb][nb][CH - 1][2 + e] : sa[mb][nb][0][2 + e]) * scale2_item;
              if (need_mask) {
                if (first_tok + 16 * mb + tau0 > pos_r[nb][e]) x0 = -INFINITY;
                if (first_tok + 16 * mb + tau1 > pos_r[nb][e]) x1 = -INFINITY;
              }
              pv[mb][nb][e][0] = x0;
              pv[mb][nb][e][1] = x1;
              mx = fmaxf(mx, fmaxf(x0, x1));
            }
            mx = rowmax8(mx);
            const float m_new = fmaxf(m[nb][e], mx);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            alpha[nb][e] = fast_exp2(m[nb][e] - m_use);
            rescale |= alpha[nb][e] != 1.f;
            float sum = 0.f;
#pragma unroll
            for (int mb = 0; mb < MB; ++mb) {
              pv[mb][nb][e][0] = fast_exp2(pv[mb][nb][e][0] - m_use);
              pv[mb][nb][e][1] = fast_exp2(pv[mb][nb][e][1] - m_use);
              sum += pv[mb][nb][e][0] + pv[mb][nb][e][1];
            }
            l[nb][e] = l[nb][e] * alpha[nb][e] + sum;
            m[nb][e] = m_new;
          }
        }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              o[mt][nb][0] *= alpha[nb][0];
              o[mt][nb][1] *= alpha[nb][1];
              o[mt][nb][2] *= alpha[nb][0];
              o[mt][nb][3] *= alpha[nb][1];
            }
        }
        // P^T B fragments: movmatrix turns (key, row-pair) into (row, key-pair)
        uint32_t pb[MB][NB][2];
#pragma unroll
        for (int mb = 0; mb < MB; ++mb)
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            if (!FP8) {
              pb[mb][nb][0] = movmatrix_trans(pack_bf16(pv[mb][nb][0][0], pv[mb][nb][1][0]));
              pb[mb][nb][1] = movmatrix_trans(pack_bf16(pv[mb][nb][0][1], pv[mb][nb][1][1]));
            } else {
              pb[mb][nb][0] = movmatrix_trans(pack_f16(pv[mb][nb][0][0], pv[mb][nb][1][0]));
              pb[mb][nb][1] = movmatrix_trans(pack_f16(pv[mb][nb][0][1], pv[mb][nb][1][1]));
            }
          }

        // ---- O^T += V^T P^T
        if (!FP8) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_bf16(o[mt][nb], vfrag[mt], pb[0][nb][0], pb[0][nb][1]);
        } else {
          // keys j4, j4+4, j4+8, j4+12 of each 16-key slice; 16 channels 16 cv ..
#pragma unroll
          for (int mb = 0; mb < MB; ++mb)
#pragma unroll
          for (int qd = 0; qd < 4; ++qd) {
            uint32_t (&w)[4][4] = vraw[mb];
            const uint32_t t0w = prmt(w[0][qd], w[1][qd], 0x5140);
            const uint32_t t1w = prmt(w[0][qd], w[1][qd], 0x7362);
            const uint32_t t2w = prmt(w[2][qd], w[3][qd], 0x5140);
            const uint32_t t3w = prmt(w[2][qd], w[3][qd], 0x7362);
            uint32_t col[4];
            col[0] = prmt(t0w, t2w, 0x5410);
            col[1] = prmt(t0w, t2w, 0x7632);
            col[2] = prmt(t1w, t3w, 0x5410);
            col[3] = prmt(t1w, t3w, 0x7632);
#pragma unroll
            for (int hm = 0; hm < 2; ++hm) {
              const int mt = 2 * qd + hm;
              uint32_t a[4];
              e4m3x4_to_f16x2x2(col[2 * hm], a[0], a[2]);
              e4m3x4_to_f16x2x2(col[2 * hm + 1], a[1], a[3]);
#pragma unroll
              for (int nb = 0; nb < NB; ++nb) mma_f16(o[mt][nb], a, pb[mb][nb][0], pb[mb][nb][1]);
            }
          }
        }
      }
      __syncwarp();
      const uint32_t cur_stage = stage;
      if (!last && lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == (uint32_t)C::kStages) { stage = 0; phase ^= 1; }
      if (!last) continue;

      // ============================ epilogue ============================
      // The last stage (held until the epilogue ends) becomes two fp32
      // buffers of kRows x 128: warps 0/1 store their rescaled O^T, warps
      // 2/3 add theirs in place (same lanes, same elements), then every
      // thread sums the two buffers. Channel blocks of 8 are XOR-swizzled by
      // row so the fragment stores are bank-conflict free.
      float* obuf = reinterpret_cast<float*>(stages + cur_stage * C::kStageBytes);
      const ItemDesc& it = meta[s].it;   // valid until this slot is released below
      const UnitDesc& u = it.u;
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) l[nb][e] = rowsum8(l[nb][e]);
      if (g8 == 0) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            red_m[warp * 16 + 8 * nb + 2 * j4 + e] = m[nb][e];
            red_l[warp * 16 + 8 * nb + 2 * j4 + e] = l[nb][e];
          }
      }
      named_barrier(1, kNCW * 32);  // red arrays written; every warp is done reading the stage
      float sc[NB][2];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int row = 8 * nb + 2 * j4 + e;
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < kNCW; ++w) M = fmaxf(M, red_m[w * 16 + row]);
          sc[nb][e] = (m[nb][e] == -INFINITY) ? 0.f : fast_exp2(m[nb][e] - M);
        }
      // element (mt, nb, k) of O^T -> swizzled offset of (row, channel)
      auto obuf_index = [&](int mt, int nb, int k) {
        const int row = 8 * nb + 2 * j4 + (k & 1);
        const int ch = FP8 ? 16 * (int)cv + 2 * mt + (k >> 1) : 16 * mt + g8 + 8 * (k >> 1);
        return row * kD + (ch ^ (((row >> 1) & 3) << 3));
      };
      float* mybuf = obuf + (warp & 1) * kRows * kD;
      if (warp < 2) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int k = 0; k < 4; ++k) mybuf[obuf_index(mt, nb, k)] = o[mt][nb][k] * sc[nb][k & 1];
      }
      named_barrier(1, kNCW * 32);
      if (warp >= 2) {
        // each group's partial sums are read before any of its stores: a read
        // placed after a store the compiler cannot tell apart waits for it
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          float prev[NB][4];
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int k = 0; k < 4; ++k) prev[nb][k] = mybuf[obuf_index(mt, nb, k)];
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int k = 0; k < 4; ++k) mybuf[obuf_index(mt, nb, k)] = prev[nb][k] + o[mt][nb][k] * sc[nb][k & 1];
        }
      }
      named_barrier(1, kNCW * 32);

      constexpr int kTpr = 128 / kRows;    // threads per row
      constexpr int kCpt = kD / kTpr;      // channels per thread (8 or 16)
      const int t = threadIdx.x;           // 0..127
      const int row = t / kTpr;
      const int c0 = (t % kTpr) * kCpt;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kNCW; ++w) M = fmaxf(M, red_m[w * 16 + row]);
      float Ls = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kNCW; ++w) {
          const float mw = red_m[w * 16 + row];
          if (mw != -INFINITY) Ls += red_l[w * 16 + row] * fast_exp2(mw - M);
        }
      }
      float acc[kCpt];
#pragma unroll
      for (int k = 0; k < kCpt; k += 8) {
        const int off = row * kD + ((c0 + k) ^ (((row >> 1) & 3) << 3));
        const float4 a0 = *reinterpret_cast<const float4*>(obuf + off);
        const float4 a1 = *reinterpret_cast<const float4*>(obuf + off + 4);
        const float4 b0 = *reinterpret_cast<const float4*>(obuf + kRows * kD + off);
        const float4 b1 = *reinterpret_cast<const float4*>(obuf + kRows * kD + off + 4);
        acc[k] = a0.x + b0.x;
        acc[k + 1] = a0.y + b0.y;
        acc[k + 2] = a0.z + b0.z;
        acc[k + 3] = a0.w + b0.w;
        acc[k + 4] = a1.x + b1.x;
        acc[k + 5] = a1.y + b1.y;
        acc[k + 6] = a1.z + b1.z;
        acc[k + 7] = a1.w + b1.w;
      }
      const float inv = Ls > 0.f ? vscale / Ls : 0.f;
      const bool valid_row = row < u.nrows;
      const int pr_ = u.row0 + row;
      const int qi = pr_ / G;
      const int head = u.g * G + (pr_ - qi * G);
      const size_t out_row = (size_t)(u.q_start + qi) * p.num_q_heads + head;
      const bool lse_lane = (t % kTpr) == 0;

      if (u.n_splits == 1) {
        if (valid_row) {
          // the row's state is final: fold in its sink, if any
          const float s2 = sink_log2(p.sinks, head);
          const float Mt = fmaxf(M, s2);
          const float a = M == -INFINITY ? 0.f : fast_exp2(M - Mt);
          const float Lt = Ls * a + (s2 == -INFINITY ? 0.f : fast_exp2(s2 - Mt));
          const float sc = Lt > 0.f ? vscale * a / Lt : 0.f;
          uint32_t packed[kCpt / 2];
#pragma unroll
          for (int k = 0; k < kCpt / 2; ++k)
            packed[k] = errored ? 0u : pack_bf16(acc[2 * k] * sc, acc[2 * k + 1] * sc);
          uint4* dst = reinterpret_cast<uint4*>(p.out + out_row * kD + c0);
#pragma unroll
          for (int k = 0; k < kCpt / 8; ++k)
            dst[k] = make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]);
          if (p.lse != nullptr && lse_lane)
            p.lse[out_row] = errored ? NAN : (Lt > 0.f ? (Mt + __log2f(Lt)) * kLn2 : -INFINITY);
        }
      } else {
        const size_t prow = (size_t)u.partial_base + (size_t)it.split * u.nrows + row;
        if (valid_row) {
          float* dst = p.po + prow * kD + c0;
#pragma unroll
          for (int k = 0; k < kCpt; k += 4)
            *reinterpret_cast<float4*>(dst + k) = make_float4(acc[k] * inv, acc[k + 1] * inv, acc[k + 2] * inv, acc[k + 3] * inv);
          if (lse_lane) p.plse[prow] = errored ? NAN : (Ls > 0.f ? M + __log2f(Ls) : -INFINITY);
        }
      }
      fence_proxy_async();          // merge-buffer writes precede the next TMA into this stage
      named_barrier(1, kNCW * 32);  // every warp is done with the merge buffer and red arrays
      if (lane == 0) {
        mbar_arrive(&empty[cur_stage]);
        mbar_arrive(&slot_empty[s]);
      }
      if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
    }
  }

  // ---- leave the queue; the last CTA out resets it for the next launch
  __syncthreads();
  if (threadIdx.x == 0 && s_flag[1]) {
    __threadfence();
    if (atomicAdd(&hdr->done_counter, 1u) == gridDim.x - 1) {
      hdr->queue_counter = 0u;
      hdr->done_counter = 0u;
      __threadfence();
    }
  }
}

}  // namespace

template <bool FP8, int NB>
static cudaError_t launch_impl(const CUtensorMap& kmap, const CUtensorMap& vmap, const GqaParams& p,
                               int grid, cudaStream_t stream) {
  using C = Cfg<FP8, NB>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(gqa_decode_kernel<FP8, NB>), C::kSmemBytes);
  if (e != cudaSuccess) return e;
  gqa_decode_kernel<FP8, NB><<<grid, kThreads, C::kSmemBytes, stream>>>(kmap, vmap, p);
  return cudaGetLastError();
}

cudaError_t launch_gqa_decode(const CUtensorMap& kmap, const CUtensorMap& vmap, const GqaParams& p,
                              bool fp8, int rows_per_unit, int grid, cudaStream_t stream) {
  if (rows_per_unit <= 8)
    return fp8 ? launch_impl<true, 1>(kmap, vmap, p, grid, stream) : launch_impl<false, 1>(kmap, vmap, p, grid, stream);
  return fp8 ? launch_impl<true, 2>(kmap, vmap, p, grid, stream) : launch_impl<false, 2>(kmap, vmap, p, grid, stream);
}

}  // namespace pd
