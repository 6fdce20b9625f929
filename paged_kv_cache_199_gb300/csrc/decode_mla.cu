// Paged MLA decode attention for sm_103a on the 5th-generation tensor cores:
// every query head attends over one shared latent KV head.
//
// What it computes: PR #4557 ("feat(cake_mla): add generated Blackwell
// TRT-LLM MLA decode backend") calls trtllm_batch_decode_with_kv_cache_mla
// over a paged latent cache whose row is 512 latent + 64 rope channels
// (PR #5552, "Kimi-K3 FP8 latent MLA"): the key is the whole 576-channel row
// and the value its first 512 channels; query rows are packed (token, head)
// pairs; the causal bound is inclusive (PR #4557 review "Exclusive causal
// bound drops the newest key").
//
// Design:
//  * one persistent CTA per SM; a unit is 64 packed query rows of one
//    request; its keys are cut into 64-token tiles;
//  * scheduler warp 8 pops items (or walks the CTA's static range), checks
//    the device metadata, prefetches page ids and TMA-loads the unit's
//    64 x 576 query block (nine 128-byte swizzled slabs); it also counts
//    split arrivals and queues the unit merge on the last one;
//  * producer warp 5 TMA-loads each 64 x 576 key tile (nine swizzled slabs,
//    two stages of 72 KB); values are the first eight slabs of the same tile;
//  * four threads issue the tcgen05 MMAs, two for S and two for O: one
//    thread issues at most one MMA per 64-76 cycles whatever its shape,
//    while the tensor core takes an M = 64, N = 64 MMA every 32 cycles when
//    more than one thread feeds it, and every stage waits for its S and its O
//    before it is refilled. Per tile, S = Q K^T is 36 MMAs of M = 64 rows,
//    N = 64 keys, K = 16: warp 4 issues the first 18 K steps into one
//    accumulator of the tile's tensor-memory S buffer, warp 6 the other 18
//    into a second (the softmax adds them). O^T += V^T P^T is 16 MMAs of
//    M = 128 latent channels, N = 64 rows, K = 16 keys: warp 7 accumulates
//    channel blocks 0-1, warp 9 blocks 2-3. V^T is the key tile read
//    MN-major, P^T the bf16 probabilities in shared memory. O^T (512 channels
//    x 64 rows, fp32) lives in tensor memory on all 128 lanes. S of tile t+1
//    is issued while the softmax of tile t runs; a stage is released when
//    the S and the O MMAs that read it are done;
//  * softmax warps 0-3 read S rows from tensor memory (row 16 w + i is lane
//    32 w + i), mask the causal tail, keep a running maximum that only moves
//    when a tile raises it by more than 2^8 (otherwise P stays below 256 and
//    nothing is rescaled), rescale O^T in tensor memory when it does, write
//    P (bf16, swizzled) for the O issuer, and run the epilogue and the
//    split merges.
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
constexpr int kRows = 64;            // packed query rows per unit
constexpr int kSoftWarps = 4;        // softmax / epilogue / merge warps 0..3
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kMmaWarp = 4;
constexpr int kProducerWarp = 5;
constexpr int kSchedulerWarp = 8;
constexpr int kOWarp = 7;
// The second S issuer on SM sub-partition 2 (warp w runs on sub-partition
// w mod 4): with both S issuers on sub-partition 0 beside softmax warp 0 and
// the scheduler alone beside softmax warp 2, mla1 measured 815-817 us against
// 809 (the kernel misses ~13 % of its instruction-cache requests)
constexpr int kMmaWarp2 = 6;         // the second S issuer
constexpr int kOWarp2 = 9;           // the second O issuer
constexpr int kSIssuers = 2;         // threads issuing S MMAs; with the O issuers, each releases every stage
constexpr int kThreads = 10 * 32;
constexpr int kSlots = 2;
constexpr int kWin = 64;             // page ids prefetched per item
constexpr int kSlabBytes = kTile * 128;                 // 8 KB: 64 rows of 128 bytes
constexpr int kPBytes = kRows * 128;                    // P: one 128-byte row per query row
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kGrowThreshold = 8.f;                   // log2 units
// tensor memory: two S buffers, each the sum of two accumulators (M = 64
// layout, 64 columns each; buffer b, accumulator a at 64 (2 b + a)), and O^T
// as four 64-column blocks of 128 channels
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;

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

// Per element type. A 576-channel row is cut into 128-byte slabs: nine for
// BF16, five for E4M3 (the fifth holds channels 512..575 and 64 zero bytes
// that TMA fills past the row end). Every MMA reads 32 bytes of a row: 16
// BF16 channels (kind::f16) or 32 E4M3 channels (kind::f8f6f4).
template <bool FP8>
struct MlaCfg {
  static constexpr int kElem = FP8 ? 1 : 2;
  static constexpr int kSlabs = FP8 ? 5 : 9;
  static constexpr int kSSteps = kDqk * kElem / 32;          // K steps of S: 36 or 18
  static constexpr int kVSlabsPerBlock = 128 * kElem / 128;  // slabs of a 128-channel block of V
  static constexpr int kVSlabs = 4 * kVSlabsPerBlock;        // slabs holding V (channels 0..511)
  static constexpr int kPVSteps = kTile * kElem / 32;        // K steps of O over one tile: 4 or 2
  static constexpr int kPVStepBytes = (32 / kElem) * 128;    // bytes of V rows per K step
  static constexpr int kStages = FP8 ? 4 : 2;   // 40 or 72 KB each
  // P buffers: E4M3 has room for two, so the softmax of tile t+1 writes one
  // while the O MMAs of tile t still read the other; with the one BF16 buffer
  // the softmax of t+1 waits for those MMAs before it writes
  static constexpr int kPBufs = FP8 ? 2 : 1;
  // How the two S issuers share the work. BF16 (two stages): each tile's S is
  // split over the K steps into two accumulators, which the softmax adds, so
  // that every stage gets its S in half the time. E4M3 (four stages): the
  // issuers take alternate stages whole; one accumulator per tile keeps the
  // softmax, which bounds that instance, at one tensor-memory read per tile.
  static constexpr bool kSplitK = !FP8;
  // O issuers: BF16 splits the four 128-channel blocks of O^T over two
  // threads; E4M3 (8 O MMAs a tile) measured faster with one.
  static constexpr int kOIssuers = FP8 ? 1 : 2;
  static constexpr int kStageBytes = kSlabs * kSlabBytes;    // 72 or 40 KB
  static constexpr int kQBytes = kSlabs * kRows * 128;       // 72 or 40 KB
  static constexpr uint32_t kIdescS = FP8 ? umma_idesc_e4m3(64, 64, 0, 0) : umma_idesc_bf16(64, 64, 0, 0);
  static constexpr uint32_t kIdescO = FP8 ? umma_idesc_e4m3(128, 64, 1, 0) : umma_idesc_bf16(128, 64, 1, 0);
  static constexpr int kOffStages = 0;
  static constexpr int kOffQ = kOffStages + kStages * kStageBytes;
  static constexpr int kOffP = kOffQ + kQBytes;
  static constexpr int kOffMeta = kOffP + kPBufs * kPBytes;
  static constexpr int kOffRed = kOffMeta + kSlots * (int)sizeof(SlotMeta);
  static constexpr int kOffInfo = kOffRed + 2 * kRows * 4 + 16;
  static constexpr int kOffBars = kOffInfo + kStages * (int)sizeof(StageInfo);
  static constexpr int kNumBars = 2 * kStages + 16;
  static constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kStages % 2 == 0, "the S buffer follows the stage's parity");
  static_assert(kSSteps % 2 == 0, "split over K, the two S issuers take half of the K steps each");
  static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");
};

template <bool FP8>
__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if constexpr (FP8)
    umma_e4m3(d, a, b, idesc, acc);
  else
    umma_bf16(d, a, b, idesc, acc);
}

// MERGE task: combine the split states of one 64-row unit (128 threads).
__device__ __noinline__ void mla_merge_unit(const MlaParams& p, const UnitDesc u) {
  const int t = threadIdx.x;   // 0..127
  const int row = t >> 1;      // 64 rows, two threads each
  const int cbase = (t & 1) * 256;
  if (row >= u.nrows) return;
  const size_t base = (size_t)u.partial_base + row;
  const int ns = u.n_splits;
  float ls[kMaxSplits];
#pragma unroll
  for (int k = 0; k < kMaxSplits; ++k) ls[k] = k < ns ? ld_cg(p.plse + base + (size_t)k * u.nrows) : -INFINITY;
  const float s2 = sink_log2(p.sinks, (u.row0 + row) % p.num_heads);
  float Mx = s2;
  bool bad = false;
#pragma unroll
  for (int k = 0; k < kMaxSplits; ++k) {
    bad |= isnan(ls[k]);
    Mx = fmaxf(Mx, ls[k]);
  }
  float w[kMaxSplits];
  float W = (bad || s2 == -INFINITY) ? 0.f : fast_exp2(s2 - Mx);
#pragma unroll
  for (int k = 0; k < kMaxSplits; ++k) {
    w[k] = (bad || ls[k] == -INFINITY || Mx == -INFINITY) ? 0.f : fast_exp2(ls[k] - Mx);
    W += w[k];
  }
  const float winv = W > 0.f ? 1.f / W : 0.f;
  const size_t out_row = (size_t)u.q_start * p.num_heads + u.row0 + row;
  for (int c = cbase; c < cbase + 256; c += 8) {
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
  if (p.lse != nullptr && (t & 1) == 0)
    p.lse[out_row] = bad ? NAN : (W > 0.f ? (Mx + __log2f(W)) * kLn2 : -INFINITY);
}

__device__ __forceinline__ uint32_t swz(int row, int chunk) { return (uint32_t)((chunk ^ (row & 7)) << 4); }

template <bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
                      const MlaParams p) {
  using C = MlaCfg<FP8>;
  constexpr int kStages = C::kStages;
  constexpr int kSlabs = C::kSlabs;
  constexpr int kStageBytes = C::kStageBytes;
  constexpr int kOffStages = C::kOffStages, kOffQ = C::kOffQ, kOffP = C::kOffP, kOffMeta = C::kOffMeta;
  constexpr int kOffRed = C::kOffRed, kOffInfo = C::kOffInfo, kOffBars = C::kOffBars;
  constexpr int kChanPerSlab = 128 / C::kElem;   // TMA x coordinate step of one slab
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem + kOffStages;
  uint8_t* qbuf = smem + kOffQ;
  uint8_t* pbuf = smem + kOffP;
  SlotMeta* meta = reinterpret_cast<SlotMeta*>(smem + kOffMeta);
  float* red_a = reinterpret_cast<float*>(smem + kOffRed);  // [64] per-row O rescale factors
  float* red_l = red_a + kRows;                              // [64] per-row 1 / l
  int* s_flag = reinterpret_cast<int*>(red_l + kRows);
  StageInfo* sinfo = reinterpret_cast<StageInfo*>(smem + kOffInfo);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* empty = full + kStages;          // each issuer (commit or arrive) + 4 softmax warps
  uint64_t* slot_full = empty + kStages;
  uint64_t* slot_empty = slot_full + kSlots;
  uint64_t* q_full = slot_empty + kSlots;    // the query block landed
  uint64_t* q_empty = q_full + 1;            // the last S of the item read it
  uint64_t* s_full = q_empty + 1;            // [2] S computed
  uint64_t* s_empty = s_full + 2;            // [2] S read back by the softmax warps
  // one full/empty pair per P buffer: with two buffers the softmax may write
  // two tiles before the O issuer looks, and one shared barrier would then
  // complete two phases and hide the first from the issuer's parity wait
  uint64_t* p_full = s_empty + 2;            // [2] P buffer b written (and O^T rescaled)
  uint64_t* p_empty = p_full + 2;            // [2] the O MMAs that read P buffer b are done
  uint64_t* o_empty = p_empty + 2;           // the epilogue read O^T
  uint64_t* mma_done = o_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  WsHeader* hdr = p.hdr;
  const int H = p.num_heads;

  if (threadIdx.x == 0) {
    s_flag[1] = 1;  // cleared by the scheduler if the workspace holds another plan
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSIssuers + C::kOIssuers + kSoftWarps);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&slot_full[s], 1);
      mbar_init(&slot_empty[s], kSoftWarps);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 2);   // both S issuers are done with the item's query block
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 2);   // both S issuers' MMAs done
      mbar_init(&s_empty[b], kSoftWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&p_full[b], kSoftWarps);
      mbar_init(&p_empty[b], C::kOIssuers);   // the O MMAs that read buffer b done
    }
    mbar_init(o_empty, kSoftWarps);
    mbar_init(mma_done, kSIssuers + C::kOIssuers);
    fence_barrier_init();
    fence_proxy_async();
  }
  __syncthreads();
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int P = p.page_size;
  const int BR = p.box_rows;

  if (warp == kSchedulerWarp) {
    // ============================== scheduler ==============================
    uint32_t s = 0, sph = 0;
    uint32_t qph = 0;       // q_empty phase (one per work item)
    bool q_loaded = false;  // the latest q_full phase carries copies of this warp
    bool dead = false, exhausted = false, first_pop = true;
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
    }
    plan_ok = __shfl_sync(0xffffffffu, plan_ok, 0);
    int used[kSlots], split_unit[kSlots], split_n[kSlots];
#pragma unroll
    for (int k = 0; k < kSlots; ++k) used[k] = 0, split_unit[k] = -1, split_n[k] = 0;
    bool took_first = false;
    while (plan_ok) {
      int merge_unit = -1;
      if (!mbar_wait(&slot_empty[s], sph ^ 1, p.wait_ns)) { dead = true; break; }
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
          took_first = true;
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
      const int tok_first = it.tile_begin * kTile;
      const int tok_end = min(it.tile_end * kTile, u.kv_len);
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
      if (lane == 0) mbar_arrive(&slot_full[s]);
      // the query block has one buffer: wait until the previous item is done with it
      if (!mbar_wait(q_empty, qph ^ 1, p.wait_ns)) { dead = true; break; }
      qph ^= 1;
      q_loaded = err == 0;
      if (lane == 0) {
        if (err) {
          mbar_arrive(q_full);
        } else {
          mbar_arrive_expect_tx(q_full, (uint32_t)C::kQBytes);
          const int grow = u.q_start * H + u.row0;   // packed (token, head) rows are contiguous
          for (int c = 0; c < kSlabs; ++c)
            tma_load_4d(qbuf + c * kRows * 128, &q_map, kChanPerSlab * c, grow, 0, 0, q_full,
                        l2_evict_last_policy());
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
    // the query copies of the last item land before the CTA exits (its phase
    // is the latest one of q_full, parity qph ^ 1)
    if (q_loaded && lane == 0) mbar_wait(q_full, qph ^ 1, kDrainLimitNs);
  } else if (warp == kMmaWarp || warp == kMmaWarp2) {
    // ================================ S issue ================================
    // One thread cannot issue tcgen05.mma faster than about one per 64-76
    // cycles whatever the shape, while the tensor core takes an M = 64,
    // N = 64 MMA every 32 cycles when more than one thread feeds it; and each
    // stage waits for its S before the softmax, P and O can follow. So every
    // tile's S is issued by two threads at once: the one of warp kMmaWarp runs
    // the first half of the K steps into accumulator 0 of the tile's S
    // buffer, the one of warp kMmaWarp2 the second half into accumulator 1;
    // the softmax adds the two.
    if (lane == 0) {
      const uint32_t me = warp == kMmaWarp ? 0u : 1u;
      constexpr int kHalf = C::kSSteps / 2;
      const uint32_t qaddr = smem_u32(qbuf), kaddr0 = smem_u32(stages);
      uint32_t stage = 0, phase = 0, qph = 0;
      uint32_t sph[2] = {0u, 0u};
      bool dead = false;
      while (true) {
        if (!mbar_wait(&full[stage], phase, p.wait_ns)) { dead = true; break; }
        const int f = sinfo[stage].flags;
        if (f & F_END) break;
        const bool ctrl = (f & (F_MERGE | F_NOP)) != 0;
        if (!ctrl && (f & F_FIRST)) {
          if (!mbar_wait(q_full, qph, p.wait_ns)) { dead = true; break; }
          qph ^= 1;
        }
        const bool mine = C::kSplitK || (stage & 1u) == me;   // alternate stages: the owner's alone
        if (!mine) {
          if (!ctrl && (f & F_LAST)) umma_commit(q_empty);
        } else if (ctrl || (f & (F_BAD | F_INVALID))) {
          mbar_arrive(&empty[stage]);
          if (!C::kSplitK) mbar_arrive(&empty[stage]);   // for the other S issuer too
          if (!ctrl && (f & F_LAST)) umma_commit(q_empty);
        } else {
          // S = Q K^T into buffer (stage & 1); the stage is released for this
          // issuer when its MMAs are done (the O issuers release it for V)
          const uint32_t sbuf = stage & 1u;
          if (!mbar_wait(&s_empty[sbuf], sph[sbuf] ^ 1, p.wait_ns)) { dead = true; break; }
          sph[sbuf] ^= 1;
          tc_fence_after();
          const uint64_t qdesc = umma_desc_sw128(qaddr, 16, 1024);
          const uint64_t kdesc = umma_desc_sw128(kaddr0 + stage * kStageBytes, 16, 1024);
          if constexpr (C::kSplitK) {
#pragma unroll
            for (int h = 0; h < kHalf; ++h) {
              const int ks = (int)me * kHalf + h;
              const uint64_t off = (uint64_t)(((ks >> 2) * kSlabBytes + (ks & 3) * 32) >> 4);
              umma<FP8>(tmem + kColS + 64 * (2 * sbuf + me), qdesc + off, kdesc + off, C::kIdescS, h > 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int ks = 0; ks < C::kSSteps; ++ks) {
              const uint64_t off = (uint64_t)(((ks >> 2) * kSlabBytes + (ks & 3) * 32) >> 4);
              umma<FP8>(tmem + kColS + 64 * 2 * sbuf, qdesc + off, kdesc + off, C::kIdescS, ks > 0 ? 1u : 0u);
            }
          }
          umma_commit(&s_full[sbuf]);
          umma_commit(&empty[stage]);
          if (!C::kSplitK) {
            umma_commit(&s_full[sbuf]);    // the counts expect both S issuers
            umma_commit(&empty[stage]);
          }
          if (f & F_LAST) umma_commit(q_empty);
        }
        if (++stage == (uint32_t)kStages) { stage = 0; phase ^= 1; }
      }
      if (dead) set_error(hdr, PD_DEV_TIMEOUT, -1);
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, kDrainLimitNs);
    }
  } else if (warp == kOWarp || (warp == kOWarp2 && C::kOIssuers == 2)) {
    // ================================ O issue ================================
    // Two threads, as for S: the one of warp kOWarp accumulates channel
    // blocks 0 and 1 of O^T, the one of warp kOWarp2 blocks 2 and 3.
    if (lane == 0) {
      constexpr int kBlocks = 4 / C::kOIssuers;   // O^T channel blocks of this issuer
      const int c0 = warp == kOWarp ? 0 : kBlocks;
      const uint32_t paddr = smem_u32(pbuf), kaddr0 = smem_u32(stages);
      uint32_t stage = 0, phase = 0, oph = 0, pv_issued = 0;
      bool dead = false, o_wait = false, first_pv = false;
      while (true) {
        if (!mbar_wait(&full[stage], phase, p.wait_ns)) { dead = true; break; }
        const int f = sinfo[stage].flags;
        if (f & F_END) break;
        const bool ctrl = (f & (F_MERGE | F_NOP)) != 0;
        if (!ctrl && (f & F_FIRST)) {
          o_wait = true;   // the item's first O MMA waits for the epilogue of the last item that had one
          first_pv = true;
        }
        if (ctrl || (f & (F_BAD | F_INVALID))) {
          mbar_arrive(&empty[stage]);
        } else {
          // O^T += V^T P^T once the softmax wrote P of this tile
          const uint32_t pb = pv_issued % C::kPBufs;
          if (!mbar_wait(&p_full[pb], (pv_issued / C::kPBufs) & 1u, p.wait_ns)) { dead = true; break; }
          if (o_wait) {
            if (!mbar_wait(o_empty, oph ^ 1, p.wait_ns)) { dead = true; break; }
            oph ^= 1;
            o_wait = false;
          }
          tc_fence_after();
          const uint32_t vbase = kaddr0 + stage * kStageBytes;
#pragma unroll
          for (int kk = 0; kk < C::kPVSteps; ++kk) {
            const uint64_t bdesc = umma_desc_sw128(paddr + pb * kPBytes + kk * 32, 16, 1024);
#pragma unroll
            for (int c = c0; c < c0 + kBlocks; ++c) {
              const uint64_t adesc = umma_desc_sw128(vbase + C::kVSlabsPerBlock * c * kSlabBytes + kk * C::kPVStepBytes,
                                                     kSlabBytes, 1024);
              umma<FP8>(tmem + kColO + 64 * c, adesc, bdesc, C::kIdescO, (first_pv && kk == 0) ? 0u : 1u);
            }
          }
          umma_commit(&empty[stage]);
          umma_commit(&p_empty[pb]);
          ++pv_issued;
          first_pv = false;
        }
        if (++stage == (uint32_t)kStages) { stage = 0; phase ^= 1; }
      }
      if (dead) set_error(hdr, PD_DEV_TIMEOUT, -1);
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, kDrainLimitNs);
    }
  } else if (warp == kProducerWarp) {
    // ============================== producer ==============================
    prefetch_tensormap(&kv_map);
    // the sibling row blocks of a request read the same tiles: keep them in L2
    const uint64_t pol = l2_evict_normal_policy();
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
        const int f = kind == T_MERGE ? F_MERGE : kind == T_NOP ? F_NOP : F_INVALID;
        if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns)) { dead = true; break; }
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
            mbar_arrive_expect_tx(&full[stage], (uint32_t)nbox * BR * 128 * kSlabs);
          }
          uint8_t* dst = stages + stage * kStageBytes;
          for (int j = 0; j < nbox; ++j) {
            const int page = __shfl_sync(0xffffffffu, j < 32 ? pg0 : pg1, j & 31);
            if (lane == 0) {
              const int slot = (tok0 + j * BR) % P;
              for (int c = 0; c < kSlabs; ++c)
                tma_load_4d(dst + c * kSlabBytes + j * BR * 128, &kv_map, kChanPerSlab * c, 0, slot, page,
                            &full[stage], pol);
            }
          }
          // BF16 whole-page tiles: bring the tile that refills this stage next
          // (one ring cycle ahead) into L2 with one untiled bulk prefetch, so
          // that the refill of the two-stage ring waits for L2 rather than
          // HBM (measured 926 -> 907 us at 512 x 4096; the four-stage E4M3
          // ring measured slower with it, and per-slab tensor prefetches
          // slower still)
          if (!FP8 && P == kTile && t + kStages < it.tile_end) {
            const int pi = (t + kStages) * kTile / P - win0;
            int pnext = 0;
            if (lane == 0) {
              pnext = pi < nwin ? m.pages[pi] : __ldg(trow + win0 + pi);
              if (pnext >= 0 && pnext < p.num_pages) {
                const uint8_t* src = p.kv_pool + (size_t)pnext * (size_t)p.page_bytes;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"((uint32_t)(kTile * kDqk * C::kElem))
                             : "memory");
              }
            }
          }
        }
        if (++stage == (uint32_t)kStages) { stage = 0; phase ^= 1; }
      }
      if (dead) break;
      if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
    }
    if (!dead && mbar_wait(&empty[stage], phase ^ 1, p.wait_ns)) {
      if (lane == 0) {
        sinfo[stage] = StageInfo{-1, 0, F_END, 0};
        mbar_arrive(&full[stage]);
      }
      if (++stage == (uint32_t)kStages) { stage = 0; phase ^= 1; }
    } else {
      dead = true;
    }
    if (dead && lane == 0) set_error(hdr, PD_DEV_TIMEOUT, -1);
    // the copies this warp put in flight land before the CTA exits (on the
    // normal path they have, and these waits return at once)
    drain_ring(full, kStages, stage, phase);
  } else if (warp < kSoftWarps) {
    // ============================== softmax / epilogue ==============================
    const int w = warp;                // tensor-memory lane quarter
    const int r = 16 * w + (lane & 15);  // the S row of this thread
    const int kh = lane >> 4;            // its key half of each tile
    const bool row_thread = lane < 16;   // writes the row's statistics
    const uint32_t tq = tmem + ((uint32_t)(32 * w) << 16);
    // E4M3: logits carry q_scale * kv_scale, values kv_scale
    const float qk_scale = FP8 ? __ldg(p.q_scale) * __ldg(p.kv_scale) : 1.f;
    const float v_scale = FP8 ? __ldg(p.kv_scale) : 1.f;
    const float scale2 = p.sm_scale * qk_scale * kLog2e;
    uint32_t stage = 0, phase = 0, s = 0, sph = 0, pv_count = 0;
    uint32_t sfph[2] = {0u, 0u};
    bool item_pv = false;
    float m = -INFINITY, l = 0.f;
    int errored = 0, kv_len = 0, pos = 0;
    bool dead = false;

    while (true) {
      if (!mbar_wait(&full[stage], phase, p.wait_ns)) { dead = true; break; }
      const StageInfo info = sinfo[stage];
      if (info.flags & F_END) break;
      if (info.flags & (F_MERGE | F_NOP)) {
        if (!mbar_wait(&slot_full[s], sph, p.wait_ns)) { dead = true; break; }
        if (info.flags & F_MERGE) mla_merge_unit(p, meta[s].it.u);
        named_barrier(1, kSoftThreads);
        if (lane == 0) {
          mbar_arrive(&empty[stage]);
          mbar_arrive(&slot_empty[s]);
        }
        if (++stage == (uint32_t)kStages) { stage = 0; phase ^= 1; }
        if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
        continue;
      }
      if (info.flags & F_FIRST) {
        if (!mbar_wait(&slot_full[s], sph, p.wait_ns)) { dead = true; break; }
        const UnitDesc& fu = meta[s].it.u;
        kv_len = fu.kv_len;
        errored = (info.flags & F_INVALID) ? 1 : 0;
        pos = fu.kv_len - fu.q_len + (fu.row0 + r) / H;
        m = -INFINITY;
        l = 0.f;
        item_pv = false;
      }
      const bool last = (info.flags & F_LAST) != 0;

      if (info.flags & (F_BAD | F_INVALID)) {
        errored = 1;
        if (lane == 0) mbar_arrive(&empty[stage]);
      } else {
        // ---- S rows of this tile from tensor memory
        const uint32_t sbuf = stage & 1u;   // the S buffer of this stage's S issuer
        if (!mbar_wait(&s_full[sbuf], sfph[sbuf], p.wait_ns)) { dead = true; break; }
        sfph[sbuf] ^= 1;
        tc_fence_after();
        uint32_t sr[32], sr2[32];   // the two accumulators of S (one with alternate stages)
        tmem_ld_16x32bx2_x32(tq + kColS + 128 * sbuf, sr);
        if constexpr (C::kSplitK) tmem_ld_16x32bx2_x32(tq + kColS + 128 * sbuf + 64, sr2);
        tmem_wait_ld(sr);
        if constexpr (C::kSplitK) tmem_wait_ld(sr2);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[sbuf]);

        // ---- value rows past the sequence end are zero (0 * stale data must stay 0)
        const int tok0 = info.tile * kTile;
        uint8_t* st = stages + stage * kStageBytes;
        if (tok0 + kTile > kv_len) {
          const int t = threadIdx.x;  // 0..127: key row t / 2, half of the value slabs each
          const int kr = t >> 1;
          constexpr int kHalf = C::kVSlabs / 2;
          if (tok0 + kr >= kv_len) {
#pragma unroll
            for (int c = kHalf * (t & 1); c < kHalf * (t & 1) + kHalf; ++c)
#pragma unroll
              for (int k = 0; k < 8; ++k)
                *reinterpret_cast<uint4*>(st + c * kSlabBytes + kr * 128 + k * 16) = make_uint4(0, 0, 0, 0);
          }
        }

        // ---- masked, scaled scores (keys 32 kh .. +32 of row r); running
        // maximum with the growth threshold, shared by the two half-warps
        // (the two accumulators' sum and the scaling run on packed pairs)
        float x[32];
        const int key0 = tok0 + 32 * kh;
        const bool need_mask = key0 + 31 > pos;
        const uint64_t scale_2 = f2pack(scale2, scale2);
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          uint64_t a = f2pack(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1]));
          if constexpr (C::kSplitK) a = f2add(a, f2pack(__uint_as_float(sr2[k]), __uint_as_float(sr2[k + 1])));
          f2unpack(f2mul(a, scale_2), x[k], x[k + 1]);
        }
        if (need_mask) {
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (key0 + k > pos) x[k] = -INFINITY;
        }
        float mt = -INFINITY, mt1 = -INFINITY;
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          mt = fmax3(mt, x[k], x[k + 1]);
          mt1 = fmax3(mt1, x[k + 2], x[k + 3]);
        }
        mt = fmaxf(mt, mt1);
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
        float alpha = 1.f;
        const bool grow = mt > m + kGrowThreshold;
        if (grow) {
          alpha = m == -INFINITY ? 0.f : fast_exp2(m - mt);
          m = mt;
        }
        const float mu = m == -INFINITY ? 0.f : m;
        // P of keys 32 kh .. +32 as the MMA will read it: BF16 (16 words) or
        // E4M3 (8 words, P <= 2^8 fits), and the row sum
        uint32_t pk[16];
        float sum = 0.f;
        if constexpr (!FP8) {
          // the row sum is taken in fp32 before the bf16 rounding of P (each
          // value within 2^-9 of the one the MMA reads; the E4M3 branch below
          // sums the codes themselves, whose rounding is 2^-4)
          const uint64_t nmu_2 = f2pack(-mu, -mu);
          uint64_t sum_2 = f2pack(0.f, 0.f);   // even and odd keys apart
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            float t0, t1;
            f2unpack(f2add(f2pack(x[2 * k], x[2 * k + 1]), nmu_2), t0, t1);
            const float p0 = fast_exp2(t0), p1 = fast_exp2(t1);
            pk[k] = pack_bf16(p0, p1);
            sum_2 = f2add(sum_2, f2pack(p0, p1));
          }
          float s0, s1;
          f2unpack(sum_2, s0, s1);
          sum = s0 + s1;
        } else {
          __half2 hs = __float2half2_rn(0.f);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t lo = pack_e4m3x2(fast_exp2(x[4 * k] - mu), fast_exp2(x[4 * k + 1] - mu));
            const uint32_t hi = pack_e4m3x2(fast_exp2(x[4 * k + 2] - mu), fast_exp2(x[4 * k + 3] - mu));
            pk[k] = lo | (hi << 16);
            uint32_t a, b;
            e4m3x4_to_f16x2x2(pk[k], a, b);   // exact
            hs = __hadd2(hs, __hadd2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b)));
          }
          sum = __low2float(hs) + __high2float(hs);
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 16);
        l = l * alpha + sum;
        const bool rescale_o = group_any(grow && item_pv, 3, kSoftThreads);

        // ---- P may be written once the O MMAs that read its buffer last are
        // done (use pv_count / kPBufs - 1), and O^T rescaled once every O MMA
        // issued so far is: S and O have separate issuers, so this tile's S
        // completing says nothing about them
        const uint32_t pb = pv_count % C::kPBufs;    // P buffer of this tile
        if (pv_count >= (uint32_t)C::kPBufs &&
            !mbar_wait(&p_empty[pb], (pv_count / C::kPBufs - 1u) & 1u, p.wait_ns)) { dead = true; break; }
        if (rescale_o && pv_count > 0) {
          const uint32_t last = pv_count - 1u;
          if (!mbar_wait(&p_empty[last % C::kPBufs], (last / C::kPBufs) & 1u, p.wait_ns)) { dead = true; break; }
        }
        uint8_t* pdst = pbuf + pb * kPBytes;
        if (rescale_o) {
          if (row_thread) red_a[r] = alpha;
          named_barrier(2, kSoftThreads);
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint32_t o[16];
              tmem_ld16(tq + kColO + 64 * c + 16 * k, o);
              tmem_wait_ld(o);
#pragma unroll
              for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * red_a[16 * k + j]);
              tmem_st16(tq + kColO + 64 * c + 16 * k, o);
            }
          }
          tmem_wait_st();
          named_barrier(2, kSoftThreads);
        }
        if constexpr (!FP8) {
#pragma unroll
          for (int j = 0; j < 4; ++j)   // keys 32 kh .. +32: bytes 64 kh .. +64 of the row
            *reinterpret_cast<uint4*>(pdst + r * 128 + swz(r, 4 * kh + j)) =
                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 2; ++j)   // keys 32 kh .. +32: bytes 32 kh .. +32 of the row
            *reinterpret_cast<uint4*>(pdst + r * 128 + swz(r, 2 * kh + j)) =
                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&p_full[pb]);
          mbar_arrive(&empty[stage]);
        }
        ++pv_count;
        item_pv = true;
      }
      if (++stage == (uint32_t)kStages) { stage = 0; phase ^= 1; }
      if (!last) continue;

      // ============================ epilogue ============================
      if (item_pv) {
        // the O MMAs of the item's last P (the latest use of its buffer)
        const uint32_t last = pv_count - 1u;
        if (!mbar_wait(&p_empty[last % C::kPBufs], (last / C::kPBufs) & 1u, p.wait_ns)) { dead = true; break; }
      }
      tc_fence_after();
      const ItemDesc& it = meta[s].it;
      const UnitDesc& u = it.u;
      const bool split = u.n_splits > 1;
      // an unsplit row's state is final: fold in its sink, if any (a split
      // unit's merge adds it once)
      const float s2 = split ? -INFINITY : sink_log2(p.sinks, (u.row0 + r) % H);
      const float Mt = fmaxf(m, s2);
      const float a = m == -INFINITY ? 0.f : fast_exp2(m - Mt);
      const float Lt = l * a + (s2 == -INFINITY ? 0.f : fast_exp2(s2 - Mt));
      const float lse2 = Lt > 0.f ? Mt + __log2f(Lt) : -INFINITY;
      if (row_thread) red_l[r] = (Lt > 0.f && !errored) ? v_scale * a / Lt : 0.f;
      named_barrier(1, kSoftThreads);
      const int nrows = u.nrows;
      const size_t out_row0 = (size_t)u.q_start * H + u.row0;
      const size_t prow0 = (size_t)u.partial_base + (size_t)it.split * nrows;
      // O^T block (32 channels of this warp x 16 rows) by block: BF16 writes
      // it straight from registers (a lane's channel of each row; the warp's
      // 32 channels of a row are contiguous), E4M3 through a 2 KB shared tile
      // of the P buffer (free: the last O MMAs are done) as 16-byte stores,
      // which measured faster for that instance (131 against 138 us at 128
      // requests; BF16 813 against 833 us the other way round)
      uint8_t* tile = pbuf + w * 2048;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        const int ch0 = 128 * c + 32 * w;
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
          // the rows' scales, read before any store: a shared-memory store the
          // compiler cannot tell apart from red_l would otherwise hold each
          // read behind the store before it (measured: the epilogue took
          // ~20000 cycles, ~9700 with the reads first)
          float sc[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) sc[j] = red_l[16 * k + j];
          uint32_t o[16] = {};
          if (!errored) {
            tmem_ld16(tq + kColO + 64 * c + 16 * k, o);
            tmem_wait_ld(o);
          }
          if constexpr (!FP8) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int row = 16 * k + j;
              const float v = errored ? 0.f : __uint_as_float(o[j]) * sc[j];
              if (row < nrows) {
                if (split)
                  p.po[(prow0 + row) * kDv + ch0 + lane] = v;
                else
                  p.out[(out_row0 + row) * kDv + ch0 + lane] = __float2bfloat16_rn(v);
              }
            }
          } else if (split) {
            // fp32 [16 rows][32 channels]
#pragma unroll
            for (int j = 0; j < 16; ++j)
              reinterpret_cast<float*>(tile)[j * 32 + lane] = errored ? 0.f : __uint_as_float(o[j]) * sc[j];
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int idx = q * 32 + lane;  // 128 chunks of 16 bytes: row idx / 8, chunk idx % 8
              const int row = 16 * k + (idx >> 3);
              const uint4 v = reinterpret_cast<const uint4*>(tile)[idx];
              if (row < nrows)
                *reinterpret_cast<uint4*>(p.po + (prow0 + row) * kDv + ch0 + 4 * (idx & 7)) = v;
            }
            __syncwarp();
          } else {
            // bf16 [16 rows][32 channels]
#pragma unroll
            for (int j = 0; j < 16; ++j)
              reinterpret_cast<__nv_bfloat16*>(tile)[j * 32 + lane] =
                  __float2bfloat16_rn(errored ? 0.f : __uint_as_float(o[j]) * sc[j]);
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const int idx = q * 32 + lane;  // 64 chunks of 16 bytes: row idx / 4, chunk idx % 4
              const int row = 16 * k + (idx >> 2);
              const uint4 v = reinterpret_cast<const uint4*>(tile)[idx];
              if (row < nrows)
                *reinterpret_cast<uint4*>(p.out + (out_row0 + row) * kDv + ch0 + 8 * (idx & 3)) = v;
            }
            __syncwarp();
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && item_pv) mbar_arrive(o_empty);   // once per item that ran O MMAs
      if (row_thread && r < nrows) {
        if (split)
          p.plse[prow0 + r] = errored ? NAN : lse2;
        else if (p.lse != nullptr)
          p.lse[out_row0 + r] = errored ? NAN : lse2 * kLn2;
      }
      named_barrier(1, kSoftThreads);  // red arrays and the slot may be reused
      if (lane == 0) mbar_arrive(&slot_empty[s]);
      if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
    }
    if (dead && lane == 0) set_error(hdr, PD_DEV_TIMEOUT, -1);
  }

  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
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

template <bool FP8>
static cudaError_t launch_impl(const CUtensorMap& kvmap, const CUtensorMap& qmap, const MlaParams& p, int grid,
                               cudaStream_t stream) {
  constexpr int smem = MlaCfg<FP8>::kSmemBytes;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(mla_decode_kernel<FP8>), smem);
  if (e != cudaSuccess) return e;
  mla_decode_kernel<FP8><<<grid, kThreads, smem, stream>>>(kvmap, qmap, p);
  return cudaGetLastError();
}

cudaError_t launch_mla_decode(const CUtensorMap& kvmap, const CUtensorMap& qmap, const MlaParams& p, bool fp8,
                              int grid, cudaStream_t stream) {
  return fp8 ? launch_impl<true>(kvmap, qmap, p, grid, stream) : launch_impl<false>(kvmap, qmap, p, grid, stream);
}

}  // namespace pd
