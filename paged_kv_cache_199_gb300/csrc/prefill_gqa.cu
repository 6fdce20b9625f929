// Paged prefill (context) attention for sm_103a on the 5th-generation tensor
// cores: GQA over BF16 K/V pages with head_dim 128 and many new query tokens
// per request.
//
// What it computes: the context call of the cake_fmha API page
// (trtllm_batch_context_with_kv_cache, the same arguments as the decode
// call): query token i of request b, which has q_len new tokens among its
// L = seq_lens[b] cached ones, attends over keys 0 .. L - q_len + i of its KV
// head (the inclusive causal bound of PR #4557's review "Exclusive causal
// bound drops the newest key").
//
// Design:
//  * one persistent CTA per SM; a unit is up to 256 packed (token, head)
//    query rows of one request and one KV head, held as two 128-row query
//    tiles A and B (each 128 / G tokens times the G query heads of the
//    group) that share every key and value tile; keys are cut into
//    128-token tiles;
//  * scheduler warp 12 pops items, checks the device metadata, prefetches
//    page ids and TMA-loads the unit's query tiles (128-byte swizzled slabs,
//    a box of 64 channels x G heads x 128 / G tokens each);
//  * producer warp 9 TMA-loads each key tile into a two-slot ring and
//    producer warp 8 each value tile into another (two 16 KB slabs of 64
//    channels each), so that key loads never wait for a value slot;
//  * two threads issue the tcgen05 MMAs: MMA warp 10 issues S_X = Q_X K^T
//    (8 MMAs of M = 128 rows, N = 128 keys, K = 16) for X = A, B of each key
//    tile, and warp 11 issues O_X += P_X V (8 MMAs of N = 128 channels,
//    K = 16 keys) as soon as the softmax of tile X wrote P_X, so that one
//    issuer's barrier waits do not hold up the other's MMAs. Tensor memory
//    holds, per query tile, one S buffer of 128 columns, whose first 64
//    columns receive P (bf16 pairs, read by the O MMAs as their A operand),
//    and O in 128 columns: all 512 columns. The S of tile X for the next
//    keys waits until O_X has read P_X, while the other tile's softmax runs;
//  * softmax warps 0-3 own the rows of query tile A and warps 4-7 those of
//    tile B (one row per thread, tensor-memory lane quarter w mod 4), so one
//    group's softmax runs while the tensor cores work for the other. The
//    running maximum moves only when a tile raises it by more than 8 in the
//    log2 domain (P stays below 2^8 otherwise), and O is rescaled in tensor
//    memory when it does; the epilogue writes bf16 rows (or fp32 split
//    states that the LSE-merge kernel combines).
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

constexpr int kTile = 128;           // keys per tile
constexpr int kD = 128;              // head_dim of Q, K and V
constexpr int kRows = 128;           // rows of a query tile (tensor-memory lanes)
constexpr int kQTiles = 2;           // query tiles per unit
constexpr int kGroupWarps = 4;       // softmax warps per query tile
constexpr int kSoftWarps = kQTiles * kGroupWarps;
constexpr int kGroupThreads = kGroupWarps * 32;
// Warp w runs on SM sub-partition w mod 4, beside softmax warps w mod 4 and
// w mod 4 + 4: the S issuer (10) and the O issuer (11) each get a
// sub-partition of their own (with both on sub-partition 0, 151.5 us against
// 147.7 for the prefill workload)
constexpr int kMmaWarp = 10;
constexpr int kKProducerWarp = 9;
constexpr int kVProducerWarp = 8;
constexpr int kSchedulerWarp = 12;
constexpr int kOWarp = 11;
constexpr int kIssuers = 2;          // S and O MMAs are issued by two threads
constexpr int kThreads = 13 * 32;
constexpr int kSlots = 2;
constexpr int kWin = 64;             // page ids prefetched per item
constexpr int kSlab = 128 * 128;     // 16 KB: 128 rows of 128 bytes (64 bf16 channels)
constexpr int kTileBytes = 2 * kSlab;
static_assert(kRows * kD * 2 == kTileBytes && kTile * kD * 2 == kTileBytes, "tiles are two 16 KB slabs");
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kGrowThreshold = 8.f;  // log2 units

// tensor memory: per query tile X, S (and then P in its first 64 columns) at
// column 256 X, O at 256 X + 128
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t col_s(int x) { return 256u * (uint32_t)x; }
__host__ __device__ constexpr uint32_t col_o(int x) { return 256u * (uint32_t)x + 128u; }

constexpr uint32_t kIdescS = umma_idesc_bf16(128, 128, 0, 0);  // Q (K-major) x K tile (K-major)
constexpr uint32_t kIdescO = umma_idesc_bf16(128, 128, 0, 1);  // P (tensor memory) x V tile (MN-major)

enum : int { F_FIRST = 1, F_LAST = 2, F_BAD = 4, F_INVALID = 8, F_END = 16 };
enum : int { T_ITEM = 0, T_END = 3 };

struct StageInfo {
  int32_t slot;
  int32_t tile;
  int32_t flags;
  int32_t nq;                        // query tiles of the stage's item
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

constexpr int kOffQ = 0;                                   // two query tiles
constexpr int kOffK = kOffQ + kQTiles * kTileBytes;
constexpr int kOffV = kOffK + kKStages * kTileBytes;
constexpr int kOffMeta = kOffV + kVStages * kTileBytes;
constexpr int kOffInfo = kOffMeta + kSlots * (int)sizeof(SlotMeta);
constexpr int kOffBars = kOffInfo + kKStages * (int)sizeof(StageInfo);
constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 2 * kSlots + 4 * kQTiles + 4;
constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 16 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

__global__ void __launch_bounds__(kThreads, 1)
    gqa_prefill_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                       const __grid_constant__ CUtensorMap q_map, const GqaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qbuf = smem + kOffQ;
  uint8_t* kring = smem + kOffK;
  uint8_t* vring = smem + kOffV;
  SlotMeta* meta = reinterpret_cast<SlotMeta*>(smem + kOffMeta);
  StageInfo* sinfo = reinterpret_cast<StageInfo*>(smem + kOffInfo);
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* kempty = kfull + kKStages;       // both issuers (commit or arrive) + 8 softmax warps
  uint64_t* vfull = kempty + kKStages;
  uint64_t* vempty = vfull + kVStages;       // the O issuer (commit after the O MMAs)
  uint64_t* slot_full = vempty + kVStages;
  uint64_t* slot_empty = slot_full + kSlots;
  uint64_t* q_full = slot_empty + kSlots;    // the query tiles landed
  uint64_t* q_empty = q_full + 1;            // the last S of the item read them
  uint64_t* s_full = q_empty + 1;            // [2] S of query tile X computed
  uint64_t* p_full = s_full + kQTiles;       // [2] P of tile X written (and O_X rescaled)
  uint64_t* o_done = p_full + kQTiles;       // [2] the O MMAs of tile X (latest issued) are done
  uint64_t* o_empty = o_done + kQTiles;      // [2] the epilogue of tile X read O_X
  uint64_t* mma_done = o_empty + kQTiles;
  int* s_flag = reinterpret_cast<int*>(mma_done + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_flag + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  WsHeader* hdr = p.hdr;
  const int G = p.group;

  if (threadIdx.x == 0) {
    s_flag[0] = 1;  // cleared by the scheduler if the workspace holds another plan
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], kIssuers + kSoftWarps);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&slot_full[s], 1);
      mbar_init(&slot_empty[s], kSoftWarps);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int x = 0; x < kQTiles; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], kGroupWarps);
      mbar_init(&o_done[x], 1);
      mbar_init(&o_empty[x], kGroupWarps);
    }
    mbar_init(mma_done, kIssuers);
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
    prefetch_tensormap(&q_map);
    uint32_t s = 0, sph = 0;
    uint32_t qph = 0;
    bool q_loaded = false;   // the latest q_full phase carries copies of this warp
    bool dead = false, first_pop = true;
    int k_next = 0, k_end = 0;
    if (p.cta_items != nullptr) {
      k_next = __ldg(&p.cta_items[blockIdx.x]);
      k_end = __ldg(&p.cta_items[blockIdx.x + 1]);
    }
    uint32_t ws_magic = 0;
    uint64_t ws_plan = 0;
    if (lane == 0) {
      ws_magic = hdr->magic;
      ws_plan = hdr->plan_id;
    }
    int plan_ok = 1;
    if (lane == 0 && (ws_magic != kWsMagic || ws_plan != p.plan_id)) {
      plan_ok = 0;
      set_error(hdr, PD_DEV_PLAN_MISMATCH, -1);
      s_flag[0] = 0;
      meta[0].kind = T_END;
      meta[0].err = 0;
      mbar_arrive(&slot_full[0]);
    }
    plan_ok = __shfl_sync(0xffffffffu, plan_ok, 0);
    while (plan_ok) {
      if (!mbar_wait(&slot_empty[s], sph ^ 1, p.wait_ns)) { dead = true; break; }
      SlotMeta& m = meta[s];
      uint32_t idx = (uint32_t)p.num_items;
      if (p.cta_items != nullptr) {
        if (k_next < k_end) idx = (uint32_t)k_next++;
      } else if (first_pop) {
        idx = blockIdx.x;
        first_pop = false;
      } else {
        if (lane == 0) idx = gridDim.x + atomicAdd(&hdr->queue_counter, 1u);
        idx = __shfl_sync(0xffffffffu, idx, 0);
      }
      if (idx >= (uint32_t)p.num_items) {
        if (lane == 0) {
          m.kind = T_END;
          m.err = 0;
          mbar_arrive(&slot_full[s]);
        }
        break;
      }
      const ItemDesc it = p.items[idx];
      const UnitDesc& u = it.u;
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
      // one query block (two tiles): wait until the previous item's last S has read it
      if (!mbar_wait(q_empty, qph ^ 1, p.wait_ns)) { dead = true; break; }
      qph ^= 1;
      q_loaded = err == 0;
      if (lane == 0) {
        if (err) {
          mbar_arrive(q_full);
        } else {
          // tile X holds rows row0 + 128 X .. + 127: tokens (row0 + 128 X) / G
          // .. + 128 / G of the group's G heads; rows past the request read
          // neighbouring tokens (or zeros past the last one), never written back
          const int nq = (u.nrows + kRows - 1) / kRows;
          mbar_arrive_expect_tx(q_full, (uint32_t)(nq * kTileBytes));
          for (int x = 0; x < nq; ++x) {
            const int tok = u.q_start + (u.row0 + kRows * x) / G;
            for (int c = 0; c < 2; ++c)
              tma_load_4d(qbuf + x * kTileBytes + c * kSlab, &q_map, 64 * c, u.g * G, tok, 0, q_full,
                          l2_evict_last_policy());
          }
        }
      }
      if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
    }
    if (dead && lane == 0) set_error(hdr, PD_DEV_TIMEOUT, -1);
    // the query copies of the last item land before the CTA exits (its phase
    // is the latest one of q_full, parity qph ^ 1)
    if (q_loaded && lane == 0) mbar_wait(q_full, qph ^ 1, kDrainLimitNs);
  } else if (warp == kMmaWarp) {
    // ================================ S issue ================================
    if (lane == 0) {
      const uint32_t qaddr = smem_u32(qbuf), kaddr0 = smem_u32(kring);
      uint32_t ks = 0, kph = 0, qph = 0;
      // S_x number n overwrites P_x of number n - 1: it waits until the O
      // MMAs that read P_x (O_x number n - 1) are done
      uint32_t n_s[kQTiles] = {0u, 0u};
      bool dead = false;
      int nq = 1;
      while (true) {
        if (!mbar_wait(&kfull[ks], kph, p.wait_ns)) { dead = true; break; }
        const StageInfo info = sinfo[ks];
        const int f = info.flags;
        if (f & F_END) break;
        if (f & F_FIRST) {
          nq = info.nq;
          if (!mbar_wait(q_full, qph, p.wait_ns)) { dead = true; break; }
          qph ^= 1;
        }
        if (f & (F_BAD | F_INVALID)) {
          mbar_arrive(&kempty[ks]);
          if (f & F_LAST) umma_commit(q_empty);
          if (++ks == (uint32_t)kKStages) { ks = 0; kph ^= 1; }
          continue;
        }
        const uint64_t kdesc = umma_desc_sw128(kaddr0 + ks * kTileBytes, 16, 1024);
        for (int x = 0; x < nq; ++x) {
          if (n_s[x] > 0 && !mbar_wait(&o_done[x], (n_s[x] - 1u) & 1u, p.wait_ns)) { dead = true; break; }
          tc_fence_after();
          const uint64_t qdesc = umma_desc_sw128(qaddr + x * kTileBytes, 16, 1024);
#pragma unroll
          for (int kc = 0; kc < kD / 16; ++kc) {
            const uint64_t off = (uint64_t)(((kc >> 2) * kSlab + (kc & 3) * 32) >> 4);
            umma_bf16(tmem + col_s(x), qdesc + off, kdesc + off, kIdescS, kc > 0 ? 1u : 0u);
          }
          umma_commit(&s_full[x]);
          ++n_s[x];
        }
        if (dead) break;
        umma_commit(&kempty[ks]);
        if (f & F_LAST) umma_commit(q_empty);
        if (++ks == (uint32_t)kKStages) { ks = 0; kph ^= 1; }
      }
      if (dead) set_error(hdr, PD_DEV_TIMEOUT, -1);
      // every MMA issued has completed before tensor memory is released
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, kDrainLimitNs);
    }
  } else if (warp == kOWarp) {
    // ================================ O issue ================================
    if (lane == 0) {
      const uint32_t vaddr0 = smem_u32(vring);
      uint32_t ks = 0, kph = 0, vcount = 0;
      uint32_t p_seen[kQTiles] = {0u, 0u};     // P tiles of tile X consumed (p_full phases)
      uint32_t o_emp[kQTiles] = {0u, 0u};      // items of tile X that ran O MMAs (o_empty phases)
      bool first_o[kQTiles] = {false, false};
      bool dead = false;
      int nq = 1;
      while (true) {
        if (!mbar_wait(&kfull[ks], kph, p.wait_ns)) { dead = true; break; }
        const StageInfo info = sinfo[ks];
        const int f = info.flags;
        if (f & F_END) break;
        mbar_arrive(&kempty[ks]);   // stage info read
        if (++ks == (uint32_t)kKStages) { ks = 0; kph ^= 1; }
        if (f & F_FIRST) {
          nq = info.nq;
          first_o[0] = first_o[1] = true;   // the item's first O of each tile starts O afresh
        }
        if (f & (F_BAD | F_INVALID)) continue;
        // O_x += P_x V as soon as the softmax of tile x wrote P_x
        const uint32_t vs = vcount % kVStages;
        if (!mbar_wait(&vfull[vs], (vcount / kVStages) & 1u, p.wait_ns)) { dead = true; break; }
        const uint32_t vbase = vaddr0 + vs * kTileBytes;
        for (int x = 0; x < nq; ++x) {
          if (!mbar_wait(&p_full[x], p_seen[x] & 1u, p.wait_ns)) { dead = true; break; }
          ++p_seen[x];
          if (first_o[x]) {   // the epilogue of the last item that ran O_x has read it
            if (!mbar_wait(&o_empty[x], (o_emp[x] & 1u) ^ 1u, p.wait_ns)) { dead = true; break; }
            ++o_emp[x];
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            // P from tensor memory: keys 16 kk .. + 16 are columns 8 kk .. + 8 of S_x
            const uint64_t bdesc = umma_desc_sw128(vbase + kk * 16 * 128, kSlab, 1024);
            umma_bf16_ts(tmem + col_o(x), tmem + col_s(x) + 8 * kk, bdesc, kIdescO,
                         (first_o[x] && kk == 0) ? 0u : 1u);
          }
          umma_commit(&o_done[x]);
          first_o[x] = false;
        }
        if (dead) break;
        umma_commit(&vempty[vs]);
        ++vcount;
      }
      if (dead) set_error(hdr, PD_DEV_TIMEOUT, -1);
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, kDrainLimitNs);
    }
  } else if (warp == kKProducerWarp || warp == kVProducerWarp) {
    // ============================== producers ==============================
    // Both walk the same items and tiles; the key producer publishes each
    // tile's flags in the key ring, the value producer fills the value ring
    // for the tiles that have data (the same page-range check skips the same
    // tiles on both sides).
    const bool is_k = warp == kKProducerWarp;
    const CUtensorMap* map = is_k ? &k_map : &v_map;
    prefetch_tensormap(map);
    // the sibling row blocks of a request read the same tiles: keep them in L2
    const uint64_t pol = l2_evict_normal_policy();
    uint32_t ks = 0, kph = 0, vcount = 0;
    uint32_t s = 0, sph = 0;
    bool dead = false;
    while (true) {
      if (!mbar_wait(&slot_full[s], sph, p.wait_ns)) { dead = true; break; }
      const SlotMeta& m = meta[s];
      if (m.kind == T_END) break;
      const ItemDesc it = m.it;
      const UnitDesc& u = it.u;
      const int nq = (u.nrows + kRows - 1) / kRows;   // query tiles of the unit
      if (m.err) {
        if (is_k) {
          if (!mbar_wait(&kempty[ks], kph ^ 1, p.wait_ns)) { dead = true; break; }
          if (lane == 0) {
            sinfo[ks] = StageInfo{(int32_t)s, it.tile_begin, F_FIRST | F_LAST | F_INVALID, nq};
            mbar_arrive(&kfull[ks]);
          }
          if (++ks == (uint32_t)kKStages) { ks = 0; kph ^= 1; }
        }
        if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
        continue;
      }
      const int L = u.kv_len;
      const int win0 = m.win0, nwin = m.nwin;
      const int32_t* trow = p.block_tables + (size_t)u.b * p.max_pages_per_seq;
      const int c1g = p.layout == PD_LAYOUT_HND ? -1 : u.g;
      for (int t = it.tile_begin; t < it.tile_end; ++t) {
        const int tok0 = t * kTile;
        const int nvalid = min(kTile, L - tok0);
        const int nbox = (nvalid + BR - 1) / BR;   // <= 128 / 8 = 16 boxes (BR >= 8)
        int pg = 0;
        if (lane < nbox) {
          const int pi = (tok0 + lane * BR) / P - win0;
          pg = pi < nwin ? m.pages[pi] : __ldg(trow + win0 + pi);
        }
        const bool bad = __any_sync(0xffffffffu, lane < nbox && (pg < 0 || pg >= p.num_pages));
        const uint32_t bytes = (uint32_t)nbox * BR * 128 * 2;
        uint8_t* dst = nullptr;
        uint64_t* bar = nullptr;
        if (is_k) {
          const int flags = (t == it.tile_begin ? F_FIRST : 0) | (t == it.tile_end - 1 ? F_LAST : 0);
          if (!mbar_wait(&kempty[ks], kph ^ 1, p.wait_ns)) { dead = true; break; }
          if (lane == 0) {
            if (bad) set_error(hdr, PD_DEV_BAD_PAGE, u.b);
            sinfo[ks] = StageInfo{(int32_t)s, t, flags | (bad ? F_BAD : 0), nq};
            if (bad)
              mbar_arrive(&kfull[ks]);
            else
              mbar_arrive_expect_tx(&kfull[ks], bytes);
          }
          if (!bad) {
            dst = kring + ks * kTileBytes;
            bar = &kfull[ks];
          }
          if (++ks == (uint32_t)kKStages) { ks = 0; kph ^= 1; }
        } else if (!bad) {
          const uint32_t vs = vcount % kVStages, vph = (vcount / kVStages) & 1u;
          if (!mbar_wait(&vempty[vs], vph ^ 1, p.wait_ns)) { dead = true; break; }
          if (lane == 0) mbar_arrive_expect_tx(&vfull[vs], bytes);
          dst = vring + vs * kTileBytes;
          bar = &vfull[vs];
          ++vcount;
        }
        if (dst != nullptr) {
          for (int j = 0; j < nbox; ++j) {
            const int page = __shfl_sync(0xffffffffu, pg, j);
            if (lane == 0) {
              const int slot = (tok0 + j * BR) % P;
              const int c1 = c1g < 0 ? slot : c1g;
              const int c2 = c1g < 0 ? u.g : slot;
              for (int c = 0; c < 2; ++c)
                tma_load_4d(dst + c * kSlab + j * BR * 128, map, 64 * c, c1, c2, page, bar, pol);
            }
          }
        }
      }
      if (dead) break;
      if (++s == (uint32_t)kSlots) { s = 0; sph ^= 1; }
    }
    if (is_k) {
      if (!dead && mbar_wait(&kempty[ks], kph ^ 1, p.wait_ns)) {
        if (lane == 0) {
          sinfo[ks] = StageInfo{-1, 0, F_END, 0};
          mbar_arrive(&kfull[ks]);
        }
        if (++ks == (uint32_t)kKStages) { ks = 0; kph ^= 1; }
      } else {
        dead = true;
      }
    }
    if (dead && lane == 0) set_error(hdr, PD_DEV_TIMEOUT, -1);
    // the copies this warp put in flight land before the CTA exits (on the
    // normal path they have, and these waits return at once)
    if (is_k)
      drain_ring(const_cast<uint64_t*>(kfull), kKStages, ks, kph);
    else
      drain_ring(const_cast<uint64_t*>(vfull), kVStages, vcount % kVStages, (vcount / kVStages) & 1u);
  } else {
    // ============================== softmax / epilogue ==============================
    const int x = warp / kGroupWarps;    // query tile of this warp's group
    const int q4 = warp % kGroupWarps;   // tensor-memory lane quarter
    const int r = 32 * q4 + lane;        // the row (lane) of this thread within tile x
    const uint32_t tq = tmem + ((uint32_t)(32 * q4) << 16);
    const uint32_t scol = tq + col_s(x), ocol = tq + col_o(x);
    const float scale2 = p.sm_scale * kLog2e;
    uint32_t ks = 0, kph = 0, s = 0, sph = 0, sfph = 0, vcount = 0, pcount = 0;
    bool item_pv = false, active = false;
    float m = -INFINITY, l = 0.f;
    int errored = 0, kv_len = 0, pos = 0;
    bool dead = false;
    while (true) {
      if (!mbar_wait(&kfull[ks], kph, p.wait_ns)) { dead = true; break; }
      const StageInfo info = sinfo[ks];
      if (info.flags & F_END) break;
      if (info.flags & F_FIRST) {
        if (!mbar_wait(&slot_full[s], sph, p.wait_ns)) { dead = true; break; }
        const UnitDesc& fu = meta[s].it.u;
        kv_len = fu.kv_len;
        errored = (info.flags & F_INVALID) ? 1 : 0;
        active = x < info.nq;
        // rows past the unit read neighbouring query rows and are never
        // written; they see the same keys as the unit's last row
        const int ur = kRows * x + r;   // row within the unit
        pos = ur < fu.nrows ? fu.kv_len - fu.q_len + (fu.row0 + ur) / G : fu.kv_len - 1;
        m = -INFINITY;
        l = 0.f;
        item_pv = false;
      }
      const bool last = (info.flags & F_LAST) != 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(&kempty[ks]);   // stage info read
      if (++ks == (uint32_t)kKStages) { ks = 0; kph ^= 1; }

      if (!active) {
        // this group has no rows in the item
      } else if (info.flags & (F_BAD | F_INVALID)) {
        errored = 1;
      } else {
        const int tok0 = info.tile * kTile;
        // ---- value rows past the sequence end are zero (0 * stale data must
        // stay 0); group A writes them, and its O MMAs go before group B's
        if (x == 0) {
          if (tok0 + kTile > kv_len) {
            const uint32_t vs = vcount % kVStages;
            if (!mbar_wait(&vfull[vs], (vcount / kVStages) & 1u, p.wait_ns)) { dead = true; break; }
            uint8_t* vt = vring + vs * kTileBytes;
            const int first = kv_len - tok0;
            // rows first .. 127 of both slabs: 16 chunks of 16 bytes per row
            for (int idx = threadIdx.x; idx < (kTile - first) * 16; idx += kGroupThreads) {
              const int row = first + (idx >> 4), c = idx & 15;
              *reinterpret_cast<uint4*>(vt + (c >> 3) * kSlab + row * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async();
          }
          ++vcount;
        }

        // ---- pass 1: the row maximum over the 128 keys (raw scores; the scale
        // is positive), 32 columns at a time; keys past the row's causal
        // bound are left out
        if (!mbar_wait(&s_full[x], sfph, p.wait_ns)) { dead = true; break; }
        sfph ^= 1;
        tc_fence_after();
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          const int kb = tok0 + 32 * c;
          // tcgen05.ld is warp-wide: the warp takes one branch, the reducing
          // load when every row of the warp sees the whole chunk
          if (__all_sync(0xffffffffu, kb + 31 <= pos)) {
            float cm;
            tmem_ld32_max(scol + 32 * c, v, cm);
            tmem_wait_ld_red(v, cm);
            mx0 = fmaxf(mx0, cm);
          } else {
            tmem_ld32(scol + 32 * c, v);
            tmem_wait_ld(v);
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              if (kb + k <= pos) mx0 = fmaxf(mx0, __uint_as_float(v[k]));
              if (kb + k + 1 <= pos) mx1 = fmaxf(mx1, __uint_as_float(v[k + 1]));
            }
          }
        }
        const float raw_max = fmaxf(mx0, mx1);
        const float mt = raw_max == -INFINITY ? -INFINITY : raw_max * scale2;
        float alpha = 1.f;
        const bool grow = mt > m + kGrowThreshold;
        if (grow) {
          alpha = m == -INFINITY ? 0.f : fast_exp2(m - mt);
          m = mt;
        }
        const float mu = m == -INFINITY ? 0.f : m;
        // ---- O_x is complete here (this S was issued after the last O_x
        // finished): rescale it in tensor memory when the maximum moved
        if (__any_sync(0xffffffffu, grow && item_pv)) {
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t o[16];
            tmem_ld16(ocol + 16 * c, o);
            tmem_wait_ld(o);
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tmem_st16(ocol + 16 * c, o);
          }
        }
        // ---- pass 2: P = 2^(s - m), 32 keys at a time, packed as bf16 pairs
        // into columns 16 c .. + 16 of the same buffer (keys 0 .. 32 c + 31
        // have been read by then); the row sum in fp32 (even and odd keys
        // apart). The scaling and the sums run on packed pairs.
        const uint64_t scale_2 = f2pack(scale2, scale2), nmu_2 = f2pack(-mu, -mu);
        uint64_t sum_2 = f2pack(0.f, 0.f);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(scol + 32 * c, v);
          tmem_wait_ld(v);
          const int kb = tok0 + 32 * c;
          const bool masked = kb + 31 > pos;
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float t0, t1;
            f2unpack(f2fma(f2pack(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])), scale_2, nmu_2), t0, t1);
            float p0 = fast_exp2(t0);
            float p1 = fast_exp2(t1);
            if (masked) {
              p0 = kb + 2 * j <= pos ? p0 : 0.f;
              p1 = kb + 2 * j + 1 <= pos ? p1 : 0.f;
            }
            pk[j] = pack_bf16(p0, p1);
            sum_2 = f2add(sum_2, f2pack(p0, p1));
          }
          tmem_st16(scol + 16 * c, pk);
        }
        float sum0, sum1;
        f2unpack(sum_2, sum0, sum1);
        l = l * alpha + (sum0 + sum1);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[x]);
        ++pcount;
        item_pv = true;
      }
      if (!last) continue;

      // ============================ epilogue ============================
      if (active) {
        if (item_pv && !mbar_wait(&o_done[x], (pcount - 1u) & 1u, p.wait_ns)) { dead = true; break; }
        tc_fence_after();
        const ItemDesc& it = meta[s].it;
        const UnitDesc& u = it.u;
        const bool split = u.n_splits > 1;
        const int ur = kRows * x + r;
        const int head = u.g * G + (u.row0 + ur) % G;
        // an unsplit row's state is final: fold in its sink, if any (the
        // merge kernel adds it once for split units)
        const float s2 = split ? -INFINITY : sink_log2(p.sinks, head);
        const float Mt = fmaxf(m, s2);
        const float a = m == -INFINITY ? 0.f : fast_exp2(m - Mt);
        const float Lt = l * a + (s2 == -INFINITY ? 0.f : fast_exp2(s2 - Mt));
        const float lse2 = Lt > 0.f ? Mt + __log2f(Lt) : -INFINITY;
        const float inv = (Lt > 0.f && !errored) ? a / Lt : 0.f;
        const bool row_ok = ur < u.nrows;
        const size_t out_row = (size_t)(u.q_start + (u.row0 + ur) / G) * p.num_q_heads + head;
        const size_t prow = (size_t)u.partial_base + (size_t)it.split * u.nrows + ur;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t o[16] = {};
          if (!errored && item_pv) {
            tmem_ld16(ocol + 16 * c, o);
            tmem_wait_ld(o);
          }
          if (!row_ok) continue;
          if (split) {
            float* dst = p.po + prow * kD + 16 * c;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<float4*>(dst + 4 * j) =
                  make_float4(__uint_as_float(o[4 * j]) * inv, __uint_as_float(o[4 * j + 1]) * inv,
                              __uint_as_float(o[4 * j + 2]) * inv, __uint_as_float(o[4 * j + 3]) * inv);
          } else {
            uint32_t b[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              b[j] = pack_bf16(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
            uint4* dst = reinterpret_cast<uint4*>(p.out + out_row * kD + 16 * c);
            dst[0] = make_uint4(b[0], b[1], b[2], b[3]);
            dst[1] = make_uint4(b[4], b[5], b[6], b[7]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && item_pv) mbar_arrive(&o_empty[x]);   // once per item that ran O_x MMAs
        if (row_ok) {
          if (split)
            p.plse[prow] = errored ? NAN : lse2;
          else if (p.lse != nullptr)
            p.lse[out_row] = errored ? NAN : lse2 * kLn2;
        }
      }
      __syncwarp();
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
  if (threadIdx.x == 0 && s_flag[0]) {
    __threadfence();
    if (atomicAdd(&hdr->done_counter, 1u) == gridDim.x - 1) {
      hdr->queue_counter = 0u;
      hdr->done_counter = 0u;
      __threadfence();
    }
  }
}

}  // namespace

cudaError_t launch_gqa_prefill(const CUtensorMap& kmap, const CUtensorMap& vmap, const CUtensorMap& qmap,
                               const GqaParams& p, int grid, cudaStream_t stream) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(gqa_prefill_kernel), kSmemBytes);
  if (e != cudaSuccess) return e;
  gqa_prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(kmap, vmap, qmap, p);
  return cudaGetLastError();
}

}  // namespace pd
