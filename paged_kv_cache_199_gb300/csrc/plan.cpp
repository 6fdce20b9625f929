// Host split planner for paged decode attention.
//
// A unit is the set of packed query rows of one request that read the same
// KV head (GQA: q_len * Hq/Hkv rows per KV head, cut into blocks of at most
// 16 rows; MLA: q_len * H rows cut into blocks of 64). A unit's key range is
// cut into at most 16 contiguous tile ranges ("splits"): the split-KV
// reducer described in PR #4557 ("Blackwell TRT-LLM MLA decode backend")
// keeps statistics for at most 16 splits because its host never asks for
// more. Every (unit, split) pair is one work item of a persistent queue; the
// items are ordered longest first, as PR #4557's persistent CLC route orders
// its work ids, with ties broken by (unit, split) index.
//
// Two schedules are considered (the queue is kept unless the static
// partition is predicted to finish at least 25% earlier):
//  * a static balanced partition: the flattened (unit, tile) sequence is cut
//    into one contiguous, equal range per CTA slot (at most 16 pieces per
//    unit); each CTA runs its own pieces, split pieces first so that their
//    merges happen early and the last pieces are whole units where possible;
//  * the shared persistent queue described below.
// For the queue the split count is not fixed per shape: the planner tries a small set of
// item-size caps, simulates the persistent queue on the device's CTA slots
// (greedy longest-processing-time list scheduling, which is what a
// longest-first atomic queue executes) with a cost model of tiles plus a
// per-item overhead plus the partial-state traffic of split units, and keeps
// the cap with the smallest predicted finish time. This replaces the pages'
// fixed per-wave cost constant (PR #5552 split planners) with the schedule
// the kernel will actually run.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <functional>
#include <new>
#include <queue>
#include <set>
#include <vector>

#include "kernels.h"
#include "paged_decode.h"
#include "plan_internal.h"

namespace pd {

int ctas_per_sm(const pd_problem& p) {
  // the GQA decode kernel sizes its pipeline for two resident CTAs per SM,
  // the MLA and prefill kernels for one
  return p.kind == PD_ATTN_GQA ? 2 : 1;
}

namespace {

// Fixed cost of one work item (query load, epilogue, slot turnaround) in units
// of one tile's streaming time; measured on GB300 at about 2-2.5 us per item
// against ~1.5 us per 32 KB tile (64 BF16 or 128 E4M3 tokens).
double item_overhead_tiles(const pd_problem&) { return 1.5; }

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

uint64_t fnv1a(uint64_t h, const void* data, size_t n) {
  const uint8_t* p = static_cast<const uint8_t*>(data);
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= 1099511628211ull;
  }
  return h;
}

struct UnitWork {
  int32_t tiles;
  int32_t nrows;
};

// Predicted finish time (in tile units) of list-scheduling `costs` (already
// sorted in decreasing order) on `slots` identical workers.
double simulate_lpt(const std::vector<double>& costs, int slots) {
  if (costs.empty()) return 0.0;
  if ((int)costs.size() <= slots) return costs.front();
  std::priority_queue<double, std::vector<double>, std::greater<double>> heap;
  for (int i = 0; i < slots; ++i) heap.push(0.0);
  double makespan = 0.0;
  for (double c : costs) {
    double t = heap.top() + c;
    heap.pop();
    heap.push(t);
    makespan = std::max(makespan, t);
  }
  return makespan;
}

int splits_for(int tiles, int cap_tiles, int max_splits) {
  if (tiles <= 0) return 1;
  int s = (tiles + cap_tiles - 1) / cap_tiles;
  return std::max(1, std::min(s, std::min(max_splits, tiles)));
}

// Cost of the item sizes produced by a cap, sorted decreasing.
std::vector<double> item_costs(const std::vector<UnitWork>& units, int cap, int max_splits,
                               double partial_tiles_per_row, double overhead) {
  std::vector<double> costs;
  costs.reserve(units.size() * 2);
  for (const UnitWork& u : units) {
    int s = splits_for(u.tiles, cap, max_splits);
    double extra = s > 1 ? 2.0 * partial_tiles_per_row * u.nrows : 0.0;
    int base = u.tiles / s, rem = u.tiles % s;
    for (int k = 0; k < s; ++k) costs.push_back((base + (k < rem ? 1 : 0)) + overhead + extra);
  }
  std::sort(costs.begin(), costs.end(), std::greater<double>());
  return costs;
}

pd_status validate(const pd_problem& p, const int32_t* seq_lens, const int32_t* q_indptr) {
  if (p.batch < 0 || p.page_size < 1 || p.max_pages_per_seq < 0 || p.max_kv_len < 0 ||
      p.num_pages < 0 || p.max_splits < 0 || p.max_splits > kMaxSplits || p.num_sms < 0 ||
      p.k_page_stride < 0 || p.v_page_stride < 0)
    return PD_ERR_INVALID_ARG;
  if (p.merge_mode != PD_MERGE_AUTO && p.merge_mode != PD_MERGE_FUSED && p.merge_mode != PD_MERGE_KERNEL)
    return PD_ERR_INVALID_ARG;
  if (p.schedule != PD_SCHED_AUTO && p.schedule != PD_SCHED_STATIC && p.schedule != PD_SCHED_QUEUE)
    return PD_ERR_INVALID_ARG;
  if (p.num_q_heads < 1 || p.num_kv_heads < 1 || p.num_q_heads % p.num_kv_heads != 0)
    return PD_ERR_INVALID_ARG;
  if ((int64_t)p.max_kv_len > (int64_t)p.max_pages_per_seq * p.page_size) return PD_ERR_INVALID_ARG;
  if (p.kind == PD_ATTN_GQA || p.kind == PD_ATTN_PREFILL) {
    if (p.layout != PD_LAYOUT_NHD && p.layout != PD_LAYOUT_HND) return PD_ERR_INVALID_ARG;
    if (p.kv_dtype != PD_KV_BF16 && p.kv_dtype != PD_KV_FP8_E4M3) return PD_ERR_INVALID_ARG;
    if (p.head_dim_qk != 128 || p.head_dim_v != 128) return PD_ERR_UNSUPPORTED;
    if (p.kind == PD_ATTN_PREFILL) {
      // tensor-core tiles: BF16 operands, 128-byte swizzled TMA boxes of >= 8
      // token rows, and 128-row query blocks made of whole groups
      if (p.kv_dtype != PD_KV_BF16) return PD_ERR_UNSUPPORTED;
      if (p.page_size % 8 != 0) return PD_ERR_UNSUPPORTED;
      if (128 % (p.num_q_heads / p.num_kv_heads) != 0) return PD_ERR_UNSUPPORTED;
    }
  } else if (p.kind == PD_ATTN_MLA) {
    if (p.num_kv_heads != 1) return PD_ERR_INVALID_ARG;
    if (p.head_dim_qk != 576 || p.head_dim_v != 512) return PD_ERR_UNSUPPORTED;
    if (p.kv_dtype != PD_KV_BF16 && p.kv_dtype != PD_KV_FP8_E4M3) return PD_ERR_INVALID_ARG;
    // key tiles are TMA boxes of >= 8 whole 128-byte rows (the swizzled operand layout)
    if (p.page_size % 8 != 0) return PD_ERR_UNSUPPORTED;
  } else {
    return PD_ERR_INVALID_ARG;
  }
  const bool gqa_like = p.kind == PD_ATTN_GQA || p.kind == PD_ATTN_PREFILL;
  const int64_t elem = (gqa_like && p.kv_dtype == PD_KV_FP8_E4M3) ? 1 : 2;
  const int64_t compact = gqa_like
                              ? (int64_t)p.page_size * p.num_kv_heads * p.head_dim_qk
                              : (int64_t)p.page_size * p.head_dim_qk;
  for (int64_t s : {p.k_page_stride, p.v_page_stride}) {
    if (s == 0) continue;
    if (s < compact || (s * elem) % 16 != 0) return PD_ERR_INVALID_ARG;
  }
  if (p.batch == 0) return PD_OK;
  if (!seq_lens) return PD_ERR_INVALID_ARG;
  if (p.num_pages < 1 || p.max_pages_per_seq < 1) return PD_ERR_INVALID_ARG;
  if (q_indptr && q_indptr[0] != 0) return PD_ERR_INVALID_ARG;
  for (int b = 0; b < p.batch; ++b) {
    int64_t ql = q_indptr ? (int64_t)q_indptr[b + 1] - q_indptr[b] : 1;
    if (ql < 0) return PD_ERR_INVALID_ARG;
    if (seq_lens[b] < 0 || seq_lens[b] > p.max_kv_len) return PD_ERR_INVALID_ARG;
    if (ql > seq_lens[b]) return PD_ERR_INVALID_ARG;  // new tokens must be in the cache
  }
  if (q_indptr && q_indptr[p.batch] > (1 << 30)) return PD_ERR_INVALID_ARG;
  return PD_OK;
}

}  // namespace
}  // namespace pd

extern "C" pd_status paged_decode_plan(const pd_problem* problem, const int32_t* seq_lens_host,
                                       const int32_t* q_indptr_host, pd_plan** plan_out) {
  using namespace pd;
  if (!problem || !plan_out) return PD_ERR_INVALID_ARG;
  *plan_out = nullptr;
  const pd_problem& p = *problem;
  pd_status st = validate(p, seq_lens_host, q_indptr_host);
  if (st != PD_OK) return st;

  pd_plan* plan = new (std::nothrow) pd_plan();
  if (!plan) return PD_ERR_INVALID_ARG;
  plan->prob = p;
  const bool mla = p.kind == PD_ATTN_MLA;
  const bool prefill = p.kind == PD_ATTN_PREFILL;
  // AUTO: split states go to the separate LSE-merge kernel, launched as a
  // programmatic dependent of the decode grid. An MLA unit's states are 64
  // rows x 512 channels per split, which that kernel spreads over many CTAs
  // (measured on GB300, FP8 latent MLA, 16 requests x 4096: 60 us against
  // 99 us with the last-arriving CTA merging). For GQA it measured no slower
  // than the last-arriver merge inside the decode kernel and faster where
  // splits are many (E4M3, 16 requests x 4096: 37.4 us against 39.5; ragged
  // batch of 128: 152 against 154-156); FUSED still selects the in-kernel merge.
  if (plan->prob.merge_mode == PD_MERGE_AUTO) plan->prob.merge_mode = PD_MERGE_KERNEL;
  // the prefill kernel leaves split states to the LSE-merge kernel
  if (prefill) plan->prob.merge_mode = PD_MERGE_KERNEL;
  if (plan->prob.k_page_stride == 0)
    plan->prob.k_page_stride = !mla ? (int64_t)p.page_size * p.num_kv_heads * p.head_dim_qk
                                    : (int64_t)p.page_size * p.head_dim_qk;
  if (plan->prob.v_page_stride == 0)
    plan->prob.v_page_stride = !mla ? (int64_t)p.page_size * p.num_kv_heads * p.head_dim_v
                                    : plan->prob.k_page_stride;
  plan->tile_tokens = mla ? kMlaTileTokens
                     : prefill ? kPrefillTileTokens
                     : p.kv_dtype == PD_KV_FP8_E4M3 ? kGqaFp8TileTokens : kGqaTileTokens;
  plan->rows_per_unit = mla ? kMlaRowsPerUnit : prefill ? kPrefillRowsPerUnit : kGqaRowsPerUnit;
  if (p.kind == PD_ATTN_GQA) {
    // the GQA kernel packs 8 or 16 query rows per unit; take 8 when every
    // request's q_len * (Hq / Hkv) fits, which halves the MMA work
    int max_rows = 0;
    for (int b = 0; b < p.batch; ++b) {
      const int ql = q_indptr_host ? q_indptr_host[b + 1] - q_indptr_host[b] : 1;
      max_rows = std::max(max_rows, ql * (p.num_q_heads / p.num_kv_heads));
    }
    plan->rows_per_unit = max_rows <= 8 ? 8 : kGqaRowsPerUnit;
  }

  int num_sms = p.num_sms;
  if (num_sms == 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
      delete plan;
      return cuda_fail(e, "SM count query");   // records the text for paged_decode_last_cuda_error
    }
  }
  plan->num_sms = num_sms;
  const int slots = num_sms * ctas_per_sm(p);

  plan->seq_lens.assign(seq_lens_host, seq_lens_host + p.batch);
  plan->q_indptr.resize(p.batch + 1);
  for (int b = 0; b <= p.batch; ++b) plan->q_indptr[b] = q_indptr_host ? q_indptr_host[b] : b;
  plan->total_q = plan->q_indptr[p.batch];

  // ---- units ---------------------------------------------------------------
  const int G = mla ? p.num_q_heads : p.num_q_heads / p.num_kv_heads;
  const int n_kv = mla ? 1 : p.num_kv_heads;
  const int T = plan->tile_tokens;
  const int R = plan->rows_per_unit;
  std::vector<UnitWork> work;
  for (int b = 0; b < p.batch; ++b) {
    const int ql = plan->q_indptr[b + 1] - plan->q_indptr[b];
    const int L = plan->seq_lens[b];
    const int rows = ql * G;
    for (int g = 0; g < n_kv; ++g) {
      for (int r0 = 0; r0 < rows; r0 += R) {
        UnitDesc u{};
        u.b = b;
        u.g = g;
        u.row0 = r0;
        u.nrows = std::min(R, rows - r0);
        u.q_start = plan->q_indptr[b];
        u.q_len = ql;
        u.kv_len = L;
        u.n_splits = 1;
        u.partial_base = -1;
        // the last query row of this block sees keys 0 .. L - ql + i_last
        const int i_last = (r0 + u.nrows - 1) / G;
        const int visible = L - ql + i_last + 1;
        plan->units.push_back(u);
        work.push_back(UnitWork{(visible + T - 1) / T, u.nrows});
      }
    }
  }

  // ---- split selection -------------------------------------------------------
  const int max_splits = p.max_splits == 0 ? kMaxSplits : p.max_splits;
  int max_tiles = 0;
  int64_t total_tiles = 0;
  for (const UnitWork& w : work) {
    max_tiles = std::max(max_tiles, w.tiles);
    total_tiles += w.tiles;
  }
  // partial-state bytes of one row relative to one tile of K/V bytes
  const double elem = p.kv_dtype == PD_KV_FP8_E4M3 ? 1.0 : 2.0;
  const double tile_bytes = mla ? (double)T * p.head_dim_qk * elem
                                : (double)T * (p.head_dim_qk + p.head_dim_v) * elem;
  const double partial_tiles_per_row = (double)p.head_dim_v * 4.0 / tile_bytes;
  const double ovh = item_overhead_tiles(p);

  int best_cap = std::max(1, max_tiles);
  if (!work.empty() && max_splits > 1) {
    std::set<int> caps;
    for (int s = 1; s <= max_splits; ++s) caps.insert(std::max(1, (max_tiles + s - 1) / s));
    for (int k = 1; k <= 32; ++k)
      caps.insert(std::max<int64_t>(1, (total_tiles + (int64_t)k * slots - 1) / ((int64_t)k * slots)));
    double best = 1e300;
    int64_t best_items = 0;
    for (int cap : caps) {
      if (cap > max_tiles) continue;
      std::vector<double> costs = item_costs(work, cap, max_splits, partial_tiles_per_row, ovh);
      double t = simulate_lpt(costs, slots);
      // prefer fewer items (less partial traffic) unless 1% faster
      if (t < best * 0.99 || (t <= best * 1.01 && (int64_t)costs.size() < best_items)) {
        best = std::min(best, t);
        best_cap = cap;
        best_items = (int64_t)costs.size();
      }
    }
  }

  // ---- static balanced partition -------------------------------------------------
  // CTA c takes tiles [bound[c], bound[c+1]) of the flattened sequence, with
  // bound[c] = floor(total c / n): every range is at least floor(total / n)
  // tiles wide. A unit of t tiles meets at most ceil(t / w) + 1 ranges of
  // width >= w, so ranges of at least t_max / (max_splits - 1) tiles keep every
  // unit within max_splits pieces: n is the largest count whose narrowest
  // range is ceil(W) tiles or more.
  std::vector<int64_t> offset(work.size() + 1, 0);
  for (size_t i = 0; i < work.size(); ++i) offset[i + 1] = offset[i] + work[i].tiles;
  bool use_static = false;
  int static_ctas = 0;
  if (!work.empty() && max_splits > 1 && p.schedule != PD_SCHED_QUEUE) {
    double W = (double)total_tiles / slots;
    const double minW = (double)max_tiles / (double)(max_splits - 1);
    W = std::max({W, minW, 1.0});
    static_ctas = (int)std::min<int64_t>(slots, total_tiles / (int64_t)std::ceil(W));
    static_ctas = std::max(1, static_ctas);
    // predicted finish: the longest range plus the per-item overhead of its pieces
    double t_static = 0.0;
    for (int c = 0; c < static_ctas; ++c) {
      const int64_t b0 = total_tiles * c / static_ctas, b1 = total_tiles * (c + 1) / static_ctas;
      const size_t u0 = std::upper_bound(offset.begin(), offset.end(), b0) - offset.begin() - 1;
      const size_t u1 = std::lower_bound(offset.begin(), offset.end(), b1) - offset.begin();
      t_static = std::max(t_static, (double)(b1 - b0) + ovh * (double)(u1 - u0) +
                                        2.0 * partial_tiles_per_row * plan->rows_per_unit);
    }
    std::vector<double> costs = item_costs(work, best_cap, max_splits, partial_tiles_per_row, ovh);
    const double t_queue = simulate_lpt(costs, slots);
    // the model leaves out the static schedule's split-piece epilogues and
    // its end-of-call merges (every CTA ends on a shared piece), which cost
    // ~15-20% on GB300 for uniform batches: take it only when clearly ahead
    use_static = p.schedule == PD_SCHED_STATIC || t_static * 1.25 <= t_queue;
  }

  // ---- items -------------------------------------------------------------------
  struct Tmp {
    double cost;
    ItemDesc it;
  };
  std::vector<Tmp> tmp;
  int64_t partial = 0;
  if (use_static) {
    // pieces per unit, in position order (split index = position)
    std::vector<std::vector<std::pair<int, int>>> pieces(work.size());  // (first tile, end tile)
    std::vector<std::vector<std::pair<int, int>>> per_cta(static_ctas);  // (unit, piece index)
    for (int c = 0; c < static_ctas; ++c) {
      const int64_t b0 = total_tiles * c / static_ctas, b1 = total_tiles * (c + 1) / static_ctas;
      size_t u = std::upper_bound(offset.begin(), offset.end(), b0) - offset.begin() - 1;
      for (int64_t pos = b0; pos < b1 && u < work.size(); ++u) {
        const int64_t end = std::min<int64_t>(b1, offset[u + 1]);
        if (end <= pos) continue;
        per_cta[c].push_back({(int)u, (int)pieces[u].size()});
        pieces[u].push_back({(int)(pos - offset[u]), (int)(end - offset[u])});
        pos = end;
      }
    }
    for (size_t ui = 0; ui < plan->units.size(); ++ui) {
      UnitDesc& u = plan->units[ui];
      const int s = (int)pieces[ui].size();
      u.n_splits = s;
      if (s > 1) {
        u.partial_base = partial;
        partial += (int64_t)s * u.nrows;
      }
      plan->max_splits_used = std::max(plan->max_splits_used, s);
    }
    plan->cta_first.assign(static_ctas + 1, 0);
    for (int c = 0; c < static_ctas; ++c) {
      std::vector<std::pair<int, int>>& v = per_cta[c];
      // the range's first and last pieces are the ones shared with the
      // neighbouring CTAs: run them first, whole units after them
      std::vector<std::pair<int, int>> ord;
      if (!v.empty()) ord.push_back(v.front());
      if (v.size() > 1) ord.push_back(v.back());
      for (size_t k = 1; k + 1 < v.size(); ++k) ord.push_back(v[k]);
      for (const auto& pc : ord) {
        const auto& rng = pieces[pc.first][pc.second];
        plan->items.push_back(ItemDesc{pc.first, rng.first, rng.second, pc.second, UnitDesc{}});
      }
      plan->cta_first[c + 1] = (int32_t)plan->items.size();
    }
    for (ItemDesc& it : plan->items) it.u = plan->units[it.unit];
    plan->partial_rows = partial;
    plan->num_ctas = static_ctas;
  } else {
  for (size_t ui = 0; ui < plan->units.size(); ++ui) {
    UnitDesc& u = plan->units[ui];
    const int tiles = work[ui].tiles;
    const int s = splits_for(tiles, best_cap, max_splits);
    u.n_splits = s;
    if (s > 1) {
      u.partial_base = partial;
      partial += (int64_t)s * u.nrows;
    }
    plan->max_splits_used = std::max(plan->max_splits_used, s);
    const int base = tiles / s, rem = tiles % s;
    int t0 = 0;
    for (int k = 0; k < s; ++k) {
      const int n = base + (k < rem ? 1 : 0);
      tmp.push_back(Tmp{(double)n, ItemDesc{(int32_t)ui, t0, t0 + n, k, UnitDesc{}}});
      t0 += n;
    }
  }
  std::stable_sort(tmp.begin(), tmp.end(), [](const Tmp& a, const Tmp& b) {
    if (a.cost != b.cost) return a.cost > b.cost;
    if (a.it.unit != b.it.unit) return a.it.unit < b.it.unit;
    return a.it.split < b.it.split;
  });
  plan->items.reserve(tmp.size());
  for (Tmp& t : tmp) {
    t.it.u = plan->units[t.it.unit];
    plan->items.push_back(t.it);
  }
  plan->partial_rows = partial;
  plan->num_ctas = (int)std::max<int64_t>(1, std::min<int64_t>(slots, (int64_t)plan->items.size()));
  }

  // ---- workspace layout + blob ---------------------------------------------------
  WsHeader& h = plan->hdr;
  std::memset(&h, 0, sizeof h);
  h.magic = kWsMagic;
  h.version = 1;
  h.error_info = -1;
  h.num_units = (int32_t)plan->units.size();
  h.num_items = (int32_t)plan->items.size();
  int64_t off = sizeof(WsHeader);
  h.units_off = off;
  off = align_up(off + (int64_t)plan->units.size() * sizeof(UnitDesc), 256);
  h.items_off = off;
  off = align_up(off + (int64_t)plan->items.size() * sizeof(ItemDesc), 256);
  h.counters_off = off;
  off = align_up(off + (int64_t)plan->units.size() * sizeof(uint32_t), 16);
  h.cta_off = plan->cta_first.empty() ? 0 : off;
  h.num_ctas = plan->num_ctas;
  const int64_t blob_end = off + (int64_t)plan->cta_first.size() * sizeof(int32_t);
  off = align_up(blob_end, 256);
  h.plse_off = off;
  off = align_up(off + partial * (int64_t)sizeof(float), 256);
  h.po_off = off;
  off = align_up(off + partial * (int64_t)p.head_dim_v * (int64_t)sizeof(float), 256);
  h.total_bytes = off;

  plan->blob.assign((size_t)blob_end, 0);
  std::memcpy(plan->blob.data() + h.units_off, plan->units.data(),
              plan->units.size() * sizeof(UnitDesc));
  std::memcpy(plan->blob.data() + h.items_off, plan->items.data(),
              plan->items.size() * sizeof(ItemDesc));
  if (h.cta_off)
    std::memcpy(plan->blob.data() + h.cta_off, plan->cta_first.data(),
                plan->cta_first.size() * sizeof(int32_t));
  uint64_t id = 1469598103934665603ull;
  id = fnv1a(id, &plan->prob, sizeof(pd_problem));
  id = fnv1a(id, &h, sizeof(WsHeader));
  id = fnv1a(id, plan->blob.data() + sizeof(WsHeader), plan->blob.size() - sizeof(WsHeader));
  id = fnv1a(id, &plan->num_ctas, sizeof(int32_t));
  plan->plan_id = id;
  h.plan_id = id;
  std::memcpy(plan->blob.data(), &h, sizeof(WsHeader));
  *plan_out = plan;
  return PD_OK;
}

extern "C" size_t paged_decode_workspace_size(const pd_plan* plan) {
  return plan ? (size_t)plan->hdr.total_bytes : 0;
}

extern "C" pd_status paged_decode_plan_get_info(const pd_plan* plan, pd_plan_info* info) {
  if (!plan || !info) return PD_ERR_INVALID_ARG;
  info->num_units = (int32_t)plan->units.size();
  info->num_items = (int32_t)plan->items.size();
  info->num_ctas = plan->num_ctas;
  info->tile_tokens = plan->tile_tokens;
  info->max_splits_used = plan->max_splits_used;
  info->rows_per_unit = plan->rows_per_unit;
  info->partial_rows = plan->partial_rows;
  info->workspace_bytes = plan->hdr.total_bytes;
  info->plan_id = plan->plan_id;
  info->merge_mode = plan->prob.merge_mode;
  info->launches_per_run = 1 + ((plan->prob.merge_mode == PD_MERGE_KERNEL && plan->partial_rows > 0) ? 1 : 0);
  return PD_OK;
}

extern "C" pd_status paged_decode_plan_get_items(const pd_plan* plan, int32_t* items_out) {
  if (!plan || !items_out) return PD_ERR_INVALID_ARG;
  for (size_t i = 0; i < plan->items.size(); ++i) {
    items_out[4 * i + 0] = plan->items[i].unit;
    items_out[4 * i + 1] = plan->items[i].tile_begin;
    items_out[4 * i + 2] = plan->items[i].tile_end;
    items_out[4 * i + 3] = plan->items[i].split;
  }
  return PD_OK;
}

extern "C" void paged_decode_plan_destroy(pd_plan* plan) { delete plan; }

extern "C" const char* pd_status_string(pd_status s) {
  switch (s) {
    case PD_OK: return "ok";
    case PD_ERR_INVALID_ARG: return "invalid argument";
    case PD_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PD_ERR_UNSUPPORTED: return "unsupported shape";
    case PD_ERR_CUDA: return "CUDA runtime error";
    case PD_ERR_DEVICE_FLAG: return "device error flag set";
  }
  return "unknown status";
}

extern "C" int32_t paged_decode_version(void) { return 0x000100; }
