// Workspace layout shared by the host planner and the CUDA kernels.
//
// The workspace is caller-owned device memory:
//   [0, 256)            WsHeader
//   units_off           UnitDesc[num_units]
//   items_off           ItemDesc[num_items]   (64 B each; queue order, or grouped by CTA)
//   cta_off             int32[num_ctas + 1]   first item of each CTA (static schedule only)
//   counters_off        uint32[num_units]     split arrival counters (self-reset)
//   plse_off            float[partial_rows]   split LSE (log2 domain)
//   po_off              float[partial_rows * head_dim_v] normalised split output
// paged_decode_plan_upload writes everything up to the counters (zeroed);
// the partial arrays need no initial value.
#pragma once
#include <stdint.h>

namespace pd {

constexpr uint32_t kWsMagic = 0x31575050u;  // "PPW1"
constexpr int kMaxSplits = 16;

struct WsHeader {
  uint32_t magic;
  uint32_t version;
  uint64_t plan_id;
  int32_t error_code;      // first device error (pd_device_error), 0 = none
  int32_t error_info;      // request index of that error, or -1
  uint32_t queue_counter;  // persistent work queue head
  uint32_t done_counter;   // CTAs that have left the queue
  int32_t num_units;
  int32_t num_items;
  int64_t units_off, items_off, counters_off, plse_off, po_off;
  int64_t total_bytes;
  int64_t cta_off;         // int32[num_ctas + 1] item ranges per CTA, or 0 (shared queue)
  int32_t num_ctas;
  int32_t pad0;
  uint8_t pad[256 - 104];
};
static_assert(sizeof(WsHeader) == 256, "header size");

// One independent unit of work: the query rows of one request that share
// one KV head (GQA) or the latent head (MLA), cut into row blocks of at most
// the kernel's MMA height.
struct UnitDesc {
  int32_t b;             // request
  int32_t g;             // kv head (GQA) / 0 (MLA)
  int32_t row0;          // first packed row of this block within (b, g)
  int32_t nrows;         // rows in this block
  int32_t q_start;       // first query row of the request (q_indptr[b])
  int32_t q_len;         // query rows of the request
  int32_t kv_len;        // seq_lens[b]
  int32_t n_splits;      // 1 = written directly to out
  int64_t partial_base;  // first partial row (splits * nrows rows), -1 if unsplit
  int32_t pad[2];
};
static_assert(sizeof(UnitDesc) == 48, "unit size");

// A work item carries a copy of its unit so that one load describes it.
struct ItemDesc {
  int32_t unit;
  int32_t tile_begin;
  int32_t tile_end;      // exclusive
  int32_t split;
  UnitDesc u;
};
static_assert(sizeof(ItemDesc) == 64, "item size");

}  // namespace pd
