// Host-side plan object shared by the planner (plan.cpp) and the launch
// code (api.cu). Not part of the public ABI.
#pragma once
#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "paged_decode.h"
#include "ws_layout.h"

namespace pd {

// Kernel geometry the planner must agree with.
constexpr int kGqaTileTokens = 64;   // tokens per pipeline stage (BF16 pools)
constexpr int kGqaFp8TileTokens = 128;  // E4M3 pools: 128-token stages of the same bytes
constexpr int kGqaRowsPerUnit = 16;  // two n8 MMA blocks of packed query rows (8 if all fit)
constexpr int kMlaTileTokens = 64;
constexpr int kMlaRowsPerUnit = 64;  // four m16 tiles of packed (token, head) rows
constexpr int kPrefillTileTokens = 128;  // keys per tensor-core tile of the prefill kernel
constexpr int kPrefillRowsPerUnit = 256; // packed (token, head) rows per prefill unit: two 128-row query tiles

}  // namespace pd

struct pd_plan {
  pd_problem prob;
  int32_t num_sms = 0;
  int32_t num_ctas = 0;
  int32_t tile_tokens = 0;
  int32_t rows_per_unit = 0;
  int32_t max_splits_used = 0;
  int64_t partial_rows = 0;
  int64_t total_q = 0;
  uint64_t plan_id = 0;
  pd::WsHeader hdr{};                 // offsets + identity, copied into the blob
  std::vector<pd::UnitDesc> units;
  std::vector<pd::ItemDesc> items;
  std::vector<int32_t> cta_first;      // static schedule: first item of each CTA (+ end), else empty
  std::vector<uint8_t> blob;          // bytes [0, end of the CTA table) of the workspace
  std::vector<int32_t> seq_lens;      // host copies the plan was built from
  std::vector<int32_t> q_indptr;
};

namespace pd {
// Number of persistent CTAs resident per SM for a problem's kernel.
int ctas_per_sm(const pd_problem& p);
}
