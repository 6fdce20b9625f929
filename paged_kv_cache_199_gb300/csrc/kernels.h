// Internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "paged_decode.h"
#include "ws_layout.h"

namespace pd {

struct GqaParams {
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* q_indptr;   // nullptr: one query row per request
  const float* k_scale;      // E4M3 pools only
  const float* v_scale;
  const float* sinks;        // [num_q_heads] sink logits (natural log), or nullptr
  __nv_bfloat16* out;
  float* lse;                // nullptr: not requested
  WsHeader* hdr;
  const UnitDesc* units;
  const ItemDesc* items;
  const int32_t* cta_items;  // static schedule: item range of each CTA; nullptr: shared queue
  uint32_t* counters;
  float* plse;
  float* po;
  uint64_t plan_id;
  int32_t num_items;
  int32_t num_q_heads;
  int32_t group;             // Hq / Hkv
  int32_t page_size;
  int32_t num_pages;
  int32_t max_pages_per_seq;
  int32_t box_rows;          // tokens per TMA box (power of two dividing page_size, <= 64)
  int32_t swizzle;           // 1: tiles use the 128-byte TMA swizzle
  int32_t layout;            // PD_LAYOUT_*
  int32_t fused_merge;       // 1: last split merges inside the kernel
  float sm_scale;
  uint64_t wait_ns;          // limit of every pipeline wait (PD_DEV_TIMEOUT past it)
};

struct MlaParams {
  const __nv_bfloat16* q;    // [total_q][H][576]
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* q_indptr;
  const float* sinks;        // [H] sink logits (natural log), or nullptr
  const float* q_scale;      // E4M3 query and latent pool: q = code * q_scale
  const float* kv_scale;     //   and kv = code * kv_scale
  __nv_bfloat16* out;        // [total_q][H][512]
  float* lse;
  WsHeader* hdr;
  const UnitDesc* units;
  const ItemDesc* items;
  const int32_t* cta_items;  // static schedule: item range of each CTA; nullptr: shared queue
  uint32_t* counters;
  float* plse;
  float* po;
  uint64_t plan_id;
  int32_t num_items;
  int32_t num_heads;
  int32_t page_size;
  int32_t num_pages;
  int32_t max_pages_per_seq;
  int32_t box_rows;
  int32_t swizzle;
  int32_t fused_merge;
  float sm_scale;
  uint64_t wait_ns;          // limit of every pipeline wait (PD_DEV_TIMEOUT past it)
  const uint8_t* kv_pool;    // the latent pool's bytes (L2 prefetch of whole pages)
  int64_t page_bytes;        // bytes of one page
};

// Merge of split partial states stored in a plan's workspace (units with
// n_splits > 1) into the output rows. LSE values there are in the log2 domain.
struct UnitMergeParams {
  const WsHeader* hdr;       // the workspace: merged only if it holds plan_id
  uint64_t plan_id;
  const UnitDesc* units;
  int32_t num_units;
  const float* plse;
  const float* po;
  const float* sinks;        // [num_q_heads] sink logits (natural log), or nullptr
  __nv_bfloat16* out;
  float* lse;
  int32_t dim;               // head_dim_v (a multiple of 4, <= 1024)
  int32_t max_rows;          // largest nrows of any unit
  int32_t num_q_heads;
  int32_t group;             // query heads per KV head (GQA) or H (MLA)
};

cudaError_t ensure_smem_attr(const void* func, int bytes);
// The pipeline wait limit the next launches get (paged_decode_set_wait_limit_ns);
// kWaitLimitNsHost (2 s, the kernels' kWaitLimitNs) unless a caller set another.
constexpr uint64_t kWaitLimitNsHost = 2000000000ull;
uint64_t wait_limit_ns();
// Records a failed CUDA call for paged_decode_last_cuda_error(); returns PD_ERR_CUDA.
pd_status cuda_fail(cudaError_t e, const char* where);
cudaError_t launch_gqa_decode(const CUtensorMap& kmap, const CUtensorMap& vmap, const GqaParams& p,
                              bool fp8, int rows_per_unit, int grid, cudaStream_t stream);
cudaError_t launch_gqa_prefill(const CUtensorMap& kmap, const CUtensorMap& vmap, const CUtensorMap& qmap,
                               const GqaParams& p, int grid, cudaStream_t stream);
cudaError_t launch_mla_decode(const CUtensorMap& kvmap, const CUtensorMap& qmap, const MlaParams& p,
                              bool fp8, int grid, cudaStream_t stream);
cudaError_t launch_unit_merge(const UnitMergeParams& p, cudaStream_t stream, bool pdl);
cudaError_t launch_merge_states(const float* v, const float* s, int num_states, int64_t rows,
                                int dim, __nv_bfloat16* out, float* lse, cudaStream_t stream);

}  // namespace pd
