// C-ABI entry points of libpaged_decode.so: argument checks, TMA descriptor
// encoding and kernel launches. No device allocation happens here.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "kernels.h"
#include "paged_decode.h"
#include "plan_internal.h"
#include "ws_layout.h"

namespace pd {

namespace {
thread_local char g_last_cuda_error[256] = "";
// limit of the kernels' pipeline waits for the next launches (0: the default)
std::atomic<uint64_t> g_wait_limit_ns{0};
}

uint64_t wait_limit_ns() {
  const uint64_t v = g_wait_limit_ns.load(std::memory_order_relaxed);
  return v == 0 ? kWaitLimitNsHost : v;
}

// Record a failed CUDA call for paged_decode_last_cuda_error() and clear the
// runtime's sticky-free error state.
pd_status cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s (%d)", where, cudaGetErrorString(e), (int)e);
  cudaGetLastError();
  return PD_ERR_CUDA;
}

cudaError_t ensure_smem_attr(const void* func, int bytes) {
  // The attribute is per device; remember which devices were configured.
  static std::mutex mu;
  static const void* done_func[64][4] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64)
    for (int i = 0; i < 4; ++i)
      if (done_func[dev][i] == func) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64)
    for (int i = 0; i < 4; ++i)
      if (done_func[dev][i] == nullptr) {
        done_func[dev][i] = func;
        break;
      }
  return cudaSuccess;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    cudaGetLastError();
  });
  return fn;
}

// Largest power of two dividing the page size, at most 64: the rows of one
// TMA box never cross a page.
int box_rows_for(int page_size) {
  int br = page_size & (-page_size);
  return br > 64 ? 64 : br;
}

// A paged pool as a 4-D tensor whose box is `box_rows` token rows of 128
// bytes: HND {D, P, Hkv, pages}, NHD {D, Hkv, P, pages}, MLA {576, 1, P, pages}.
bool encode_pool_map(CUtensorMap* map, const void* base, bool fp8, int layout, int64_t num_pages,
                     int64_t page_size, int64_t num_kv_heads, int64_t head_dim, int64_t page_stride,
                     int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t e = fp8 ? 1 : 2;
  cuuint64_t dims[4];
  cuuint64_t strides[3];
  cuuint32_t box[4];
  const cuuint32_t elem_strides[4] = {1, 1, 1, 1};
  dims[0] = (cuuint64_t)head_dim;
  box[0] = (cuuint32_t)(128 / e);
  if (layout == PD_LAYOUT_HND) {
    dims[1] = page_size;
    dims[2] = num_kv_heads;
    strides[0] = head_dim * e;
    strides[1] = page_size * head_dim * e;
    box[1] = box_rows;
    box[2] = 1;
  } else {
    dims[1] = num_kv_heads;
    dims[2] = page_size;
    strides[0] = head_dim * e;
    strides[1] = num_kv_heads * head_dim * e;
    box[1] = 1;
    box[2] = box_rows;
  }
  dims[3] = num_pages;
  strides[2] = page_stride * e;
  box[3] = 1;
  const CUtensorMapSwizzle swz = box_rows >= 8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                  const_cast<void*>(base), dims, strides, box, elem_strides,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// MLA query rows [total_q * H][576] as a 2-D tensor (padded to 4-D) read in
// 64-row x 64-channel swizzled boxes.
bool encode_mla_query_map(CUtensorMap* map, const void* q, int64_t rows, bool fp8) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t e = fp8 ? 1 : 2;   // E4M3: boxes of 128 channels; the fifth reads zeros past 576
  const cuuint64_t dims[4] = {576, (cuuint64_t)rows, 1, 1};
  const cuuint64_t strides[3] = {576 * e, (cuuint64_t)rows * 576 * e, (cuuint64_t)rows * 576 * e};
  const cuuint32_t box[4] = {(cuuint32_t)(128 / e), 64, 1, 1};
  const cuuint32_t elem_strides[4] = {1, 1, 1, 1};
  return fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q),
            dims, strides, box, elem_strides,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// GQA query rows [total_q][Hq][128] read as 128 packed (token, head) rows:
// a box of 64 channels x `group` heads x 128 / group tokens per slab.
bool encode_prefill_query_map(CUtensorMap* map, const void* q, int64_t total_q, int num_q_heads, int group) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {128, (cuuint64_t)num_q_heads, (cuuint64_t)total_q, 1};
  const cuuint64_t strides[3] = {128 * 2, (cuuint64_t)num_q_heads * 128 * 2,
                                 (cuuint64_t)total_q * num_q_heads * 128 * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)group, (cuuint32_t)(128 / group), 1};
  const cuuint32_t elem_strides[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, elem_strides,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct WsPtrs {
  WsHeader* hdr;
  const UnitDesc* units;
  const ItemDesc* items;
  const int32_t* cta_items;
  uint32_t* counters;
  float* plse;
  float* po;
};

WsPtrs ws_ptrs(const pd_plan* plan, void* ws) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  const WsHeader& h = plan->hdr;
  return WsPtrs{reinterpret_cast<WsHeader*>(b), reinterpret_cast<const UnitDesc*>(b + h.units_off),
                reinterpret_cast<const ItemDesc*>(b + h.items_off),
                h.cta_off ? reinterpret_cast<const int32_t*>(b + h.cta_off) : nullptr,
                reinterpret_cast<uint32_t*>(b + h.counters_off), reinterpret_cast<float*>(b + h.plse_off),
                reinterpret_cast<float*>(b + h.po_off)};
}

pd_status check_workspace(const pd_plan* plan, const void* ws, size_t bytes) {
  if (!ws || !aligned16(ws)) return PD_ERR_INVALID_ARG;
  if (bytes < (size_t)plan->hdr.total_bytes) return PD_ERR_WORKSPACE_TOO_SMALL;
  return PD_OK;
}

pd_status launch_merge_if_needed(const pd_plan* plan, const WsPtrs& w, void* out, float* lse,
                                 const float* sinks, cudaStream_t stream) {
  if (plan->prob.merge_mode != PD_MERGE_KERNEL || plan->partial_rows == 0) return PD_OK;
  const bool mla = plan->prob.kind == PD_ATTN_MLA;
  UnitMergeParams mp{};
  mp.hdr = w.hdr;
  mp.plan_id = plan->plan_id;
  mp.units = w.units;
  mp.num_units = (int32_t)plan->units.size();
  mp.plse = w.plse;
  mp.po = w.po;
  mp.sinks = sinks;
  mp.out = static_cast<__nv_bfloat16*>(out);
  mp.lse = lse;
  mp.dim = plan->prob.head_dim_v;
  mp.max_rows = plan->rows_per_unit;
  mp.num_q_heads = plan->prob.num_q_heads;
  mp.group = mla ? plan->prob.num_q_heads : plan->prob.num_q_heads / plan->prob.num_kv_heads;
  const cudaError_t e = launch_unit_merge(mp, stream, true);
  return e == cudaSuccess ? PD_OK : cuda_fail(e, "LSE merge launch");
}

}  // namespace
}  // namespace pd

using namespace pd;

extern "C" pd_status paged_decode_plan_upload(const pd_plan* plan, void* workspace,
                                              size_t workspace_bytes, pd_stream_t stream) {
  if (!plan) return PD_ERR_INVALID_ARG;
  pd_status st = check_workspace(plan, workspace, workspace_bytes);
  if (st != PD_OK) return st;
  const cudaError_t e = cudaMemcpyAsync(workspace, plan->blob.data(), plan->blob.size(),
                                        cudaMemcpyHostToDevice, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "plan upload");
  return PD_OK;
}

namespace pd {
namespace {

pd_status run_gqa(const pd_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                  const int32_t* block_tables, const int32_t* seq_lens, const int32_t* q_indptr,
                  float sm_scale, const float* k_scale, const float* v_scale, const float* sinks,
                  void* out, float* lse, void* workspace, size_t workspace_bytes, pd_stream_t stream) {
  if (!plan || plan->prob.kind != PD_ATTN_GQA) return PD_ERR_INVALID_ARG;
  pd_status st = check_workspace(plan, workspace, workspace_bytes);
  if (st != PD_OK) return st;
  if (plan->items.empty()) return PD_OK;
  const pd_problem& pr = plan->prob;
  const bool fp8 = pr.kv_dtype == PD_KV_FP8_E4M3;
  if (!q || !k_pool || !v_pool || !block_tables || !seq_lens || !out) return PD_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out)) return PD_ERR_INVALID_ARG;
  if (fp8 && (!k_scale || !v_scale)) return PD_ERR_INVALID_ARG;
  if (!(sm_scale == sm_scale)) return PD_ERR_INVALID_ARG;

  const int br = box_rows_for(pr.page_size);
  CUtensorMap kmap, vmap;
  if (!encode_pool_map(&kmap, k_pool, fp8, pr.layout, pr.num_pages, pr.page_size, pr.num_kv_heads,
                       pr.head_dim_qk, pr.k_page_stride, br) ||
      !encode_pool_map(&vmap, v_pool, fp8, pr.layout, pr.num_pages, pr.page_size, pr.num_kv_heads,
                       pr.head_dim_v, pr.v_page_stride, br))
    return cuda_fail(cudaErrorInvalidValue, "K/V tensor map encoding");

  const WsPtrs w = ws_ptrs(plan, workspace);
  GqaParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.q_indptr = q_indptr;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.sinks = sinks;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.hdr = w.hdr;
  p.units = w.units;
  p.items = w.items;
  p.cta_items = w.cta_items;
  p.counters = w.counters;
  p.plse = w.plse;
  p.po = w.po;
  p.plan_id = plan->plan_id;
  p.num_items = (int32_t)plan->items.size();
  p.num_q_heads = pr.num_q_heads;
  p.group = pr.num_q_heads / pr.num_kv_heads;
  p.page_size = pr.page_size;
  p.num_pages = pr.num_pages;
  p.max_pages_per_seq = pr.max_pages_per_seq;
  p.box_rows = br;
  p.swizzle = br >= 8 ? 1 : 0;
  p.layout = pr.layout;
  p.fused_merge = pr.merge_mode == PD_MERGE_FUSED ? 1 : 0;
  p.sm_scale = sm_scale;
  p.wait_ns = wait_limit_ns();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = launch_gqa_decode(kmap, vmap, p, fp8, plan->rows_per_unit, plan->num_ctas, s);
  if (e != cudaSuccess) return cuda_fail(e, "GQA decode launch");
  return launch_merge_if_needed(plan, w, out, lse, sinks, s);
}

pd_status run_mla(const pd_plan* plan, const void* q, const void* kv_pool, const int32_t* block_tables,
                  const int32_t* seq_lens, const int32_t* q_indptr, float sm_scale, const float* sinks,
                  bool fp8, const float* q_scale, const float* kv_scale, void* out, float* lse,
                  void* workspace, size_t workspace_bytes, pd_stream_t stream) {
  if (!plan || plan->prob.kind != PD_ATTN_MLA) return PD_ERR_INVALID_ARG;
  if (fp8 != (plan->prob.kv_dtype == PD_KV_FP8_E4M3)) return PD_ERR_INVALID_ARG;
  if (fp8 && (!q_scale || !kv_scale)) return PD_ERR_INVALID_ARG;
  pd_status st = check_workspace(plan, workspace, workspace_bytes);
  if (st != PD_OK) return st;
  if (plan->items.empty()) return PD_OK;
  const pd_problem& pr = plan->prob;
  if (!q || !kv_pool || !block_tables || !seq_lens || !out) return PD_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_pool) || !aligned16(out)) return PD_ERR_INVALID_ARG;
  if (!(sm_scale == sm_scale)) return PD_ERR_INVALID_ARG;
  const int br = box_rows_for(pr.page_size);
  CUtensorMap kvmap, qmap;
  // the latent pool is an NHD pool with one head of 576 channels
  if (!encode_pool_map(&kvmap, kv_pool, fp8, PD_LAYOUT_NHD, pr.num_pages, pr.page_size, 1,
                       pr.head_dim_qk, pr.k_page_stride, br) ||
      !encode_mla_query_map(&qmap, q, plan->total_q * pr.num_q_heads, fp8))
    return cuda_fail(cudaErrorInvalidValue, "MLA tensor map encoding");
  const WsPtrs w = ws_ptrs(plan, workspace);
  MlaParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.q_indptr = q_indptr;
  p.sinks = sinks;
  p.q_scale = q_scale;
  p.kv_scale = kv_scale;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.hdr = w.hdr;
  p.units = w.units;
  p.items = w.items;
  p.cta_items = w.cta_items;
  p.counters = w.counters;
  p.plse = w.plse;
  p.po = w.po;
  p.plan_id = plan->plan_id;
  p.num_items = (int32_t)plan->items.size();
  p.num_heads = pr.num_q_heads;
  p.kv_pool = static_cast<const uint8_t*>(kv_pool);
  p.page_bytes = pr.k_page_stride * (fp8 ? 1 : 2);
  p.page_size = pr.page_size;
  p.num_pages = pr.num_pages;
  p.max_pages_per_seq = pr.max_pages_per_seq;
  p.box_rows = br;
  p.swizzle = br >= 8 ? 1 : 0;
  p.fused_merge = pr.merge_mode == PD_MERGE_FUSED ? 1 : 0;
  p.sm_scale = sm_scale;
  p.wait_ns = wait_limit_ns();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_mla_decode(kvmap, qmap, p, fp8, plan->num_ctas, s);
  if (e != cudaSuccess) return cuda_fail(e, "MLA decode launch");
  return launch_merge_if_needed(plan, w, out, lse, sinks, s);
}

pd_status run_prefill(const pd_plan* plan, const void* q, const void* k_pool, const void* v_pool,
                      const int32_t* block_tables, const int32_t* seq_lens, const int32_t* q_indptr,
                      float sm_scale, const float* sinks, void* out, float* lse, void* workspace,
                      size_t workspace_bytes, pd_stream_t stream) {
  if (!plan || plan->prob.kind != PD_ATTN_PREFILL) return PD_ERR_INVALID_ARG;
  pd_status st = check_workspace(plan, workspace, workspace_bytes);
  if (st != PD_OK) return st;
  if (plan->items.empty()) return PD_OK;
  const pd_problem& pr = plan->prob;
  if (!q || !k_pool || !v_pool || !block_tables || !seq_lens || !out) return PD_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out)) return PD_ERR_INVALID_ARG;
  // the kernel takes row maxima of the raw scores, which needs a positive scale
  if (!(sm_scale > 0.f) || !(sm_scale < INFINITY)) return PD_ERR_INVALID_ARG;
  const int br = box_rows_for(pr.page_size);   // >= 8: the plan requires page_size % 8 == 0
  const int group = pr.num_q_heads / pr.num_kv_heads;
  CUtensorMap kmap, vmap, qmap;
  if (!encode_pool_map(&kmap, k_pool, false, pr.layout, pr.num_pages, pr.page_size, pr.num_kv_heads,
                       pr.head_dim_qk, pr.k_page_stride, br) ||
      !encode_pool_map(&vmap, v_pool, false, pr.layout, pr.num_pages, pr.page_size, pr.num_kv_heads,
                       pr.head_dim_v, pr.v_page_stride, br) ||
      !encode_prefill_query_map(&qmap, q, plan->total_q, pr.num_q_heads, group))
    return cuda_fail(cudaErrorInvalidValue, "prefill tensor map encoding");
  const WsPtrs w = ws_ptrs(plan, workspace);
  GqaParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.q_indptr = q_indptr;
  p.sinks = sinks;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.hdr = w.hdr;
  p.units = w.units;
  p.items = w.items;
  p.cta_items = w.cta_items;
  p.counters = w.counters;
  p.plse = w.plse;
  p.po = w.po;
  p.plan_id = plan->plan_id;
  p.num_items = (int32_t)plan->items.size();
  p.num_q_heads = pr.num_q_heads;
  p.group = group;
  p.page_size = pr.page_size;
  p.num_pages = pr.num_pages;
  p.max_pages_per_seq = pr.max_pages_per_seq;
  p.box_rows = br;
  p.swizzle = 1;
  p.layout = pr.layout;
  p.fused_merge = 0;
  p.sm_scale = sm_scale;
  p.wait_ns = wait_limit_ns();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = launch_gqa_prefill(kmap, vmap, qmap, p, plan->num_ctas, s);
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return launch_merge_if_needed(plan, w, out, lse, sinks, s);
}

}  // namespace
}  // namespace pd

extern "C" pd_status paged_decode_run(const pd_plan* plan, const void* q, const void* k_pool,
                                      const void* v_pool, const int32_t* block_tables,
                                      const int32_t* seq_lens, const int32_t* q_indptr,
                                      float sm_scale, const float* k_scale, const float* v_scale,
                                      void* out, float* lse, void* workspace,
                                      size_t workspace_bytes, pd_stream_t stream) {
  return pd::run_gqa(plan, q, k_pool, v_pool, block_tables, seq_lens, q_indptr, sm_scale, k_scale, v_scale,
                     nullptr, out, lse, workspace, workspace_bytes, stream);
}

extern "C" pd_status paged_decode_run_sinks(const pd_plan* plan, const void* q, const void* k_pool,
                                            const void* v_pool, const int32_t* block_tables,
                                            const int32_t* seq_lens, const int32_t* q_indptr,
                                            float sm_scale, const float* k_scale, const float* v_scale,
                                            const float* sinks, void* out, float* lse, void* workspace,
                                            size_t workspace_bytes, pd_stream_t stream) {
  if (!sinks) return PD_ERR_INVALID_ARG;
  return pd::run_gqa(plan, q, k_pool, v_pool, block_tables, seq_lens, q_indptr, sm_scale, k_scale, v_scale,
                     sinks, out, lse, workspace, workspace_bytes, stream);
}

extern "C" pd_status paged_prefill_run(const pd_plan* plan, const void* q, const void* k_pool,
                                       const void* v_pool, const int32_t* block_tables,
                                       const int32_t* seq_lens, const int32_t* q_indptr, float sm_scale,
                                       const float* sinks, void* out, float* lse, void* workspace,
                                       size_t workspace_bytes, pd_stream_t stream) {
  return pd::run_prefill(plan, q, k_pool, v_pool, block_tables, seq_lens, q_indptr, sm_scale, sinks, out, lse,
                         workspace, workspace_bytes, stream);
}

extern "C" pd_status mla_decode_run(const pd_plan* plan, const void* q, const void* kv_pool,
                                    const int32_t* block_tables, const int32_t* seq_lens,
                                    const int32_t* q_indptr, float sm_scale, void* out, float* lse,
                                    void* workspace, size_t workspace_bytes, pd_stream_t stream) {
  return pd::run_mla(plan, q, kv_pool, block_tables, seq_lens, q_indptr, sm_scale, nullptr, false, nullptr,
                     nullptr, out, lse, workspace, workspace_bytes, stream);
}

extern "C" pd_status mla_decode_run_fp8(const pd_plan* plan, const void* q, const void* kv_pool,
                                        const int32_t* block_tables, const int32_t* seq_lens,
                                        const int32_t* q_indptr, float sm_scale, const float* q_scale,
                                        const float* kv_scale, const float* sinks, void* out, float* lse,
                                        void* workspace, size_t workspace_bytes, pd_stream_t stream) {
  return pd::run_mla(plan, q, kv_pool, block_tables, seq_lens, q_indptr, sm_scale, sinks, true, q_scale,
                     kv_scale, out, lse, workspace, workspace_bytes, stream);
}

extern "C" pd_status mla_decode_run_sinks(const pd_plan* plan, const void* q, const void* kv_pool,
                                          const int32_t* block_tables, const int32_t* seq_lens,
                                          const int32_t* q_indptr, float sm_scale, const float* sinks,
                                          void* out, float* lse, void* workspace, size_t workspace_bytes,
                                          pd_stream_t stream) {
  if (!sinks) return PD_ERR_INVALID_ARG;
  return pd::run_mla(plan, q, kv_pool, block_tables, seq_lens, q_indptr, sm_scale, sinks, false, nullptr,
                     nullptr, out, lse, workspace, workspace_bytes, stream);
}

extern "C" pd_status paged_decode_merge_states(const float* v_states, const float* s_states,
                                               int32_t num_states, int64_t rows, int32_t dim,
                                               void* out, float* lse_out, pd_stream_t stream) {
  if (num_states < 1 || num_states > 64 || rows < 0 || dim < 8 || dim > 1024 || dim % 8 != 0)
    return PD_ERR_INVALID_ARG;
  if (rows == 0) return PD_OK;
  if (!v_states || !s_states || !out || !aligned16(v_states) || !aligned16(out)) return PD_ERR_INVALID_ARG;
  const cudaError_t e = launch_merge_states(v_states, s_states, num_states, rows, dim,
                                            static_cast<__nv_bfloat16*>(out), lse_out,
                                            reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "LSE merge launch");
  return PD_OK;
}

extern "C" pd_status paged_decode_read_error(void* workspace, int32_t* code_out, int32_t* info_out,
                                             pd_stream_t stream) {
  if (!workspace || !code_out) return PD_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  int32_t buf[2] = {0, -1};
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(buf, &hdr->error_code, sizeof buf, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  const int32_t clear[2] = {0, -1};
  e = cudaMemcpy(&hdr->error_code, clear, sizeof clear, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clear error word");
  *code_out = buf[0];
  if (info_out) *info_out = buf[1];
  return buf[0] == PD_DEV_OK ? PD_OK : PD_ERR_DEVICE_FLAG;
}

extern "C" const char* paged_decode_last_cuda_error(void) { return pd::g_last_cuda_error; }

extern "C" pd_status paged_decode_set_wait_limit_ns(uint64_t limit_ns) {
  pd::g_wait_limit_ns.store(limit_ns, std::memory_order_relaxed);
  return PD_OK;
}
