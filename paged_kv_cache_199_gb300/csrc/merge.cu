// LSE merge of split attention states (the split-KV combine step).
//
// PR #4557 ("Blackwell TRT-LLM MLA decode backend") pairs its split-KV
// attention kernel with a reducer, and PR #5552 launches warp-per-row merge
// kernels as programmatic dependents of the attention kernel. The merge of
// states s over disjoint key ranges is
//   lse = log sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) out_s,
// with empty states (lse_s = -inf) carrying no weight.
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "device_common.cuh"
#include "kernels.h"
#include "ws_layout.h"

namespace pd {
namespace {

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* dst, float a, float b, float c, float d) {
  *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16(a, b), pack_bf16(c, d));
}

// One thread per (unit row, 4 channels); blocks are laid out over the units
// in plan order (threads of unsplit units exit at once). All split LSEs and
// partial outputs of a row are loaded before any is used, so a row costs two
// dependent L2 round trips whatever its split count.
__global__ void __launch_bounds__(256) unit_merge_kernel(const UnitMergeParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the decode grid's writes are visible
  // a workspace that holds another plan has no states of this one (the
  // decode kernel has set the error word): write nothing
  if (p.hdr->magic != kWsMagic || p.hdr->plan_id != p.plan_id) return;
  const int per_row = p.dim / 4;                      // threads per row
  const int rows_per_block = blockDim.x / per_row;
  const int unit = blockIdx.x;
  const UnitDesc u = p.units[unit];
  if (u.n_splits <= 1) return;
  const int r = blockIdx.y * rows_per_block + (int)threadIdx.x / per_row;
  if (r >= u.nrows) return;
  const int c = ((int)threadIdx.x % per_row) * 4;
  const size_t base = (size_t)u.partial_base + r;
  const int ns = u.n_splits;
  float ls[kMaxSplits];
#pragma unroll
  for (int k = 0; k < kMaxSplits; ++k) ls[k] = k < ns ? p.plse[base + (size_t)k * u.nrows] : -INFINITY;
  float4 v[kMaxSplits];
#pragma unroll
  for (int k = 0; k < kMaxSplits; ++k)
    v[k] = k < ns ? *reinterpret_cast<const float4*>(p.po + (base + (size_t)k * u.nrows) * p.dim + c)
                  : make_float4(0.f, 0.f, 0.f, 0.f);
  const int pr = u.row0 + r;
  const int qi = pr / p.group;
  const int head = u.g * p.group + (pr - qi * p.group);
  const float s2 = sink_log2(p.sinks, head);
  float Mx = s2;
  bool bad = false;
#pragma unroll
  for (int k = 0; k < kMaxSplits; ++k) {
    bad |= isnan(ls[k]);
    Mx = fmaxf(Mx, ls[k]);
  }
  float W = (bad || s2 == -INFINITY) ? 0.f : fast_exp2(s2 - Mx);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!bad && Mx != -INFINITY) {
#pragma unroll
    for (int k = 0; k < kMaxSplits; ++k) {
      const float w = ls[k] == -INFINITY ? 0.f : fast_exp2(ls[k] - Mx);
      W += w;
      acc.x += w * v[k].x;
      acc.y += w * v[k].y;
      acc.z += w * v[k].z;
      acc.w += w * v[k].w;
    }
  }
  const float winv = W > 0.f ? 1.f / W : 0.f;
  const size_t out_row = (size_t)(u.q_start + qi) * p.num_q_heads + head;
  if (bad) {
    store_bf16x4(p.out + out_row * p.dim + c, 0.f, 0.f, 0.f, 0.f);
  } else {
    store_bf16x4(p.out + out_row * p.dim + c, acc.x * winv, acc.y * winv, acc.z * winv, acc.w * winv);
  }
  if (p.lse != nullptr && c == 0)
    p.lse[out_row] = bad ? NAN : (W > 0.f ? (Mx + __log2f(W)) * kLn2 : -INFINITY);
}

// General states: v [S][rows][dim], s [S][rows] natural-log LSE. One warp per row.
__global__ void __launch_bounds__(256) merge_states_kernel(const float* __restrict__ v,
                                                           const float* __restrict__ s, int S,
                                                           int64_t rows, int dim,
                                                           __nv_bfloat16* __restrict__ out,
                                                           float* __restrict__ lse) {
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float Mx = -INFINITY;
  for (int k = 0; k < S; ++k) Mx = fmaxf(Mx, s[(int64_t)k * rows + row] * kLog2e);
  float W = 0.f;
  if (Mx != -INFINITY)
    for (int k = 0; k < S; ++k) {
      const float x = s[(int64_t)k * rows + row] * kLog2e;
      if (x != -INFINITY) W += fast_exp2(x - Mx);
    }
  const float winv = W > 0.f ? 1.f / W : 0.f;
  for (int c = lane * 8; c < dim; c += 256) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (Mx != -INFINITY)
      for (int k = 0; k < S; ++k) {
        const float x = s[(int64_t)k * rows + row] * kLog2e;
        if (x == -INFINITY) continue;
        const float w = fast_exp2(x - Mx) * winv;
        const float4* src = reinterpret_cast<const float4*>(v + ((int64_t)k * rows + row) * dim + c);
        const float4 a = src[0], b = src[1];
        acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
        acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
      }
    __nv_bfloat16* dst = out + row * dim + c;
    *reinterpret_cast<uint4*>(dst) = make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]),
                                                pack_bf16(acc[4], acc[5]), pack_bf16(acc[6], acc[7]));
  }
  if (lse != nullptr && lane == 0) lse[row] = W > 0.f ? (Mx + __log2f(W)) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_unit_merge(const UnitMergeParams& p, cudaStream_t stream, bool pdl) {
  if (p.num_units == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  const int per_row = p.dim / 4;
  const int rows_per_block = 256 / per_row;
  cfg.gridDim = dim3((unsigned)p.num_units, (unsigned)((p.max_rows + rows_per_block - 1) / rows_per_block));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, unit_merge_kernel, p);
}

cudaError_t launch_merge_states(const float* v, const float* s, int num_states, int64_t rows,
                                int dim, __nv_bfloat16* out, float* lse, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const int warps = 8;
  const unsigned grid = (unsigned)((rows + warps - 1) / warps);
  merge_states_kernel<<<grid, warps * 32, 0, stream>>>(v, s, num_states, rows, dim, out, lse);
  return cudaGetLastError();
}

}  // namespace pd
