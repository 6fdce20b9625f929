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

// One warp per unit row; blocks of eight rows are laid out over the units in
// plan order (warps of unsplit units exit at once). Lane k reads split k's
// LSE, so the row's maximum and weight sum are warp reductions; each lane
// then reads its 16-byte column groups of the row's partial outputs, four
// splits' loads in flight before they are used. The plan check and the unit
// descriptor are read together: the states follow one round trip later.
constexpr int kMergeRowsPerBlock = 8;
constexpr int kMergeSplitBatch = 4;    // splits whose loads are in flight together
constexpr int kMergeVecPerLane = 4;    // 16-byte column groups per lane and pass (512 channels)
static_assert(kMaxSplits <= 32, "one lane per split's LSE");

__global__ void __launch_bounds__(kMergeRowsPerBlock * 32) unit_merge_kernel(const UnitMergeParams p) {
  const int lane = threadIdx.x & 31;
  const int unit = blockIdx.x;
  const int r = blockIdx.y * kMergeRowsPerBlock + (int)(threadIdx.x >> 5);
  // The plan header, the unit descriptors and the sinks were in place before
  // the decode grid started and it does not write them, so they are read
  // before the wait for its states (one round trip less after it ends).
  const uint32_t magic = p.hdr->magic;
  const uint64_t plan_id = p.hdr->plan_id;
  const UnitDesc u = p.units[unit];
  // a workspace that holds another plan has no states of this one (the
  // decode kernel has set the error word): write nothing
  if (magic != kWsMagic || plan_id != p.plan_id) return;
  if (u.n_splits <= 1 || r >= u.nrows) return;
  const int pr = u.row0 + r;
  const int qi = pr / p.group;
  const int head = u.g * p.group + (pr - qi * p.group);
  const float s2 = sink_log2(p.sinks, head);
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the decode grid's writes are visible
  const int ns = u.n_splits;   // <= kMaxSplits <= 32
  const size_t base = (size_t)u.partial_base + r;
  const int nvec = p.dim / 4;                         // 16-byte column groups of a row
  // column groups f0 + lane + 32 j of splits k0 .. k0 + 3
  auto load_batch = [&](int f0, int k0, float4 (&v)[kMergeSplitBatch][kMergeVecPerLane]) {
#pragma unroll
    for (int k = 0; k < kMergeSplitBatch; ++k)
#pragma unroll
      for (int j = 0; j < kMergeVecPerLane; ++j) {
        const int f = f0 + lane + 32 * j;
        v[k][j] = (k0 + k < ns && f < nvec)
                      ? *reinterpret_cast<const float4*>(p.po + (base + (size_t)(k0 + k) * u.nrows) * p.dim + 4 * f)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
  };
  // the LSEs and the first batch of partial outputs are read together
  const float lk = lane < ns ? p.plse[base + (size_t)lane * u.nrows] : -INFINITY;
  float4 v[kMergeSplitBatch][kMergeVecPerLane];
  load_batch(0, 0, v);
  const bool bad = __any_sync(0xffffffffu, isnan(lk));
  float Mx = lk;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, o));
  Mx = fmaxf(Mx, s2);
  const float wk = (bad || lk == -INFINITY || Mx == -INFINITY) ? 0.f : fast_exp2(lk - Mx);
  float W = wk;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
  if (!bad && s2 != -INFINITY) W += fast_exp2(s2 - Mx);
  const float winv = W > 0.f ? 1.f / W : 0.f;
  const size_t out_row = (size_t)(u.q_start + qi) * p.num_q_heads + head;
  for (int f0 = 0; f0 < nvec; f0 += 32 * kMergeVecPerLane) {
    float4 acc[kMergeVecPerLane];
#pragma unroll
    for (int j = 0; j < kMergeVecPerLane; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    // a NaN state (an errored split) or no weight at all gives a zero row
    for (int k0 = 0; k0 < ns && !bad && Mx != -INFINITY; k0 += kMergeSplitBatch) {
      if (f0 != 0 || k0 != 0) load_batch(f0, k0, v);
#pragma unroll
      for (int k = 0; k < kMergeSplitBatch; ++k) {
        const float w = __shfl_sync(0xffffffffu, wk, (k0 + k) & 31);   // 0 past the splits, and if bad
#pragma unroll
        for (int j = 0; j < kMergeVecPerLane; ++j) {
          acc[j].x += w * v[k][j].x;
          acc[j].y += w * v[k][j].y;
          acc[j].z += w * v[k][j].z;
          acc[j].w += w * v[k][j].w;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kMergeVecPerLane; ++j) {
      const int f = f0 + lane + 32 * j;
      if (f < nvec)
        store_bf16x4(p.out + out_row * p.dim + 4 * f, acc[j].x * winv, acc[j].y * winv, acc[j].z * winv,
                     acc[j].w * winv);
    }
  }
  if (p.lse != nullptr && lane == 0)
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
  cfg.gridDim = dim3((unsigned)p.num_units, (unsigned)((p.max_rows + kMergeRowsPerBlock - 1) / kMergeRowsPerBlock));
  cfg.blockDim = dim3(kMergeRowsPerBlock * 32);
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
