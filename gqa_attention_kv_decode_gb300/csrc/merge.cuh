// merge.cuh -- the log-sum-exp merge of split-KV decode partials, shared by
// the fp32/bf16 and the 4-bit decode paths.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "ptx.cuh"

namespace gqa {
namespace {

__device__ __forceinline__ float load_f(const float* p) { return *p; }
__device__ __forceinline__ float load_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// What the merge needs to know about one decode call.  The split kernel
// writes, for query-head row bh = b*Hq + h and split s < n_used(b),
// ml[bh*n_split + s] = (max in log2 units, sum) and
// part_o[(bh*n_split + s)*D + d] = unnormalised output.
struct MergeParams {
  void* o;
  const int32_t* kv_lens;
  int Hq, max_kv_len, chunk, n_split;
  const float2* ml;
  const float* part_o;
};

// Merges the split partials of one (request, query head) row, after the split
// kernel has finished (programmatic dependent launch: the grid may start
// early; griddepcontrol.wait returns once the split kernel's writes are
// visible).  All partial loads of a thread are issued before the weights are
// known, so the merge costs about one L2 round trip.
//   w_s = 2^(m_s - M) / sum_s l_s 2^(m_s - M),   o = sum_s w_s o_s,   M = max_s m_s
template <typename T, int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(const MergeParams p) {
  constexpr int D4 = D / 4;
  constexpr int NSG = 256 / D4;  // split groups: thread (sg, c4) sums splits sg, sg + NSG, ...
  constexpr int PRE = 8;         // partials held in registers per thread
  __shared__ float w_s[1024];
  __shared__ float4 red[NSG][D4];
  const int bh = blockIdx.x;
  const int b = bh / p.Hq;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c4 = tid % D4, sg = tid / D4;
  grid_launch_dependents();  // the next call's split kernel may start staging
  grid_dependency_wait();
  int L = p.kv_lens ? p.kv_lens[b] : p.max_kv_len;
  L = L < 0 ? 0 : (L > p.max_kv_len ? p.max_kv_len : L);
  const int n_used = (L + p.chunk - 1) / p.chunk;
  if (n_used <= 1) return;  // written by the split kernel itself
  const float2* ml = p.ml + size_t(bh) * p.n_split;
  const float4* po = reinterpret_cast<const float4*>(p.part_o + size_t(bh) * p.n_split * D) + c4;
  float4 x[PRE];
#pragma unroll
  for (int k = 0; k < PRE; ++k) {
    const int sidx = sg + k * NSG;
    x[k] = sidx < n_used ? __ldcg(po + size_t(sidx) * D4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (warp == 0) {
    // (m, l) of splits lane, lane + 32, ...: the first ML_REG of them stay in
    // registers between the max and the weights, the rest are read twice
    constexpr int ML_REG = 4;
    float2 mlr[ML_REG];
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < ML_REG; ++k) {
      const int sidx = lane + 32 * k;
      mlr[k] = sidx < n_used ? __ldcg(&ml[sidx]) : make_float2(-INFINITY, 0.f);
      M = fmaxf(M, mlr[k].x);
    }
    for (int sidx = lane + 32 * ML_REG; sidx < n_used; sidx += 32) M = fmaxf(M, __ldcg(&ml[sidx]).x);
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
    float Ls = 0.f;
#pragma unroll
    for (int k = 0; k < ML_REG; ++k) {
      const int sidx = lane + 32 * k;
      if (sidx < n_used) {
        const float w = fast_exp2(mlr[k].x - M);
        w_s[sidx] = w;
        Ls += mlr[k].y * w;
      }
    }
    for (int sidx = lane + 32 * ML_REG; sidx < n_used; sidx += 32) {
      const float2 v = __ldcg(&ml[sidx]);
      const float w = fast_exp2(v.x - M);
      w_s[sidx] = w;
      Ls += v.y * w;
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, m);
    const float inv = 1.f / Ls;
    for (int sidx = lane; sidx < n_used; sidx += 32) w_s[sidx] *= inv;
  }
  __syncthreads();
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < PRE; ++k) {
    const int sidx = sg + k * NSG;
    if (sidx < n_used) {
      const float w = w_s[sidx];
      acc.x += x[k].x * w;
      acc.y += x[k].y * w;
      acc.z += x[k].z * w;
      acc.w += x[k].w * w;
    }
  }
  for (int sidx = sg + PRE * NSG; sidx < n_used; sidx += NSG) {
    const float4 v = __ldcg(po + size_t(sidx) * D4);
    const float w = w_s[sidx];
    acc.x += v.x * w;
    acc.y += v.y * w;
    acc.z += v.z * w;
    acc.w += v.w * w;
  }
  red[sg][c4] = acc;
  __syncthreads();
  if (tid < D4) {
    float4 t = red[0][tid];
#pragma unroll
    for (int k = 1; k < NSG; ++k) {
      const float4 v = red[k][tid];
      t.x += v.x;
      t.y += v.y;
      t.z += v.z;
      t.w += v.w;
    }
    T* dst = static_cast<T*>(p.o) + size_t(bh) * D + tid * 4;
    store_f(dst + 0, t.x);
    store_f(dst + 1, t.y);
    store_f(dst + 2, t.z);
    store_f(dst + 3, t.w);
  }
}

// Launches `kern` with programmatic stream serialisation: the grid may start
// once every CTA of the preceding grid in the stream has called
// griddepcontrol.launch_dependents (or exited), and must itself call
// griddepcontrol.wait before it touches memory that grid may write.
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The merge grid (one CTA per request and query head) overlaps the split
// kernel's tail; the kernel itself waits for the split kernel's results.
template <typename T, int D>
cudaError_t launch_merge(const MergeParams& p, int rows, cudaStream_t stream) {
  return launch_pdl(decode_merge_kernel<T, D>, dim3(rows), dim3(256), 0, stream, p);
}

}  // namespace
}  // namespace gqa
