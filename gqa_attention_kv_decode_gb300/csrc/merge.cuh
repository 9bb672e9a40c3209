// merge.cuh -- the log-sum-exp merge of split-KV decode partials, shared by
// the fp32/bf16 and the 4-bit decode paths.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "gqa_attn.h"
#include "ptx.cuh"

namespace gqa {
namespace {

__device__ __forceinline__ float load_f(const float* p) { return *p; }
__device__ __forceinline__ float load_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// What the merge needs to know about one decode call.  The split kernel
// writes, for query-head row bh = b*Hq + h and split s < n_used(b) =
// min(n_split, ceil(L_b / chunk)),
// ml[bh*n_split + s] = (max in log2 units, sum) and
// part_o[(bh*n_split + s)*D + d] = unnormalised output.
struct MergeParams {
  void* o;
  const int32_t* kv_lens;
  int Hq, max_kv_len, chunk, n_split;  // n_split: partial slots per row
  const float2* ml;
  const float* part_o;
  // 4-bit cache + residual window (n_quant != nullptr): the 4-bit part of
  // request b has clamp(n_quant[b], 0, max_quant) keys in min(n_split - 1,
  // ceil(that / chunk)) splits, the window clamp(kv_lens[b] - that, 0,
  // res_cap) keys in one more slot;
  // every used slot holds a partial, even when there is only one.
  const int32_t* n_quant = nullptr;
  int max_quant = 0, res_cap = 0;
  uint32_t* status = nullptr;
  int kv_period = 0;  // > 0: layers stacked along the batch axis share kv_lens[b % kv_period]
};

// Merges the split partials of one (request, query head) row, after the split
// kernel has finished (programmatic dependent launch: the grid may start
// early; griddepcontrol.wait returns once the split kernel's writes are
// visible).  Thread (sg, c4) owns columns 4c4..4c4+3 of splits sg, sg + NSG,
// ...; it loads their partials and (m, l) pairs in one round trip and
// combines them online (running maximum), so no block-wide maximum is needed
// before the sums.  One barrier later, NSG per-thread states per column are
// combined with the log-sum-exp rule:
//   M = max_s m_s,   o = sum_s o_s 2^(m_s - M) / sum_s l_s 2^(m_s - M).
// The summation order is fixed, so the result is deterministic.
template <typename T, int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(const MergeParams p) {
  constexpr int D4 = D / 4;
  constexpr int NSG = 256 / D4;  // split groups: thread (sg, c4) takes splits sg, sg + NSG, ...
  constexpr int PRE = 8;         // partials per thread loaded before any is used
  __shared__ float4 red_o[NSG][D4];
  __shared__ float2 red_ml[NSG];
  const int bh = blockIdx.x;
  const int b = bh / p.Hq;
  const int tid = threadIdx.x;
  const int c4 = tid % D4, sg = tid / D4;
  grid_launch_dependents();  // the next call's split kernel may start staging
  grid_dependency_wait();
  // The first PRE partials of every split group are loaded for all planned
  // slots at once, together with the request's length, so that the two
  // round trips overlap; slots past the request's splits are masked below.
  const float2* ml = p.ml + size_t(bh) * p.n_split;
  const float4* po = reinterpret_cast<const float4*>(p.part_o + size_t(bh) * p.n_split * D) + c4;
  float4 x[PRE];
  float2 mlv[PRE];
#pragma unroll
  for (int k = 0; k < PRE; ++k) {
    const int sidx = sg + k * NSG;
    const bool in = sidx < p.n_split;
    x[k] = in ? __ldcg(po + size_t(sidx) * D4) : make_float4(0.f, 0.f, 0.f, 0.f);
    mlv[k] = in ? __ldcg(&ml[sidx]) : make_float2(-INFINITY, 0.f);
  }
  int L = p.kv_lens ? p.kv_lens[p.kv_period > 0 ? b % p.kv_period : b] : p.max_kv_len;
  int n_used;
  if (p.n_quant != nullptr) {
    L = L < 0 ? 0 : L;
    int nq = p.n_quant[b];
    nq = nq < 0 ? 0 : (nq > p.max_quant ? p.max_quant : nq);
    int lr = L - nq;
    lr = lr < 0 ? 0 : (lr > p.res_cap ? p.res_cap : lr);
    n_used = min(p.n_split - 1, (nq + p.chunk - 1) / p.chunk) + (lr > 0 ? 1 : 0);
    if (n_used == 0) {  // no key at all: zeros
      if (tid == 0) atomicOr(p.status, GQA_DEV_EMPTY_REQUEST);
      if (tid < D4) {
        T* dst = static_cast<T*>(p.o) + size_t(bh) * D + tid * 4;
        for (int e = 0; e < 4; ++e) store_f(dst + e, 0.f);
      }
      return;
    }
  } else {
    L = L < 0 ? 0 : (L > p.max_kv_len ? p.max_kv_len : L);
    n_used = min(p.n_split, (L + p.chunk - 1) / p.chunk);
    if (n_used <= 1) return;  // written by the split kernel itself
  }
#pragma unroll
  for (int k = 0; k < PRE; ++k)
    if (sg + k * NSG >= n_used) {  // loaded above, but not a split of this request
      x[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      mlv[k] = make_float2(-INFINITY, 0.f);
    }
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < PRE; ++k) M = fmaxf(M, mlv[k].x);
  float Ls = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < PRE; ++k) {
    const float w = mlv[k].x == -INFINITY ? 0.f : fast_exp2(mlv[k].x - M);
    Ls += mlv[k].y * w;
    acc.x += x[k].x * w;
    acc.y += x[k].y * w;
    acc.z += x[k].z * w;
    acc.w += x[k].w * w;
  }
  // more splits than PRE * NSG: one at a time, raising the maximum as needed
  for (int sidx = sg + PRE * NSG; sidx < n_used; sidx += NSG) {
    const float4 v = __ldcg(po + size_t(sidx) * D4);
    const float2 m = __ldcg(&ml[sidx]);
    if (m.x > M) {
      const float a = M == -INFINITY ? 0.f : fast_exp2(M - m.x);
      Ls *= a;
      acc.x *= a;
      acc.y *= a;
      acc.z *= a;
      acc.w *= a;
      M = m.x;
    }
    const float w = fast_exp2(m.x - M);
    Ls += m.y * w;
    acc.x += v.x * w;
    acc.y += v.y * w;
    acc.z += v.z * w;
    acc.w += v.w * w;
  }
  red_o[sg][c4] = acc;
  if (c4 == 0) red_ml[sg] = make_float2(M, Ls);
  __syncthreads();
  if (tid < D4) {
    float Mg = red_ml[0].x;
#pragma unroll
    for (int k = 1; k < NSG; ++k) Mg = fmaxf(Mg, red_ml[k].x);
    float den = 0.f;
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < NSG; ++k) {
      const float2 mk = red_ml[k];
      const float w = mk.x == -INFINITY ? 0.f : fast_exp2(mk.x - Mg);
      const float4 v = red_o[k][tid];
      den += mk.y * w;
      t.x += v.x * w;
      t.y += v.y * w;
      t.z += v.z * w;
      t.w += v.w * w;
    }
    const float inv = 1.f / den;
    T* dst = static_cast<T*>(p.o) + size_t(bh) * D + tid * 4;
    store_f(dst + 0, t.x * inv);
    store_f(dst + 1, t.y * inv);
    store_f(dst + 2, t.z * inv);
    store_f(dst + 3, t.w * inv);
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
