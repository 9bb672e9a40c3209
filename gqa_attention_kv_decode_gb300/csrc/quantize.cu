// quantize.cu -- 4-bit group-affine quantization of KV rows on the GPU
// ("Batching Decode Attention Across Requests ...", VeloxQuant-MLX blog,
// "Part 4": re-quantizing the whole growing history every step cost more than
// the attention itself; only the newly aged, group-aligned block of tokens is
// quantized each step).  This kernel quantizes `rows` rows of every head of a
// bf16 source into rows [dst_row0, dst_row0 + rows) of a 4-bit cache: a full
// cache at prefill time, or one flushed block per decode step.
//
// Per group of 64 consecutive elements along D (the pages give the format
// x = code * scale + bias and no quantizer; the reading used everywhere in
// this library): scale = fp16((max - min) / 15), bias = fp16(min), r = the
// fp32 reciprocal of the scale, code = clamp(round_half_even((x - bias) * r),
// 0, 15), 0 when the scale is 0.  The arithmetic is IEEE fp32 with
// round-to-nearest operations, so the integer codes are a deterministic
// function of the input.
//
// A lane loads 16 bytes (8 elements); D/8 lanes hold a row and 8 lanes a
// group, whose minimum and maximum come from three xor shuffles.  A warp keeps
// UNR such loads in flight (4 rows at D = 128) before it computes.  Codes are
// written as 4 bytes per lane (one contiguous D/2-byte run per row), the
// group's scale and bias by its first lane.  HBM-bound: 2D bytes read,
// D/2 + 4 D/64 written per row.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gqa_attn.h"
#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

struct QuantParams {
  const __nv_bfloat16* src;
  uint8_t* codes;
  __half* scale;
  __half* bias;
  long long src_head_rows, dst_head_rows, dst_row0;
  long long heads, rows;
};

template <int D>
__global__ void __launch_bounds__(256) quantize_q4_kernel(const QuantParams p) {
  constexpr int LPR = D / 8;          // lanes per row (8 elements a lane)
  constexpr int RPL = 32 / LPR;       // rows per warp-wide load
  constexpr int UNR = 2;              // loads in flight per lane
  constexpr int NG = D / 64;          // groups per row
  const int lane = threadIdx.x & 31;
  const long long total = p.heads * p.rows;
  const long long row0 = ((long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5)) * (RPL * UNR);
  const int col = lane % LPR;         // 8-element chunk of the row
  uint4 w[UNR];
  long long rows[UNR];
#pragma unroll
  for (int u = 0; u < UNR; ++u) {
    rows[u] = row0 + u * RPL + lane / LPR;
    if (rows[u] < total) {
      const long long head = rows[u] / p.rows, r = rows[u] % p.rows;
      w[u] = *reinterpret_cast<const uint4*>(p.src + (head * p.src_head_rows + r) * D + col * 8);
    } else {
      w[u] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int u = 0; u < UNR; ++u) {
    float x[8];
    const uint32_t ww[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = bf16x2_to_float2(ww[i]);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
    float lo = fminf(fminf(fminf(x[0], x[1]), fminf(x[2], x[3])), fminf(fminf(x[4], x[5]), fminf(x[6], x[7])));
    float hi = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])), fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) {  // the 8 lanes of a group
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, m));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, m));
    }
    if (rows[u] >= total) continue;
    const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), 15.f));
    const __half b16 = __float2half_rn(lo);
    const float s = __half2float(s16), bb = __half2float(b16);
    const float rcp = __frcp_rn(s);
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // clamping to [0, 15] before rounding gives the same codes as after it
      const float t = fminf(fmaxf(__fmul_rn(__fsub_rn(x[i], bb), rcp), 0.f), 15.f);
      const uint32_t q = __float2uint_rn(t);
      packed |= (s > 0.f ? q : 0u) << (4 * i);
    }
    const long long head = rows[u] / p.rows, r = rows[u] % p.rows;
    const long long drow = head * p.dst_head_rows + p.dst_row0 + r;
    *reinterpret_cast<uint32_t*>(p.codes + drow * (D / 2) + col * 4) = packed;
    if ((col & 7) == 0) {
      p.scale[drow * NG + col / 8] = s16;
      p.bias[drow * NG + col / 8] = b16;
    }
  }
}

}  // namespace
}  // namespace gqa

using namespace gqa;

extern "C" GQA_ATTN_API int gqa_attn_quantize_q4(const void* src, int64_t src_head_rows, uint8_t* codes,
                                                 uint16_t* scale, uint16_t* bias, int64_t dst_head_rows,
                                                 int64_t dst_row0, int heads, int rows, int D,
                                                 int group_size, void* stream) {
  if (heads < 1 || rows < 1 || (D != 64 && D != 128) || group_size != 64) return GQA_ERR_INVALID_ARG;
  if (rows > src_head_rows || dst_row0 < 0 || dst_row0 + rows > dst_head_rows) return GQA_ERR_INVALID_ARG;
  const long long total = (long long)heads * rows;
  const long long rows_per_cta = 8LL * (D == 128 ? 4 : 8);  // 8 warps x (rows per load x loads in flight)
  if ((total + rows_per_cta - 1) / rows_per_cta > 0x7fffffffLL) return GQA_ERR_INVALID_ARG;
  if (src == nullptr || codes == nullptr || scale == nullptr || bias == nullptr) return GQA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) % 16) != 0 || (reinterpret_cast<uintptr_t>(codes) % 4) != 0 ||
      (reinterpret_cast<uintptr_t>(scale) % 2) != 0 || (reinterpret_cast<uintptr_t>(bias) % 2) != 0)
    return GQA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  for (const void* ptr : {static_cast<const void*>(src), static_cast<const void*>(codes),
                          static_cast<const void*>(scale), static_cast<const void*>(bias)}) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
      cudaGetLastError();
      return GQA_ERR_NOT_DEVICE_PTR;
    }
    if (!((attr.type == cudaMemoryTypeDevice && attr.device == dev) || attr.type == cudaMemoryTypeManaged))
      return GQA_ERR_NOT_DEVICE_PTR;
  }
  QuantParams p;
  p.src = static_cast<const __nv_bfloat16*>(src);
  p.codes = codes;
  p.scale = reinterpret_cast<__half*>(scale);
  p.bias = reinterpret_cast<__half*>(bias);
  p.src_head_rows = src_head_rows;
  p.dst_head_rows = dst_head_rows;
  p.dst_row0 = dst_row0;
  p.heads = heads;
  p.rows = rows;
  const unsigned grid = unsigned((total + rows_per_cta - 1) / rows_per_cta);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (D == 128)
    quantize_q4_kernel<128><<<grid, 256, 0, s>>>(p);
  else
    quantize_q4_kernel<64><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}
