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
// this library): scale = fp16((max - min) / 15), bias = fp16(min),
// code = clamp(round_half_even((x - bias) / scale), 0, 15), 0 when the scale
// is 0, with the subtraction and the division each one IEEE fp32 operation
// rounded to nearest.  The codes are a deterministic function of the input.
//
// The division is formed without a divide instruction.  With y = RN(1/s),
// q0 = RN(d y) is within 2^-22 |q| of the exact quotient q = d / s, and one
// residual step q1 = RN(q0 + RN(d - s q0) y) (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990) brings the value before its last rounding within about
// 2^-44 |q| of q.  That last rounding returns RN(q), because q is never that
// close to a midpoint mid between two consecutive floats: d has 24 significant
// bits and s (fp16) 11, so d - mid s is a nonzero multiple of
// 2^(e_q + e_s - 34) and |q - mid| >= 2^(e_q - 35).  So q1 is exactly the
// quotient a correctly rounded fp32 division returns, and the ties of
// round-half-even are decided on the same value.
//
// A lane holds 32 elements (four 16-byte loads of one row); D/32 lanes hold a
// row and 2 lanes a group, whose minimum and maximum come from one xor
// shuffle.  The per-group work (the scale's division, the reciprocal, the
// fp16 roundings) is one instruction stream for all lanes of a warp, so more
// elements per lane divide its cost: a 16,384-token cache at B = 4, Hkv = 8
// took 43.7 us with 8 elements a lane and 37.5 us with 16 or 32; a 64-token
// flush 6.7 us with 16 and 6.1 with 32.  A lane keeps two rows (128 bytes)
// in flight before it computes: 35.5 us (one row 37.6, four 37.5, the
// registers then limiting the CTAs per SM).  Codes are written as 16 bytes
// per lane (one contiguous D/2-byte run per row), the group's scale and bias
// by its first lane.  HBM-bound: 2D bytes read,
// D/2 + 4 D/64 written per row.  The grid is (row blocks, heads), so no lane
// divides to find its head.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gqa_attn.h"
#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kQuantEpl = 32;  // elements a lane quantizes (16 or 32)

struct QuantParams {
  const __nv_bfloat16* src;
  uint8_t* codes;
  __half* scale;
  __half* bias;
  long long src_head_rows, dst_head_rows, dst_row0;
  long long heads, rows;
};

template <int D>
struct QuantCfg {
  static constexpr int EPL = kQuantEpl;  // elements a lane holds
  static constexpr int NV = EPL / 8;     // 16-byte loads per lane and row
  static constexpr int LPR = D / EPL;    // lanes per row
  static constexpr int LPG = 64 / EPL;   // lanes per group
  static constexpr int RPL = 32 / LPR;   // rows per warp-wide load
  static constexpr int UNR = 64 / EPL;   // rows in flight per lane (128 bytes)
  static constexpr int ROWS_PER_CTA = 8 * RPL * UNR;  // 8 warps
};

template <int D>
__global__ void __launch_bounds__(256) quantize_q4_kernel(const QuantParams p) {
  constexpr int EPL = QuantCfg<D>::EPL;
  constexpr int NV = QuantCfg<D>::NV;
  constexpr int LPR = QuantCfg<D>::LPR;
  constexpr int LPG = QuantCfg<D>::LPG;
  constexpr int RPL = QuantCfg<D>::RPL;
  constexpr int UNR = QuantCfg<D>::UNR;
  constexpr int NG = D / 64;          // groups per row
  const int lane = threadIdx.x & 31;
  // launched with programmatic stream serialisation: the next grid may start
  // launching now; the previous one must be complete before any global access
  grid_launch_dependents();
  grid_dependency_wait();
  const long long head = blockIdx.y + (long long)gridDim.y * blockIdx.z;
  if (head >= p.heads) return;
  const int row0 = (int(blockIdx.x) * 8 + (int(threadIdx.x) >> 5)) * (RPL * UNR);
  const int col = lane % LPR;         // 16-element chunk of the row
  const __nv_bfloat16* src = p.src + head * p.src_head_rows * D + col * EPL;
  const long long dst0 = head * p.dst_head_rows + p.dst_row0;
  uint4 w[UNR][NV];
  int rows[UNR];
#pragma unroll
  for (int u = 0; u < UNR; ++u) {
    rows[u] = row0 + u * RPL + lane / LPR;
    const uint4* s4 = reinterpret_cast<const uint4*>(src + (long long)rows[u] * D);
#pragma unroll
    for (int k = 0; k < NV; ++k) w[u][k] = rows[u] < p.rows ? s4[k] : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int u = 0; u < UNR; ++u) {
    uint32_t ww[EPL / 2];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      ww[4 * k] = w[u][k].x;
      ww[4 * k + 1] = w[u][k].y;
      ww[4 * k + 2] = w[u][k].z;
      ww[4 * k + 3] = w[u][k].w;
    }
    // group minimum and maximum on the bf16 pairs (exact), carried through the
    // shuffles as one (min, -max) pair
    __nv_bfloat162 mn = *reinterpret_cast<const __nv_bfloat162*>(&ww[0]), mx = mn;
#pragma unroll
    for (int i = 1; i < EPL / 2; ++i) {
      const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&ww[i]);
      mn = __hmin2(mn, x);
      mx = __hmax2(mx, x);
    }
    const __nv_bfloat162 nmx = __hneg2(mx);
    __nv_bfloat162 v = __hmin2(__lows2bfloat162(mn, nmx), __highs2bfloat162(mn, nmx));  // (lo, -hi)
#pragma unroll
    for (int m = 1; m < LPG; m <<= 1) {  // the lanes of a group
      const uint32_t o = __shfl_xor_sync(0xffffffffu, *reinterpret_cast<const uint32_t*>(&v), m);
      v = __hmin2(v, *reinterpret_cast<const __nv_bfloat162*>(&o));
    }
    if (rows[u] >= p.rows) continue;
    const float lo = __bfloat162float(__low2bfloat16(v)), hi = -__bfloat162float(__high2bfloat16(v));
    const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), 15.f));
    const __half b16 = __float2half_rn(lo);
    const float s = __half2float(s16), bb = __half2float(b16);
    const float rcp = __frcp_rn(s);
    // with an infinite scale or bias the quotients are 0, +-inf or NaN, which
    // the reciprocal product already gives exactly; the residual step would
    // turn them into NaN
    const bool corr = fabsf(s) < INFINITY && fabsf(bb) < INFINITY;
    // per pair: d = x - bias (x + (-bias) is x - bias), q = d / scale as
    // above, rounded to the nearest integer, ties to even, by the saturating
    // conversion (negative values and NaN give 0), then capped at 15
    const float2 nb = make_float2(-bb, -bb), r2 = make_float2(rcp, rcp), ns2 = make_float2(-s, -s);
    uint32_t packed[EPL / 8];
#pragma unroll
    for (int k = 0; k < EPL / 8; ++k) packed[k] = 0u;
#pragma unroll
    for (int i = 0; i < EPL / 2; ++i) {
      const float2 d = __fadd2_rn(bf16x2_to_float2(ww[i]), nb);
      float2 t = __fmul2_rn(d, r2);
      if (corr) t = __ffma2_rn(__ffma2_rn(t, ns2, d), r2, t);
      const uint32_t k0 = min(__float2uint_rn(t.x), 15u), k1 = min(__float2uint_rn(t.y), 15u);
      packed[i / 4] += (k0 + 16u * k1) << (8 * (i % 4));
    }
    const long long drow = dst0 + rows[u];
    uint32_t* cdst = reinterpret_cast<uint32_t*>(p.codes + drow * (D / 2) + col * (EPL / 2));  // (4-byte aligned)
#pragma unroll
    for (int k = 0; k < EPL / 8; ++k) cdst[k] = (s > 0.f) ? packed[k] : 0u;
    if ((col % LPG) == 0) {
      p.scale[drow * NG + col / LPG] = s16;
      p.bias[drow * NG + col / LPG] = b16;
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
  const int rows_per_cta = D == 128 ? QuantCfg<128>::ROWS_PER_CTA : QuantCfg<64>::ROWS_PER_CTA;
  if (heads > 65535LL * 65535LL) return GQA_ERR_INVALID_ARG;
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
  // (row blocks of a head, heads): heads spill from y into z past 65535
  const dim3 grid(unsigned((rows + rows_per_cta - 1) / rows_per_cta), unsigned(heads < 65535 ? heads : 65535),
                  unsigned((heads + 65534) / 65535));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = D == 128 ? cudaLaunchKernelEx(&cfg, quantize_q4_kernel<128>, p)
                                 : cudaLaunchKernelEx(&cfg, quantize_q4_kernel<64>, p);
  return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}
