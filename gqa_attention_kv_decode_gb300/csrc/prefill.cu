// prefill.cu -- causal / chunked GQA prefill on the tcgen05 tensor cores of
// sm_103a ("Fused attention makes a 4,096-token Qwen2 prefill on Metal 4.5x
// faster", "Cause and workaround": one pass over the grouped KV heads, the
// causal mask applied inside the kernel with the queries aligned to the end
// of the keys, no score matrix in memory).
//
// One CTA computes a 128-row query tile of one query head h; it reads KV head
// g = h / n_rep directly (no repeat_kv).  Per KV tile of 128 keys:
//   1. S = Q K^T     tcgen05.mma (M=128, N=128, K=64) into tensor memory,
//                    Q and K staged by TMA in 128-byte-swizzled shared memory;
//   2. softmax       each thread owns one query row = one TMEM lane: it loads
//                    its 128 scores, applies the end-aligned causal mask,
//                    keeps a running maximum (raised lazily, by > 2^8) and
//                    sum, and writes P (bf16) to shared memory in the
//                    swizzled K-major layout the tensor core reads;
//   3. O += P V      tcgen05.mma (M=128, N=64, K=128) into tensor memory,
//                    V read MN-major straight from its TMA tile.
// KV tiles entirely above the diagonal are never loaded; tiles entirely below
// it are not masked.  K and V tiles are double-buffered.  At the end O is
// divided by the row sum and written as bf16.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cmath>
#include <mutex>

#include "gqa_attn.h"
#include "internal.h"
#include "tc.cuh"

namespace gqa {
namespace {

constexpr int BM = 128;                    // query rows per tile (TMEM lanes)
constexpr int BN = 128;                    // keys per KV tile
constexpr int HD = 64;                     // head dimension
constexpr int TILE_BYTES = BM * HD * 2;    // one 128 x 64 bf16 tile: 16 KiB
constexpr uint32_t TMEM_COLS = 256;        // S: columns [0,128), O: [128,192)
constexpr uint32_t IDESC_S = idesc_bf16(BM, BN, false, false);
constexpr uint32_t IDESC_O = idesc_bf16(BM, HD, false, true);

// shared memory (offsets from a 1024-byte aligned base)
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE_BYTES;       // 2 stages
constexpr int OFF_V = OFF_K + 2 * TILE_BYTES;   // 2 stages
constexpr int OFF_P = OFF_V + 2 * TILE_BYTES;   // 2 blocks of 64 keys
constexpr int OFF_BAR = OFF_P + 2 * TILE_BYTES;
constexpr int SMEM_BYTES = OFF_BAR + 128 + 1024;  // + alignment slack

struct PrefillParams {
  __nv_bfloat16* o;
  int Hq, Hkv, n_rep, q_len, kv_len, n_qtiles, causal;
  float qk_scale_log2;  // scale * log2(e)
  uint64_t wait_limit_ns;
};

// Bounded wait shared by the whole CTA: once one thread gives up, the
// others stop waiting too (the results are then poisoned with NaN).
__device__ __forceinline__ void cta_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         uint64_t limit_ns) {
  if (*abort_flag) return;
  if (!mbar_wait_bounded(bar, parity, limit_ns)) *abort_flag = 1;
}

__global__ void __launch_bounds__(128, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int qt = p.n_qtiles - 1 - int(blockIdx.x);  // longest causal rows first
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int g = h / p.n_rep;
  const int m0 = qt * BM;
  const int off = p.kv_len - p.q_len;  // query row i sits at key position off + i

  int n_kv = (p.kv_len + BN - 1) / BN;
  if (p.causal) n_kv = min(n_kv, (off + min(m0 + BM - 1, p.q_len - 1)) / BN + 1);

  uint64_t* bar_q = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* bar_k = bar_q + 1;  // [2]
  uint64_t* bar_v = bar_q + 3;  // [2]
  uint64_t* bar_s = bar_q + 5;
  uint64_t* bar_o = bar_q + 6;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + 72);

  const int kv_head = b * p.Hkv + g;
  auto load_kv = [&](int j) {
    const int st = j & 1;
    mbar_arrive_expect_tx(&bar_k[st], TILE_BYTES);
    tma_load_3d(smem + OFF_K + st * TILE_BYTES, &tmK, 0, j * BN, kv_head, &bar_k[st]);
    mbar_arrive_expect_tx(&bar_v[st], TILE_BYTES);
    tma_load_3d(smem + OFF_V + st * TILE_BYTES, &tmV, 0, j * BN, kv_head, &bar_v[st]);
  };

  if (warp == 0) {
    tmem_alloc(tslot, TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 32) {
    for (int i = 0; i < 7; ++i) mbar_init(&bar_q[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    mbar_arrive_expect_tx(bar_q, TILE_BYTES);
    tma_load_3d(smem + OFF_Q, &tmQ, 0, m0, b * p.Hq + h, bar_q);
    for (int j = 0; j < 2 && j < n_kv; ++j) load_kv(j);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tS = tmem;
  const uint32_t tO = tmem + 128;
  const uint32_t lane_off = uint32_t(warp * 32) << 16;  // this warp's TMEM lanes

  const int r = tid;             // query row within the tile = TMEM lane
  const int qi = m0 + r;         // query row
  const int last_key = p.causal ? min(off + qi, p.kv_len - 1) : p.kv_len - 1;
  float m_ref = -INFINITY, lsum = 0.f;
  const uint32_t q_addr = smem_u32(smem + OFF_Q);
  const uint32_t p_addr = smem_u32(smem + OFF_P);

  for (int j = 0; j < n_kv; ++j) {
    const int st = j & 1;
    const uint32_t ph = uint32_t(j >> 1) & 1u;
    if (tid == 0) {
      if (j == 0) cta_wait(bar_q, 0, abort_flag, p.wait_limit_ns);
      cta_wait(&bar_k[st], ph, abort_flag, p.wait_limit_ns);
      tc_fence_after();
      const uint32_t k_addr = smem_u32(smem + OFF_K + st * TILE_BYTES);
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk)
        mma_bf16(tS, sdesc_sw128(q_addr + kk * 32), sdesc_sw128(k_addr + kk * 32), IDESC_S, kk > 0);
      mma_commit(bar_s);
    }
    cta_wait(bar_s, uint32_t(j) & 1u, abort_flag, p.wait_limit_ns);
    tc_fence_after();

    // ---- softmax of row r over keys n0 .. n0+127 ----
    const int n0 = j * BN;
    const bool masked = (n0 + BN - 1 > last_key);
    uint32_t sr[4][32];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32(tS + lane_off + c * 32, sr[c]);
    tmem_wait_ld();
    float tmax = -INFINITY;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        float s = __uint_as_float(sr[c][e]) * p.qk_scale_log2;
        if (masked && n0 + c * 32 + e > last_key) s = -INFINITY;
        sr[c][e] = __float_as_uint(s);
        tmax = fmaxf(tmax, s);
      }
    float alpha = 1.f;
    const bool resc = tmax > m_ref + 8.f;
    if (resc) {
      alpha = fast_exp2(m_ref - tmax);
      m_ref = tmax;
    }
    if (j > 0) {
      // the previous P.V must be done before P is overwritten or O rescaled;
      // its K/V stage is then free for tile j+1
      cta_wait(bar_o, uint32_t(j - 1) & 1u, abort_flag, p.wait_limit_ns);
      tc_fence_after();
      if (tid == 32 && j + 1 < n_kv) load_kv(j + 1);
      if (__any_sync(0xffffffffu, resc)) {
        uint32_t o[2][32];
        tmem_ld32(tO + lane_off, o[0]);
        tmem_ld32(tO + lane_off + 32, o[1]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) o[c][e] = __float_as_uint(__uint_as_float(o[c][e]) * alpha);
        tmem_st32(tO + lane_off, o[0]);
        tmem_st32(tO + lane_off + 32, o[1]);
        tmem_wait_st();
      }
    }
    lsum *= alpha;
    // P (bf16) into two 128-byte-swizzled K-major blocks of 64 keys
#pragma unroll
    for (int c = 0; c < 4; ++c) {
#pragma unroll
      for (int e8 = 0; e8 < 4; ++e8) {  // 8 keys = one 16-byte chunk
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float p0 = fast_exp2(__uint_as_float(sr[c][e8 * 8 + 2 * u]) - m_ref);
          const float p1 = fast_exp2(__uint_as_float(sr[c][e8 * 8 + 2 * u + 1]) - m_ref);
          lsum += p0 + p1;
          const __nv_bfloat162 pk = __floats2bfloat162_rn(p0, p1);
          w[u] = *reinterpret_cast<const uint32_t*>(&pk);
        }
        const int key = c * 32 + e8 * 8;
        const int blk = key >> 6;
        const int chunk = (key & 63) >> 3;
        unsigned char* dst = smem + OFF_P + blk * TILE_BYTES + r * 128 + ((chunk ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      cta_wait(&bar_v[st], ph, abort_flag, p.wait_limit_ns);
      const uint32_t v_addr = smem_u32(smem + OFF_V + st * TILE_BYTES);
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk)
        mma_bf16(tO, sdesc_sw128(p_addr + (kk >> 2) * TILE_BYTES + (kk & 3) * 32),
                 sdesc_sw128(v_addr + kk * 16 * 128), IDESC_O, (j > 0 || kk > 0) ? 1u : 0u);
      mma_commit(bar_o);
    }
  }

  // ---- epilogue: O / l, bf16, to global memory ----
  cta_wait(bar_o, uint32_t(n_kv - 1) & 1u, abort_flag, p.wait_limit_ns);
  tc_fence_after();
  uint32_t o[2][32];
  tmem_ld32(tO + lane_off, o[0]);
  tmem_ld32(tO + lane_off + 32, o[1]);
  tmem_wait_ld();
  const bool bad = *abort_flag != 0;
  if (qi < p.q_len) {
    const float inv = bad ? __int_as_float(0x7fc00000) : 1.f / lsum;
    uint4* dst = reinterpret_cast<uint4*>(p.o + ((size_t(b) * p.Hq + h) * p.q_len + qi) * HD);
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int e8 = 0; e8 < 4; ++e8) {
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const __nv_bfloat162 pk =
              __floats2bfloat162_rn(__uint_as_float(o[c][e8 * 8 + 2 * u]) * inv,
                                    __uint_as_float(o[c][e8 * 8 + 2 * u + 1]) * inv);
          w[u] = *reinterpret_cast<const uint32_t*>(&pk);
        }
        dst[c * 4 + e8] = make_uint4(w[0], w[1], w[2], w[3]);
      }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// [heads][row_pitch rows][64] bf16 viewed as a 3-D tensor of which only the
// first `rows` rows of each head exist; boxes of 128 rows x 64, 128-byte
// swizzle.  Rows past `rows` (e.g. cache rows past kv_len, which may hold
// anything) are never read: the copy fills them with zeros, so they add
// exactly nothing to P.V.
bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_pitch, uint64_t heads) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {HD, rows, heads};
  cuuint64_t strides[2] = {HD * 2, row_pitch * HD * 2};
  cuuint32_t box[3] = {HD, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  if (a.D != HD) return cudaErrorNotSupported;
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, a.q, a.q_len, a.q_len, uint64_t(a.B) * a.Hq) ||
      !make_map(&tk, a.k, a.kv_len, a.S_cap, uint64_t(a.B) * a.Hkv) ||
      !make_map(&tv, a.v, a.kv_len, a.S_cap, uint64_t(a.B) * a.Hkv))
    return cudaErrorInvalidValue;
  PrefillParams p;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.n_rep = a.Hq / a.Hkv;
  p.q_len = a.q_len;
  p.kv_len = a.kv_len;
  p.n_qtiles = (a.q_len + BM - 1) / BM;
  p.causal = a.causal;
  p.qk_scale_log2 = float(double(a.scale) * 1.4426950408889634);
  p.wait_limit_ns = kWaitLimitNs;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const dim3 grid(p.n_qtiles, a.Hq, a.B);
  prefill_kernel<<<grid, 128, SMEM_BYTES, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace gqa
