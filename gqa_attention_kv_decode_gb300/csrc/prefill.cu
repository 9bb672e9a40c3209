// prefill.cu -- causal / chunked GQA prefill on the tcgen05 tensor cores of
// sm_103a ("Fused attention makes a 4,096-token Qwen2 prefill on Metal 4.5x
// faster", "Cause and workaround": one pass over the grouped KV heads, the
// causal mask applied inside the kernel with the queries aligned to the end
// of the keys, no score matrix in memory).
//
// One CTA computes two consecutive 128-row query tiles (A and B) of one query
// head h and reads KV head g = h / n_rep directly (no repeat_kv).  Warp roles:
//   warp 8     TMA: Q_A, Q_B once, then K and V tiles of 128 keys (4 stages);
//   warp 9     MMA issue (one thread): S_t = Q_t K^T (M=128, N=128, K=64) and
//              O_t += P_t V (M=128, N=64, K=128) with tcgen05.mma; S, P and O
//              live in tensor memory, V is read MN-major from its TMA tile;
//   warps 0-3  softmax of tile A, warps 4-7 softmax of tile B: a thread owns
//              one query row = one TMEM lane.  In one pass over a tile it
//              loads the row's scores, exponentiates them against the running
//              maximum with the (end-aligned, causal) mask and writes P (bf16)
//              back to tensor memory, where the P.V MMA reads it as its A
//              operand.  The running maximum is raised lazily: only when a
//              tile exceeds it by more than 2^8 does the warp rescale O in
//              TMEM and redo that tile (the first tile takes its own maximum).
// While one tile's softmax runs, the tensor core works on the other tile
// (ping-pong), so MMA and exponentials overlap.  KV tiles entirely above the
// diagonal are never loaded; tiles entirely below it are not masked.
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
constexpr int NTHR = 320;                  // 8 softmax warps + TMA warp + MMA warp
constexpr uint32_t TMEM_COLS = 512;        // S_A [0,128) S_B [128,256) O_A, O_B [256,384) P_A, P_B [384,512)
constexpr uint32_t IDESC_S = idesc_bf16(BM, BN, false, false);
constexpr uint32_t IDESC_O = idesc_bf16(BM, HD, false, true);

// shared memory (offsets from a 1024-byte aligned base)
constexpr int NST = 4;                          // K/V stages: tiles j+1..j+3 in flight
constexpr int OFF_Q = 0;                        // Q_A, Q_B
constexpr int OFF_K = OFF_Q + 2 * TILE_BYTES;   // NST stages
constexpr int OFF_V = OFF_K + NST * TILE_BYTES; // NST stages
constexpr int OFF_BAR = OFF_V + NST * TILE_BYTES;
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");

// mbarrier slots
constexpr int B_Q = 0, B_KF = 1, B_VF = B_KF + NST, B_KE = B_VF + NST, B_S = B_KE + NST, B_P = B_S + 2,
              B_O = B_P + 2, N_BARS = B_O + 2;
static_assert(N_BARS * 8 <= 192, "barrier area");

struct PrefillParams {
  __nv_bfloat16* o;
  int Hq, Hkv, n_rep, q_len, kv_len, n_pairs, causal;
  float qk_scale_log2;  // scale * log2(e)
  uint64_t wait_limit_ns;
};

// Bounded wait shared by the whole CTA: once one thread gives up, the
// others stop waiting too and the outputs are poisoned with NaN.
__device__ __forceinline__ void cta_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         uint64_t limit_ns) {
  if (*abort_flag) return;
  if (!mbar_wait_bounded(bar, parity, limit_ns)) *abort_flag = 1;
}

__global__ void __launch_bounds__(NTHR, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int pair = p.n_pairs - 1 - int(blockIdx.x);  // longest causal rows first
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int g = h / p.n_rep;
  const int m0 = pair * 2 * BM;
  const int off = p.kv_len - p.q_len;  // query row i sits at key position off + i

  auto nkv_for = [&](int mstart) -> int {
    if (mstart >= p.q_len) return 0;
    int n = (p.kv_len + BN - 1) / BN;
    if (p.causal) n = min(n, (off + min(mstart + BM - 1, p.q_len - 1)) / BN + 1);
    return n;
  };
  const int nkv0 = nkv_for(m0), nkv1 = nkv_for(m0 + BM);
  const int nkv_max = max(nkv0, nkv1);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 192);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + 200);

  if (warp == 9) {
    tmem_alloc(tslot, TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 256) {
    for (int i = 0; i < N_BARS; ++i) mbar_init(&bars[i], (i == B_P || i == B_P + 1) ? 4 : 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 8) {
    // ---------------- TMA ----------------
    if (lane == 0) {
      const int kv_head = b * p.Hkv + g;
      mbar_arrive_expect_tx(&bars[B_Q], 2 * TILE_BYTES);
      tma_load_3d(smem + OFF_Q, &tmQ, 0, m0, b * p.Hq + h, &bars[B_Q]);
      tma_load_3d(smem + OFF_Q + TILE_BYTES, &tmQ, 0, m0 + BM, b * p.Hq + h, &bars[B_Q]);
      for (int j = 0; j < nkv_max; ++j) {
        const int st = j % NST;
        if (j >= NST) cta_wait(&bars[B_KE + st], uint32_t(j / NST - 1) & 1u, abort_flag, p.wait_limit_ns);
        if (*abort_flag) break;
        mbar_arrive_expect_tx(&bars[B_KF + st], TILE_BYTES);
        tma_load_3d(smem + OFF_K + st * TILE_BYTES, &tmK, 0, j * BN, kv_head, &bars[B_KF + st]);
        mbar_arrive_expect_tx(&bars[B_VF + st], TILE_BYTES);
        tma_load_3d(smem + OFF_V + st * TILE_BYTES, &tmV, 0, j * BN, kv_head, &bars[B_VF + st]);
      }
    }
  } else if (warp == 9) {
    // ---------------- MMA issue ----------------
    if (lane == 0) {
      const uint32_t q_addr = smem_u32(smem + OFF_Q);
      auto issue_s = [&](int t, int j) {
        const uint32_t qa = q_addr + t * TILE_BYTES;
        const uint32_t ka = smem_u32(smem + OFF_K + (j % NST) * TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          mma_bf16(tmem + t * 128, sdesc_sw128(qa + kk * 32), sdesc_sw128(ka + kk * 32), IDESC_S, kk > 0);
        mma_commit(&bars[B_S + t]);
      };
      cta_wait(&bars[B_Q], 0, abort_flag, p.wait_limit_ns);
      cta_wait(&bars[B_KF], 0, abort_flag, p.wait_limit_ns);
      tc_fence_after();
      if (nkv0 > 0) issue_s(0, 0);
      if (nkv1 > 0) issue_s(1, 0);
      for (int j = 0; j < nkv_max; ++j) {
        const int st = j % NST;
        bool v_ready = false, k_next = false;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int nkv_t = t == 0 ? nkv0 : nkv1;
          if (j >= nkv_t) continue;
          cta_wait(&bars[B_P + t], uint32_t(j) & 1u, abort_flag, p.wait_limit_ns);
          if (!v_ready) {
            cta_wait(&bars[B_VF + st], uint32_t(j / NST) & 1u, abort_flag, p.wait_limit_ns);
            v_ready = true;
          }
          tc_fence_after();
          const uint32_t va = smem_u32(smem + OFF_V + st * TILE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)  // P_t (bf16, TMEM) x V (MN-major, smem)
            mma_bf16_ts(tmem + 256 + t * 64, tmem + 384 + t * 64 + kk * 8, sdesc_sw128(va + kk * 16 * 128),
                        IDESC_O, (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bars[B_O + t]);
          if (j + 1 < nkv_t) {
            if (!k_next) {
              cta_wait(&bars[B_KF + (j + 1) % NST], uint32_t((j + 1) / NST) & 1u, abort_flag, p.wait_limit_ns);
              tc_fence_after();
              k_next = true;
            }
            issue_s(t, j + 1);
          }
        }
        mma_commit(&bars[B_KE + st]);  // stage st is free once everything issued so far is done
      }
    }
  } else {
    // ---------------- softmax of tile t = warp / 4 ----------------
    const int t = warp >> 2;
    const int nkv = t == 0 ? nkv0 : nkv1;
    const int r = tid & (BM - 1);
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + t * 128 + lane_off;
    const uint32_t tO = tmem + 256 + t * 64 + lane_off;
    const int qi = m0 + t * BM + r;
    const int last_key = p.causal ? min(off + qi, p.kv_len - 1) : p.kv_len - 1;
    const uint32_t tP = tmem + 384 + t * 64 + lane_off;
    float m_ref = -INFINITY, lsum = 0.f;
    const float2 cc = make_float2(p.qk_scale_log2, p.qk_scale_log2);
    // One pass over a tile: P = 2^(s*c - m_ref) (masked keys 0) written to
    // tensor memory as bf16 pairs (the A operand of O += P V); returns the
    // tile's sum of P and its raw score maximum.
    auto tile_pass = [&](int n0, bool warp_masked, float2& tsum) -> float {
      const float2 mm = make_float2(-m_ref, -m_ref);
      float rmax = -INFINITY;
      tsum = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t sr[32];
        tmem_ld32(tS + c * 32, sr);
        tmem_wait_ld();
        uint32_t pw[16];  // these 32 keys as bf16 pairs
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          float s0 = __uint_as_float(sr[2 * u]), s1 = __uint_as_float(sr[2 * u + 1]);
          if (warp_masked) {
            if (n0 + c * 32 + 2 * u > last_key) s0 = -INFINITY;
            if (n0 + c * 32 + 2 * u + 1 > last_key) s1 = -INFINITY;
          }
          rmax = max3f(rmax, s0, s1);
          const float2 x = ffma2(make_float2(s0, s1), cc, mm);
          const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
          tsum = __fadd2_rn(tsum, make_float2(p0, p1));
          const __nv_bfloat162 pk = __floats2bfloat162_rn(p0, p1);
          pw[u] = *reinterpret_cast<const uint32_t*>(&pk);
        }
        tmem_st16(tP + c * 16, pw);
      }
      return rmax;
    };
    for (int j = 0; j < nkv; ++j) {
      cta_wait(&bars[B_S + t], uint32_t(j) & 1u, abort_flag, p.wait_limit_ns);
      // P_t and O_t are free once the previous P.V of this tile is done (it
      // was issued before this tile's S, so this wait does not stall)
      if (j > 0) cta_wait(&bars[B_O + t], uint32_t(j - 1) & 1u, abort_flag, p.wait_limit_ns);
      tc_fence_after();
      const int n0 = j * BN;
      const bool warp_masked = __any_sync(0xffffffffu, n0 + BN - 1 > last_key);  // diagonal / tail
      if (j == 0) {
        // first tile: the reference is this tile's own maximum
        float rmax = -INFINITY;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t sr[2][32];
          tmem_ld32(tS + half * 64, sr[0]);
          tmem_ld32(tS + half * 64 + 32, sr[1]);
          tmem_wait_ld();
#pragma unroll
          for (int cc2 = 0; cc2 < 2; ++cc2)
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float s = __uint_as_float(sr[cc2][e]);
              rmax = fmaxf(rmax, (warp_masked && n0 + (half * 2 + cc2) * 32 + e > last_key) ? -INFINITY : s);
            }
        }
        m_ref = rmax * p.qk_scale_log2;
      }
      float2 tsum;
      const float tmax = tile_pass(n0, warp_masked, tsum) * p.qk_scale_log2;
      const bool resc = tmax > m_ref + 8.f;
      if (__any_sync(0xffffffffu, resc)) {
        // a row's maximum rose by more than 2^8: raise its reference, rescale
        // its O and redo the tile (whole warp, as TMEM access is warp-wide)
        const float alpha = resc ? fast_exp2(m_ref - tmax) : 1.f;
        if (resc) m_ref = tmax;
#pragma unroll
        for (int c = 0; c < 2; ++c) {  // 32 columns at a time keeps the register count down
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + c * 32, o);
        }
        tmem_wait_st();
        lsum *= alpha;
        tile_pass(n0, warp_masked, tsum);
      }
      lsum += tsum.x + tsum.y;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_P + t]);
    }
    // ---- epilogue: O / l, bf16, to global memory ----
    if (nkv > 0) {
      cta_wait(&bars[B_O + t], uint32_t(nkv - 1) & 1u, abort_flag, p.wait_limit_ns);
      tc_fence_after();
      const float inv = *abort_flag ? __int_as_float(0x7fc00000) : 1.f / lsum;
      uint4* dst = reinterpret_cast<uint4*>(p.o + ((size_t(b) * p.Hq + h) * p.q_len + qi) * HD);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_wait_ld();
        if (qi < p.q_len) {
#pragma unroll
          for (int e8 = 0; e8 < 4; ++e8) {
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const __nv_bfloat162 pk = __floats2bfloat162_rn(__uint_as_float(o[e8 * 8 + 2 * u]) * inv,
                                                              __uint_as_float(o[e8 * 8 + 2 * u + 1]) * inv);
              w[u] = *reinterpret_cast<const uint32_t*>(&pk);
            }
            dst[c * 4 + e8] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) tmem_dealloc(tmem, TMEM_COLS);
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
  p.n_pairs = (a.q_len + 2 * BM - 1) / (2 * BM);
  p.causal = a.causal;
  p.qk_scale_log2 = float(double(a.scale) * 1.4426950408889634);
  p.wait_limit_ns = kWaitLimitNs;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const dim3 grid(p.n_pairs, a.Hq, a.B);
  prefill_kernel<<<grid, NTHR, SMEM_BYTES, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace gqa
