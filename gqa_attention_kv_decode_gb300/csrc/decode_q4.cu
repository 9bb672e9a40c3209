// decode_q4.cu -- single-token GQA decode over a 4-bit group-affine KV cache,
// dequantised inside the attention loop, with both products on the tensor
// cores (mma.sync m16n8k16, fp32 accumulation; sm_103a).
//
// The cache stores, per (request, KV head, token), D/2 bytes of 4-bit codes
// (element 2t in the low nibble of byte t) and one fp16 scale and bias per
// group of 64 elements: x = code * scale + bias ("Batching Decode Attention
// Across Requests ...", VeloxQuant-MLX blog, "The setup" and "Part 4": the
// fused decode-attend reads the codes directly instead of materialising an
// fp16 copy).  No dequantised row is ever formed.  The affine term is folded
// out of both products, per group g:
//   q . k_j       = s_jg * (sum_{i in g} q_i c_ji) + b_jg * (sum_{i in g} q_i)
//   sum_j p_j v_j = sum_j (p_j s_jg) c_j + sum_j p_j b_jg
// so the tensor cores only ever see the integer codes.
//
//   S^T = K Q^T   fp16: M = the warp's 16 keys, N = 8 query heads, K = 16
//                 dims.  A code enters as an exact fp16 value: the nibble in
//                 bits 0-3 of a half-word under the exponent of 1024 gives
//                 1024 + c, the nibble in bits 4-7 under the exponent of 64
//                 gives 64 + c (one mask-and-or per pair of codes, one shift
//                 per word).  The k index is a permutation of the dims that
//                 puts a thread's 4 codes of a k-step in 2 bytes of one
//                 word.  q is scaled by 2^-e (exact, e per CTA) to stay below
//                 2^14 in fp16; the offsets are removed with the per-group
//                 sums of q (1024 sum_even q + 64 sum_odd q).
//   O^T = V^T P^T bf16: M = 16 dims of one group, N = 8 query heads, K = 16
//                 keys.  A code enters as the bf16 value 128 + c (a byte
//                 permute, a shift and a mask per pair).  The B operand
//                 p_j s_jg (bf16, for range) is built in the layout of the
//                 score accumulators and transposed to the B-fragment layout
//                 with movmatrix.  Its rounding (2^-9 of each weight) is
//                 multiplied by the code, so the codes are centred: one extra
//                 MMA per group whose A operand is the constant 136 leaves
//                 sum_j (c_j - 8) B_j, and the bias sums take
//                 p_j (b_jg + 8 s_jg) with p_j s_jg before its rounding.
//                 That halves the worst case (|c - 8| <= 8 against c <= 15):
//                 a head whose weight sits on a few keys came 2.7e-2 off the
//                 oracle before.
//
// The CTA structure is the one of the other decode kernels: 4 warps, tiles of
// 64 keys (warp w takes keys 16w..16w+15), tiles dealt round-robin to the
// splits, six bulk copies per stage (codes, scales and biases of K and V), a
// per-warp online softmax in base 2, warps merged in shared memory, and split
// partials merged by the shared merge kernel.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>
#include <type_traits>

#include "gqa_attn.h"
#include "internal.h"
#include "merge.cuh"
#include "ptx.cuh"

namespace gqa {
namespace {

struct Q4Params {
  const __nv_bfloat16* q;
  const uint8_t* kc;
  const __half* ks;
  const __half* kb;
  const uint8_t* vc;
  const __half* vs;
  const __half* vb;
  __nv_bfloat16* o;
  const int32_t* kv_lens;
  int B, Hq, Hkv, n_rep, n_hc, nrep_cta, S_cap, max_kv_len, chunk, n_split;
  float qscale;  // scale * log2(e)
  uint32_t* status;
  float2* ml;
  float* part_o;
  uint64_t wait_limit_ns;
  uint64_t test_stall_ns;  // 0, or (tests) a wait that nothing ends, see the kernel
  int n_slots;        // partial slots per (request, head) row in the workspace
  int force_partial;  // write partials even for a one-split request (a residual window follows)
};

template <int D, int NSTAGE>
struct Q4Cfg {
  static constexpr int TILE = 64;          // keys per tile
  static constexpr int NW = 4;             // warps; warp w takes keys [16w, 16w + 16)
  static constexpr int NTHR = 32 * NW;
  static constexpr int CB = D / 2;         // code bytes per key row
  static constexpr int NG = D / 64;        // groups per row
  static constexpr int GB = NG * 2;        // bytes of fp16 scales (or biases) per row
  static constexpr int SROUND = 16 / GB;   // rows per 16 bytes of scales
  static constexpr int KSTEPS = D / 16;    // k-steps of S = Q K^T
  static constexpr int MT = D / 16;        // M-tiles of O^T = V^T P^T
  static constexpr int OFF_KC = 0;
  static constexpr int OFF_KS = OFF_KC + TILE * CB;
  static constexpr int OFF_KB = OFF_KS + TILE * GB;
  static constexpr int OFF_VC = OFF_KB + TILE * GB;
  static constexpr int OFF_VS = OFF_VC + TILE * CB;
  static constexpr int OFF_VB = OFF_VS + TILE * GB;
  static constexpr int STAGEB = OFF_VB + TILE * GB;
  static constexpr int SCW = 4 * 16 * NG;  // fp32 scales/biases of one warp's 16 keys: [array][key][group]
  static constexpr int OFF_SC = NSTAGE * STAGEB;
  static constexpr int OFF_QA = OFF_SC + NW * SCW * 4;   // q fragments: [KSTEPS/2][lane][4] words
  static constexpr int OFF_BAR = OFF_QA + KSTEPS / 2 * 32 * 16;
  static constexpr int OFF_REL = OFF_BAR + (NSTAGE + 1) * 8;  // after full[NSTAGE + 1]
  static constexpr int OFF_FLAG = OFF_REL + ((NSTAGE * 4 + 15) / 16) * 16;
  static constexpr int SMEM = OFF_FLAG + 16;
  static constexpr int MERGE_FLOATS = NW * (8 * D + 16);  // per warp: O[8][D], m[8], l[8]
  static_assert(D == 64 || D == 128, "head dimension");
  static_assert(CB % 16 == 0 && STAGEB % 16 == 0 && TILE % SROUND == 0, "bulk copy alignment");
  static_assert(OFF_KS % 8 == 0 && OFF_KB % 8 == 0 && OFF_VS % 8 == 0 && OFF_VB % 8 == 0, "scale staging loads");
  static_assert(MERGE_FLOATS * 4 <= NSTAGE * STAGEB, "warp-merge scratch fits in the stages");
};

// Key row (within a warp's 16) behind k index kk of the P.V product and
// behind column kk % 8 of S n-tile kk / 8.  Swapping 2<->3 and 6<->7 (mod 8)
// spreads the four rows a V-code load touches over both bank halves.
__device__ __forceinline__ int key_of(int kk) { return kk ^ ((kk >> 1) & 1); }

// D (+)= A B, m16n8k16, fp32 accumulation; bf16 or fp16 inputs.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 8x8 transpose of 16-bit elements across the warp: in, thread (r, c) holds
// row r, columns 2c and 2c+1; out, it holds row r of the transpose.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float2 f16x2_to_float2(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// Codes as exact MMA operands.  bf16: the nibble at bits 0-3 (and 16-19) of
// w under the exponent of 128 gives 128 + c.  fp16: under the exponent of
// 1024 the nibble at bits 0-3 gives 1024 + c, and under the exponent of 64
// the nibble at bits 4-7 gives 64 + c (its mantissa is 16c, scaled by 2^-4).
constexpr uint32_t kBf128x2 = 0x43004300u;
constexpr uint32_t kBf136x2 = 0x43084308u;  // 136 = 128 + 8: the centre of the codes above the offset
__device__ __forceinline__ uint32_t nib_lo_bf16(uint32_t w) { return (w & 0x000F000Fu) | kBf128x2; }
__device__ __forceinline__ uint32_t nib_lo_f16(uint32_t w) { return (w & 0x000F000Fu) | 0x64006400u; }
__device__ __forceinline__ uint32_t nib_hi_f16(uint32_t w) { return (w & 0x00F000F0u) | 0x54005400u; }

template <int D, int NSTAGE>
__global__ void __launch_bounds__(Q4Cfg<D, NSTAGE>::NTHR, 4)
    decode_q4_mma_kernel(const Q4Params p) {
  using C = Q4Cfg<D, NSTAGE>;
  constexpr int TILE = C::TILE;
  constexpr int NG = C::NG;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int split = blockIdx.x;
  const int g = blockIdx.y / p.n_hc;
  const int hc = blockIdx.y % p.n_hc;
  const int b = blockIdx.z;
  const int h0 = g * p.n_rep + hc * p.nrep_cta;
  const int nh = min(p.nrep_cta, p.n_rep - hc * p.nrep_cta);
  const size_t head_row0 = (size_t(b) * p.Hkv + g) * size_t(p.S_cap);
  const unsigned char* kc = p.kc + head_row0 * C::CB;
  const unsigned char* vc = p.vc + head_row0 * C::CB;
  const unsigned char* ks = reinterpret_cast<const unsigned char*>(p.ks) + head_row0 * C::GB;
  const unsigned char* kb = reinterpret_cast<const unsigned char*>(p.kb) + head_row0 * C::GB;
  const unsigned char* vs = reinterpret_cast<const unsigned char*>(p.vs) + head_row0 * C::GB;
  const unsigned char* vb = reinterpret_cast<const unsigned char*>(p.vb) + head_row0 * C::GB;

  // Launched early (programmatic dependent launch): while the previous grid
  // in the stream may still run, only prefetch this split's first code tile
  // into L2 (as if kv_len were max_kv_len).  One tile, not NSTAGE: more
  // competes for HBM with the previous call's last CTAs (B = 4, S = 16,384:
  // 29.4 against 30.0 us per call).
  if (tid == 0 && hc == 0) {
    for (int t = 0; t < 1; ++t) {
      const int row0 = (split + t * p.n_split) * TILE;
      if (row0 >= p.max_kv_len) break;
      const uint32_t cbytes = uint32_t(min(TILE, p.max_kv_len - row0)) * C::CB;
      prefetch_l2_bulk(kc + size_t(row0) * C::CB, cbytes);
      prefetch_l2_bulk(vc + size_t(row0) * C::CB, cbytes);
    }
  }
  if (tid == 32)  // and this CTA's query rows
    prefetch_l2_bulk(p.q + (size_t(b) * p.Hq + h0) * D, uint32_t(nh * D * 2));
  grid_dependency_wait();

  int L = p.kv_lens ? p.kv_lens[b] : p.max_kv_len;
  if (L < 0 || L > p.max_kv_len) {
    if (split == 0 && blockIdx.y == 0 && tid == 0) atomicOr(p.status, GQA_DEV_KVLEN_CLAMPED);
    L = L < 0 ? 0 : p.max_kv_len;
  }
  if (L == 0) {  // no visible key: the output row is zeros
    if (p.force_partial) return;  // no 4-bit keys: the window (or the merge) has the row
    if (split == 0) {
      if (blockIdx.y == 0 && tid == 0) atomicOr(p.status, GQA_DEV_EMPTY_REQUEST);
      for (int e = tid; e < nh * D; e += C::NTHR)
        p.o[(size_t(b) * p.Hq + h0 + e / D) * D + e % D] = __float2bfloat16_rn(0.f);
    }
    return;
  }
  // min(n_split, ceil(L / chunk))
  const int n_used = L > p.chunk * p.n_split ? p.n_split : (L + p.chunk - 1) / p.chunk;
  if (split >= n_used) return;
  const int nt_all = (L + TILE - 1) / TILE;
  const int nt = (nt_all - split + n_used - 1) / n_used;  // tiles split, split + n_used, ...

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  int* rel = reinterpret_cast<int*>(smem + C::OFF_REL);
  volatile int* flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);  // [0] abort [2] issued

  // k-th tile of this split into stage st: codes, scales and biases of K and
  // V.  Scale/bias copies are rounded up to whole 16-byte pieces; S_cap is a
  // multiple of 8 (checked on the host), so they stay inside the cache.
  auto issue = [&](int kt, int st, uint64_t pol) {
    const int row0 = (split + kt * n_used) * TILE;
    const int nrows = min(TILE, L - row0);
    const uint32_t cbytes = uint32_t(nrows) * C::CB;
    const uint32_t sbytes = uint32_t((nrows + C::SROUND - 1) / C::SROUND * C::SROUND) * C::GB;
    unsigned char* dst = smem + st * C::STAGEB;
    mbar_arrive_expect_tx(&full[st], 2 * cbytes + 4 * sbytes);
    bulk_g2s(dst + C::OFF_KC, kc + size_t(row0) * C::CB, cbytes, &full[st], pol);
    bulk_g2s(dst + C::OFF_KS, ks + size_t(row0) * C::GB, sbytes, &full[st], pol);
    bulk_g2s(dst + C::OFF_KB, kb + size_t(row0) * C::GB, sbytes, &full[st], pol);
    bulk_g2s(dst + C::OFF_VC, vc + size_t(row0) * C::CB, cbytes, &full[st], pol);
    bulk_g2s(dst + C::OFF_VS, vs + size_t(row0) * C::GB, sbytes, &full[st], pol);
    bulk_g2s(dst + C::OFF_VB, vb + size_t(row0) * C::GB, sbytes, &full[st], pol);
  };
  const uint64_t pol = l2_policy_evict_first();
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      rel[s] = 0;
    }
    fence_barrier_init();
    flag[0] = 0;
    flag[1] = 0;
    for (int t = 0; t < NSTAGE && t < nt; ++t) issue(t, t, pol);
    flag[2] = min(NSTAGE, nt);
    if (p.test_stall_ns != 0) {
      // Test only (gqa_attn_set_wait_test): wait, with the test's
      // limit, on a barrier that nothing arrives on, as on a copy that never
      // lands, and give up as such a wait does.  Every CTA then takes the
      // path of a lost copy: no partials, the status bit, its copies drained
      // (with the ordinary limit) before it returns.
      mbar_init(&full[NSTAGE], 1);
      if (!mbar_wait_bounded(&full[NSTAGE], 0u, p.test_stall_ns)) flag[0] = 1;
    }
  }

  // ---- q of head r as fp16 B fragments of S^T = K Q^T.  Thread (r, c)
  // owns dims 64G + 16c + [0, 16) of every group G; k-step 4G + 2wi + u maps
  // its k indices (2c, 2c+1, 2c+8, 2c+9) to dims base + 2u + (0, 4, 1, 5),
  // base = 64G + 16c + 8wi, matching the code bytes the A side reads (below).
  // q is scaled by 2^-e (exact; e is the same for the whole CTA) so that its
  // largest element stays below 2^14; the scores are scaled back by 2^e. ----
  const int r = lane >> 2, c = lane & 3;
  float sq;                 // scale * log2(e) * 2^e
  float2 qoffL, qoffH;      // per group: -sq (1024 sum_even q + 64 sum_odd q), heads 2c, 2c+1
  float2 qbL, qbH;          // per group: sq * sum q, heads 2c, 2c+1
  {
    const uint4* qrow = reinterpret_cast<const uint4*>(p.q + (size_t(b) * p.Hq + h0 + min(r, nh - 1)) * D);
    uint4 xq[NG][2];  // bf16 q, dims 64G + 16c + 8wi + [0, 8)
    float amax = 0.f;
#pragma unroll
    for (int G = 0; G < NG; ++G)
#pragma unroll
      for (int wi = 0; wi < 2; ++wi) {
        xq[G][wi] = r < nh ? qrow[(64 * G + 16 * c + 8 * wi) / 8] : make_uint4(0u, 0u, 0u, 0u);
        // |q| as bf16 bit patterns: unsigned order is value order
        const uint32_t m = __vmaxu2(__vmaxu2(xq[G][wi].x & 0x7fff7fffu, xq[G][wi].y & 0x7fff7fffu),
                                    __vmaxu2(xq[G][wi].z & 0x7fff7fffu, xq[G][wi].w & 0x7fff7fffu));
        const float2 f = bf16x2_to_float2(m);
        amax = fmaxf(amax, fmaxf(f.x, f.y));
      }
#pragma unroll
    for (int m = 1; m <= 16; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    const int e = amax >= 16384.f ? min(ilogbf(amax) - 13, 100) : 0;
    const float down = __int_as_float((127 - e) << 23), up = __int_as_float((127 + e) << 23);
    sq = p.qscale * up;
    uint32_t qa[C::KSTEPS][2];
    float qoff[NG], qbs[NG];  // head r
#pragma unroll
    for (int G = 0; G < NG; ++G) {
      float se = 0.f, so = 0.f;  // sums of the fp16 operands over even and odd dims
#pragma unroll
      for (int wi = 0; wi < 2; ++wi) {
        const uint32_t xw[4] = {xq[G][wi].x, xq[G][wi].y, xq[G][wi].z, xq[G][wi].w};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          // dims 2u, 2u+1 (word u) and 2u+4, 2u+5 (word u+2) of the 8
          const float2 lo = bf16x2_to_float2(xw[u]), hi = bf16x2_to_float2(xw[u + 2]);
          qa[4 * G + 2 * wi + u][0] = pack_f16(lo.x * down, hi.x * down);
          qa[4 * G + 2 * wi + u][1] = pack_f16(lo.y * down, hi.y * down);
          const float2 a0 = f16x2_to_float2(qa[4 * G + 2 * wi + u][0]);
          const float2 a2 = f16x2_to_float2(qa[4 * G + 2 * wi + u][1]);
          se += a0.x + a0.y;
          so += a2.x + a2.y;
        }
      }
      se += __shfl_xor_sync(0xffffffffu, se, 1);
      se += __shfl_xor_sync(0xffffffffu, se, 2);
      so += __shfl_xor_sync(0xffffffffu, so, 1);
      so += __shfl_xor_sync(0xffffffffu, so, 2);
      // even dims enter as 1024 + c, odd dims as 64 + c
      qoff[G] = -sq * (1024.f * se + 64.f * so);
      qbs[G] = sq * (se + so);
    }
    // this thread's scores belong to heads 2c and 2c+1, held by lanes 8c, 8c+4
    qoffL.x = __shfl_sync(0xffffffffu, qoff[0], 8 * c);
    qoffH.x = __shfl_sync(0xffffffffu, qoff[0], 8 * c + 4);
    qbL.x = __shfl_sync(0xffffffffu, qbs[0], 8 * c);
    qbH.x = __shfl_sync(0xffffffffu, qbs[0], 8 * c + 4);
    qoffL.y = __shfl_sync(0xffffffffu, qoff[NG - 1], 8 * c);
    qoffH.y = __shfl_sync(0xffffffffu, qoff[NG - 1], 8 * c + 4);
    qbL.y = __shfl_sync(0xffffffffu, qbs[NG - 1], 8 * c);
    qbH.y = __shfl_sync(0xffffffffu, qbs[NG - 1], 8 * c + 4);
    // every warp holds the same fragments: one copy in shared memory, read
    // back at each tile (keeps 16 registers free in the tile loop)
    if (warp == 0) {
      uint4* qs4 = reinterpret_cast<uint4*>(smem + C::OFF_QA);
#pragma unroll
      for (int j = 0; j < C::KSTEPS / 2; ++j)
        qs4[j * 32 + lane] = make_uint4(qa[2 * j][0], qa[2 * j][1], qa[2 * j + 1][0], qa[2 * j + 1][1]);
    }
  }
  __syncthreads();

  const int kb0 = warp * 16;  // this warp's first key in every tile
  // S^T rows r and r+8 are keys kA, kB; the P.V k indices 2c, 2c+1, 2c+8, 2c+9
  // are keys kv[0..3]
  const int kA = key_of(r), kB = key_of(r + 8);
  int kv[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) kv[i] = key_of(8 * (i >> 1) + 2 * c + (i & 1));
  // fp32 scale staging: lane l converts array l/8 (K scale, K bias, V scale,
  // V bias) of keys 2(l%8), 2(l%8)+1
  float* scw = reinterpret_cast<float*>(smem + C::OFF_SC) + warp * C::SCW;
  const int sarr = lane >> 3, skey = 2 * (lane & 7);
  const int soff = sarr == 0 ? C::OFF_KS : sarr == 1 ? C::OFF_KB : sarr == 2 ? C::OFF_VS : C::OFF_VB;
  auto sc2 = [&](int arr, int key) -> float2 {  // (group 0, group NG-1) of one staged array
    if constexpr (NG == 2) return *reinterpret_cast<const float2*>(scw + (arr * 16 + key) * 2);
    const float x = scw[arr * 16 + key];
    return make_float2(x, 0.f);
  };

  // online-softmax state of heads 2c (L) and 2c+1 (H); the same on the 8 lanes of a column
  float m_refL = -INFINITY, m_refH = -INFINITY, lsumL = 0.f, lsumH = 0.f;
  float2 baccL = make_float2(0.f, 0.f), baccH = make_float2(0.f, 0.f);  // sum_j p_j (b_jG + 8 s_jG) (this thread's keys)
  float oacc[C::MT][4];  // O^T: dims (mt, r / r+8) x heads (2c, 2c+1)
  float corr[NG][4];     // 136 * sum_j B[j][head], heads (2c, 2c+1)
#pragma unroll
  for (int G = 0; G < NG; ++G) corr[G][0] = corr[G][1] = corr[G][2] = corr[G][3] = 0.f;
#pragma unroll
  for (int j = 0; j < C::MT; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;

  // One warp tile (16 keys).  FULL: all 16 keys lie below kv_len, so no
  // score needs masking and no scale can be garbage.
  auto tile = [&](const unsigned char* S, int wvalid, auto full_tag) {
    constexpr bool FULL = decltype(full_tag)::value;
    // ---- S^T = K Q^T: M = 16 keys (rows r, r+8 = keys kA, kB), N = 8 heads ----
    float sacc[NG][4];
    {
      uint32_t qa[C::KSTEPS][2];
#pragma unroll
      for (int j = 0; j < C::KSTEPS / 2; ++j) {
        const uint4 v = reinterpret_cast<const uint4*>(smem + C::OFF_QA)[j * 32 + lane];
        qa[2 * j][0] = v.x;
        qa[2 * j][1] = v.y;
        qa[2 * j + 1][0] = v.z;
        qa[2 * j + 1][1] = v.w;
      }
      const unsigned char* ka = S + C::OFF_KC + (kb0 + kA) * C::CB + 8 * c;
      const unsigned char* kbp = S + C::OFF_KC + (kb0 + kB) * C::CB + 8 * c;
#pragma unroll
      for (int G = 0; G < NG; ++G) {
        sacc[G][0] = sacc[G][1] = sacc[G][2] = sacc[G][3] = 0.f;
        const uint2 wa = *reinterpret_cast<const uint2*>(ka + 32 * G);
        const uint2 wb = *reinterpret_cast<const uint2*>(kbp + 32 * G);
#pragma unroll
        for (int wi = 0; wi < 2; ++wi) {
          const uint32_t x = wi ? wa.y : wa.x, y = wi ? wb.y : wb.x;
          const uint32_t x8 = x >> 8, y8 = y >> 8;
          const int k0 = 4 * G + 2 * wi;
          // k-step k0: codes of bytes 0 and 2; k-step k0 + 1: bytes 1 and 3
          mma_f16(sacc[G], nib_lo_f16(x), nib_lo_f16(y), nib_hi_f16(x), nib_hi_f16(y), qa[k0][0], qa[k0][1]);
          mma_f16(sacc[G], nib_lo_f16(x8), nib_lo_f16(y8), nib_hi_f16(x8), nib_hi_f16(y8), qa[k0 + 1][0],
                  qa[k0 + 1][1]);
        }
      }
    }
    // ---- scores (base 2): [0] (kA, 2c), [1] (kA, 2c+1), [2] (kB, 2c), [3] (kB, 2c+1) ----
    const float2 ksA = sc2(0, kA), kbA = sc2(1, kA), ksB = sc2(0, kB), kbB = sc2(1, kB);
    float sv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 ks2 = i < 2 ? ksA : ksB, kb2 = i < 2 ? kbA : kbB;
      const float2 off = (i & 1) ? qoffH : qoffL, qq = (i & 1) ? qbH : qbL;
      const float2 t2 = ffma2(make_float2(sacc[0][i], sacc[NG - 1][i]), make_float2(sq, sq), off);
      const float2 s2 = ffma2(kb2, qq, __fmul2_rn(ks2, t2));
      const float s = NG == 2 ? s2.x + s2.y : s2.x;
      sv[i] = (FULL || (i < 2 ? kA : kB) < wvalid) ? s : -INFINITY;
    }
    // lazy reference: raised only when a tile's maximum exceeds it by 2^8.
    // Whether any column's maximum does is decided from each lane's own
    // scores; the maxima over the 8 lanes of a column are formed only then.
    float mL = fmaxf(sv[0], sv[2]), mH = fmaxf(sv[1], sv[3]);
    if (__any_sync(0xffffffffu, mL > m_refL + 8.f || mH > m_refH + 8.f)) {
#pragma unroll
      for (int m = 4; m <= 16; m <<= 1) {
        mL = fmaxf(mL, __shfl_xor_sync(0xffffffffu, mL, m));
        mH = fmaxf(mH, __shfl_xor_sync(0xffffffffu, mH, m));
      }
      const bool rL = mL > m_refL + 8.f, rH = mH > m_refH + 8.f;
      const float aL = rL ? fast_exp2(m_refL - mL) : 1.f;
      const float aH = rH ? fast_exp2(m_refH - mH) : 1.f;
      if (rL) m_refL = mL;
      if (rH) m_refH = mH;
      lsumL *= aL;
      lsumH *= aH;
      baccL = __fmul2_rn(baccL, make_float2(aL, aL));
      baccH = __fmul2_rn(baccH, make_float2(aH, aH));
#pragma unroll
      for (int j = 0; j < C::MT; ++j) {
        oacc[j][0] *= aL;
        oacc[j][1] *= aH;
        oacc[j][2] *= aL;
        oacc[j][3] *= aH;
      }
#pragma unroll
      for (int G = 0; G < NG; ++G) {
        corr[G][0] *= aL;
        corr[G][1] *= aH;
      }
    }
    const float muL = m_refL == -INFINITY ? 0.f : m_refL;
    const float muH = m_refH == -INFINITY ? 0.f : m_refH;
    float pv[4];
    pv[0] = fast_exp2(sv[0] - muL);
    pv[1] = fast_exp2(sv[1] - muH);
    pv[2] = fast_exp2(sv[2] - muL);
    pv[3] = fast_exp2(sv[3] - muH);
    lsumL += pv[0] + pv[2];
    lsumH += pv[1] + pv[3];
    // ---- B operand of O^T += V^T P^T: p_j s_jG, transposed from (key, head
    // pair) to (head, key pair) by movmatrix; and the bias sums.  Keys past
    // kv_len (p = 0) may have any scale and bias, NaN included, so their
    // terms are selected away rather than multiplied by zero. ----
    uint32_t bp[NG][2];
    {
      const float2 vsA = sc2(2, kA), vbA = sc2(3, kA), vsB = sc2(2, kB), vbB = sc2(3, kB);
      const bool liveA = FULL || kA < wvalid, liveB = FULL || kB < wvalid;
      const float2 pA = make_float2(pv[0], pv[1]), pB = make_float2(pv[2], pv[3]);
      float2 wA[NG], wB[NG];
#pragma unroll
      for (int G = 0; G < NG; ++G) {
        const float sa = G == 0 ? vsA.x : vsA.y, sb = G == 0 ? vsB.x : vsB.y;
        wA[G] = liveA ? __fmul2_rn(pA, make_float2(sa, sa)) : make_float2(0.f, 0.f);
        wB[G] = liveB ? __fmul2_rn(pB, make_float2(sb, sb)) : make_float2(0.f, 0.f);
        bp[G][0] = movmatrix_t(pack_bf16(wA[G].x, wA[G].y));
        bp[G][1] = movmatrix_t(pack_bf16(wB[G].x, wB[G].y));
      }
      if (liveA) {
        baccL = ffma2(make_float2(pv[0], pv[0]), vbA, baccL);
        baccH = ffma2(make_float2(pv[1], pv[1]), vbA, baccH);
      }
      if (liveB) {
        baccL = ffma2(make_float2(pv[2], pv[2]), vbB, baccL);
        baccH = ffma2(make_float2(pv[3], pv[3]), vbB, baccH);
      }
      // the centre of the codes, 8 p_j s_jG, from the unrounded weights (0
      // for keys past kv_len)
      const float2 eight = make_float2(8.f, 8.f);
      baccL = ffma2(eight, make_float2(wA[0].x + wB[0].x, wA[NG - 1].x + wB[NG - 1].x), baccL);
      baccH = ffma2(eight, make_float2(wA[0].y + wB[0].y, wA[NG - 1].y + wB[NG - 1].y), baccH);
    }
    // ---- O^T += V^T P^T.  Thread (r, c) reads, for keys kv[0..3], the
    // code bytes 32G + 4r .. +3 of every group G; M-tile 4G + m takes byte
    // m: its low nibble is dim 64G + 8r + 2m (row r of the tile), its high
    // nibble dim 64G + 8r + 2m + 1 (row r + 8). ----
#pragma unroll
    for (int G = 0; G < NG; ++G) {
      uint32_t wv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        wv[i] = *reinterpret_cast<const uint32_t*>(S + C::OFF_VC + (kb0 + kv[i]) * C::CB + 32 * G + 4 * r);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t sel = 0x4400u | (0x1111u * uint32_t(m));  // bytes (m, m, 4+m, 4+m)
        const uint32_t x01 = __byte_perm(wv[0], wv[1], sel);
        const uint32_t x23 = __byte_perm(wv[2], wv[3], sel);
        mma_bf16(oacc[4 * G + m], nib_lo_bf16(x01), nib_lo_bf16(x01 >> 4), nib_lo_bf16(x23),
                 nib_lo_bf16(x23 >> 4), bp[G][0], bp[G][1]);
      }
      mma_bf16(corr[G], kBf136x2, kBf136x2, kBf136x2, kBf136x2, bp[G][0], bp[G][1]);
    }
  };

  int st = 0;
  uint32_t phase = 0;
  for (int t = 0; t < nt; ++t) {
    const bool ok = wait_or_abort(&full[st], phase, flag, p.wait_limit_ns);
    if (!__all_sync(0xffffffffu, ok)) break;
    const int wvalid = min(TILE, L - (split + t * n_used) * TILE) - kb0;  // valid keys among this warp's 16
    const unsigned char* S = smem + st * C::STAGEB;
    if (wvalid > 0) {
      // this warp's 16 scales and biases of each kind, as fp32
      if constexpr (NG == 2) {
        const uint2 h = *reinterpret_cast<const uint2*>(S + soff + (kb0 + skey) * C::GB);
        const float2 a = f16x2_to_float2(h.x), bb = f16x2_to_float2(h.y);
        *reinterpret_cast<float4*>(scw + (sarr * 16 + skey) * 2) = make_float4(a.x, a.y, bb.x, bb.y);
      } else {
        const uint32_t h = *reinterpret_cast<const uint32_t*>(S + soff + (kb0 + skey) * C::GB);
        *reinterpret_cast<float2*>(scw + sarr * 16 + skey) = f16x2_to_float2(h);
      }
      __syncwarp();
      if (wvalid >= 16)
        tile(S, wvalid, std::true_type{});
      else
        tile(S, wvalid, std::false_type{});
    }
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&rel[st], 1) == C::NW - 1) {  // the last warp done with the stage refills it
        rel[st] = 0;
        if (t + NSTAGE < nt && !flag[0]) {
          issue(t + NSTAGE, st, pol);
          atomicMax(const_cast<int*>(&flag[2]), t + NSTAGE + 1);
        }
      }
    }
    if (++st == NSTAGE) {
      st = 0;
      phase ^= 1u;
    }
  }
  // totals over the 8 lanes of each column (this thread's keys -> all keys)
#pragma unroll
  for (int m = 4; m <= 16; m <<= 1) {
    lsumL += __shfl_xor_sync(0xffffffffu, lsumL, m);
    lsumH += __shfl_xor_sync(0xffffffffu, lsumH, m);
    baccL.x += __shfl_xor_sync(0xffffffffu, baccL.x, m);
    baccL.y += __shfl_xor_sync(0xffffffffu, baccL.y, m);
    baccH.x += __shfl_xor_sync(0xffffffffu, baccH.x, m);
    baccH.y += __shfl_xor_sync(0xffffffffu, baccH.y, m);
  }
  __syncthreads();  // every warp has left the tile loop

  if (flag[0]) {  // a tile copy did not arrive in time
    if (tid == 0) {
      atomicOr(p.status, GQA_DEV_WAIT_TIMEOUT);
      const int issued = flag[2];
      for (int s = 0; s < NSTAGE && s < issued; ++s) {  // let the last copy on each stage land
        const int u = s + ((issued - 1 - s) / NSTAGE) * NSTAGE;
        mbar_wait_bounded(&full[s], uint32_t(u / NSTAGE) & 1u, p.wait_limit_ns);
      }
    }
    __syncthreads();
    return;
  }
  // every issued copy has landed: the stages can hold the warp-merge scratch
  float* merge_s = reinterpret_cast<float*>(smem);  // [warp][head][D]
  float* mw = merge_s + C::NW * 8 * D;              // [warp][head] maxima
  float* lw = mw + C::NW * 8;                       // [warp][head] sums
  {
    const int hA = 2 * c, hB = 2 * c + 1;
#pragma unroll
    for (int G = 0; G < NG; ++G)
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float* a = oacc[4 * G + m];
        const int d = 64 * G + 8 * r + 2 * m;
        const float offA = (G == 0 ? baccL.x : baccL.y) - corr[G][0];
        const float offB = (G == 0 ? baccH.x : baccH.y) - corr[G][1];
        *reinterpret_cast<float2*>(merge_s + (warp * 8 + hA) * D + d) = make_float2(a[0] + offA, a[2] + offA);
        *reinterpret_cast<float2*>(merge_s + (warp * 8 + hB) * D + d) = make_float2(a[1] + offB, a[3] + offB);
      }
    if (r == 0) {
      mw[warp * 8 + hA] = m_refL;
      mw[warp * 8 + hB] = m_refH;
      lw[warp * 8 + hA] = lsumL;
      lw[warp * 8 + hB] = lsumH;
    }
  }
  __syncthreads();
  // let the merge kernel's CTAs be scheduled while this grid drains
  grid_launch_dependents();

  // ---- merge the warps, then write O or this split's partial ----
  const size_t ws_row = size_t(b) * p.Hq + h0;  // first query head of this CTA
  for (int e = tid; e < nh * D; e += C::NTHR) {
    const int h = e / D, d = e % D;
    float M = mw[h];
#pragma unroll
    for (int w = 1; w < C::NW; ++w) M = fmaxf(M, mw[w * 8 + h]);
    float lt = 0.f, sum = 0.f;
#pragma unroll
    for (int w = 0; w < C::NW; ++w) {
      const float mwv = mw[w * 8 + h];
      const float ew = mwv == -INFINITY ? 0.f : fast_exp2(mwv - M);
      lt += lw[w * 8 + h] * ew;
      sum += merge_s[(w * 8 + h) * D + d] * ew;
    }
    if (n_used == 1 && !p.force_partial) {
      p.o[(ws_row + h) * D + d] = __float2bfloat16_rn(sum / lt);
    } else {
      p.part_o[((ws_row + h) * p.n_slots + split) * D + d] = sum;
      if (d == 0) p.ml[(ws_row + h) * p.n_slots + split] = make_float2(M, lt);
    }
  }
}

template <int D, int NSTAGE>
cudaError_t launch_q4_mma(const Q4Params& p, dim3 grid, cudaStream_t stream) {
  using C = Q4Cfg<D, NSTAGE>;
  auto kern = decode_q4_mma_kernel<D, NSTAGE>;
  static std::once_flag once;  // per instantiation; the attributes are per function
  static cudaError_t cfg_err = cudaSuccess;
  std::call_once(once, [&] {
    cfg_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (cfg_err == cudaSuccess)  // four CTAs per SM need the largest shared-memory carveout
      cfg_err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
  });
  if (cfg_err != cudaSuccess) return cfg_err;
  return launch_pdl(kern, grid, dim3(C::NTHR), C::SMEM, stream, p);
}

// Stages per head size: 5 x 9 KiB (D = 128) or 8 x 4.5 KiB (D = 64) keep four
// CTAs on an SM.
constexpr int kQ4Stages128 = 5;
constexpr int kQ4Stages64 = 8;

}  // namespace

int decode_q4_tile_rows(int D) { return D == 128 ? Q4Cfg<128, kQ4Stages128>::TILE : Q4Cfg<64, kQ4Stages64>::TILE; }

int decode_q4_ctas_per_sm() { return 4; }

cudaError_t launch_decode_q4(const DecodeQ4Args& a, cudaStream_t stream) {
  Q4Params p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.kc = a.k_codes;
  p.ks = reinterpret_cast<const __half*>(a.k_scale);
  p.kb = reinterpret_cast<const __half*>(a.k_bias);
  p.vc = a.v_codes;
  p.vs = reinterpret_cast<const __half*>(a.v_scale);
  p.vb = reinterpret_cast<const __half*>(a.v_bias);
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.kv_lens = a.kv_lens;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.n_rep = a.Hq / a.Hkv;
  p.n_hc = a.plan.n_hc;
  p.nrep_cta = a.plan.nrep_cta;
  p.S_cap = a.S_cap;
  p.max_kv_len = a.max_kv_len;
  p.chunk = a.plan.chunk;
  p.n_split = a.plan.n_split;
  p.n_slots = a.n_slots > 0 ? a.n_slots : a.plan.n_split;
  p.force_partial = a.force_partial;
  p.qscale = float(double(a.scale) * 1.4426950408889634);
  const WorkspaceLayout w = workspace_layout(a.B, a.Hq, a.Hkv, a.plan.n_hc, p.n_slots, a.D);
  unsigned char* ws = static_cast<unsigned char*>(a.workspace);
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.ml = reinterpret_cast<float2*>(ws + w.off_ml);
  p.part_o = reinterpret_cast<float*>(ws + w.off_o);
  p.wait_limit_ns = kWaitLimitNs;
  p.test_stall_ns = wait_test_ns();
  const dim3 grid(a.plan.n_split, a.Hkv * a.plan.n_hc, a.B);
  cudaError_t e = a.D == 128 ? launch_q4_mma<128, kQ4Stages128>(p, grid, stream)
                             : launch_q4_mma<64, kQ4Stages64>(p, grid, stream);
  if (e != cudaSuccess || a.plan.n_split == 1 || a.force_partial) return e;
  MergeParams m;
  m.o = p.o;
  m.kv_lens = p.kv_lens;
  m.Hq = p.Hq;
  m.max_kv_len = p.max_kv_len;
  m.chunk = p.chunk;
  m.n_split = p.n_split;
  m.ml = p.ml;
  m.part_o = p.part_o;
  const int rows = a.B * a.Hq;
  return a.D == 128 ? launch_merge<__nv_bfloat16, 128>(m, rows, stream)
                    : launch_merge<__nv_bfloat16, 64>(m, rows, stream);
}

}  // namespace gqa


namespace gqa {

// A 4-bit cache followed by an unquantized (bf16) residual window: the window
// kernel (decode_mma.cu) writes one partial per row into the slot after the
// 4-bit splits, the 4-bit kernel writes all its splits as partials, and the
// merge combines them.  Launch order: window, 4-bit splits, merge (each
// waits for the previous grid; the window grid is small, and the 4-bit
// grid's L2 prefetch overlaps it).
cudaError_t launch_decode_q4_residual(const DecodeQ4Args& aq, const DecodeArgs& ar, cudaStream_t stream) {
  const int n_slots = aq.plan.n_split + 1;
  cudaError_t e = launch_decode_mma_residual(ar, aq.kv_lens, aq.max_kv_len, aq.plan.chunk, n_slots, stream);
  if (e != cudaSuccess) return e;
  DecodeQ4Args a = aq;
  a.n_slots = n_slots;
  a.force_partial = 1;
  e = launch_decode_q4(a, stream);
  if (e != cudaSuccess) return e;
  const WorkspaceLayout w = workspace_layout(a.B, a.Hq, a.Hkv, a.plan.n_hc, n_slots, a.D);
  unsigned char* ws = static_cast<unsigned char*>(a.workspace);
  MergeParams m;
  m.o = a.o;
  m.kv_lens = ar.kv_lens;
  m.Hq = a.Hq;
  m.max_kv_len = a.max_kv_len;
  m.chunk = a.plan.chunk;
  m.n_split = n_slots;
  m.ml = reinterpret_cast<const float2*>(ws + w.off_ml);
  m.part_o = reinterpret_cast<const float*>(ws + w.off_o);
  m.n_quant = aq.kv_lens;
  m.max_quant = aq.max_kv_len;
  m.res_cap = ar.max_kv_len;
  m.status = reinterpret_cast<uint32_t*>(ws);
  const int rows = a.B * a.Hq;
  return a.D == 128 ? launch_merge<__nv_bfloat16, 128>(m, rows, stream)
                    : launch_merge<__nv_bfloat16, 64>(m, rows, stream);
}

}  // namespace gqa
