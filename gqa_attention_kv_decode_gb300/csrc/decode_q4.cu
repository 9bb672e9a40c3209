// decode_q4.cu -- single-token GQA decode over a 4-bit group-affine KV cache,
// dequantised inside the attention loop (sm_103a).
//
// The cache stores, per (request, KV head, token), D/2 bytes of 4-bit codes
// (element 2t in the low nibble of byte t) and one fp16 scale and bias per
// group of 64 elements: x = code * scale + bias ("Batching Decode Attention
// Across Requests ...", VeloxQuant-MLX blog, "The setup" and "Part 4": the
// fused decode-attend reads the codes directly instead of materialising an
// fp16 copy).  No dequantised row is ever stored: the affine term is folded
// out of both dot products,
//   q . k_j       = sum_g s_jg * (sum_{i in g} q_i c_ji) + b_jg * (sum_{i in g} q_i)
//   sum_j p_j v_j = sum_j (p_j s_jg) c_j + sum_j p_j b_jg      (per group g)
// so each code costs one multiply-add per query head and a conversion.
//
// The CTA structure is the one of the fp32/bf16 decode kernel: 4 warps, tiles
// of 64 rows streamed by bulk copies (codes, scales and biases of K and V: six
// copies per stage), tiles dealt round-robin to the splits, a per-warp online
// softmax in base 2, warps merged in shared memory, and split partials merged
// by the shared merge kernel.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

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
};

template <int D, int NREP, int NSTAGE>
struct Q4Cfg {
  static constexpr int CB = D / 2;         // code bytes per row
  static constexpr int NG = D / 64;        // groups per row
  static constexpr int GB = NG * 2;        // bytes of fp16 scales (or biases) per row
  static constexpr int SROUND = 16 / GB;   // rows per 16 bytes of scales
  static constexpr int NCW = 4;
  static constexpr int NTHR = 32 * NCW;
  static constexpr int DSQ = CB / 16;      // lanes per row in the score phase (32 codes each)
  static constexpr int RGW = 32 / DSQ;     // row groups per warp
  static constexpr int R = D == 128 ? 2 : 1;
  static constexpr int TW = RGW * R;       // rows per warp per tile
  static constexpr int TILE = NCW * TW;
  static constexpr int NREP_P = NREP <= 1 ? 1 : NREP <= 2 ? 2 : NREP <= 4 ? 4 : 8;
  static constexpr int V0 = R * NREP_P;
  static constexpr int VP = V0 > DSQ ? V0 : DSQ;
  static constexpr int NV = VP / DSQ;      // complete scores per lane after the butterfly
  static constexpr int G = NREP_P / NV;    // lanes whose ds agree modulo G hold the same heads
  static constexpr int LPRV = CB / 8;      // lanes per row in P.V (16 codes each)
  static constexpr int RPW = 32 / LPRV;
  static constexpr int OFF_KC = 0;
  static constexpr int OFF_KS = OFF_KC + TILE * CB;
  static constexpr int OFF_KB = OFF_KS + TILE * GB;
  static constexpr int OFF_VC = OFF_KB + TILE * GB;
  static constexpr int OFF_VS = OFF_VC + TILE * CB;
  static constexpr int OFF_VB = OFF_VS + TILE * GB;
  static constexpr int STAGEB = OFF_VB + TILE * GB;
  static constexpr int OFF_Q = NSTAGE * STAGEB;
  static constexpr int OFF_QSUM = OFF_Q + NREP_P * D * 4;
  static constexpr int OFF_P = OFF_QSUM + ((NREP_P * DSQ * 4 + 15) / 16) * 16;
  static constexpr int OFF_BAR = OFF_P + NCW * TW * NREP_P * 4;
  static constexpr int OFF_FLAG = OFF_BAR + NSTAGE * 8 + ((NSTAGE * 4 + 7) / 8) * 8;
  static constexpr int SMEM = OFF_FLAG + 16;
  static constexpr int MERGE_FLOATS = NCW * (NREP_P * D + 2 * NREP_P);
  static_assert(CB % 16 == 0 && DSQ >= 1, "a row is whole 16-byte chunks");
  static_assert(TILE % SROUND == 0 && STAGEB % 16 == 0, "bulk copy alignment");
  static_assert(G >= 1 && G <= DSQ && NV <= NREP_P, "head layout");
  static_assert(MERGE_FLOATS * 4 <= NSTAGE * STAGEB, "warp-merge scratch must fit");
};

// Two codes of each byte of `w` as float pairs: {low nibble, high nibble}.
// A code c becomes the float 2^23 + c by placing it under the exponent bits
// of 2^23, then 2^23 is subtracted exactly.
__device__ __forceinline__ void codes8(uint32_t w, float2 (&out)[4]) {
  const uint32_t lo = w & 0x0F0F0F0Fu;
  const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
  const float2 off = make_float2(-8388608.f, -8388608.f);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float a = __uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7440u | t));
    const float b = __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7440u | t));
    out[t] = __fadd2_rn(make_float2(a, b), off);
  }
}

template <int D, int NREP, int NSTAGE>
__global__ void __launch_bounds__(Q4Cfg<D, NREP, NSTAGE>::NTHR, 2)
    decode_q4_split_kernel(const Q4Params p) {
  using C = Q4Cfg<D, NREP, NSTAGE>;
  constexpr int TILE = C::TILE;
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

  // As in the fp32/bf16 decode kernel: while the previous grid in the stream
  // may still run, only prefetch this split's first code tiles into L2.
  if (tid == 0 && hc == 0) {
    for (int t = 0; t < NSTAGE; ++t) {
      const int row0 = (split + t * p.n_split) * TILE;
      if (row0 >= p.max_kv_len) break;
      const uint32_t cbytes = uint32_t(min(TILE, p.max_kv_len - row0)) * C::CB;
      prefetch_l2_bulk(kc + size_t(row0) * C::CB, cbytes);
      prefetch_l2_bulk(vc + size_t(row0) * C::CB, cbytes);
    }
  }
  grid_dependency_wait();

  int L = p.kv_lens ? p.kv_lens[b] : p.max_kv_len;
  if (L < 0 || L > p.max_kv_len) {
    if (split == 0 && blockIdx.y == 0 && tid == 0) atomicOr(p.status, GQA_DEV_KVLEN_CLAMPED);
    L = L < 0 ? 0 : p.max_kv_len;
  }
  if (L == 0) {
    if (split == 0) {
      if (blockIdx.y == 0 && tid == 0) atomicOr(p.status, GQA_DEV_EMPTY_REQUEST);
      for (int e = tid; e < nh * D; e += C::NTHR)
        p.o[(size_t(b) * p.Hq + h0 + e / D) * D + e % D] = __float2bfloat16_rn(0.f);
    }
    return;
  }
  const int n_used = (L + p.chunk - 1) / p.chunk;
  if (split >= n_used) return;
  const int nt_all = (L + TILE - 1) / TILE;
  const int nt = (nt_all - split + n_used - 1) / n_used;

  float* q_s = reinterpret_cast<float*>(smem + C::OFF_Q);
  float* qsum_s = reinterpret_cast<float*>(smem + C::OFF_QSUM);
  float* p_s = reinterpret_cast<float*>(smem + C::OFF_P);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  int* rel = reinterpret_cast<int*>(smem + C::OFF_BAR + NSTAGE * 8);
  volatile int* flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);

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
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      rel[s] = 0;
    }
    fence_barrier_init();
    flag[0] = 0;
    const uint64_t pol = l2_policy_evict_first();
    for (int t = 0; t < NSTAGE && t < nt; ++t) issue(t, t, pol);
    flag[2] = min(NSTAGE, nt);
  }
  // q rows (scaled, fp32), laid out so that the DSQ lanes sharing a K row
  // read consecutive 16-byte pieces: element d = 32*c + 8*w + 4*half + j of
  // head h sits at ((h*4 + w)*2 + half)*DSQ*4 + c*4 + j; and the sums of q
  // over each 32-code chunk c.
  auto qidx = [](int h, int d) {
    const int c = d >> 5, w = (d >> 3) & 3, half = (d >> 2) & 1, j = d & 3;
    return ((h * 4 + w) * 2 + half) * C::DSQ * 4 + c * 4 + j;
  };
  {
    const uint32_t* qg = reinterpret_cast<const uint32_t*>(p.q + (size_t(b) * p.Hq + h0) * D);
    for (int e2 = tid; e2 < C::NREP_P * D / 2; e2 += C::NTHR) {
      const int h = (2 * e2) / D, d = (2 * e2) % D;
      const float2 v = h < nh ? bf16x2_to_float2(qg[e2]) : make_float2(0.f, 0.f);
      q_s[qidx(h, d)] = v.x * p.qscale;
      q_s[qidx(h, d + 1)] = v.y * p.qscale;
    }
  }
  __syncthreads();
  if (tid < C::NREP_P * C::DSQ) {
    const int h = tid / C::DSQ, c = tid % C::DSQ;
    float sum = 0.f;
    for (int i = 0; i < 32; ++i) sum += q_s[qidx(h, 32 * c + i)];
    qsum_s[h * C::DSQ + c] = sum;
  }
  __syncthreads();

  const uint64_t pol = l2_policy_evict_first();
  const int ds = lane % C::DSQ;  // 16-byte chunk of a K row (32 codes)
  const int rg = lane / C::DSQ;
  const int gk = ds / 2;         // group of that chunk
  const int cp = lane % C::LPRV; // 8-byte chunk of a V row (16 codes)
  const int rsub = lane / C::LPRV;
  const int gv = cp / 4;         // group of that chunk
  float* pw = p_s + warp * C::TW * C::NREP_P;
  float mref[C::NV], lsum[C::NV], bsum[C::NV][C::NG];
#pragma unroll
  for (int i = 0; i < C::NV; ++i) {
    mref[i] = -INFINITY;
    lsum[i] = 0.f;
#pragma unroll
    for (int gg = 0; gg < C::NG; ++gg) bsum[i][gg] = 0.f;
  }
  float2 acc_o[NREP][8];
#pragma unroll
  for (int h = 0; h < NREP; ++h)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc_o[h][j] = make_float2(0.f, 0.f);

  for (int t = 0; t < nt; ++t) {
    const int st = t % NSTAGE;
    const bool ok = wait_or_abort(&full[st], uint32_t(t / NSTAGE) & 1u, flag, p.wait_limit_ns);
    if (!__all_sync(0xffffffffu, ok)) break;
    const int nvalid = min(TILE, L - (split + t * n_used) * TILE);
    const int wrow0 = warp * C::TW;
    const int wvalid = min(C::TW, nvalid - wrow0);
    const unsigned char* S = smem + st * C::STAGEB;
    const __half* Ksc = reinterpret_cast<const __half*>(S + C::OFF_KS);
    const __half* Kbi = reinterpret_cast<const __half*>(S + C::OFF_KB);
    const __half* Vsc = reinterpret_cast<const __half*>(S + C::OFF_VS);
    if (wvalid > 0) {
      // ---- scores: lane ds owns 32 codes (one group) of R rows ----
      float2 acc[C::R][NREP];
#pragma unroll
      for (int r = 0; r < C::R; ++r)
#pragma unroll
        for (int h = 0; h < NREP; ++h) acc[r][h] = make_float2(0.f, 0.f);
      uint4 raw[C::R];
#pragma unroll
      for (int r = 0; r < C::R; ++r)
        raw[r] = *reinterpret_cast<const uint4*>(S + C::OFF_KC + (wrow0 + rg * C::R + r) * C::CB + ds * 16);
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        float2 cf[C::R][4];
#pragma unroll
        for (int r = 0; r < C::R; ++r) {
          const uint32_t word = w == 0 ? raw[r].x : w == 1 ? raw[r].y : w == 2 ? raw[r].z : raw[r].w;
          codes8(word, cf[r]);
        }
#pragma unroll
        for (int h = 0; h < NREP; ++h) {
          const float4 qa = *reinterpret_cast<const float4*>(q_s + ((h * 4 + w) * 2 + 0) * C::DSQ * 4 + ds * 4);
          const float4 qb = *reinterpret_cast<const float4*>(q_s + ((h * 4 + w) * 2 + 1) * C::DSQ * 4 + ds * 4);
#pragma unroll
          for (int r = 0; r < C::R; ++r) {
            acc[r][h] = ffma2(cf[r][0], make_float2(qa.x, qa.y), acc[r][h]);
            acc[r][h] = ffma2(cf[r][1], make_float2(qa.z, qa.w), acc[r][h]);
            acc[r][h] = ffma2(cf[r][2], make_float2(qb.x, qb.y), acc[r][h]);
            acc[r][h] = ffma2(cf[r][3], make_float2(qb.z, qb.w), acc[r][h]);
          }
        }
      }
      float v[C::VP];
#pragma unroll
      for (int r = 0; r < C::R; ++r) {
        const int row = wrow0 + rg * C::R + r;
        const float sc = __half2float(Ksc[row * C::NG + gk]);
        const float bi = __half2float(Kbi[row * C::NG + gk]);
#pragma unroll
        for (int h = 0; h < C::NREP_P; ++h)
          v[r * C::NREP_P + h] =
              h < NREP ? sc * (acc[r][h].x + acc[r][h].y) + bi * qsum_s[h * C::DSQ + ds] : 0.f;
      }
#pragma unroll
      for (int i = C::V0; i < C::VP; ++i) v[i] = 0.f;
      // transposing butterfly over the DSQ lanes of a row
#pragma unroll
      for (int m = C::DSQ / 2, n = C::VP; m >= 1; m >>= 1, n >>= 1) {
        const bool hi = (ds & m) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
          const float mine = hi ? v[n / 2 + i] : v[i];
          const float send = hi ? v[i] : v[n / 2 + i];
          v[i] = mine + __shfl_xor_sync(0xffffffffu, send, m);
        }
      }
      float sc[C::NV], mx[C::NV], alpha[C::NV];
      int rloc[C::NV];
#pragma unroll
      for (int i = 0; i < C::NV; ++i) {
        const int idx = ds * C::NV + i;
        const int r = idx / C::NREP_P, h = idx % C::NREP_P;
        rloc[i] = rg * C::R + r;
        const bool valid = (idx < C::V0) && (h < nh) && (rloc[i] < wvalid);
        sc[i] = valid ? v[i] : -INFINITY;
        mx[i] = sc[i];
      }
#pragma unroll
      for (int m = C::G; m <= 16; m <<= 1)
#pragma unroll
        for (int i = 0; i < C::NV; ++i) mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], m));
      bool rescale = false;
#pragma unroll
      for (int i = 0; i < C::NV; ++i) {
        alpha[i] = 1.f;
        if (mx[i] > mref[i] + 8.f) {
          alpha[i] = fast_exp2(mref[i] - mx[i]);
          mref[i] = mx[i];
          rescale = true;
        }
        const float pv = sc[i] == -INFINITY ? 0.f : fast_exp2(sc[i] - mref[i]);
        lsum[i] = lsum[i] * alpha[i] + pv;
        const int idx = ds * C::NV + i;
        const int rr = idx < C::V0 ? rloc[i] : 0;
        const __half* vb_row = reinterpret_cast<const __half*>(S + C::OFF_VB) + (wrow0 + rr) * C::NG;
#pragma unroll
        for (int gg = 0; gg < C::NG; ++gg)
          bsum[i][gg] = bsum[i][gg] * alpha[i] + (pv != 0.f ? pv * __half2float(vb_row[gg]) : 0.f);
        if (idx < C::V0) pw[rloc[i] * C::NREP_P + idx % C::NREP_P] = pv;
      }
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int h = 0; h < NREP; ++h) {
          const float a = __shfl_sync(0xffffffffu, alpha[h % C::NV], h / C::NV);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            acc_o[h][j].x *= a;
            acc_o[h][j].y *= a;
          }
        }
      }
      __syncwarp();
      // ---- P.V: lane owns 16 codes (one group) of a V row, every head ----
      for (int j = rsub; j < wvalid; j += C::RPW) {
        const int row = wrow0 + j;
        const uint2 raw2 = *reinterpret_cast<const uint2*>(S + C::OFF_VC + row * C::CB + cp * 8);
        float2 cf[8];
        codes8(raw2.x, *reinterpret_cast<float2(*)[4]>(&cf[0]));
        codes8(raw2.y, *reinterpret_cast<float2(*)[4]>(&cf[4]));
        const float s = __half2float(Vsc[row * C::NG + gv]);
#pragma unroll
        for (int h = 0; h < NREP; ++h) {
          const float wgt = pw[j * C::NREP_P + h] * s;
          const float2 w2 = make_float2(wgt, wgt);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) acc_o[h][jj] = ffma2(cf[jj], w2, acc_o[h][jj]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&rel[st], 1) == C::NCW - 1) {
        rel[st] = 0;
        if (t + NSTAGE < nt && !flag[0]) {
          issue(t + NSTAGE, st, pol);
          atomicMax(const_cast<int*>(&flag[2]), t + NSTAGE + 1);
        }
      }
    }
  }

  // ---- warp totals; bias sums folded into the lanes that own rsub == 0 ----
#pragma unroll
  for (int m = C::G; m <= 16; m <<= 1)
#pragma unroll
    for (int i = 0; i < C::NV; ++i) {
      lsum[i] += __shfl_xor_sync(0xffffffffu, lsum[i], m);
#pragma unroll
      for (int gg = 0; gg < C::NG; ++gg) bsum[i][gg] += __shfl_xor_sync(0xffffffffu, bsum[i][gg], m);
    }
#pragma unroll
  for (int m = 16; m >= C::LPRV; m >>= 1)
#pragma unroll
    for (int h = 0; h < NREP; ++h)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc_o[h][j].x += __shfl_xor_sync(0xffffffffu, acc_o[h][j].x, m);
        acc_o[h][j].y += __shfl_xor_sync(0xffffffffu, acc_o[h][j].y, m);
      }
#pragma unroll
  for (int h = 0; h < NREP; ++h) {
    float bh = 0.f;
#pragma unroll
    for (int gg = 0; gg < C::NG; ++gg) {
      const float x = __shfl_sync(0xffffffffu, bsum[h % C::NV][gg], h / C::NV);
      if (gg == gv) bh = x;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      acc_o[h][j].x += bh;
      acc_o[h][j].y += bh;
    }
  }
  __syncthreads();  // every warp has left the tile loop

  if (flag[0]) {
    if (tid == 0) {
      atomicOr(p.status, GQA_DEV_WAIT_TIMEOUT);
      const int issued = flag[2];
      for (int s = 0; s < NSTAGE && s < issued; ++s) {
        const int u = s + ((issued - 1 - s) / NSTAGE) * NSTAGE;
        mbar_wait_bounded(&full[s], uint32_t(u / NSTAGE) & 1u, p.wait_limit_ns);
      }
    }
    __syncthreads();
    return;
  }
  float* merge_s = reinterpret_cast<float*>(smem);
  float* mw = merge_s + C::NCW * C::NREP_P * D;
  float* lw = mw + C::NCW * C::NREP_P;
  if (rsub == 0)
#pragma unroll
    for (int h = 0; h < NREP; ++h)
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<float2*>(merge_s + (warp * C::NREP_P + h) * D + cp * 16 + 2 * j) = acc_o[h][j];
  if (lane < C::G)
#pragma unroll
    for (int i = 0; i < C::NV; ++i) {
      mw[warp * C::NREP_P + lane * C::NV + i] = mref[i];
      lw[warp * C::NREP_P + lane * C::NV + i] = lsum[i];
    }
  __syncthreads();
  grid_launch_dependents();

  const size_t ws_row = size_t(b) * p.Hq + h0;
  for (int e = tid; e < nh * D; e += C::NTHR) {
    const int h = e / D, d = e % D;
    float M = mw[h];
#pragma unroll
    for (int w = 1; w < C::NCW; ++w) M = fmaxf(M, mw[w * C::NREP_P + h]);
    float lt = 0.f, sum = 0.f;
#pragma unroll
    for (int w = 0; w < C::NCW; ++w) {
      const float mwv = mw[w * C::NREP_P + h];
      const float ew = mwv == -INFINITY ? 0.f : fast_exp2(mwv - M);
      lt += lw[w * C::NREP_P + h] * ew;
      sum += merge_s[(w * C::NREP_P + h) * D + d] * ew;
    }
    if (n_used == 1) {
      p.o[(ws_row + h) * D + d] = __float2bfloat16_rn(sum / lt);
    } else {
      p.part_o[((ws_row + h) * p.n_split + split) * D + d] = sum;
      if (d == 0) p.ml[(ws_row + h) * p.n_split + split] = make_float2(M, lt);
    }
  }
}

template <int D, int NREP, int NSTAGE>
cudaError_t launch_q4_one(const Q4Params& p, dim3 grid, cudaStream_t stream) {
  using C = Q4Cfg<D, NREP, NSTAGE>;
  auto kern = decode_q4_split_kernel<D, NREP, NSTAGE>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return launch_pdl(kern, grid, dim3(C::NTHR), C::SMEM, stream, p);
}

constexpr int kQ4Stages = 8;

template <int D>
cudaError_t dispatch_q4(const Q4Params& p, dim3 grid, cudaStream_t s) {
  switch (p.nrep_cta) {
    case 1: return launch_q4_one<D, 1, kQ4Stages>(p, grid, s);
    case 2: return launch_q4_one<D, 2, kQ4Stages>(p, grid, s);
    case 3:
    case 4: return launch_q4_one<D, 4, kQ4Stages>(p, grid, s);
    default: return launch_q4_one<D, 8, kQ4Stages>(p, grid, s);
  }
}

}  // namespace

int decode_q4_tile_rows(int D) { return D == 128 ? Q4Cfg<128, 8, kQ4Stages>::TILE : Q4Cfg<64, 8, kQ4Stages>::TILE; }

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
  p.qscale = float(double(a.scale) * 1.4426950408889634);
  const WorkspaceLayout w = workspace_layout(a.B, a.Hq, a.Hkv, a.plan.n_hc, a.plan.n_split, a.D);
  unsigned char* ws = static_cast<unsigned char*>(a.workspace);
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.ml = reinterpret_cast<float2*>(ws + w.off_ml);
  p.part_o = reinterpret_cast<float*>(ws + w.off_o);
  p.wait_limit_ns = kWaitLimitNs;
  const dim3 grid(a.plan.n_split, a.Hkv * a.plan.n_hc, a.B);
  cudaError_t e = a.D == 128 ? dispatch_q4<128>(p, grid, stream) : dispatch_q4<64>(p, grid, stream);
  if (e != cudaSuccess || a.plan.n_split == 1) return e;
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
