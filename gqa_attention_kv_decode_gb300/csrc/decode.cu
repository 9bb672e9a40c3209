// decode.cu -- split-KV single-token GQA decode for sm_103a (fp32 / bf16 KV).
//
// One CTA serves one (request b, KV head g, query-head chunk, key split).  All
// the query heads that share KV head g (n_rep = Hq / Hkv of them, up to 8 per
// CTA) are computed together, so every K and V byte is read from HBM once
// ("2x Faster Qwen2 Decode on Metal in Candle", "Why It Matters": the fused
// kernel indexes the unexpanded KV heads through the head ratio and never
// copies them).
//
// Data flow per CTA:
//   * the split's key rows [s0, s1) are streamed in tiles of TILE rows; each
//     tile of K and of V is one contiguous bulk (TMA) copy into shared memory
//     (rows of a head are contiguous: "Fused attention makes a 4,096-token
//     Qwen2 prefill ...", "Cause and workaround", item 3), NSTAGE tiles in
//     flight, completion tracked by mbarriers with bounded waits;
//   * scores: 8 lanes share a key row (each 16-byte chunk of the row read by
//     one lane, conflict-free), a thread owns R rows x all heads, q is read
//     from shared memory as broadcasts, products accumulate with packed
//     fp32x2 FMAs; the 8 partial dot products are summed by a transposing
//     butterfly, after which each lane owns NV complete scores;
//   * online softmax in base 2 (q is pre-scaled by scale*log2(e)) with a lazy
//     reference: the running maximum is only raised, and the accumulators
//     rescaled, when a tile's maximum exceeds it by more than 2^8;
//   * P.V: a lane owns one 16-byte column chunk of V for every head, rows are
//     spread over row slots, p is broadcast from shared memory;
//   * the split's (max, sum, unnormalised o) go to the workspace and are
//     merged by a two-level log-sum-exp tree inside the same kernel: the last
//     CTA of each group of 8 splits merges the group, the last group merges
//     the groups and writes O.  A request that fits one split writes O
//     directly.
#include <cuda_bf16.h>

#include <cmath>

#include "gqa_attn.h"
#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

struct DecodeParams {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  const int32_t* kv_lens;
  int B, Hq, Hkv, n_rep, n_hc, nrep_cta, S_cap, max_kv_len, chunk, n_split;
  float qscale;  // scale * log2(e)
  uint32_t* status;
  int32_t* counters;
  float2* ml;
  float* part_o;
  float2* ml1;  // level-1 merged partials [B][Hq][n_groups_max]
  float* o1;    // [B][Hq][n_groups_max][D]
  int n_groups_max;
  uint64_t wait_limit_ns;
};

__device__ __forceinline__ float load_f(const float* p) { return *p; }
__device__ __forceinline__ float load_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <typename T, int D, int NREP, int TILE, int NSTAGE>
struct Cfg {
  static constexpr int E = sizeof(T);
  static constexpr int ROWB = D * E;     // bytes per key row
  static constexpr int NCH = ROWB / 16;  // 16-byte chunks per row
  static constexpr int EPC = 16 / E;     // elements per chunk
  static constexpr int NPART = EPC / 4;  // float4 pieces of q per chunk
  static constexpr int NTHR = 128;
  static constexpr int NWARP = NTHR / 32;
  static constexpr int DS = 8;           // lanes sharing a row in the score phase
  static constexpr int NIT = NCH / DS;
  static constexpr int RG = NTHR / DS;   // row groups
  static constexpr int R = TILE / RG;    // rows per thread in the score phase
  static constexpr int NREP_P = NREP <= 1 ? 1 : NREP <= 2 ? 2 : NREP <= 4 ? 4 : 8;
  static constexpr int VP = (R * NREP_P > 8) ? R * NREP_P : 8;
  static constexpr int NV = VP / 8;      // complete scores per lane after the butterfly
  static constexpr int G = NREP_P / NV;  // distinct head sets among the 8 lanes of a row group
  static constexpr int LPR = NCH;        // lanes per row in the P.V phase
  static constexpr int SLOTS = NTHR / LPR;
  static constexpr int TILEB = TILE * ROWB;
  static constexpr int STAGEB = 2 * TILEB;
  static constexpr int OFF_Q = NSTAGE * STAGEB;
  static constexpr int OFF_P = OFF_Q + NREP_P * D * 4;
  static constexpr int OFF_WMAX = OFF_P + TILE * NREP_P * 8;
  static constexpr int OFF_WSUM = OFF_WMAX + NWARP * 8 * 4;
  static constexpr int OFF_BAR = OFF_WSUM + NWARP * 8 * 4;
  static constexpr int OFF_FLAG = OFF_BAR + NSTAGE * 8;
  static constexpr int SMEM = OFF_FLAG + 16;
  static_assert(NCH % DS == 0, "row must split into 8 lanes of 16-byte chunks");
  static_assert(R >= 1 && R * RG == TILE && R <= 8, "tile must give 1..8 rows per thread");
  static_assert(NV <= NREP_P, "head layout");
  static_assert(SLOTS * NREP_P * D * 4 <= NSTAGE * STAGEB, "reduction scratch must fit");
  static_assert((128 * 8 + 16) * 4 <= NSTAGE * STAGEB, "merge weights must fit");
  static_assert(NREP >= 1 && NREP <= 8, "at most 8 query heads per CTA");
};

template <typename T, int D, int NREP, int TILE, int NSTAGE>
__global__ void __launch_bounds__(128) decode_split_kernel(const DecodeParams p) {
  using C = Cfg<T, D, NREP, TILE, NSTAGE>;
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

  int L = p.kv_lens ? p.kv_lens[b] : p.max_kv_len;
  if (L < 0 || L > p.max_kv_len) {
    if (split == 0 && blockIdx.y == 0 && tid == 0) atomicOr(p.status, GQA_DEV_KVLEN_CLAMPED);
    L = L < 0 ? 0 : p.max_kv_len;
  }
  T* out = static_cast<T*>(p.o);
  if (L == 0) {  // no visible key: the output row is zeros
    if (split == 0) {
      if (blockIdx.y == 0 && tid == 0) atomicOr(p.status, GQA_DEV_EMPTY_REQUEST);
      for (int e = tid; e < nh * D; e += C::NTHR)
        store_f(out + (size_t(b) * p.Hq + h0 + e / D) * D + e % D, 0.f);
    }
    return;
  }
  const int n_used = (L + p.chunk - 1) / p.chunk;
  if (split >= n_used) return;
  const int s0 = split * p.chunk;
  const int s1 = min(s0 + p.chunk, L);
  const int nt = (s1 - s0 + TILE - 1) / TILE;

  float* q_s = reinterpret_cast<float*>(smem + C::OFF_Q);
  float2* p_s = reinterpret_cast<float2*>(smem + C::OFF_P);
  float* wmax = reinterpret_cast<float*>(smem + C::OFF_WMAX);
  float* wsum = reinterpret_cast<float*>(smem + C::OFF_WSUM);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  volatile int* flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);

  const size_t head_row0 = (size_t(b) * p.Hkv + g) * size_t(p.S_cap);
  const unsigned char* kbase = static_cast<const unsigned char*>(p.k) + head_row0 * C::ROWB;
  const unsigned char* vbase = static_cast<const unsigned char*>(p.v) + head_row0 * C::ROWB;

  auto issue = [&](int t, int st, uint64_t pol) {
    const int row0 = s0 + t * TILE;
    const uint32_t bytes = uint32_t(min(TILE, s1 - row0)) * C::ROWB;
    unsigned char* dst = smem + st * C::STAGEB;
    mbar_arrive_expect_tx(&bar[st], 2 * bytes);
    bulk_g2s(dst, kbase + size_t(row0) * C::ROWB, bytes, &bar[st], pol);
    bulk_g2s(dst + C::TILEB, vbase + size_t(row0) * C::ROWB, bytes, &bar[st], pol);
  };

  uint64_t pol = 0;
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&bar[s], 1);
    fence_barrier_init();
    flag[0] = 0;
    pol = l2_policy_evict_first();
    for (int t = 0; t < NSTAGE && t < nt; ++t) issue(t, t, pol);
  }
  // q rows of this CTA's heads, pre-scaled, laid out so that the 8 lanes of a
  // row group read 8 consecutive 16-byte pieces: [h][part][chunk][4]
  {
    const T* qg = static_cast<const T*>(p.q);
    for (int e = tid; e < C::NREP_P * D; e += C::NTHR) {
      const int h = e / D, d = e % D;
      const float val = h < nh ? load_f(qg + (size_t(b) * p.Hq + h0 + h) * D + d) * p.qscale : 0.f;
      const int c = d / C::EPC, part = (d % C::EPC) / 4, j = d % 4;
      q_s[((h * C::NPART + part) * C::NCH + c) * 4 + j] = val;
    }
  }
  __syncthreads();

  const int ds = tid & 7;
  const int rg = tid >> 3;
  const int cp = tid % C::LPR;
  const int slot = tid / C::LPR;

  // Running reference (log2 units) of head hl; other heads' values are
  // fetched from lane h by shuffle (keeps them out of local memory).
  const int hl = lane % C::NREP_P;
  float my_mref = -INFINITY;
  float l_part[C::NV];
#pragma unroll
  for (int i = 0; i < C::NV; ++i) l_part[i] = 0.f;
  float2 acc_o[NREP][C::EPC / 2];
#pragma unroll
  for (int h = 0; h < NREP; ++h)
#pragma unroll
    for (int j = 0; j < C::EPC / 2; ++j) acc_o[h][j] = make_float2(0.f, 0.f);

  for (int t = 0; t < nt; ++t) {
    const int st = t % NSTAGE;
    const uint32_t par = uint32_t(t / NSTAGE) & 1u;
    if (!mbar_wait_bounded(&bar[st], par, p.wait_limit_ns)) flag[0] = 1;
    const int nvalid = min(TILE, s1 - (s0 + t * TILE));
    const unsigned char* Ks = smem + st * C::STAGEB;
    const unsigned char* Vs = Ks + C::TILEB;

    // ---- scores: R rows x NREP heads per thread, D split over 8 lanes ----
    float2 acc[C::R][NREP];
#pragma unroll
    for (int r = 0; r < C::R; ++r)
#pragma unroll
      for (int h = 0; h < NREP; ++h) acc[r][h] = make_float2(0.f, 0.f);
#pragma unroll
    for (int it = 0; it < C::NIT; ++it) {
      const int c = it * C::DS + ds;
      float2 kf[C::R][C::EPC / 2];
#pragma unroll
      for (int r = 0; r < C::R; ++r) {
        const uint4 raw = *reinterpret_cast<const uint4*>(Ks + (rg * C::R + r) * C::ROWB + c * 16);
        if constexpr (sizeof(T) == 4) {
          kf[r][0] = make_float2(__uint_as_float(raw.x), __uint_as_float(raw.y));
          kf[r][1] = make_float2(__uint_as_float(raw.z), __uint_as_float(raw.w));
        } else {
          kf[r][0] = bf16x2_to_float2(raw.x);
          kf[r][1] = bf16x2_to_float2(raw.y);
          kf[r][2] = bf16x2_to_float2(raw.z);
          kf[r][3] = bf16x2_to_float2(raw.w);
        }
      }
#pragma unroll
      for (int h = 0; h < NREP; ++h) {
#pragma unroll
        for (int part = 0; part < C::NPART; ++part) {
          const float4 qv =
              *reinterpret_cast<const float4*>(q_s + ((h * C::NPART + part) * C::NCH + c) * 4);
          const float2 qa = make_float2(qv.x, qv.y), qb = make_float2(qv.z, qv.w);
#pragma unroll
          for (int r = 0; r < C::R; ++r) {
            acc[r][h] = ffma2(kf[r][2 * part], qa, acc[r][h]);
            acc[r][h] = ffma2(kf[r][2 * part + 1], qb, acc[r][h]);
          }
        }
      }
    }
    // transposing butterfly over the 8 lanes of the row group: afterwards
    // lane ds holds the complete scores with flat index ds*NV + i, where the
    // flat index of (row r, head h) is r*NREP_P + h.
    float v[C::VP];
#pragma unroll
    for (int r = 0; r < C::R; ++r)
#pragma unroll
      for (int h = 0; h < C::NREP_P; ++h)
        v[r * C::NREP_P + h] = h < NREP ? acc[r][h].x + acc[r][h].y : 0.f;
#pragma unroll
    for (int i = C::R * C::NREP_P; i < C::VP; ++i) v[i] = 0.f;
#pragma unroll
    for (int m = 4, n = C::VP; m >= 1; m >>= 1, n >>= 1) {
      const bool hi = (ds & m) != 0;
#pragma unroll
      for (int i = 0; i < n / 2; ++i) {
        const float mine = hi ? v[n / 2 + i] : v[i];
        const float send = hi ? v[i] : v[n / 2 + i];
        v[i] = mine + __shfl_xor_sync(0xffffffffu, send, m);
      }
    }
    float s[C::NV];
    int hd[C::NV];
    int rowi[C::NV];
#pragma unroll
    for (int i = 0; i < C::NV; ++i) {
      const int idx = ds * C::NV + i;
      const int r = idx / C::NREP_P;
      hd[i] = idx % C::NREP_P;
      rowi[i] = rg * C::R + r;
      const bool valid = (idx < C::R * C::NREP_P) && (hd[i] < nh) && (rowi[i] < nvalid);
      s[i] = valid ? v[i] : -INFINITY;
    }
    // per-head tile maximum: lanes whose ds agree modulo G hold the same heads
    {
      float mx[C::NV];
#pragma unroll
      for (int i = 0; i < C::NV; ++i) mx[i] = s[i];
#pragma unroll
      for (int m = C::G; m <= 16; m <<= 1)
#pragma unroll
        for (int i = 0; i < C::NV; ++i) mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], m));
      if (lane < C::G)
#pragma unroll
        for (int i = 0; i < C::NV; ++i) wmax[warp * 8 + lane * C::NV + i] = mx[i];
    }
    __syncthreads();
    if (flag[0]) {  // a tile copy did not arrive in time: record it and stop
      if (tid == 0) {
        atomicOr(p.status, GQA_DEV_WAIT_TIMEOUT);
        for (int u = t; u < nt && u < t + NSTAGE; ++u)  // let issued copies land
          mbar_wait_bounded(&bar[u % NSTAGE], uint32_t(u / NSTAGE) & 1u, p.wait_limit_ns);
      }
      __syncthreads();
      return;
    }
    float my_alpha = 1.f;
    {
      float tm = wmax[hl];
#pragma unroll
      for (int w = 1; w < C::NWARP; ++w) tm = fmaxf(tm, wmax[w * 8 + hl]);
      if (tm > my_mref + 8.f) {
        my_alpha = fast_exp2(my_mref - tm);
        my_mref = tm;
      }
    }
    const bool any = __any_sync(0xffffffffu, my_alpha != 1.f);
#pragma unroll
    for (int i = 0; i < C::NV; ++i) {
      const float mr = __shfl_sync(0xffffffffu, my_mref, hd[i]);
      const float al = __shfl_sync(0xffffffffu, my_alpha, hd[i]);
      const float pv = s[i] == -INFINITY ? 0.f : fast_exp2(s[i] - mr);
      l_part[i] = l_part[i] * al + pv;
      if (ds * C::NV + i < C::R * C::NREP_P) p_s[rowi[i] * C::NREP_P + hd[i]] = make_float2(pv, pv);
    }
    if (any) {
#pragma unroll
      for (int h = 0; h < NREP; ++h) {
        const float a = __shfl_sync(0xffffffffu, my_alpha, h);
#pragma unroll
        for (int j = 0; j < C::EPC / 2; ++j) {
          acc_o[h][j].x *= a;
          acc_o[h][j].y *= a;
        }
      }
    }
    __syncthreads();

    // ---- P.V: lane owns one 16-byte column chunk for every head ----
    for (int row = slot; row < nvalid; row += C::SLOTS) {
      const uint4 raw = *reinterpret_cast<const uint4*>(Vs + row * C::ROWB + cp * 16);
      float2 vf[C::EPC / 2];
      if constexpr (sizeof(T) == 4) {
        vf[0] = make_float2(__uint_as_float(raw.x), __uint_as_float(raw.y));
        vf[1] = make_float2(__uint_as_float(raw.z), __uint_as_float(raw.w));
      } else {
        vf[0] = bf16x2_to_float2(raw.x);
        vf[1] = bf16x2_to_float2(raw.y);
        vf[2] = bf16x2_to_float2(raw.z);
        vf[3] = bf16x2_to_float2(raw.w);
      }
      const float2* prow = p_s + row * C::NREP_P;
      if constexpr (C::NREP_P == 1) {
        const float2 pp = prow[0];
#pragma unroll
        for (int j = 0; j < C::EPC / 2; ++j) acc_o[0][j] = ffma2(vf[j], pp, acc_o[0][j]);
      } else {
#pragma unroll
        for (int h2 = 0; h2 < C::NREP_P / 2; ++h2) {
          if (2 * h2 >= NREP) break;
          const float4 pp = reinterpret_cast<const float4*>(prow)[h2];
#pragma unroll
          for (int j = 0; j < C::EPC / 2; ++j) {
            acc_o[2 * h2][j] = ffma2(vf[j], make_float2(pp.x, pp.y), acc_o[2 * h2][j]);
            if (2 * h2 + 1 < NREP)
              acc_o[2 * h2 + 1][j] = ffma2(vf[j], make_float2(pp.z, pp.w), acc_o[2 * h2 + 1][j]);
          }
        }
      }
    }
    __syncthreads();
    if (tid == 0 && t + NSTAGE < nt) issue(t + NSTAGE, st, pol);
  }

  // ---- per-CTA reduction: softmax sums and row slots of o ----
  {
    float ls[C::NV];
#pragma unroll
    for (int i = 0; i < C::NV; ++i) ls[i] = l_part[i];
#pragma unroll
    for (int m = C::G; m <= 16; m <<= 1)
#pragma unroll
      for (int i = 0; i < C::NV; ++i) ls[i] += __shfl_xor_sync(0xffffffffu, ls[i], m);
    if (lane < C::G)
#pragma unroll
      for (int i = 0; i < C::NV; ++i) wsum[warp * 8 + lane * C::NV + i] = ls[i];
  }
  if (warp == 0 && lane < C::NREP_P) wmax[lane] = my_mref;  // final references
  float* red = reinterpret_cast<float*>(smem);  // all tile copies have been consumed
#pragma unroll
  for (int h = 0; h < NREP; ++h)
#pragma unroll
    for (int j = 0; j < C::EPC / 2; ++j)
      *reinterpret_cast<float2*>(red + (slot * C::NREP_P + h) * D + cp * C::EPC + 2 * j) = acc_o[h][j];
  __syncthreads();

  const size_t ws_row = size_t(b) * p.Hq + h0;  // first query head of this CTA
  for (int e = tid; e < nh * D; e += C::NTHR) {
    const int h = e / D, d = e % D;
    float sum = 0.f;
#pragma unroll
    for (int sl = 0; sl < C::SLOTS; ++sl) sum += red[(sl * C::NREP_P + h) * D + d];
    float lt = 0.f;
#pragma unroll
    for (int w = 0; w < C::NWARP; ++w) lt += wsum[w * 8 + h];
    if (n_used == 1) {
      store_f(out + (ws_row + h) * D + d, sum / lt);
    } else {
      p.part_o[((ws_row + h) * p.n_split + split) * D + d] = sum;
      if (d == 0) {
        p.ml[(ws_row + h) * p.n_split + split] = make_float2(wmax[h], lt);
      }
    }
  }
  if (n_used == 1) return;

  // ---- combine: a two-level tree over groups of GS splits ----
  // The last CTA of a group to arrive merges the group's partials (at most
  // GS of them); with one group that merge is final.  Otherwise it writes a
  // level-1 partial, and the last group to finish merges the level-1
  // partials.  Merges run in split order, so the result does not depend on
  // which CTA arrives last.  Counters are reset by the CTA that consumes them.
  constexpr int GS = 8;
  const int n_groups = (n_used + GS - 1) / GS;
  const int grp = split / GS;
  const int gsize = min(GS, n_used - grp * GS);
  int32_t* cnt = p.counters + ((size_t(b) * p.Hkv + g) * p.n_hc + hc) * (p.n_groups_max + 1);
  float* wts = reinterpret_cast<float*>(smem);  // [<=128 sources][8 heads] merge weights
  float* stat = wts + 128 * 8;                  // merged max [8], merged sum [8]

  // Merges sources [first, first+count) of the per-head lists (ml, o) whose
  // head stride is `hs` slots.  final: normalise and write O; otherwise write
  // the unnormalised level-1 partial into slot `grp`.
  auto merge = [&](const float2* mlb, const float* ob, int hs, int first, int count, bool final_) {
    for (int h = warp; h < nh; h += C::NWARP) {
      const float2* mlh = mlb + (ws_row + h) * hs + first;
      float M = -INFINITY;
      for (int sidx = lane; sidx < count; sidx += 32) M = fmaxf(M, __ldcg(&mlh[sidx]).x);
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
      float Ls = 0.f;
      for (int sidx = lane; sidx < count; sidx += 32) {
        const float2 x = __ldcg(&mlh[sidx]);
        const float w = fast_exp2(x.x - M);
        wts[sidx * 8 + h] = w;
        Ls += x.y * w;
      }
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, m);
      if (final_) {
        const float inv = 1.f / Ls;
        for (int sidx = lane; sidx < count; sidx += 32) wts[sidx * 8 + h] *= inv;
      } else if (lane == 0) {
        stat[h] = M;
        stat[8 + h] = Ls;
      }
    }
    __syncthreads();
    constexpr int D4 = D / 4;
    for (int pos = tid; pos < nh * D4; pos += C::NTHR) {
      const int h = pos / D4, c4 = pos % D4;
      const float4* src = reinterpret_cast<const float4*>(ob + ((ws_row + h) * hs + first) * D) + c4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
      for (int sidx = 0; sidx < count; ++sidx) {
        const float4 x = __ldcg(src + size_t(sidx) * D4);
        const float w = wts[sidx * 8 + h];
        acc.x += x.x * w;
        acc.y += x.y * w;
        acc.z += x.z * w;
        acc.w += x.w * w;
      }
      if (final_) {
        T* dst = out + (ws_row + h) * D + c4 * 4;
        store_f(dst + 0, acc.x);
        store_f(dst + 1, acc.y);
        store_f(dst + 2, acc.z);
        store_f(dst + 3, acc.w);
      } else {
        reinterpret_cast<float4*>(p.o1 + ((ws_row + h) * p.n_groups_max + grp) * D)[c4] = acc;
      }
    }
    if (!final_ && tid < nh)
      p.ml1[(ws_row + tid) * p.n_groups_max + grp] = make_float2(stat[tid], stat[8 + tid]);
  };

  __threadfence();
  __syncthreads();
  if (tid == 0) flag[1] = (atomicAdd(&cnt[grp], 1) == gsize - 1);
  __syncthreads();
  if (!flag[1]) return;
  __threadfence();
  if (tid == 0) cnt[grp] = 0;
  if (n_groups == 1) {
    merge(p.ml, p.part_o, p.n_split, 0, n_used, true);
    return;
  }
  merge(p.ml, p.part_o, p.n_split, grp * GS, gsize, false);
  __threadfence();
  __syncthreads();
  if (tid == 0) flag[1] = (atomicAdd(&cnt[p.n_groups_max], 1) == n_groups - 1);
  __syncthreads();
  if (!flag[1]) return;
  __threadfence();
  if (tid == 0) cnt[p.n_groups_max] = 0;
  merge(p.ml1, p.o1, p.n_groups_max, 0, n_groups, true);
}

template <typename T, int D, int NREP, int TILE, int NSTAGE>
cudaError_t launch_one(const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  using C = Cfg<T, D, NREP, TILE, NSTAGE>;
  auto kern = decode_split_kernel<T, D, NREP, TILE, NSTAGE>;
  static bool configured = false;  // per instantiation; attribute is per-function
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  kern<<<grid, C::NTHR, C::SMEM, stream>>>(p);
  return cudaGetLastError();
}

// Per (dtype, D): tile height and pipeline depth.  A stage (K + V tile) is
// 32 KiB for the 128-dim heads; three stages keep ~64 KiB in flight per CTA
// and two CTAs fit on an SM.
template <typename T, int D>
struct TileCfg;
template <> struct TileCfg<float, 128> { static constexpr int TILE = 32, NSTAGE = 3; };
template <> struct TileCfg<__nv_bfloat16, 128> { static constexpr int TILE = 64, NSTAGE = 3; };
template <> struct TileCfg<float, 64> { static constexpr int TILE = 64, NSTAGE = 3; };
template <> struct TileCfg<__nv_bfloat16, 64> { static constexpr int TILE = 64, NSTAGE = 4; };

template <typename T, int D>
cudaError_t dispatch_nrep(const DecodeParams& p, dim3 grid, cudaStream_t s) {
  constexpr int TL = TileCfg<T, D>::TILE, NS = TileCfg<T, D>::NSTAGE;
  switch (p.nrep_cta) {
    case 1: return launch_one<T, D, 1, TL, NS>(p, grid, s);
    case 2: return launch_one<T, D, 2, TL, NS>(p, grid, s);
    case 3:
    case 4: return launch_one<T, D, 4, TL, NS>(p, grid, s);
    case 5:
    case 6:
    case 7: return launch_one<T, D, 7, TL, NS>(p, grid, s);
    default: return launch_one<T, D, 8, TL, NS>(p, grid, s);
  }
}

}  // namespace

int decode_tile_rows(int dtype, int D) {
  if (dtype == GQA_F32) return D == 128 ? TileCfg<float, 128>::TILE : TileCfg<float, 64>::TILE;
  return D == 128 ? TileCfg<__nv_bfloat16, 128>::TILE : TileCfg<__nv_bfloat16, 64>::TILE;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  DecodeParams p;
  p.q = a.q;
  p.k = a.k;
  p.v = a.v;
  p.o = a.o;
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
  p.n_groups_max = w.n_groups_max;
  unsigned char* ws = static_cast<unsigned char*>(a.workspace);
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.counters = reinterpret_cast<int32_t*>(ws + w.off_counters);
  p.ml = reinterpret_cast<float2*>(ws + w.off_ml);
  p.part_o = reinterpret_cast<float*>(ws + w.off_o);
  p.ml1 = reinterpret_cast<float2*>(ws + w.off_ml1);
  p.o1 = reinterpret_cast<float*>(ws + w.off_o1);
  p.wait_limit_ns = kWaitLimitNs;
  const dim3 grid(a.plan.n_split, a.Hkv * a.plan.n_hc, a.B);
  if (a.dtype == GQA_F32)
    return a.D == 128 ? dispatch_nrep<float, 128>(p, grid, stream)
                      : dispatch_nrep<float, 64>(p, grid, stream);
  return a.D == 128 ? dispatch_nrep<__nv_bfloat16, 128>(p, grid, stream)
                    : dispatch_nrep<__nv_bfloat16, 64>(p, grid, stream);
}

}  // namespace gqa
