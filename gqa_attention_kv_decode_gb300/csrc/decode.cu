// decode.cu -- split-KV single-token GQA decode for sm_103a on the CUDA cores
// (fp32 KV caches; bf16 caches run on the tensor cores, decode_mma.cu).
//
// One CTA serves one (request b, KV head g, query-head chunk, key split).  All
// the query heads that share KV head g (n_rep = Hq / Hkv of them, up to 8 per
// CTA) are computed together, so every K and V byte is read from HBM once
// ("2x Faster Qwen2 Decode on Metal in Candle", "Why It Matters": the fused
// kernel indexes the unexpanded KV heads through the head ratio and never
// copies them).
//
// Data flow per CTA:
//   * the split's key rows are streamed in tiles of TILE rows, tiles dealt
//     round-robin to the splits; each
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
//   * a request that fits one split writes O directly; otherwise each split
//     writes (max, sum, unnormalised o) to the workspace and a second, small
//     kernel (one CTA per request and query head, launched with programmatic
//     dependent launch) merges them with the log-sum-exp rule, in split order.
#include <cuda_bf16.h>

#include <cmath>
#include <mutex>

#include "gqa_attn.h"
#include "internal.h"
#include "merge.cuh"
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
  float2* ml;     // [B][Hq][n_split] (max in log2 units, sum)
  float* part_o;  // [B][Hq][n_split][D] unnormalised partial outputs
  uint64_t wait_limit_ns;
  uint64_t test_stall_ns;  // 0, or (tests) a wait that nothing ends, see the kernel
  // paged cache (PAGED kernels): k and v are pools [num_blocks][Hkv][block_size][D]
  const int32_t* block_table;  // [B][max_blocks]
  int block_size, max_blocks, num_blocks;
  const void* k_new;  // [B][Hkv][D]: token appended at row kv_lens[b] - 1, or null
  const void* v_new;
  int kv_period;  // > 0: layers stacked along the batch axis share kv_lens[b % kv_period]
  // call boundary (see the kernel): 1 for a long context with few units --
  // trigger the merge's launch at the start and start two tiles towards L2
  int long_few;
};


template <typename T, int D, int NREP, int R_, int NSTAGE>
struct Cfg {
  static constexpr int E = sizeof(T);
  static constexpr int ROWB = D * E;     // bytes per key row
  static constexpr int NCH = ROWB / 16;  // 16-byte chunks per row
  static constexpr int EPC = 16 / E;     // elements per chunk
  static constexpr int NPART = EPC / 4;  // float4 pieces of q per chunk
  static constexpr int NCW = 8;          // warps; each owns an eighth of every tile's rows
  static constexpr int NWARP = NCW;
  static constexpr int NTHR = 32 * NWARP;
  static constexpr int DS = 8;           // lanes sharing a row in the score phase
  static constexpr int NIT = NCH / DS;
  static constexpr int R = R_;           // rows per lane in the score phase
  static constexpr int TW = 4 * R;       // rows per consumer warp per tile
  static constexpr int TILE = NCW * TW;
  static constexpr int NREP_P = NREP <= 1 ? 1 : NREP <= 2 ? 2 : NREP <= 4 ? 4 : 8;
  static constexpr int VP = (R * NREP_P > 8) ? R * NREP_P : 8;
  static constexpr int NV = VP / 8;      // complete scores per lane after the butterfly
  static constexpr int G = NREP_P / NV;  // distinct head sets among the 8 lanes of a row group
  static constexpr int LPR = NCH;        // lanes per row in the P.V phase
  static constexpr int RPW = 32 / LPR;   // rows a warp covers per P.V step
  static constexpr int TILEB = TILE * ROWB;
  static constexpr int STAGEB = 2 * TILEB;
  static constexpr int OFF_Q = NSTAGE * STAGEB;
  static constexpr int OFF_P = OFF_Q + NREP_P * D * 4;
  static constexpr int OFF_BAR = OFF_P + NCW * TW * NREP_P * 8;
  static constexpr int OFF_FLAG = OFF_BAR + (NSTAGE + 1) * 8 + NSTAGE * 4;  // full[NSTAGE + 1], rel[NSTAGE]
  static constexpr int SMEM = OFF_FLAG + 16;
  static constexpr int MERGE_FLOATS = NCW * (NREP_P * D + 2 * NREP_P);
  static_assert(NCH % DS == 0, "row must split into 8 lanes of 16-byte chunks");
  static_assert(LPR <= 32 && 32 % LPR == 0, "a warp covers whole rows in P.V");
  static_assert(TW % RPW == 0, "P.V steps tile the warp's rows");
  static_assert(NV <= NREP_P && R <= 8, "head layout");
  static_assert(MERGE_FLOATS * 4 <= NSTAGE * STAGEB, "warp-merge scratch must fit");
  static_assert((128 * 8 + 16) * 4 <= NSTAGE * STAGEB, "split-merge weights must fit");
  static_assert(NREP >= 1 && NREP <= 8, "at most 8 query heads per CTA");
};

// PAGED: K and V are block pools addressed through the block table; a tile
// (a multiple of which the block size is) never crosses a block.  With k_new
// the CTA that owns row kv_len - 1 writes the new token into its tile in
// shared memory and into the pool.
// A long context with few (request, KV head) units: the call-boundary
// settings of decode_split_kernel for it (see there).
constexpr int kLongFewUnits = 16, kLongFewKeys = 8192;

template <typename T, int D, int NREP, int R_, int NSTAGE, bool PAGED>
__global__ void __launch_bounds__(Cfg<T, D, NREP, R_, NSTAGE>::NTHR, 1)
    decode_split_kernel(const DecodeParams p) {
  using C = Cfg<T, D, NREP, R_, NSTAGE>;
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
  const size_t head_row0 = PAGED ? 0 : (size_t(b) * p.Hkv + g) * size_t(p.S_cap);
  const unsigned char* kbase = static_cast<const unsigned char*>(p.k) + head_row0 * C::ROWB;
  const unsigned char* vbase = static_cast<const unsigned char*>(p.v) + head_row0 * C::ROWB;

  // This grid may have been launched while the previous one in the stream
  // (usually the merge of the previous call) is still running.  Until
  // grid_dependency_wait() returns nothing may be read or written; the first
  // tile this split will copy (assuming kv_len = max_kv_len, which only the
  // ragged case can make wrong) is meanwhile prefetched into L2.  One tile,
  // not NSTAGE: more competes for HBM with the previous call's last CTAs,
  // which are on the critical path (28-call sequences at 32,768 keys: 26.4
  // against 26.5 us per call with plain launches, 25.9 against 27.7 in a
  // CUDA graph; no prefetch: 27.4 / 26.9).  A long context with few units
  // (p.long_few) prefetches two tiles and lets the merge kernel's CTAs be
  // scheduled at once, so that they are resident when this grid ends:
  // 32,768 keys 25.6 / 26.3 us (graph / plain launches), 8192 keys 11.3 /
  // 12.0 against 11.8 / 12.2; at 128 and 2048 keys that measured slower.
  if (p.long_few) grid_launch_dependents();
  if (!PAGED && tid == 0 && hc == 0) {  // (a paged cache's rows are known only after the wait)
    for (int t = 0; t < (p.long_few ? 2 : 1); ++t) {
      const int row0 = (split + t * p.n_split) * TILE;
      if (row0 >= p.max_kv_len) break;
      const uint32_t bytes = uint32_t(min(TILE, p.max_kv_len - row0)) * C::ROWB;
      prefetch_l2_bulk(kbase + size_t(row0) * C::ROWB, bytes);
      prefetch_l2_bulk(vbase + size_t(row0) * C::ROWB, bytes);
    }
  }
  if (tid == 32)  // and this CTA's query rows (a prefetch only warms L2; it reads nothing early)
    prefetch_l2_bulk(static_cast<const T*>(p.q) + (size_t(b) * p.Hq + h0) * D, uint32_t(nh * D * C::E));
  grid_dependency_wait();

  int L = p.kv_lens ? p.kv_lens[p.kv_period > 0 ? b % p.kv_period : b] : p.max_kv_len;
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
  // min(n_split, ceil(L / chunk))
  const int n_used = L > p.chunk * p.n_split ? p.n_split : (L + p.chunk - 1) / p.chunk;
  if (split >= n_used) return;
  // Tiles are dealt round-robin to the request's n_used splits: split s
  // takes tiles s, s + n_used, ...  At any moment the CTAs of one head then
  // stream one dense region of the cache instead of n_used far-apart ones.
  const int nt_all = (L + TILE - 1) / TILE;
  const int nt = (nt_all - split + n_used - 1) / n_used;

  float* q_s = reinterpret_cast<float*>(smem + C::OFF_Q);
  float2* p_s = reinterpret_cast<float2*>(smem + C::OFF_P);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);   // copy landed
  int* rel = reinterpret_cast<int*>(smem + C::OFF_BAR + (NSTAGE + 1) * 8);  // warps done with a stage
  volatile int* flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);  // [0] abort [2] issued

  // Byte offset of key row `row` of this (request, KV head) in K or V.  For a
  // paged cache the block id comes from the table; an id outside the pool is
  // reported and replaced by block 0, so no copy ever leaves the pool.
  auto row_offset = [&](int row) -> size_t {
    if constexpr (PAGED) {
      int blk = p.block_table[size_t(b) * p.max_blocks + row / p.block_size];
      if (blk < 0 || blk >= p.num_blocks) {
        atomicOr(p.status, GQA_DEV_BAD_BLOCK);
        blk = 0;
      }
      return ((size_t(blk) * p.Hkv + g) * p.block_size + row % p.block_size) * C::ROWB;
    } else {
      return size_t(row) * C::ROWB;
    }
  };
  // Copy k-th tile of this split into stage st (one elected thread).
  auto issue = [&](int kt, int st, uint64_t pol) {
    const int row0 = (split + kt * n_used) * TILE;
    const uint32_t bytes = uint32_t(min(TILE, L - row0)) * C::ROWB;
    unsigned char* dst = smem + st * C::STAGEB;
    const size_t off = row_offset(row0);
    mbar_arrive_expect_tx(&full[st], 2 * bytes);
    bulk_g2s(dst, kbase + off, bytes, &full[st], pol);
    bulk_g2s(dst + C::TILEB, vbase + off, bytes, &full[st], pol);
  };
  // The appended token (row L - 1) lies in tile (L - 1) / TILE, which is
  // tile t_new of split ((L - 1) / TILE) % n_used.
  int t_new = -1;
  if (PAGED && p.k_new != nullptr && ((L - 1) / TILE) % n_used == split) t_new = ((L - 1) / TILE) / n_used;
  if (tid == 0) {  // barriers, then the first NSTAGE copies before q is staged
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      rel[s] = 0;
    }
    fence_barrier_init();
    flag[0] = 0;
    flag[1] = 0;
    const uint64_t pol = l2_policy_evict_first();
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
  // q rows of this CTA's heads (contiguous in memory), pre-scaled, laid out so
  // that the 8 lanes of a row group read 8 consecutive 16-byte pieces:
  // [h][part][chunk][4].  Every thread issues its (at most two) 16-byte loads
  // before storing anything, so staging costs one memory round trip.
  {
    constexpr int NVEC_MAX = (C::NREP_P * D * C::E / 16 + C::NTHR - 1) / C::NTHR;
    const int nvec = nh * D * C::E / 16;
    const uint4* qg = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) +
                                                     (size_t(b) * p.Hq + h0) * D);
    uint4 raw[NVEC_MAX];
#pragma unroll
    for (int k = 0; k < NVEC_MAX; ++k) {
      const int vi = tid + k * C::NTHR;
      if (vi < nvec) raw[k] = qg[vi];
    }
#pragma unroll
    for (int k = 0; k < NVEC_MAX; ++k) {
      const int vi = tid + k * C::NTHR;
      if (vi < nvec) {
        const int h = vi / C::NCH, c = vi % C::NCH;  // one 16-byte vector = one chunk
        float* dst = q_s + (h * C::NPART * C::NCH + c) * 4;
        if constexpr (sizeof(T) == 4) {
          *reinterpret_cast<float4*>(dst) =
              make_float4(__uint_as_float(raw[k].x) * p.qscale, __uint_as_float(raw[k].y) * p.qscale,
                          __uint_as_float(raw[k].z) * p.qscale, __uint_as_float(raw[k].w) * p.qscale);
        } else {
          const float2 a0 = bf16x2_to_float2(raw[k].x), a1 = bf16x2_to_float2(raw[k].y);
          const float2 a2 = bf16x2_to_float2(raw[k].z), a3 = bf16x2_to_float2(raw[k].w);
          *reinterpret_cast<float4*>(dst) =
              make_float4(a0.x * p.qscale, a0.y * p.qscale, a1.x * p.qscale, a1.y * p.qscale);
          *reinterpret_cast<float4*>(dst + C::NCH * 4) =
              make_float4(a2.x * p.qscale, a2.y * p.qscale, a3.x * p.qscale, a3.y * p.qscale);
        }
      }
    }
    for (int e = nh * D + tid; e < C::NREP_P * D; e += C::NTHR) q_s[e] = 0.f;  // padded heads
  }
  __syncthreads();

  float* merge_s = reinterpret_cast<float*>(smem);  // aliases the stages after the loop
  // ---- every warp: rows [warp*TW, warp*TW + TW) of each tile.  The last
  // warp to finish with a stage refills it (no dedicated producer). ----
  const uint64_t pol = l2_policy_evict_first();
    const int ds = lane & 7;
    const int rg = lane >> 3;
    const int cp = lane % C::LPR;
    const int rsub = lane / C::LPR;
    float2* pw = p_s + warp * C::TW * C::NREP_P;
    float mref[C::NV], lsum[C::NV];
#pragma unroll
    for (int i = 0; i < C::NV; ++i) {
      mref[i] = -INFINITY;
      lsum[i] = 0.f;
    }
    float2 acc_o[NREP][C::EPC / 2];
#pragma unroll
    for (int h = 0; h < NREP; ++h)
#pragma unroll
      for (int j = 0; j < C::EPC / 2; ++j) acc_o[h][j] = make_float2(0.f, 0.f);

    for (int t = 0; t < nt; ++t) {
      const int st = t % NSTAGE;
      const bool ok = wait_or_abort(&full[st], uint32_t(t / NSTAGE) & 1u, flag, p.wait_limit_ns);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (PAGED && t == t_new && warp == ((L - 1) % TILE) / C::TW) {
        // the warp that reads row L - 1 puts the new token there (over the
        // stale cache row just copied) and into the pool
        const int r = (L - 1) % TILE;
        if (lane < C::NCH) {
          const size_t src = (size_t(b) * p.Hkv + g) * C::ROWB + lane * 16;
          const uint4 kx = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(p.k_new) + src);
          const uint4 vx = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(p.v_new) + src);
          *reinterpret_cast<uint4*>(smem + st * C::STAGEB + r * C::ROWB + lane * 16) = kx;
          *reinterpret_cast<uint4*>(smem + st * C::STAGEB + C::TILEB + r * C::ROWB + lane * 16) = vx;
          const size_t off = row_offset(L - 1) + lane * 16;
          *reinterpret_cast<uint4*>(const_cast<unsigned char*>(kbase) + off) = kx;
          *reinterpret_cast<uint4*>(const_cast<unsigned char*>(vbase) + off) = vx;
        }
        fence_proxy_async_smem();  // before the stage can be refilled by a copy
        __syncwarp();
      }
      const int nvalid = min(TILE, L - (split + t * n_used) * TILE);
      const int wrow0 = warp * C::TW;
      const int wvalid = min(C::TW, nvalid - wrow0);
      const unsigned char* Ks = smem + st * C::STAGEB + wrow0 * C::ROWB;
      const unsigned char* Vs = smem + st * C::STAGEB + C::TILEB + wrow0 * C::ROWB;
      if (wvalid > 0) {
        // ---- scores: R rows x NREP heads per lane, D split over 8 lanes ----
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
        // transposing butterfly over the 8 lanes of a row group: afterwards
        // lane ds holds the complete scores with flat index ds*NV + i, where
        // the flat index of (row r, head h) is r*NREP_P + h.
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
        // ---- online softmax over this warp's rows (base 2, lazy reference) ----
        float sc[C::NV], mx[C::NV], alpha[C::NV];
#pragma unroll
        for (int i = 0; i < C::NV; ++i) {
          const int idx = ds * C::NV + i;
          const int r = idx / C::NREP_P, h = idx % C::NREP_P;
          const bool valid = (idx < C::R * C::NREP_P) && (h < nh) && (rg * C::R + r < wvalid);
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
          if (idx < C::R * C::NREP_P)
            pw[(rg * C::R + idx / C::NREP_P) * C::NREP_P + idx % C::NREP_P] = make_float2(pv, pv);
        }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int h = 0; h < NREP; ++h) {
            const float a = __shfl_sync(0xffffffffu, alpha[h % C::NV], h / C::NV);
#pragma unroll
            for (int j = 0; j < C::EPC / 2; ++j) {
              acc_o[h][j].x *= a;
              acc_o[h][j].y *= a;
            }
          }
        }
        __syncwarp();
        // ---- P.V: lane owns one 16-byte column chunk for every head ----
        for (int j = rsub; j < wvalid; j += C::RPW) {
          const uint4 raw = *reinterpret_cast<const uint4*>(Vs + j * C::ROWB + cp * 16);
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
          const float2* prow = pw + j * C::NREP_P;
          if constexpr (C::NREP_P == 1) {
            const float2 pp = prow[0];
#pragma unroll
            for (int jj = 0; jj < C::EPC / 2; ++jj) acc_o[0][jj] = ffma2(vf[jj], pp, acc_o[0][jj]);
          } else {
#pragma unroll
            for (int h2 = 0; h2 < C::NREP_P / 2; ++h2) {
              if (2 * h2 >= NREP) break;
              const float4 pp = reinterpret_cast<const float4*>(prow)[h2];
#pragma unroll
              for (int jj = 0; jj < C::EPC / 2; ++jj) {
                acc_o[2 * h2][jj] = ffma2(vf[jj], make_float2(pp.x, pp.y), acc_o[2 * h2][jj]);
                if (2 * h2 + 1 < NREP)
                  acc_o[2 * h2 + 1][jj] = ffma2(vf[jj], make_float2(pp.z, pp.w), acc_o[2 * h2 + 1][jj]);
              }
            }
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

    // ---- this warp's (max, sum, o) into the merge scratch ----
#pragma unroll
    for (int m = C::G; m <= 16; m <<= 1)
#pragma unroll
      for (int i = 0; i < C::NV; ++i) lsum[i] += __shfl_xor_sync(0xffffffffu, lsum[i], m);
#pragma unroll
    for (int m = 16; m >= C::LPR; m >>= 1)
#pragma unroll
      for (int h = 0; h < NREP; ++h)
#pragma unroll
        for (int j = 0; j < C::EPC / 2; ++j) {
          acc_o[h][j].x += __shfl_xor_sync(0xffffffffu, acc_o[h][j].x, m);
          acc_o[h][j].y += __shfl_xor_sync(0xffffffffu, acc_o[h][j].y, m);
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
  // all issued copies have landed: the stages can hold the merge scratch
  {
    float* mw = merge_s + C::NCW * C::NREP_P * D;
    float* lw = mw + C::NCW * C::NREP_P;
    if (rsub == 0)
#pragma unroll
      for (int h = 0; h < NREP; ++h)
#pragma unroll
        for (int j = 0; j < C::EPC / 2; ++j)
          *reinterpret_cast<float2*>(merge_s + (warp * C::NREP_P + h) * D + (lane % C::LPR) * C::EPC +
                                     2 * j) = acc_o[h][j];
    if (lane < C::G)
#pragma unroll
      for (int i = 0; i < C::NV; ++i) {
        mw[warp * C::NREP_P + lane * C::NV + i] = mref[i];
        lw[warp * C::NREP_P + lane * C::NV + i] = lsum[i];
      }
  }
  __syncthreads();
  // let the merge kernel's CTAs be scheduled while this grid drains
  if (!p.long_few) grid_launch_dependents();

  // ---- merge the consumer warps, then write O or this split's partial ----
  const size_t ws_row = size_t(b) * p.Hq + h0;  // first query head of this CTA
  {
    const float* mw = merge_s + C::NCW * C::NREP_P * D;
    const float* lw = mw + C::NCW * C::NREP_P;
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
        store_f(out + (ws_row + h) * D + d, sum / lt);
      } else {
        p.part_o[((ws_row + h) * p.n_split + split) * D + d] = sum;
        if (d == 0) p.ml[(ws_row + h) * p.n_split + split] = make_float2(M, lt);
      }
    }
  }
}

template <typename T, int D, int NREP, int R, int NSTAGE, bool PAGED>
cudaError_t launch_one(const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  using C = Cfg<T, D, NREP, R, NSTAGE>;
  auto kern = decode_split_kernel<T, D, NREP, R, NSTAGE, PAGED>;
  static std::once_flag once;  // per instantiation; the attributes are per function
  static cudaError_t cfg_err = cudaSuccess;
  std::call_once(once, [&] {
    cfg_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (cfg_err == cudaSuccess)  // the largest shared-memory carveout
      cfg_err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
  });
  if (cfg_err != cudaSuccess) return cfg_err;
  return launch_pdl(kern, grid, dim3(C::NTHR), C::SMEM, stream, p);
}

// Per (dtype, D): tile height and pipeline depth.  A stage (K + V tile) is
// 64 KiB; three stages keep 192 KiB in flight, so one CTA of 8 warps fills
// an SM and the grid is one CTA per SM.  One large CTA per SM (rather than
// two of 4 warps) halves the split partials the merge reads and evens out the
// bandwidth each CTA gets, so the CTAs of a call finish closer together.
template <typename T, int D>
struct TileCfg;
template <> struct TileCfg<float, 128> { static constexpr int R = 2, NSTAGE = 3, TILE = 64; };
template <> struct TileCfg<float, 64> { static constexpr int R = 4, NSTAGE = 3, TILE = 128; };

template <typename T, int D, bool PAGED>
cudaError_t dispatch_nrep(const DecodeParams& p, dim3 grid, cudaStream_t s) {
  constexpr int TL = TileCfg<T, D>::R, NS = TileCfg<T, D>::NSTAGE;
  static_assert(Cfg<T, D, 8, TL, NS>::TILE == TileCfg<T, D>::TILE, "tile height");
  switch (p.nrep_cta) {
    case 1: return launch_one<T, D, 1, TL, NS, PAGED>(p, grid, s);
    case 2: return launch_one<T, D, 2, TL, NS, PAGED>(p, grid, s);
    case 3:
    case 4: return launch_one<T, D, 4, TL, NS, PAGED>(p, grid, s);
    case 5:
    case 6:
    case 7: return launch_one<T, D, 7, TL, NS, PAGED>(p, grid, s);
    default: return launch_one<T, D, 8, TL, NS, PAGED>(p, grid, s);
  }
}

}  // namespace

// bf16 caches run on the tensor cores (decode_mma.cu), whose kernel shape
// (tile height, CTAs per SM) depends on the problem.
int decode_ctas_per_sm(int dtype, bool paged, long units, int max_kv_len) {
  return dtype == GQA_F32 ? 1 : decode_mma_ctas_per_sm(paged, units, max_kv_len);
}

int decode_tile_rows(int dtype, int D, bool paged, long units, int max_kv_len) {
  if (dtype == GQA_F32) return D == 128 ? TileCfg<float, 128>::TILE : TileCfg<float, 64>::TILE;
  return decode_mma_tile_rows(paged, units, max_kv_len);
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
  unsigned char* ws = static_cast<unsigned char*>(a.workspace);
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.ml = reinterpret_cast<float2*>(ws + w.off_ml);
  p.part_o = reinterpret_cast<float*>(ws + w.off_o);
  p.wait_limit_ns = kWaitLimitNs;
  p.test_stall_ns = wait_test_ns();
  p.block_table = a.block_table;
  p.block_size = a.block_size;
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  p.k_new = a.k_new;
  p.v_new = a.v_new;
  p.kv_period = a.kv_period;
  p.long_few = (a.block_table == nullptr && long(a.B) * a.Hkv * a.plan.n_hc <= kLongFewUnits &&
                a.max_kv_len >= kLongFewKeys) ? 1 : 0;
  const dim3 grid(a.plan.n_split, a.Hkv * a.plan.n_hc, a.B);
  cudaError_t e;
  if (a.dtype != GQA_F32)
    e = launch_decode_mma(a, stream);
  else if (a.block_table != nullptr)
    e = a.D == 128 ? dispatch_nrep<float, 128, true>(p, grid, stream) : dispatch_nrep<float, 64, true>(p, grid, stream);
  else
    e = a.D == 128 ? dispatch_nrep<float, 128, false>(p, grid, stream) : dispatch_nrep<float, 64, false>(p, grid, stream);
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
  m.kv_period = a.kv_period;
  const int rows = a.B * a.Hq;
  if (a.dtype == GQA_F32)
    return a.D == 128 ? launch_merge<float, 128>(m, rows, stream) : launch_merge<float, 64>(m, rows, stream);
  return a.D == 128 ? launch_merge<__nv_bfloat16, 128>(m, rows, stream)
                    : launch_merge<__nv_bfloat16, 64>(m, rows, stream);
}

}  // namespace gqa
