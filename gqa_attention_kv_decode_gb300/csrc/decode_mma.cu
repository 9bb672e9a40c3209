// decode_mma.cu -- single-token GQA decode over a bf16 KV cache with the
// score and P.V products on the tensor cores (mma.sync m16n8k16, bf16 in,
// fp32 accumulate) ("2x Faster Qwen2 Decode on Metal in Candle", "Why It
// Matters": one pass over the grouped KV heads, no repeat_kv copy, no score
// matrix in memory).
//
// With a bf16 cache every KV byte carries twice the multiply-adds of an fp32
// one, and on the CUDA cores the kernel runs out of issue slots before HBM
// runs out of bandwidth.  Here the query heads of one KV head are the M rows
// of an m16n8k16 product (up to 8 heads; the other rows are zero):
//   S = Q K^T   per warp: 16 keys x D dims, B fragments read with ldmatrix,
//   O += P V    P taken straight from the score accumulators (their layout
//               is the A-operand layout of the next product), V fragments
//               read with ldmatrix.trans.
// The CTA structure is the one of the CUDA-core kernel: 4 warps and tiles of
// 64 keys (or, for one long request, 8 warps and tiles of 128 keys), warp w
// taking keys 16w..16w+15 of every tile, tiles dealt round-robin to the
// splits, a per-warp online softmax in base 2, warps merged in shared
// memory, and split partials merged by the shared merge kernel.  K and V
// tiles arrive by tiled TMA with 128-byte swizzle (rows of 128 bytes, 16-byte
// chunks XOR-ed with the row index), so the 8 rows an ldmatrix reads sit in 8
// different bank groups.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cmath>
#include <mutex>

#include "gqa_attn.h"
#include "internal.h"
#include "merge.cuh"
#include "ptx.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace gqa {
namespace {

struct MmaParams {
  const __nv_bfloat16* q;
  __nv_bfloat16* o;
  const int32_t* kv_lens;
  const unsigned char* k;  // row-contiguous cache, for the L2 prefetch of the first tiles
  const unsigned char* v;
  int B, Hq, Hkv, n_rep, n_hc, nrep_cta, S_cap, max_kv_len, chunk, n_split;
  float qscale;  // scale * log2(e)
  uint32_t* status;
  float2* ml;
  float* part_o;
  uint64_t wait_limit_ns;
  uint64_t test_stall_ns;  // 0, or (tests) a wait that nothing ends, see the kernel
  // paged cache (PAGED kernels): the tensor maps span the pools
  // [num_blocks * Hkv][block_size][D]
  const int32_t* block_table;  // [B][max_blocks]
  int block_size, max_blocks, num_blocks;
  const __nv_bfloat16* k_new;  // [B][Hkv][D]: token appended at row kv_lens[b] - 1, or null
  const __nv_bfloat16* v_new;
  unsigned char* k_pool;       // pool bases, written by the append
  unsigned char* v_pool;
  // residual window after a 4-bit cache (len_sub != nullptr): the request
  // attends rows [0, kv_lens[b] - clamp(len_sub[b], 0, max_sub)) of this
  // cache, and its partial goes to slot min(n_slots - 1, ceil(that clamp /
  // slot_chunk)), the one after the 4-bit splits the request uses
  const int32_t* len_sub;
  int max_sub, slot_chunk;
  int n_slots;        // partial slots per (request, head) row
  int force_partial;  // write a partial even for a one-split request
  int kv_period;      // > 0: layers stacked along the batch axis share kv_lens[b % kv_period]
};

// Two shapes of the contiguous-cache kernel.  For long contexts with few
// (request, KV head) units -- a single long request -- 8 warps per CTA, one
// CTA per SM, tiles of 128 keys: half the split partials for the merge to
// read and twice the keys per split (7B geometry, 32K keys: 15.25 -> 14.7 us
// per call).  Otherwise two 4-warp CTAs per SM with tiles of 64 keys: more
// CTAs to spread a short context over (a single SM streams only about
// 40 GB/s, so short contexts need many SMs), and with many units, multi-wave
// grids whose two CTAs per SM overlap each other's ramps and tails (Qwen3-4B
// ragged B = 4..64: the 8-warp shape was 18-20 % slower; 7B geometry at 2K
// keys: 7.1 against 5.7 us per call).
constexpr int kWideUnits = 16;      // units up to which the 8-warp shape may be used
constexpr int kWideMinKeys = 8192;  // and keys from which it is used

template <int D, int NSTAGE, int NW_>
struct MmaCfg {
  static constexpr int NW = NW_;              // warps; warp w takes keys [16w, 16w + 16)
  static constexpr int TILE = 16 * NW;        // keys per tile
  static constexpr int NTHR = 32 * NW;
  static constexpr int HALVES = D / 64;       // 128-byte columns per key row
  static constexpr int BOX = TILE * 128;      // one column of the tile: TILE rows x 128 bytes
  static constexpr int SUB = TILE / 64;       // TMA boxes (64 rows x 128 bytes) per column
  static constexpr int TILEB = HALVES * BOX;  // K (or V) tile
  static constexpr int STAGEB = 2 * TILEB;    // K + V
  static constexpr int OFF_BAR = NSTAGE * STAGEB;
  static constexpr int OFF_REL = OFF_BAR + (NSTAGE + 1) * 8;  // after full[NSTAGE + 1]
  static constexpr int OFF_FLAG = OFF_REL + NSTAGE * 4;
  static constexpr int SMEM = OFF_FLAG + 16 + 1024;  // + slack for the 1024-byte alignment of the boxes
  static constexpr int KSTEPS = D / 16;       // k-steps of S = Q K^T
  static constexpr int NT_O = D / 8;          // n-tiles of O
  static constexpr int MERGE_FLOATS = NW * (8 * D + 16);  // per warp: O[8][D], m[8], l[8]
  static_assert(D == 64 || D == 128, "head dimension");
  static_assert(MERGE_FLOATS * 4 <= NSTAGE * STAGEB, "warp-merge scratch fits in the stages");
};

// Byte offset of 16-byte chunk `chunk` (0..7) of key row `row` inside a
// 128-byte-swizzled box: the chunk index is XOR-ed with the row index mod 8.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return uint32_t(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D (+)= A B with A rows 8..15 zero (only 8 query heads per CTA): the A
// registers a1, a3 of those rows are passed as zero.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// PAGED: K and V tiles come from block pools through the block table (a tile
// never crosses a block); with k_new the CTA that owns row kv_len - 1 writes
// the new token into its tile in shared memory and into the pool.
template <int D, int NSTAGE, int NW, bool PAGED>
__global__ void __launch_bounds__(MmaCfg<D, NSTAGE, NW>::NTHR, 8 / NW)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const MmaParams p) {
  using C = MmaCfg<D, NSTAGE, NW>;
  constexpr int TILE = C::TILE;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int split = blockIdx.x;
  const int g = blockIdx.y / p.n_hc;
  const int hc = blockIdx.y % p.n_hc;
  const int b = blockIdx.z;
  const int h0 = g * p.n_rep + hc * p.nrep_cta;
  const int nh = min(p.nrep_cta, p.n_rep - hc * p.nrep_cta);
  const int kv_head = b * p.Hkv + g;
  const size_t head_row0 = size_t(kv_head) * size_t(p.S_cap);

  // Launched early (programmatic dependent launch): until the wait returns,
  // only prefetch the first tiles of this split into L2 (as if kv_len were
  // max_kv_len) and the tensor maps.  Two tiles for the 8-warp shape (one
  // long request; 28-call sequences at 32,768 keys in a CUDA graph: 14.5 us
  // per call, 14.8 with all three stages, 15.3 with five tiles; plain
  // launches 14.8 with two or three, 15.4 with one), one for the 4-warp
  // shape, where more competes for HBM with the previous call's last CTAs
  // (Qwen3-4B ragged B = 64: 166.0 against 171.3 us per call).
  if (tid == 0 && hc == 0) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    constexpr int kPrefetchTiles = NW == 8 ? 2 : 1;
    for (int t = 0; t < (PAGED ? 0 : kPrefetchTiles); ++t) {  // (a paged cache's rows are known only after the wait)
      const int row0 = (split + t * p.n_split) * TILE;
      if (row0 >= p.max_kv_len) break;
      const uint32_t bytes = uint32_t(min(TILE, p.max_kv_len - row0)) * D * 2;
      prefetch_l2_bulk(p.k + (head_row0 + row0) * D * 2, bytes);
      prefetch_l2_bulk(p.v + (head_row0 + row0) * D * 2, bytes);
    }
  }
  if (tid == 32)  // and this CTA's query rows
    prefetch_l2_bulk(p.q + (size_t(b) * p.Hq + h0) * D, uint32_t(nh * D * 2));
  // The 8-warp shape (one long request) lets the merge kernel's CTAs be
  // scheduled at once; they wait for this grid anyway, and being resident
  // when it ends shortens the hand-off (32,768 keys in a CUDA graph: 14.30
  // against 14.52 us per call; the 4-warp shape, ragged batches, measured
  // slower that way and triggers near its end, below).
  if constexpr (NW == 8) grid_launch_dependents();
  grid_dependency_wait();

  int L = p.kv_lens ? p.kv_lens[p.kv_period > 0 ? b % p.kv_period : b] : p.max_kv_len;
  int slot0 = 0;
  if (p.len_sub != nullptr) {
    const int nq = p.len_sub[b];
    const int nqc = nq < 0 ? 0 : (nq > p.max_sub ? p.max_sub : nq);
    if ((nqc != nq || L < 0) && split == 0 && blockIdx.y == 0 && tid == 0)
      atomicOr(p.status, GQA_DEV_KVLEN_CLAMPED);
    slot0 = min(p.n_slots - 1, (nqc + p.slot_chunk - 1) / p.slot_chunk);  // the 4-bit splits used
    L = max(L, 0) - nqc;
    if (L < 0) L = 0;
  }
  if (L < 0 || L > p.max_kv_len) {
    if (split == 0 && blockIdx.y == 0 && tid == 0) atomicOr(p.status, GQA_DEV_KVLEN_CLAMPED);
    L = L < 0 ? 0 : p.max_kv_len;
  }
  if (L == 0) {  // no visible key: the output row is zeros
    if (p.force_partial) return;  // (the merge writes it)
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

  // k-th tile of this split into stage st: K then V, each HALVES boxes of
  // 64 keys x 64 dims.  Rows past S_cap arrive as zeros; rows in [L, S_cap)
  // arrive as whatever the cache holds there (masked below).
  // (row within the map, map head) of key row `row`.  For a paged cache the
  // block id comes from the table; an id outside the pool is reported and
  // replaced by block 0.
  auto map_coord = [&](int row, int& mrow, int& mhead) {
    if constexpr (PAGED) {
      int blk = p.block_table[size_t(b) * p.max_blocks + row / p.block_size];
      if (blk < 0 || blk >= p.num_blocks) {
        atomicOr(p.status, GQA_DEV_BAD_BLOCK);
        blk = 0;
      }
      mrow = row % p.block_size;
      mhead = blk * p.Hkv + g;
    } else {
      mrow = row;
      mhead = kv_head;
    }
  };
  auto issue = [&](int kt, int st) {
    const int row0 = (split + kt * n_used) * TILE;
    int mrow, mhead;
    map_coord(row0, mrow, mhead);
    unsigned char* dst = smem + st * C::STAGEB;
    mbar_arrive_expect_tx(&full[st], C::STAGEB);
#pragma unroll
    for (int hf = 0; hf < C::HALVES; ++hf)
#pragma unroll
      for (int sb = 0; sb < C::SUB; ++sb)
        tma_load_3d(dst + hf * C::BOX + sb * 8192, &tmK, hf * 64, mrow + sb * 64, mhead, &full[st]);
#pragma unroll
    for (int hf = 0; hf < C::HALVES; ++hf)
#pragma unroll
      for (int sb = 0; sb < C::SUB; ++sb)
        tma_load_3d(dst + C::TILEB + hf * C::BOX + sb * 8192, &tmV, hf * 64, mrow + sb * 64, mhead, &full[st]);
  };
  // The appended token (row L - 1) lies in tile (L - 1) / TILE, which is
  // tile t_new of split ((L - 1) / TILE) % n_used.
  int t_new = -1;
  if (PAGED && p.k_new != nullptr && ((L - 1) / TILE) % n_used == split) t_new = ((L - 1) / TILE) / n_used;
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      rel[s] = 0;
    }
    fence_barrier_init();
    flag[0] = 0;
    flag[1] = 0;
    for (int t = 0; t < NSTAGE && t < nt; ++t) issue(t, t);
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
  // Q as A fragments: row = query head lane/4 (zero past nh), k = dims.
  const int r = lane >> 2, c = lane & 3;
  uint32_t qa[C::KSTEPS][2];
  {
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + (size_t(b) * p.Hq + h0 + min(r, nh - 1)) * D);
#pragma unroll
    for (int ks = 0; ks < C::KSTEPS; ++ks) {
      qa[ks][0] = r < nh ? qrow[(16 * ks + 2 * c) / 2] : 0u;
      qa[ks][1] = r < nh ? qrow[(16 * ks + 8 + 2 * c) / 2] : 0u;
    }
  }
  __syncthreads();

  const uint32_t sbase = smem_u32(smem);
  const int kb = warp * 16;  // this warp's first key in every tile
  const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: matrix and row this lane addresses
  float m_ref = -INFINITY, lsum = 0.f;  // head r; m_ref is the same on the 4 lanes of the head
  float oacc[C::NT_O][4];
#pragma unroll
  for (int j = 0; j < C::NT_O; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;

  for (int t = 0; t < nt; ++t) {
    const int st = t % NSTAGE;
    const bool ok = wait_or_abort(&full[st], uint32_t(t / NSTAGE) & 1u, flag, p.wait_limit_ns);
    if (!__all_sync(0xffffffffu, ok)) break;
    const int row0 = (split + t * n_used) * TILE;
    const int wvalid = min(TILE, L - row0) - kb;  // valid keys among this warp's 16
    const uint32_t kaddr = sbase + st * C::STAGEB, vaddr = kaddr + C::TILEB;
    if (PAGED && t == t_new && warp == ((L - 1) % TILE) / 16) {
      // the warp that reads row L - 1 puts the new token there (over the
      // stale cache row just copied; 128-byte swizzled layout) and into the pool
      const int r = (L - 1) % TILE;
      if (lane < C::HALVES * 8) {
        const int hf = lane >> 3, ch = lane & 7;
        const size_t src = (size_t(b) * p.Hkv + g) * D + hf * 64 + ch * 8;
        const uint4 kx = *reinterpret_cast<const uint4*>(p.k_new + src);
        const uint4 vx = *reinterpret_cast<const uint4*>(p.v_new + src);
        unsigned char* kt = smem + st * C::STAGEB + hf * C::BOX + swz(r, ch);
        *reinterpret_cast<uint4*>(kt) = kx;
        *reinterpret_cast<uint4*>(kt + C::TILEB) = vx;
        int mrow, mhead;
        map_coord(L - 1, mrow, mhead);
        const size_t dst = ((size_t(mhead) * p.block_size + mrow) * D + hf * 64 + ch * 8) * 2;
        *reinterpret_cast<uint4*>(p.k_pool + dst) = kx;
        *reinterpret_cast<uint4*>(p.v_pool + dst) = vx;
      }
      fence_proxy_async_smem();  // before the stage can be refilled by TMA
      __syncwarp();
    }
    if (wvalid > 0) {
      if (wvalid < 16) {
        // V rows past kv_len may hold anything (NaN included): 0 x NaN would
        // reach O, so those rows are zeroed (their P is 0)
        unsigned char* vt = smem + st * C::STAGEB + C::TILEB;
        const int nchunk = (16 - wvalid) * C::HALVES * 8;
        for (int i = lane; i < nchunk; i += 32) {
          const int row = kb + wvalid + i / (C::HALVES * 8), rem = i % (C::HALVES * 8);
          *reinterpret_cast<uint4*>(vt + (rem / 8) * C::BOX + row * 128 + (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();  // before the stage can be refilled by TMA
        __syncwarp();
      }
      // ---- S = Q K^T over this warp's 16 keys (two n-tiles of 8) ----
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < C::KSTEPS; ++ks) {
        const int key = kb + 8 * (mi >> 1) + rr, d = 16 * ks + 8 * (mi & 1);
        uint32_t b00, b01, b10, b11;
        ldsm_x4(kaddr + (d / 64) * C::BOX + swz(key, (d % 64) / 8), b00, b01, b10, b11);
        mma_16816(sacc[0], qa[ks][0], qa[ks][1], b00, b01);
        mma_16816(sacc[1], qa[ks][0], qa[ks][1], b10, b11);
      }
      // scores of head r for keys kb + {2c, 2c+1, 8+2c, 9+2c}, base 2
      float sv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int kl = 8 * (i >> 1) + 2 * c + (i & 1);
        sv[i] = kl < wvalid ? sacc[i >> 1][i & 1] * p.qscale : -INFINITY;
      }
      float mx = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      // lazy reference: raised only when a tile's maximum exceeds it by 2^8
      const bool resc = mx > m_ref + 8.f;
      if (__any_sync(0xffffffffu, resc)) {
        const float alpha = resc ? fast_exp2(m_ref - mx) : 1.f;
        if (resc) m_ref = mx;
        lsum *= alpha;
#pragma unroll
        for (int j = 0; j < C::NT_O; ++j) {
          oacc[j][0] *= alpha;
          oacc[j][1] *= alpha;
        }
      }
      const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
      float pv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pv[i] = fast_exp2(sv[i] - m_use);
      lsum += (pv[0] + pv[1]) + (pv[2] + pv[3]);
      const uint32_t pa0 = pack_bf16(pv[0], pv[1]), pa2 = pack_bf16(pv[2], pv[3]);
      // ---- O += P V: pairs of 8-dim n-tiles ----
#pragma unroll
      for (int jj = 0; jj < C::NT_O / 2; ++jj) {
        const int key = kb + 8 * (mi & 1) + rr, d = 16 * jj + 8 * (mi >> 1);
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(vaddr + (d / 64) * C::BOX + swz(key, (d % 64) / 8), v0, v1, v2, v3);
        mma_16816(oacc[2 * jj], pa0, pa2, v0, v1);
        mma_16816(oacc[2 * jj + 1], pa0, pa2, v2, v3);
      }
    }
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&rel[st], 1) == C::NW - 1) {  // the last warp done with the stage refills it
        rel[st] = 0;
        if (t + NSTAGE < nt && !flag[0]) {
          issue(t + NSTAGE, st);
          atomicMax(const_cast<int*>(&flag[2]), t + NSTAGE + 1);
        }
      }
    }
  }
  lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
  lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
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
#pragma unroll
  for (int j = 0; j < C::NT_O; ++j)
    *reinterpret_cast<float2*>(merge_s + (warp * 8 + r) * D + 8 * j + 2 * c) = make_float2(oacc[j][0], oacc[j][1]);
  if (c == 0) {
    mw[warp * 8 + r] = m_ref;
    lw[warp * 8 + r] = lsum;
  }
  __syncthreads();
  // let the merge kernel's CTAs be scheduled while this grid drains
  if constexpr (NW != 8) grid_launch_dependents();

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
      p.part_o[((ws_row + h) * p.n_slots + slot0 + split) * D + d] = sum;
      if (d == 0) p.ml[(ws_row + h) * p.n_slots + slot0 + split] = make_float2(M, lt);
    }
  }
}

// Tensor maps of the K and V caches, [B*Hkv][S_cap][D] bf16 as a 3-D tensor
// with 64-row x 64-dim boxes and 128-byte swizzle.  Encoding one costs about
// a microsecond of host time, so the maps of recently used caches are kept
// (keyed by base address and shape; a map holds no data, only the layout).
struct MapEntry {
  const void* base;
  int D, S_cap, heads;
  CUtensorMap map;
};
constexpr int kMapCache = 128;

bool kv_map(CUtensorMap* out, const void* base, int D, int S_cap, int heads) {
  static std::mutex mu;
  static MapEntry cache[kMapCache];
  static int used = 0, next = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].base == base && cache[i].D == D && cache[i].S_cap == S_cap && cache[i].heads == heads) {
      *out = cache[i].map;
      return true;
    }
  CUtensorMap m;
  if (!encode_bf16_rows(&m, base, uint64_t(D), uint64_t(S_cap), uint64_t(S_cap), uint64_t(heads), 64, 64))
    return false;
  MapEntry& e = cache[next];
  e.base = base;
  e.D = D;
  e.S_cap = S_cap;
  e.heads = heads;
  e.map = m;
  next = (next + 1) % kMapCache;
  if (used < kMapCache) ++used;
  *out = m;
  return true;
}

template <int D, int NSTAGE, int NW, bool PAGED>
cudaError_t launch_mma(const CUtensorMap& tk, const CUtensorMap& tv, const MmaParams& p, dim3 grid,
                       cudaStream_t stream) {
  using C = MmaCfg<D, NSTAGE, NW>;
  auto kern = decode_mma_kernel<D, NSTAGE, NW, PAGED>;
  static std::once_flag once;
  static cudaError_t cfg_err = cudaSuccess;
  std::call_once(once, [&] {
    cfg_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (cfg_err == cudaSuccess)  // two CTAs per SM need the largest shared-memory carveout
      cfg_err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
  });
  if (cfg_err != cudaSuccess) return cfg_err;
  return launch_pdl(kern, grid, dim3(C::NTHR), C::SMEM, stream, tk, tv, p);
}

}  // namespace

// Tile height (16 keys per warp) and CTAs per SM of the kernel shape used for
// `units` (request, KV head chunk) pairs and `max_kv_len` keys; the paged
// kernel always has 4 warps, so that a 64-row block holds whole tiles.
static bool wide_shape(bool paged, long units, int max_kv_len) {
  return !paged && units <= kWideUnits && max_kv_len >= kWideMinKeys;
}
int decode_mma_tile_rows(bool paged, long units, int max_kv_len) {
  return wide_shape(paged, units, max_kv_len) ? 128 : 64;
}
int decode_mma_ctas_per_sm(bool paged, long units, int max_kv_len) {
  return wide_shape(paged, units, max_kv_len) ? 1 : 2;
}

cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t stream) {
  if (a.D != 64 && a.D != 128) return cudaErrorNotSupported;
  CUtensorMap tk, tv;
  const bool paged = a.block_table != nullptr;
  const int heads = paged ? a.num_blocks * a.Hkv : a.B * a.Hkv;
  const int rows = paged ? a.block_size : a.S_cap;
  if (!kv_map(&tk, a.k, a.D, rows, heads) || !kv_map(&tv, a.v, a.D, rows, heads)) return cudaErrorInvalidValue;
  MmaParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.kv_lens = a.kv_lens;
  p.k = static_cast<const unsigned char*>(a.k);
  p.v = static_cast<const unsigned char*>(a.v);
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
  const WorkspaceLayout w =
      workspace_layout(a.B, a.Hq, a.Hkv, a.plan.n_hc, a.n_slots > 0 ? a.n_slots : a.plan.n_split, a.D);
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
  p.k_new = static_cast<const __nv_bfloat16*>(a.k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(a.v_new);
  p.k_pool = static_cast<unsigned char*>(const_cast<void*>(a.k));
  p.v_pool = static_cast<unsigned char*>(const_cast<void*>(a.v));
  p.len_sub = a.len_sub;
  p.max_sub = a.max_sub;
  p.slot_chunk = a.slot_chunk > 0 ? a.slot_chunk : 1;
  p.n_slots = a.n_slots > 0 ? a.n_slots : a.plan.n_split;
  p.force_partial = a.force_partial;
  p.kv_period = a.kv_period;
  const dim3 grid(a.plan.n_split, a.Hkv * a.plan.n_hc, a.B);
  if (paged)
    return a.D == 128 ? launch_mma<128, 3, 4, true>(tk, tv, p, grid, stream)
                      : launch_mma<64, 6, 4, true>(tk, tv, p, grid, stream);
  // the shape follows the plan's tile height
  if (a.plan.tile == 128)
    return a.D == 128 ? launch_mma<128, 3, 8, false>(tk, tv, p, grid, stream)
                      : launch_mma<64, 6, 8, false>(tk, tv, p, grid, stream);
  if (a.plan.tile != 64) return cudaErrorInvalidValue;
  return a.D == 128 ? launch_mma<128, 3, 4, false>(tk, tv, p, grid, stream)
                    : launch_mma<64, 6, 4, false>(tk, tv, p, grid, stream);
}

}  // namespace gqa


namespace gqa {

cudaError_t launch_decode_mma_residual(const DecodeArgs& a, const int32_t* n_quant, int max_quant, int slot_chunk,
                                       int n_slots, cudaStream_t stream) {
  DecodeArgs r = a;
  r.len_sub = n_quant;
  r.max_sub = max_quant;
  r.slot_chunk = slot_chunk;
  r.n_slots = n_slots;
  r.force_partial = 1;
  return launch_decode_mma(r, stream);
}

}  // namespace gqa
