// prefill.cu -- causal / chunked GQA prefill on the tcgen05 tensor cores of
// sm_103a ("Fused attention makes a 4,096-token Qwen2 prefill on Metal 4.5x
// faster", "Cause and workaround": one pass over the grouped KV heads, the
// causal mask applied inside the kernel with the queries aligned to the end
// of the keys, no score matrix in memory).  Head dimension 64 or 128.
//
// One CTA computes two consecutive 128-row query tiles (A and B) of one query
// head h and reads KV head g = h / n_rep directly (no repeat_kv).  Roles:
//   warpgroup 2, warp 8   TMA: Q_A, Q_B once, then K and V tiles of 128 keys
//                         through 4 shared-memory stages (2 at D = 128);
//   warpgroup 2, warp 9   MMA issue of S_t = Q_t K^T (M=128, N=128, K=D);
//   warps 10, 11          MMA issue of O_t += P_t V (M=128, N=64 per
//                         64-column half of O, K=128) for t = A, B; S, P and
//                         O live in tensor memory, V is read MN-major from its
//                         TMA tile;
//   warpgroup 0 / 1       softmax of tile A / B: a thread owns one query row
//                         (one TMEM lane).  It loads the row's 128 scores into
//                         registers and at once hands the S columns back, so
//                         the tensor core computes the next S while the
//                         exponentials of this one run (at D = 128, where P
//                         takes over the S columns, once P.V has read P).
//                         P (bf16) goes back to tensor memory in two halves
//                         of 64 keys, each of which releases its half of the
//                         P.V product.
// The running maximum is raised lazily: only when a tile's maximum exceeds it
// by more than 2^8 is O rescaled (in TMEM).  KV tiles entirely above the
// diagonal are never loaded; only tiles that cross it are masked.  Warpgroup
// 2 gives registers to the softmax warpgroups (setmaxnreg), which hold a
// whole score row.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <cstdlib>
#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <vector>

#include "gqa_attn.h"
#include "internal.h"
#include "tc.cuh"
#include "tmap.cuh"

namespace gqa {
namespace {

constexpr int BM = 128;                    // query rows per tile (TMEM lanes)
constexpr int BN = 128;                    // keys per KV tile
constexpr int NTHR = 384;                  // three warpgroups
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC_S = idesc_bf16(BM, BN, false, false);
constexpr uint32_t IDESC_O = idesc_bf16(BM, 64, false, true);  // one 64-column half of O per instruction
constexpr int kMinShareTiles = 6;          // KV tiles per cluster share, at least
constexpr int BOX_BYTES = 128 * 128;       // one TMA box: 128 rows x 64 bf16 columns (128 bytes), 16 KiB

// Layout for head dimension HD (64 or 128).  A Q, K or V tile is HD/64 boxes
// of 64 columns side by side in shared memory.
//   tensor memory, HD = 64:  S_A [0,128) S_B [128,256) O_A [256,320) O_B [320,384)
//                            P_A [384,448) P_B [448,512)
//   tensor memory, HD = 128: S_A [0,128) S_B [128,256) O_A [256,384) O_B [384,512);
//                            P_t overwrites the first 64 columns of S_t (the
//                            row's scores are in registers by then), so the
//                            next S_t waits until P_t V has been computed
//   shared memory: Q_A, Q_B, then NST stages of K and NST of V (4 stages at
//                  HD = 64, 161 KB; 2 at HD = 128, 193 KB)
template <int HD_>
struct PfCfg {
  static constexpr int HD = HD_;
  static constexpr int NBOX = HD / 64;
  static constexpr int TILE_BYTES = NBOX * BOX_BYTES;
  static constexpr int NST = HD == 64 ? 4 : 2;
  static constexpr bool P_ALIAS = HD == 128;
  static constexpr uint32_t TM_S = 0, TM_O = 256, TM_P = P_ALIAS ? 0u : 384u;
  static constexpr uint32_t P_STRIDE = P_ALIAS ? 128u : 64u;  // columns from P_A to P_B
  // Register split.  The kernel is compiled for 384 threads x 168 registers
  // (65,536 / 384, rounded down to a multiple of 8); the shares must not add
  // up to more: 128 x 56 + 256 x 224 = 64,512.  A softmax thread holds a
  // 128-score row (at HD = 128 it also walks a 128-column O row, 32 columns
  // at a time, and spilled with 208); the MMA-issue code fits in 56.  At
  // HD = 64, 56 / 224 measured 0.4% faster than 72 / 208.
  static constexpr int REG_CTRL = 56, REG_SOFTMAX = 224;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NST * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + NST * TILE_BYTES;
  static constexpr int OFF_ILV = OFF_BAR + 256;              // (m, l) of 128 rows, single-tile units
  static constexpr int OFF_LIM = OFF_ILV + 1024;             // per softmax thread: last key - first key
  static constexpr int SMEM_BYTES = OFF_LIM + 1024 + 1024;   // + alignment slack
  // mbarrier slots ([t] = per query tile)
  //   B_S[t]   S_t ready (MMA commit)           B_SC[t]  S_t read by all 4 warps
  //   B_P0[t]  P_t keys 0..63 stored            B_P1[t]  P_t keys 64..127 stored
  //   B_O0[t]  P.V over keys 0..63 done         B_O1[t]  P.V over all keys done
  //   B_DRAIN  after a timed-out wait: the MMA-issuing warps' work is done
  //   B_STALL  nothing arrives on it (the failure-path test waits on it)
  static constexpr int B_Q = 0, B_KF = 1, B_VF = B_KF + NST, B_KE = B_VF + NST, B_S = B_KE + NST,
                       B_SC = B_S + 2, B_P0 = B_SC + 2, B_P1 = B_P0 + 2, B_O0 = B_P1 + 2, B_O1 = B_O0 + 2,
                       B_DRAIN = B_O1 + 2, B_STALL = B_DRAIN + 1, N_BARS = B_STALL + 1;
  static constexpr int OFF_TSLOT = 8 * N_BARS, OFF_ABORT = OFF_TSLOT + 8, OFF_UNIT = OFF_ABORT + 4,
                       OFF_ISSUED = OFF_UNIT + 8;
  // Split-KV exchange (after the main loop, over Q and the K/V stages): a
  // partial row is (O[HD], m, l) padded to HD/4 + 1 float4 chunks; a unit is
  // 32 rows of one tile, stored chunk-major ([chunk][row][4]) so that the 32
  // lanes of a warp write one 512-byte run per remote store; the 8 units of a
  // CTA are spread over the cluster.  With ks CTAs in a cluster a rank
  // finishes ceil(8/ks) units and holds ks of those per rank.
  static constexpr int XCHUNKS = HD / 4 + 1, XUNIT = XCHUNKS * 32 * 4;  // floats per unit
  static constexpr int X_MAX_UNITS = OFF_BAR / (XUNIT * 4);
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
  static_assert(OFF_ISSUED + 4 <= 256, "barrier area");
  static_assert(HD == 64 || HD == 128, "head dimension");
  static_assert(128 * REG_CTRL + 256 * REG_SOFTMAX <= NTHR * 168, "register split exceeds the launch allocation");
};
// Cluster sizes whose exchange fits: every size up to 8 at HD = 64 (at most
// 14 units), 1-5 and 8 at HD = 128 (10 units for 5, 12 and 14 for 6 and 7).
__host__ __device__ constexpr bool kv_split_fits(int units_max, int ks) {
  return ks * ((8 + ks - 1) / ks) <= units_max;
}
static_assert(kv_split_fits(PfCfg<64>::X_MAX_UNITS, 7), "every cluster size fits at HD = 64");
static_assert(kv_split_fits(PfCfg<128>::X_MAX_UNITS, 5) && kv_split_fits(PfCfg<128>::X_MAX_UNITS, 8),
              "cluster sizes 5 and 8 fit at HD = 128");
// float offset of chunk c of row `lane` in unit (src, slot) of the exchange
template <int HD>
__device__ __forceinline__ int xidx(int src, int slot, int units_per_rank, int c, int lane) {
  return (((src * units_per_rank + slot) * PfCfg<HD>::XCHUNKS + c) * 32 + lane) * 4;
}

// Status of the prefill calls on this device (GQA_DEV_* bits), OR-accumulated
// by every prefill kernel until gqa_attn_clear_prefill_status.
__device__ uint32_t g_prefill_status = 0;

struct PrefillParams {
  __nv_bfloat16* o;
  int Hq, Hkv, n_rep, q_len, kv_len, n_pairs, causal;
  // Work units on grid y (see prefill_kernel): pairs of query tiles below
  // ilv_from, and single query tiles of the pairs from ilv_from on, whose KV
  // tiles the two softmax warpgroups share out (even / odd); n_first pairs
  // are scheduled before those single tiles.
  int n_tiles, ilv_from, n_first;
  int kv_splits;        // CTAs of a cluster sharing one pair's KV tiles (1 to 8)
  float qk_scale_log2;  // scale * log2(e)
  uint64_t wait_limit_ns;
  uint64_t test_stall_ns;  // 0, or (tests) a wait that nothing ends, see the TMA role
  int q_pitch;          // rows per head of Q and O
  // per-request lengths (varlen; null: q_len, kv_len for every request):
  // request b has clamp(kv_lens[b], 0, kv_len) keys and clamp(q_lens[b], 0,
  // min(q_len, its keys)) queries, aligned to the end of its keys
  const int32_t* q_lens;
  const int32_t* kv_lens;
};

// Bounded wait shared by the whole CTA: once one thread gives up, the
// others stop waiting too and the outputs are poisoned with NaN.  A phase
// that has already completed costs one probe.
__device__ __forceinline__ void cta_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return;
  if (*abort_flag) return;
  if (!mbar_wait_bounded(bar, parity, limit_ns)) *abort_flag = 1;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster executes each of these exactly
// once per exchange (no thread skips one), so the barrier always completes.
__device__ __forceinline__ void cluster_sync_all() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// Address of this CTA's shared-memory location `p` in the CTA of `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}
__device__ __forceinline__ void dsmem_st4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

template <int N>
__device__ __forceinline__ void set_max_regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void set_max_regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Named barriers 2 and 3 alternate the exponentials of the two softmax
// warpgroups (256 threads each: 128 wait, the other 128 arrive).
constexpr int BAR_TURN_A = 2, BAR_TURN_B = 3;
// Named barrier 4: slot 1 of a single-tile unit has left its (m, l) for slot 0.
constexpr int BAR_ILV = 4;
__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Exponentials of 64 scores s[0..63] of one row against the reference m
// (P = 2^(s*c - m)), packed as 32 bf16 pairs; their sum is added to acc.
__device__ __forceinline__ void exp_half(const uint32_t* s, float2 c, float2 mm, uint32_t (&pw)[32],
                                         float2 (&acc)[4]) {
#pragma unroll
  for (int u = 0; u < 32; ++u) {
    const float2 x = ffma2(make_float2(__uint_as_float(s[2 * u]), __uint_as_float(s[2 * u + 1])), c, mm);
    const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
    acc[u & 3] = __fadd2_rn(acc[u & 3], make_float2(p0, p1));
    const __nv_bfloat162 pk = __floats2bfloat162_rn(p0, p1);
    pw[u] = *reinterpret_cast<const uint32_t*>(&pk);
  }
}

// After a timed-out wait: lets the copies still in flight land before the
// shared memory is released -- Q, and the last of the n_issued K/V tiles in
// each of the NST stages.  Out of line: it runs only on that path, and
// inlined it cost the D = 128 kernel 2% in the hot loop.
template <int NST>
__device__ __noinline__ void drain_copies(uint64_t* bars, int b_q, int b_kf, int b_vf, int n_issued,
                                          uint64_t limit_ns) {
  mbar_wait_bounded(&bars[b_q], 0u, limit_ns);
  for (int s = 0; s < NST && s < n_issued; ++s) {
    const int u = s + ((n_issued - 1 - s) / NST) * NST;
    mbar_wait_bounded(&bars[b_kf + s], uint32_t(u / NST) & 1u, limit_ns);
    mbar_wait_bounded(&bars[b_vf + s], uint32_t(u / NST) & 1u, limit_ns);
  }
}

// Test only (gqa_attn_set_wait_test): waits, with the test's limit, on a
// barrier that nothing arrives on, as on a copy that never lands, and gives
// up as such a wait does.  Out of line, like the drain.
__device__ __noinline__ void stall_test(uint64_t* bar, uint64_t stall_ns, volatile int* abort_flag) {
  if (!mbar_wait_bounded(bar, 0u, stall_ns)) *abort_flag = 1;
}

// HD: head dimension (64 or 128).  SPLIT: the pair's KV range is shared by a
// cluster of p.kv_splits CTAs whose partial rows are merged through
// distributed shared memory.  ILV: the grid also holds single-tile units (see
// below); a launch without them uses the ILV = false kernel, whose code is
// that of pairs alone (the unit bookkeeping costs the pair loop registers).
template <int HD, bool SPLIT, bool ILV>
__global__ void __launch_bounds__(NTHR, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using C = PfCfg<HD>;
  constexpr int NBOX = C::NBOX, TILE_BYTES = C::TILE_BYTES, NST = C::NST;
  constexpr int OFF_Q = C::OFF_Q, OFF_K = C::OFF_K, OFF_V = C::OFF_V, OFF_BAR = C::OFF_BAR;
  constexpr int B_Q = C::B_Q, B_KF = C::B_KF, B_VF = C::B_VF, B_KE = C::B_KE, B_S = C::B_S, B_SC = C::B_SC,
                B_P0 = C::B_P0, B_P1 = C::B_P1, B_O0 = C::B_O0, B_O1 = C::B_O1, B_DRAIN = C::B_DRAIN;
  constexpr uint32_t TM_S = C::TM_S, TM_O = C::TM_O, TM_P = C::TM_P;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // Blocks start in the order of their linear index (x fastest), and the
  // units on y are ordered longest first for a causal mask, so the short
  // ones fill in behind the long ones.  A unit is either a pair of query
  // tiles (A, B) over the same KV tiles, or a single query tile ("ilv")
  // whose KV tiles are dealt to the two softmax warpgroups in turn (slot 0
  // the even ones, slot 1 the odd ones), which halves the iterations of the
  // longest causal tiles; the two slots' partial rows are combined at the
  // end.  Order on y: n_first pairs (ilv_from - 1 downwards), the single
  // tiles (the last tile downwards), then the remaining pairs.
  const int ks = SPLIT ? p.kv_splits : 1;
  const int upr = (8 + ks - 1) / ks;  // exchange units a rank finishes
  const int rank = SPLIT ? int(cluster_rank()) : 0;
  static_assert(!(SPLIT && ILV), "a cluster split runs pairs only");
  bool ilv = false;
  int m0;
  if constexpr (ILV) {
    const int n_ilv = max(0, p.n_tiles - 2 * p.ilv_from);
    const int y = int(blockIdx.y);
    ilv = y >= p.n_first && y < p.n_first + n_ilv;
    m0 = ilv ? (p.n_tiles - 1 - (y - p.n_first)) * BM : (p.ilv_from - 1 - (y < p.n_first ? y : y - n_ilv)) * 2 * BM;
  } else {
    m0 = (p.n_pairs - 1 - int(blockIdx.y)) * 2 * BM;
  }
  const int bh = int(blockIdx.x) / ks;  // a cluster = ks consecutive x
  const int h = bh % p.Hq;
  const int b = bh / p.Hq;
  const int g = h / p.n_rep;
  // Launched with programmatic stream serialisation: the next grid in the
  // stream may start launching at once (its CTAs wait in the same way), and
  // nothing the previous grid writes is read or written before it is done.
  // With uniform lengths the wait comes after the tensor-memory allocation
  // and barrier set-up below, which overlap the previous grid's tail; the
  // per-request lengths are global data, so that case waits here.
  grid_launch_dependents();
  if (p.q_lens != nullptr) grid_dependency_wait();
  int q_len = p.q_len, kv_len = p.kv_len;
  if (p.q_lens != nullptr) {
    const int kv_raw = p.kv_lens[b], q_raw = p.q_lens[b];
    kv_len = min(max(kv_raw, 0), p.kv_len);
    q_len = min(max(q_raw, 0), min(p.q_len, kv_len));
    if (threadIdx.x == 0 && blockIdx.y == 0 && (kv_raw != kv_len || q_raw != q_len))
      atomicOr(&g_prefill_status, GQA_DEV_KVLEN_CLAMPED);
    // a pair past this request's queries has nothing to do (the CTAs of a
    // cluster share the pair, so they leave together)
    if (m0 >= q_len) return;
  }
  const int off = kv_len - q_len;  // query row i sits at key position off + i

  auto nkv_for = [&](int mstart) -> int {
    if (mstart >= q_len) return 0;
    int n = (kv_len + BN - 1) / BN;
    if (p.causal) n = min(n, (off + min(mstart + BM - 1, q_len - 1)) / BN + 1);
    return n;
  };
  // The pair's KV tiles [0, nkv_all) are cut into ks contiguous shares; this
  // CTA takes share `rank`, [j_lo, j_hi).  Below, j counts tiles of the share
  // (barrier phases, stages) and j_lo + j is the tile's position in the keys.
  // nkv0, nkv1: the KV tiles of slot 0 and slot 1 (tiles A and B of a pair;
  // the even and odd tiles of a single-tile unit).
  const int nkv_a = nkv_for(m0), nkv_b = ilv ? 0 : nkv_for(m0 + BM);
  const int nkv_all = max(nkv_a, nkv_b);
  const int j_lo = SPLIT ? nkv_all * rank / ks : 0;
  const int j_hi = SPLIT ? nkv_all * (rank + 1) / ks : nkv_all;
  const int nkv0 = SPLIT ? max(0, min(nkv_a, j_hi) - j_lo) : ilv ? (nkv_all + 1) / 2 : nkv_a;
  const int nkv1 = SPLIT ? max(0, min(nkv_b, j_hi) - j_lo) : ilv ? nkv_all / 2 : nkv_b;
  const int nkv_max = j_hi - j_lo;
  // KV tile j of the unit belongs to slot t as the slot's iteration li
  auto active = [&](int j, int t) -> bool { return ilv ? (j & 1) == t : j < (t == 0 ? nkv0 : nkv1); };
  auto local_it = [&](int j) -> int { return ilv ? j >> 1 : j; };

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + C::OFF_TSLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + C::OFF_ABORT);
  volatile int* unit_info = reinterpret_cast<volatile int*>(smem + OFF_BAR + C::OFF_UNIT);

  if (warp == 9) {
    tmem_alloc(tslot, TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 256) {
    for (int i = 0; i < C::N_BARS; ++i) {
      const bool per_warp = (i >= B_SC && i < B_O0);  // arrivals of the 4 softmax warps of a tile
      const bool three = (i >= B_KE && i < B_KE + NST) || i == B_DRAIN;  // the three MMA-issuing warps
      mbar_init(&bars[i], per_warp ? 4 : three ? 3 : 1);
    }
    *abort_flag = 0;
    if (ILV) {
      unit_info[0] = m0;  // read back by the softmax epilogue (see there)
      unit_info[1] = int(ilv);
    }
    fence_barrier_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (p.q_lens == nullptr) grid_dependency_wait();

  if (warp >= 8) {
    set_max_regs_dec<C::REG_CTRL>();
    if (warp == 8 && lane == 0) {
      // ---------------- TMA ----------------
      const int kv_head = b * p.Hkv + g;
      const int n_q = ilv ? 1 : 2;  // a single-tile unit reads Q_A only
      int n_issued = 0;
      // (test only: Q is in flight, no K/V tile yet)
      if (p.test_stall_ns != 0) stall_test(&bars[C::B_STALL], p.test_stall_ns, abort_flag);
      mbar_arrive_expect_tx(&bars[B_Q], n_q * TILE_BYTES);
      for (int t = 0; t < n_q; ++t)
#pragma unroll
        for (int bx = 0; bx < NBOX; ++bx)
          tma_load_3d(smem + OFF_Q + t * TILE_BYTES + bx * BOX_BYTES, &tmQ, bx * 64, m0 + t * BM, b * p.Hq + h,
                      &bars[B_Q]);
      for (int j = 0; j < nkv_max; ++j) {
        const int st = j % NST;
        if (j >= NST) cta_wait(&bars[B_KE + st], uint32_t(j / NST - 1) & 1u, abort_flag, p.wait_limit_ns);
        if (*abort_flag) break;
        mbar_arrive_expect_tx(&bars[B_KF + st], TILE_BYTES);
#pragma unroll
        for (int bx = 0; bx < NBOX; ++bx)
          tma_load_3d(smem + OFF_K + st * TILE_BYTES + bx * BOX_BYTES, &tmK, bx * 64, (j_lo + j) * BN, kv_head,
                      &bars[B_KF + st]);
        mbar_arrive_expect_tx(&bars[B_VF + st], TILE_BYTES);
#pragma unroll
        for (int bx = 0; bx < NBOX; ++bx)
          tma_load_3d(smem + OFF_V + st * TILE_BYTES + bx * BOX_BYTES, &tmV, bx * 64, (j_lo + j) * BN, kv_head,
                      &bars[B_VF + st]);
        n_issued = j + 1;
      }
      // the K/V tiles copied, for the drain after a timed-out wait
      *reinterpret_cast<volatile int*>(smem + OFF_BAR + C::OFF_ISSUED) = n_issued;
    } else if (warp == 9) {
      // ---------------- MMA issue: S_t = Q_t K^T ----------------
      // Three warps issue tcgen05.mma (this one the scores, warps 10 and 11
      // the P.V products of tiles A and B), so that no single instruction
      // stream has to wait for all six hand-offs of an iteration.  Each runs
      // its loop warp-wide (waits, descriptors, loop control in step) and one
      // elected lane issues each tcgen05 instruction.
      const uint64_t qdesc = sdesc_sw128(smem_u32(smem + OFF_Q));
      const uint64_t kdesc = sdesc_sw128(smem_u32(smem + OFF_K));
      constexpr uint64_t TILE_STEP = TILE_BYTES >> 4;  // descriptor units (16 B) per tile / stage
      constexpr uint64_t K_KSTEP = 32 >> 4;             // per 16-deep slice of the head dimension
      constexpr uint64_t BOX_STEP = BOX_BYTES >> 4;     // per 64 dims (the next box)
      cta_wait(&bars[B_Q], 0, abort_flag, p.wait_limit_ns);
      for (int j = 0; j < nkv_max; ++j) {
        const int st = j % NST;
        cta_wait(&bars[B_KF + st], uint32_t(j / NST) & 1u, abort_flag, p.wait_limit_ns);
        const uint64_t kd = kdesc + st * TILE_STEP;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!active(j, t)) continue;
          const int li = local_it(j);
          // S_t(li) overwrites S_t(li-1), which its softmax must have read,
          // and, where P_t lives in the S_t columns, P_t(li-1), which the
          // P.V product of iteration li-1 must have read
          if (li > 0) {
            cta_wait(&bars[B_SC + t], uint32_t(li - 1) & 1u, abort_flag, p.wait_limit_ns);
            if (C::P_ALIAS) cta_wait(&bars[B_O1 + t], uint32_t(li - 1) & 1u, abort_flag, p.wait_limit_ns);
          }
          tc_fence_after();
          const uint64_t qd = qdesc + (ilv ? 0 : t) * TILE_STEP;
          const uint32_t d = tmem + TM_S + t * 128;
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint64_t koff = (kk / 4) * BOX_STEP + (kk % 4) * K_KSTEP;
            mma_bf16_warp(d, qd + koff, kd + koff, IDESC_S, kk > 0 ? 1u : 0u);
          }
          mma_commit_warp(&bars[B_S + t]);
        }
        mma_commit_warp(&bars[B_KE + st]);  // K of stage st is no longer needed once these are done
      }
    } else if (warp >= 10) {
      // ---------------- MMA issue: O_t += P_t V, t = warp - 10 ----------------
      const int t = warp - 10;
      const uint64_t vdesc = sdesc_sw128(smem_u32(smem + OFF_V));
      constexpr uint64_t TILE_STEP = TILE_BYTES >> 4;
      constexpr uint64_t V_KSTEP = 2048 >> 4;  // 16 keys of the MN-major V tile
      constexpr uint64_t BOX_STEP = BOX_BYTES >> 4;  // the next 64 dims of V
      const uint32_t d = tmem + TM_O + t * HD, a = tmem + TM_P + t * C::P_STRIDE;
      // Per-request lengths: the V map spans the whole cache, so the last KV
      // tile may hold rows past kv_len (anything, NaN included; their P is 0
      // but 0 * NaN is NaN).  Both P.V warps zero those rows first.
      const int j_zero = (p.q_lens != nullptr && kv_len % BN != 0) ? (kv_len - 1) / BN - j_lo : -1;
      for (int j = 0; j < nkv_max; ++j) {
        const int st = j % NST;
        // Waited for even past this tile's last KV tile: the load of tile j
        // orders this warp's arrival on B_KE[st] after the previous phase,
        // so one warp can never arrive twice within a phase.
        cta_wait(&bars[B_VF + st], uint32_t(j / NST) & 1u, abort_flag, p.wait_limit_ns);
        if (j == j_zero) {
          unsigned char* vt = smem + OFF_V + st * TILE_BYTES;
          const int r0 = kv_len % BN;  // first row to clear (rows are 128 bytes; swizzle stays inside a row)
          const int per_box = (BN - r0) * 8;  // 16-byte chunks to clear in each box
          for (int i = (warp - 10) * 32 + lane; i < per_box * NBOX; i += 64) {
            const int bx = i / per_box, k = i % per_box;
            *reinterpret_cast<uint4*>(vt + bx * BOX_BYTES + (r0 + k / 8) * 128 + (k % 8) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          asm volatile("bar.sync 1, 64;" ::: "memory");  // both P.V warps are done clearing
        }
        if (active(j, t)) {
          const int li = local_it(j);
          const uint64_t vd = vdesc + st * TILE_STEP;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            cta_wait(&bars[(half ? B_P1 : B_P0) + t], uint32_t(li) & 1u, abort_flag, p.wait_limit_ns);
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
              for (int bx = 0; bx < NBOX; ++bx)  // O columns [64 bx, 64 bx + 64) from V box bx
                mma_bf16_ts_warp(d + bx * 64, a + half * 32 + kk * 8, vd + bx * BOX_STEP + (half * 4 + kk) * V_KSTEP,
                                 IDESC_O, (li > 0 || half > 0 || kk > 0) ? 1u : 0u);
            mma_commit_warp(&bars[(half ? B_O1 : B_O0) + t]);
          }
        }
        mma_commit_warp(&bars[B_KE + st]);  // V of stage st is no longer needed (for this tile)
      }
    }
    if (SPLIT) {  // the two exchange barriers of the split-KV epilogue (below)
      cluster_sync_all();
      cluster_sync_all();
    }
  } else {
    // ---------------- softmax of tile t = warp / 4 ----------------
    set_max_regs_inc<C::REG_SOFTMAX>();
    const int t = warp >> 2;
    const int nkv = t == 0 ? nkv0 : nkv1;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + TM_S + t * 128 + lane_off;
    const uint32_t tO = tmem + TM_O + t * HD + lane_off;
    const uint32_t tP = tmem + TM_P + t * C::P_STRIDE + lane_off;
    const float c = p.qk_scale_log2;  // > 0 (the scale is checked on the host)
    // Masking.  Key n0_first + j * n0_step is the first of this slot's j-th
    // KV tile; the row's last visible key is last_key.  Kept through the
    // loop is only j_diag, the first iteration whose tile the diagonal (or
    // kv_len) may cross for this row; last_key - n0_first waits in shared
    // memory for the few iterations that mask (the loop holds a whole score
    // row in registers and has none to spare).
    // (ILV kernel; pairs alone keep qi and last_key and mask tile j iff
    // (j_lo + j) * BN + BN - 1 > last_key)
    const int qi = m0 + (ilv ? 0 : t * BM) + (tid & (BM - 1));
    const int last_key = p.causal ? min(off + qi, kv_len - 1) : kv_len - 1;
    int j_diag = 0;
    if constexpr (ILV) {
      const int n0_first = (ilv ? t : 0) * BN, n0_step = ilv ? 2 * BN : BN;
      const int x = last_key - (BN - 1) - n0_first;  // tile j is masked iff j * n0_step > x
      j_diag = x < 0 ? 0 : x / n0_step + 1;
      reinterpret_cast<int*>(smem + C::OFF_LIM)[tid] = last_key - n0_first;
    }
    float m_ref = -INFINITY, lsum = 0.f;
    // The two warpgroups share the schedulers, the XU and the FMA pipe; run
    // together their exponentials take twice as long while their P stores
    // and waits leave those pipes idle.  For the tiles both have (j < nmin)
    // they take turns: A computes the exponentials of tile j while B stores
    // and loads, then B while A does.  The trip counts are fixed per CTA, so
    // every bar.sync meets exactly 128 arrivals: A syncs on TURN_A nmin times
    // and B arrives on it nmin times (once before its loop); B syncs on TURN_B
    // nmin times and A arrives on it nmin times.
    const int nmin = min(nkv0, nkv1);
    if (t == 1 && nmin > 0) named_bar_arrive(BAR_TURN_A, 256);
    for (int j = 0; j < nkv; ++j) {
      cta_wait(&bars[B_S + t], uint32_t(j) & 1u, abort_flag, p.wait_limit_ns);
      tc_fence_after();
      // the row's 128 scores, with the maximum of each 32 from the load itself
      uint32_t s[BN];
      float rmx[4];
      tmem_ld32_max(tS, *reinterpret_cast<uint32_t(*)[32]>(s), rmx[0]);
      tmem_ld32_max(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(s + 32), rmx[1]);
      tmem_ld32_max(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(s + 64), rmx[2]);
      tmem_ld32_max(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(s + 96), rmx[3]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_SC + t]);  // the S columns may be overwritten now

      const bool cross = ILV ? j >= j_diag : (j_lo + j) * BN + BN - 1 > last_key;
      if (__any_sync(0xffffffffu, cross)) {  // the diagonal (or the end) crosses this tile
        // mask (keys past last_key), then take the maximum again over what is left
        const int lim = ILV ? reinterpret_cast<const volatile int*>(smem + C::OFF_LIM)[tid] -
                                  j * (unit_info[1] ? 2 * BN : BN)
                            : last_key - (j_lo + j) * BN;  // last_key - (first key of the tile)
#pragma unroll
        for (int e = 0; e < BN; ++e)
          if (e > lim) s[e] = 0xff800000u;  // -inf
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int e = 0; e < BN; e += 8) {
          mx[0] = max3f(mx[0], __uint_as_float(s[e]), __uint_as_float(s[e + 1]));
          mx[1] = max3f(mx[1], __uint_as_float(s[e + 2]), __uint_as_float(s[e + 3]));
          mx[2] = max3f(mx[2], __uint_as_float(s[e + 4]), __uint_as_float(s[e + 5]));
          mx[3] = max3f(mx[3], __uint_as_float(s[e + 6]), __uint_as_float(s[e + 7]));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) rmx[i] = mx[i];
      }
      const float tmax = max3f(rmx[0], rmx[1], fmaxf(rmx[2], rmx[3])) * c;
      if (j == 0) {
        // The first tile of the share.  Without a split it holds key 0, which
        // every row sees; with one (or for the odd KV tiles of a single-tile
        // unit), a row may see no key of the share at all (then every later
        // tile of the share is masked for it too): its reference stays -inf
        // and its exponentials use 0 instead.
        m_ref = tmax;
      } else {
        const bool resc = tmax > m_ref + 8.f;
        if (__any_sync(0xffffffffu, resc)) {
          // a row's maximum rose by more than 2^8: raise its reference and
          // rescale its O once the previous P.V is done (whole warp, as TMEM
          // access is warp-wide)
          cta_wait(&bars[B_O1 + t], uint32_t(j - 1) & 1u, abort_flag, p.wait_limit_ns);
          tc_fence_after();
          const float alpha = resc ? fast_exp2(m_ref - tmax) : 1.f;
          if (resc) m_ref = tmax;
#pragma unroll
          for (int cc = 0; cc < HD / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + cc * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + cc * 32, o);
          }
          tmem_wait_st();
          lsum *= alpha;
        }
      }
      // (-inf only for a row that has seen no key of this slot yet, possible
      // with a KV split or for the odd tiles of a single-tile unit)
      const float m_use = ((SPLIT || ILV) && m_ref == -INFINITY) ? 0.f : m_ref;
      float mu = m_use;
      if (j < nmin) named_bar_sync(t == 0 ? BAR_TURN_A : BAR_TURN_B, 256);  // this warpgroup's turn
      // the exponentials depend on mu: keep the compiler from starting them
      // before the turn begins
      asm volatile("" : "+f"(mu));
      const float2 cc2 = make_float2(c, c), mm = make_float2(-mu, -mu);
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pw[32];
        exp_half(s + half * 64, cc2, mm, pw, acc);
        // after the last exponentials of the tile (their sums are inputs
        // here, so none is moved past the hand-over): the other's turn
        if (half == 1 && j < nmin) {
          asm volatile("" ::"f"(acc[0].x), "f"(acc[0].y), "f"(acc[1].x), "f"(acc[1].y), "f"(acc[2].x),
                       "f"(acc[2].y), "f"(acc[3].x), "f"(acc[3].y));
          if (t == 0 || j < nmin - 1) named_bar_arrive(t == 0 ? BAR_TURN_B : BAR_TURN_A, 256);
        }
        // P_t half may be overwritten once the previous P.V has read it
        if (j > 0) cta_wait(&bars[(half ? B_O1 : B_O0) + t], uint32_t(j - 1) & 1u, abort_flag, p.wait_limit_ns);
        tc_fence_after();
        tmem_st32(tP + half * 32, pw);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[(half ? B_P1 : B_P0) + t]);
      }
      lsum += (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y) + (acc[2].x + acc[2].y) + (acc[3].x + acc[3].y);
    }
    if (nkv > 0) {
      cta_wait(&bars[B_O1 + t], uint32_t(nkv - 1) & 1u, abort_flag, p.wait_limit_ns);
      tc_fence_after();
    }

    // ---- epilogue: O / l, bf16, to global memory ----
    // The unit's first query row and kind, read back from shared memory
    // rather than kept in registers through the loop, which uses nearly all
    // of this warpgroup's registers.
    const bool ilv_e = ILV && unit_info[1] != 0;
    const int qi_e = ILV ? unit_info[0] + (ilv_e ? 0 : t * BM) + (tid & (BM - 1)) : qi;
    if (ILV && ilv_e) {
      // Single-tile unit: slot 1 hands its rows' (m, l) to slot 0 through
      // shared memory; slot 0 reads both O accumulators from tensor memory
      // (its warps reach the same lanes) and combines them:
      //   M = max(m0, m1),  w_s = 2^(m_s - M),  O = (w0 O0 + w1 O1) / (w0 l0 + w1 l1).
      float2* mlx = reinterpret_cast<float2*>(smem + C::OFF_ILV);
      if (t == 1) {
        mlx[tid & (BM - 1)] = make_float2(m_ref, lsum);
        tc_fence_before();
        named_bar_arrive(BAR_ILV, 256);
      } else {
        named_bar_sync(BAR_ILV, 256);
        tc_fence_after();
        const float2 x1 = mlx[tid & (BM - 1)];
        const bool has1 = nkv1 > 0;  // the same for the whole CTA (O1 is never written otherwise)
        const float M = fmaxf(m_ref, x1.x);
        // (exactly 1 for the slot holding the larger reference)
        const float w0 = m_ref == -INFINITY ? 0.f : m_ref == M ? 1.f : fast_exp2(m_ref - M);
        const float w1 = (!has1 || x1.x == -INFINITY) ? 0.f : x1.x == M ? 1.f : fast_exp2(x1.x - M);
        const float inv = *abort_flag ? __int_as_float(0x7fc00000) : 1.f / (w0 * lsum + w1 * x1.y);
        const float a0 = w0 * inv, a1 = w1 * inv;
        __nv_bfloat16* const orow = p.o + ((size_t(b) * p.Hq + h) * p.q_pitch + qi_e) * HD;
#pragma unroll
        for (int cc = 0; cc < HD / 32; ++cc) {
          uint32_t o0[32], o1[32];
          tmem_ld32(tO + cc * 32, o0);
          if (has1) tmem_ld32(tO + HD + cc * 32, o1);
          tmem_wait_ld();
          if (qi_e < q_len) {
#pragma unroll
            for (int e8 = 0; e8 < 4; ++e8) {
              uint32_t w[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int e = e8 * 8 + 2 * u;
                float v0 = __uint_as_float(o0[e]) * a0, v1 = __uint_as_float(o0[e + 1]) * a0;
                if (has1) {
                  v0 = fmaf(__uint_as_float(o1[e]), a1, v0);
                  v1 = fmaf(__uint_as_float(o1[e + 1]), a1, v1);
                }
                const __nv_bfloat162 pk = __floats2bfloat162_rn(v0, v1);
                w[u] = *reinterpret_cast<const uint32_t*>(&pk);
              }
              reinterpret_cast<uint4*>(orow)[cc * 4 + e8] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
    } else if (!SPLIT) {
      if (nkv > 0) {
        __nv_bfloat16* const orow = p.o + ((size_t(b) * p.Hq + h) * p.q_pitch + qi_e) * HD;
        const float inv = *abort_flag ? __int_as_float(0x7fc00000) : 1.f / lsum;
#pragma unroll
        for (int cc = 0; cc < HD / 32; ++cc) {  // 32 columns at a time keeps the register count down
          uint32_t o[32];
          tmem_ld32(tO + cc * 32, o);
          tmem_wait_ld();
          if (qi_e < q_len) {
#pragma unroll
            for (int e8 = 0; e8 < 4; ++e8) {
              uint32_t w[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const __nv_bfloat162 pk = __floats2bfloat162_rn(__uint_as_float(o[e8 * 8 + 2 * u]) * inv,
                                                                __uint_as_float(o[e8 * 8 + 2 * u + 1]) * inv);
                w[u] = *reinterpret_cast<const uint32_t*>(&pk);
              }
              reinterpret_cast<uint4*>(orow)[cc * 4 + e8] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
    } else {
      // Split KV: every softmax thread sends its row's partial (O, m, l) to
      // the CTA of the cluster that finishes this 32-row unit (unit u = warp,
      // finished by rank u % ks, slot u / ks), which merges the ks partials
      //   M = max m_s,  w_s = 2^(m_s - M),  O = sum w_s O_s / sum w_s l_s.
      float* xbuf = reinterpret_cast<float*>(smem + OFF_Q);  // Q and the K/V stages are free after the loop
      cluster_sync_all();  // every CTA of the cluster is done with its stages
      {
        const int dst_rank = warp % ks, slot = warp / ks;
        const float* loc = xbuf + xidx<HD>(rank, slot, upr, 0, lane);
        const uint32_t ra = dsmem_addr(loc, uint32_t(dst_rank));
#pragma unroll
        for (int cc = 0; cc < HD / 32; ++cc) {
          uint32_t o[32];
          if (nkv > 0) {
            tmem_ld32(tO + cc * 32, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0u;
          }
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4)
            dsmem_st4(ra + (cc * 8 + e4) * 512,
                      make_float4(__uint_as_float(o[4 * e4]), __uint_as_float(o[4 * e4 + 1]),
                                  __uint_as_float(o[4 * e4 + 2]), __uint_as_float(o[4 * e4 + 3])));
        }
        dsmem_st4(ra + (HD / 4) * 512, make_float4(m_ref, lsum, 0.f, 0.f));
      }
      cluster_sync_all();  // every partial has arrived
      if (warp % ks == rank && qi_e < q_len) {
        __nv_bfloat16* const orow = p.o + ((size_t(b) * p.Hq + h) * p.q_pitch + qi_e) * HD;
        const int slot = warp / ks;
        float M = -INFINITY;
        for (int src = 0; src < ks; ++src) M = fmaxf(M, xbuf[xidx<HD>(src, slot, upr, HD / 4, lane)]);
        float w_src[8], L = 0.f;
#pragma unroll
        for (int src = 0; src < 8; ++src) {
          const float ms = src < ks ? xbuf[xidx<HD>(src, slot, upr, HD / 4, lane)] : -INFINITY;
          w_src[src] = ms == -INFINITY ? 0.f : fast_exp2(ms - M);
          if (src < ks) L += xbuf[xidx<HD>(src, slot, upr, HD / 4, lane) + 1] * w_src[src];
        }
        const float inv = *abort_flag ? __int_as_float(0x7fc00000) : 1.f / L;
#pragma unroll
        for (int e8 = 0; e8 < HD / 8; ++e8) {  // 8 output columns at a time
          float acc8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int src = 0; src < 8; ++src) {
            if (src < ks) {
              const float4 v0 = *reinterpret_cast<const float4*>(xbuf + xidx<HD>(src, slot, upr, 2 * e8, lane));
              const float4 v1 = *reinterpret_cast<const float4*>(xbuf + xidx<HD>(src, slot, upr, 2 * e8 + 1, lane));
              const float w = w_src[src];
              acc8[0] += v0.x * w; acc8[1] += v0.y * w; acc8[2] += v0.z * w; acc8[3] += v0.w * w;
              acc8[4] += v1.x * w; acc8[5] += v1.y * w; acc8[6] += v1.z * w; acc8[7] += v1.w * w;
            }
          }
          uint32_t wd[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const __nv_bfloat162 pk = __floats2bfloat162_rn(acc8[2 * u] * inv, acc8[2 * u + 1] * inv);
            wd[u] = *reinterpret_cast<const uint32_t*>(&pk);
          }
          reinterpret_cast<uint4*>(orow)[e8] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // After a wait that timed out, tensor-core work may still be in flight:
  // the three issuing warps wait (bounded) for all of their own before the
  // tensor memory is released, and the call is flagged.  (Otherwise every
  // MMA has been waited for by the softmax warps already.)
  if (*abort_flag) {
    if (warp >= 9 && warp <= 11) {
      mma_commit_warp(&bars[B_DRAIN]);
      mbar_wait_bounded(&bars[B_DRAIN], 0, p.wait_limit_ns);
    }
    if (warp == 8 && lane == 0)  // and the copies in flight land before the shared memory is released
      drain_copies<NST>(bars, B_Q, B_KF, B_VF, *reinterpret_cast<volatile int*>(smem + OFF_BAR + C::OFF_ISSUED),
                        p.wait_limit_ns);
    if (tid == 0) atomicOr(&g_prefill_status, GQA_DEV_WAIT_TIMEOUT);
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 9) tmem_dealloc(tmem, TMEM_COLS);
}

// Q, K, V as [heads][row_pitch rows][hd] bf16 with only the first `rows` rows
// of a head readable (cache rows past kv_len arrive as zeros and add exactly
// nothing to P.V); boxes of 128 rows x 64 columns (128 bytes, the widest a
// 128-byte swizzle takes), hd / 64 of them side by side for a tile.
bool make_map(CUtensorMap* map, const void* base, int hd, uint64_t rows, uint64_t row_pitch, uint64_t heads) {
  return encode_bf16_rows(map, base, uint64_t(hd), rows, row_pitch, heads, 64, 128);
}

// Work units of a launch with uniform lengths: the first pair run as single
// query tiles (ilv_from) and the pairs scheduled before those (n_first).
struct UnitPlan {
  int ilv_from, n_first;
};

// KV tiles that query tile t of a head needs (uniform lengths).
long tile_kv_tiles(long t, long q_len, long kv_len, bool causal) {
  const long m = t * BM;
  if (m >= q_len) return 0;
  long n = (kv_len + BN - 1) / BN;
  if (causal) n = std::min(n, (kv_len - q_len + std::min(m + BM - 1, q_len - 1)) / BN + 1);
  return n;
}

// The pairs scheduled before the single tiles: those longer than every
// single tile (so that the grid runs longest first).
int pairs_first(int ilv_from, long n_tiles, long q_len, long kv_len, bool causal) {
  long max_single = 0;
  for (long t = 2L * ilv_from; t < n_tiles; ++t)
    max_single = std::max(max_single, (tile_kv_tiles(t, q_len, kv_len, causal) + 1) / 2);
  int n = 0;
  for (long pr = ilv_from - 1; pr >= 0; --pr) {
    const long it = std::max(tile_kv_tiles(2 * pr, q_len, kv_len, causal),
                             tile_kv_tiles(2 * pr + 1, q_len, kv_len, causal));
    if (it <= max_single) break;
    ++n;
  }
  return n;
}

// Planner (D = 64): list-schedule the units of each candidate first
// single-tile pair on the SMs in launch order and keep the shortest
// makespan, ties going to pairs alone.  The costs, in iterations of the
// pair-only kernel, were fitted to a sweep of every candidate at 513 to
// 8192 causal queries (model against measurement within about 1 us): a
// unit's set-up and epilogue 3.3, a two-tile iteration 1.0, and 1.074 for
// every iteration of the kernel that holds single-tile units (its unit
// bookkeeping costs the softmax loop registers).  Only causal grids of a
// few waves can gain (the longest pairs bound them); the result is cached
// per shape.  At D = 128 single tiles did not pay in any case measured.
UnitPlan plan_units(long q_len, long kv_len, bool causal, long heads, int sms) {
  const int n_pairs = int((q_len + 2 * BM - 1) / (2 * BM));
  const long n_tiles = (q_len + BM - 1) / BM;
  UnitPlan none{n_pairs, 0};
  if (!causal || long(n_pairs) * heads > 16L * sms || n_tiles > 65535) return none;
  static std::mutex mu;
  static std::map<std::array<long, 5>, UnitPlan> cache;
  const std::array<long, 5> key{q_len, kv_len, long(causal), heads, long(sms)};
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  constexpr double kSetup = 3.3, kIlvKernel = 1.074;
  std::vector<long> pair_it(n_pairs), single_it(n_tiles);
  for (int pr = 0; pr < n_pairs; ++pr)
    pair_it[pr] = std::max(tile_kv_tiles(2L * pr, q_len, kv_len, causal),
                           tile_kv_tiles(2L * pr + 1, q_len, kv_len, causal));
  for (long t = 0; t < n_tiles; ++t) single_it[t] = (tile_kv_tiles(t, q_len, kv_len, causal) + 1) / 2;
  UnitPlan best = none;
  double best_span = 0.0;
  std::vector<double> sm_free;
  for (int from = n_pairs; from >= 0; --from) {
    const int n_first = pairs_first(from, n_tiles, q_len, kv_len, causal);
    std::vector<long> order;  // unit costs in launch order (y), each for every head
    for (int i = 0; i < n_first; ++i) order.push_back(pair_it[from - 1 - i]);
    for (long t = n_tiles - 1; t >= 2L * from; --t) order.push_back(single_it[t]);
    for (int pr = from - 1 - n_first; pr >= 0; --pr) order.push_back(pair_it[pr]);
    const double per_it = from == n_pairs ? 1.0 : kIlvKernel;
    sm_free.assign(size_t(sms), 0.0);
    std::priority_queue<double, std::vector<double>, std::greater<double>> q(sm_free.begin(), sm_free.end());
    double span = 0.0;
    for (const long c : order)
      for (long hh = 0; hh < heads; ++hh) {
        const double start = q.top();
        q.pop();
        const double end = start + kSetup + per_it * double(c);
        span = std::max(span, end);
        q.push(end);
      }
    if (from == n_pairs || span < best_span - 1e-9) {
      best_span = span;
      best = UnitPlan{from, n_first};
    }
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() >= 1024) cache.clear();
  cache[key] = best;
  return best;
}

template <int HD>
cudaError_t launch_prefill_hd(const PrefillArgs& a, cudaStream_t stream) {
  using C = PfCfg<HD>;
  CUtensorMap tq, tk, tv;
  // uniform lengths: the K/V maps end at kv_len, so rows past it arrive as
  // zeros; per-request lengths: the maps span the whole buffers and the
  // kernel masks and clears what lies past each request's lengths
  const bool varlen = a.q_lens != nullptr;
  const uint64_t q_rows = a.q_len, kv_rows = varlen ? uint64_t(a.S_cap) : uint64_t(a.kv_len);
  if (!make_map(&tq, a.q, HD, q_rows, a.q_len, uint64_t(a.B) * a.Hq) ||
      !make_map(&tk, a.k, HD, kv_rows, a.S_cap, uint64_t(a.B) * a.Hkv) ||
      !make_map(&tv, a.v, HD, kv_rows, a.S_cap, uint64_t(a.B) * a.Hkv))
    return cudaErrorInvalidValue;
  PrefillParams p;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.n_rep = a.Hq / a.Hkv;
  p.q_len = a.q_len;
  p.kv_len = varlen ? a.S_cap : a.kv_len;
  p.q_pitch = a.q_len;
  p.q_lens = a.q_lens;
  p.kv_lens = a.kv_lens;
  p.n_pairs = (a.q_len + 2 * BM - 1) / (2 * BM);
  p.causal = a.causal;
  p.qk_scale_log2 = float(double(a.scale) * 1.4426950408889634);
  p.wait_limit_ns = kWaitLimitNs;
  p.test_stall_ns = wait_test_ns();
  // Split the KV range of a pair over a cluster when the pairs alone leave
  // SMs idle: as many CTAs per pair (up to 8) as keep the grid within one
  // wave and every share at kMinShareTiles KV tiles or more.  (Beyond one
  // wave a cluster has to wait for SMs of one GPC to free up together, which
  // costs more than the split gains: T=4097 took 49 us unsplit, 68 us split
  // in two.)  At HD = 128 the exchange holds no more than 5 CTAs' units
  // except for 8, so 6 and 7 become 5.
  {
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long pairs = long(a.B) * a.Hq * p.n_pairs;
    const int kv_tiles = (a.kv_len + BN - 1) / BN;
    int ks = 1;
    if (pairs * 2 <= sms)
      ks = int(std::min<long>({8L, sms / pairs, std::max<long>(1L, kv_tiles / kMinShareTiles)}));
    if (const int v = prefill_kv_split_override(); v >= 1 && v <= 8) ks = v;  // tuning and tests only
    while (!kv_split_fits(C::X_MAX_UNITS, ks)) --ks;
    p.kv_splits = ks;
    // work units: pairs, and for the longest causal tiles single tiles
    p.n_tiles = (a.q_len + BM - 1) / BM;
    UnitPlan up{p.n_pairs, 0};
    if (ks == 1 && !varlen) {
      const int forced = prefill_interleave_override();  // tuning and tests only
      if (forced >= 0) {
        up.ilv_from = std::min(forced, p.n_pairs);
        up.n_first = pairs_first(up.ilv_from, p.n_tiles, a.q_len, a.kv_len, a.causal != 0);
      } else if (HD == 64) {
        up = plan_units(a.q_len, a.kv_len, a.causal != 0, long(a.B) * a.Hq, sms);
      }
      if (std::max(0, p.n_tiles - 2 * up.ilv_from) + up.ilv_from > 65535) up = UnitPlan{p.n_pairs, 0};
    }
    p.ilv_from = up.ilv_from;
    p.n_first = up.n_first;
  }
  static std::once_flag once;
  static cudaError_t cfg_err = cudaSuccess;
  std::call_once(once, [&] {
    for (const void* k : {reinterpret_cast<const void*>(prefill_kernel<HD, false, false>),
                          reinterpret_cast<const void*>(prefill_kernel<HD, true, false>),
                          reinterpret_cast<const void*>(prefill_kernel<HD, false, true>)})
      if (cfg_err == cudaSuccess)
        cfg_err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  });
  if (cfg_err != cudaSuccess) return cfg_err;
  const dim3 grid(a.B * a.Hq * p.kv_splits, std::max(0, p.n_tiles - 2 * p.ilv_from) + p.ilv_from);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(NTHR);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = p.kv_splits;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  if (p.kv_splits == 1) {
    cfg.numAttrs = 1;
    if (p.n_tiles - 2 * p.ilv_from > 0)  // single-tile units in the grid
      return cudaLaunchKernelEx(&cfg, prefill_kernel<HD, false, true>, tq, tk, tv, p);
    return cudaLaunchKernelEx(&cfg, prefill_kernel<HD, false, false>, tq, tk, tv, p);
  }
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, prefill_kernel<HD, true, false>, tq, tk, tv, p);
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  if (a.D == 64) return launch_prefill_hd<64>(a, stream);
  if (a.D == 128) return launch_prefill_hd<128>(a, stream);
  return cudaErrorNotSupported;
}

}  // namespace gqa

using namespace gqa;

extern "C" GQA_ATTN_API int gqa_attn_read_prefill_status(uint32_t* out, void* stream) {
  if (out == nullptr) return GQA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyFromSymbolAsync(out, g_prefill_status, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return GQA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GQA_ERR_CUDA;
  return GQA_OK;
}

extern "C" GQA_ATTN_API int gqa_attn_clear_prefill_status(void* stream) {
  static const uint32_t zero = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyToSymbolAsync(g_prefill_status, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return GQA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GQA_ERR_CUDA;
  return GQA_OK;
}
