// internal.h -- host-side plumbing shared by the C ABI and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace gqa {

// Workspace layout (all offsets 256-byte aligned):
//   [0, 256)   uint32 device status word (GQA_DEV_* bits) + padding
//   ml         float2 [B][Hq][n_split]      per-split (max in log2 units, sum)
//   part_o     float  [B][Hq][n_split][D]   per-split unnormalised outputs
// Nothing in it has to start at zero except the status word.
struct WorkspaceLayout {
  size_t off_ml, off_o, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WorkspaceLayout workspace_layout(int B, int Hq, int Hkv, int n_hc, int n_split, int D) {
  (void)Hkv;
  (void)n_hc;
  WorkspaceLayout w;
  const size_t bh = size_t(B) * Hq;
  w.off_ml = 256;
  w.off_o = align256(w.off_ml + sizeof(float) * 2 * bh * n_split);
  w.total = align256(w.off_o + sizeof(float) * bh * n_split * D);
  return w;
}

// The split plan: a request of L keys uses n_used = min(n_split,
// ceil(L / chunk)) splits (grid x < n_used), and its tiles are dealt to them
// round-robin.
struct SplitPlan {
  int tile;     // rows per shared-memory tile
  int chunk;    // rows per split that count towards n_used
  int n_split;  // grid.x
  int n_hc;     // query-head chunks per KV head (n_rep > 8)
  int nrep_cta; // query heads one CTA serves (<= 8)
};

// ctas_per_sm: how many CTAs of the kernel an SM holds at once; the grid is
// sized for about that many per SM.
SplitPlan plan_splits(int B, int Hq, int Hkv, int max_kv_len, int tile, int num_sms, int ctas_per_sm = 2);

int device_sm_count();

// The prefill KV-split cluster size forced by gqa_attn_set_plan_override, or
// 0 (the planner decides).
int prefill_kv_split_override();
// Forced first interleaved pair of prefill (>= 0), or -1 for the planner's choice.
int prefill_interleave_override();
uint64_t wait_test_ns();  // gqa_attn_set_wait_test; 0 = off

// Shape, dtype and pointer checks shared by gqa_attn_decode and
// gqa_attn_decode_noalloc (everything but the workspace); GQA_OK or an error.
int validate_decode_args(const void* q, const void* k, const void* v, const void* o, const int32_t* kv_lens,
                         int B, int Hq, int Hkv, int D, int S_cap, int max_kv_len, float scale, int dtype);

struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  const int32_t* kv_lens;
  int B, Hq, Hkv, D, S_cap, max_kv_len;
  float scale;
  int dtype;
  void* workspace;
  SplitPlan plan;
  // paged cache (block_table != nullptr): k and v are pools
  // [num_blocks][Hkv][block_size][D]; k_new / v_new (or null) is appended at
  // row kv_lens[b] - 1 of each request before it attends
  const int32_t* block_table = nullptr;
  int block_size = 0, max_blocks = 0, num_blocks = 0;
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  // residual window after a 4-bit cache (bf16 kernel only): see
  // launch_decode_mma_residual
  const int32_t* len_sub = nullptr;
  int max_sub = 0, slot_chunk = 0, n_slots = 0, force_partial = 0;
  // layers stacked along the batch axis (kv_period = requests per layer):
  // request b reads kv_lens[b % kv_period]
  int kv_period = 0;
};

// Tile height (rows) of the decode kernel for this dtype / head size, and how
// many of its CTAs an SM holds.
// `units`: (request, KV head chunk) pairs of one call, B * Hkv * n_hc.
int decode_tile_rows(int dtype, int D, bool paged, long units, int max_kv_len);
int decode_ctas_per_sm(int dtype, bool paged, long units, int max_kv_len);
int decode_mma_tile_rows(bool paged, long units, int max_kv_len);
int decode_mma_ctas_per_sm(bool paged, long units, int max_kv_len);
// The decode plan of one layer call (contiguous or paged cache).
SplitPlan decode_plan(int B, int Hq, int Hkv, int D, int max_kv_len, int dtype, bool paged);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t stream);  // bf16 caches (tensor cores)

struct DecodeQ4Args {
  const void* q;
  const uint8_t* k_codes;
  const uint16_t* k_scale;
  const uint16_t* k_bias;
  const uint8_t* v_codes;
  const uint16_t* v_scale;
  const uint16_t* v_bias;
  void* o;
  const int32_t* kv_lens;
  int B, Hq, Hkv, D, S_cap, max_kv_len;
  float scale;
  void* workspace;
  SplitPlan plan;
  int n_slots = 0;        // partial slots per row (0: plan.n_split)
  int force_partial = 0;  // write partials even for one split, and launch no merge
};

// The residual window of a 4-bit cache: request b attends rows
// [0, kv_lens[b] - clamp(n_quant[b], 0, max_quant)) of a.k / a.v (bf16,
// S_cap = the window capacity) and writes its partial into slot
// ceil(clamp(n_quant[b]) / slot_chunk) of n_slots.
cudaError_t launch_decode_mma_residual(const DecodeArgs& a, const int32_t* n_quant, int max_quant, int slot_chunk,
                                       int n_slots, cudaStream_t stream);
// A 4-bit cache (aq, with aq.kv_lens = n_quant) followed by a bf16 window (ar).
cudaError_t launch_decode_q4_residual(const DecodeQ4Args& aq, const DecodeArgs& ar, cudaStream_t stream);

int decode_q4_tile_rows(int D);
int decode_q4_ctas_per_sm();
cudaError_t launch_decode_q4(const DecodeQ4Args& a, cudaStream_t stream);

struct PrefillArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  int B, Hq, Hkv, D, q_len, kv_len, S_cap;
  float scale;
  int causal;
  // per-request lengths (device int32 [B]) or null; with them q_len is the
  // rows per head of Q and O and every request may use up to S_cap keys
  const int32_t* q_lens = nullptr;
  const int32_t* kv_lens = nullptr;
};

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);

// Upper bound on the time a kernel waits for one of its own tile copies
// before it records GQA_DEV_WAIT_TIMEOUT and stops (nanoseconds).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

}  // namespace gqa
