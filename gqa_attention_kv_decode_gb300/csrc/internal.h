// internal.h -- host-side plumbing shared by the C ABI and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace gqa {

// Workspace layout (all offsets 256-byte aligned):
//   [0, 256)   uint32 device status word (GQA_DEV_* bits) + padding
//   counters   int32 [B][Hkv][n_hc][n_groups_max + 1] arrival counters of the
//              merge tree (self-resetting: each is zeroed by its consumer)
//   ml         float2 [B][Hq][n_split]      per-split (max in log2 units, sum)
//   part_o     float  [B][Hq][n_split][D]   per-split unnormalised outputs
//   ml1, o1    the same per group of 8 splits [B][Hq][n_groups_max](...)
struct WorkspaceLayout {
  int n_groups_max;
  size_t off_counters, off_ml, off_o, off_ml1, off_o1, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WorkspaceLayout workspace_layout(int B, int Hq, int Hkv, int n_hc, int n_split, int D) {
  WorkspaceLayout w;
  w.n_groups_max = (n_split + 7) / 8;
  const size_t bh = size_t(B) * Hq;
  w.off_counters = 256;
  w.off_ml = align256(w.off_counters + sizeof(int32_t) * size_t(B) * Hkv * n_hc * (w.n_groups_max + 1));
  w.off_o = align256(w.off_ml + sizeof(float) * 2 * bh * n_split);
  w.off_ml1 = align256(w.off_o + sizeof(float) * bh * n_split * D);
  w.off_o1 = align256(w.off_ml1 + sizeof(float) * 2 * bh * w.n_groups_max);
  w.total = align256(w.off_o1 + sizeof(float) * bh * w.n_groups_max * D);
  return w;
}

// The split plan: keys of every request are cut into chunks of `chunk` rows
// (a multiple of the kernel's tile); chunk s of request b goes to grid x = s.
struct SplitPlan {
  int tile;     // rows per shared-memory tile
  int chunk;    // rows per split
  int n_split;  // grid.x
  int n_hc;     // query-head chunks per KV head (n_rep > 8)
  int nrep_cta; // query heads one CTA serves (<= 8)
};

SplitPlan plan_splits(int B, int Hq, int Hkv, int max_kv_len, int tile, int num_sms);

int device_sm_count();

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
};

// Tile height (rows) of the decode kernel for this dtype / head size.
int decode_tile_rows(int dtype, int D);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

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
};

int decode_q4_tile_rows(int D);
cudaError_t launch_decode_q4(const DecodeQ4Args& a, cudaStream_t stream);

struct PrefillArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  int B, Hq, Hkv, D, q_len, kv_len, S_cap;
  float scale;
  int causal;
};

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);

// Upper bound on the time a kernel waits for one of its own tile copies
// before it records GQA_DEV_WAIT_TIMEOUT and stops (nanoseconds).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

}  // namespace gqa
