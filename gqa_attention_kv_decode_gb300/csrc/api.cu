// api.cu -- the extern "C" boundary of libgqa_attn.so: argument validation,
// the split-KV planner, workspace sizing and kernel dispatch.  Every check
// runs on the host before anything is launched.
#include <cuda_runtime.h>

#include <algorithm>

#include <atomic>
#include <cmath>
#include <mutex>

#include "gqa_attn.h"
#include "internal.h"

namespace gqa {

int device_sm_count() {
  static std::atomic<int> cache[64];  // 0 until queried (zero-initialised as a static)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

static long ceil_div(long a, long b) { return (a + b - 1) / b; }

// Plan overrides (gqa_attn_set_plan_override); 0 = the planner decides.
static std::atomic<int> g_decode_splits_override{0};
static std::atomic<int> g_prefill_kv_split_override{0};

int prefill_kv_split_override() { return g_prefill_kv_split_override.load(std::memory_order_relaxed); }
static std::atomic<int> g_prefill_interleave_override{-1};
int prefill_interleave_override() { return g_prefill_interleave_override.load(std::memory_order_relaxed); }
// Failure-path test (gqa_attn_set_wait_test); 0 = off.
static std::atomic<uint64_t> g_wait_test_ns{0};
uint64_t wait_test_ns() { return g_wait_test_ns.load(std::memory_order_relaxed); }

// Chooses how many key splits each (request, KV head) gets so that the grid
// covers at most ctas_per_sm CTAs per SM (one wave) when requests are few and
// short, while a split stays at least one tile and at most 1024 rows long (so
// the splits of long, ragged requests balance across the SMs).  A split count
// set with gqa_attn_set_plan_override (tuning and tests only) replaces the
// planner's choice.
SplitPlan plan_splits(int B, int Hq, int Hkv, int max_kv_len, int tile, int num_sms, int ctas_per_sm) {
  SplitPlan p;
  const int n_rep = Hq / Hkv;
  p.tile = tile;
  p.n_hc = (n_rep + 7) / 8;
  p.nrep_cta = int(ceil_div(n_rep, p.n_hc));
  const long units = long(B) * Hkv * p.n_hc;
  const long target = long(ctas_per_sm > 0 ? ctas_per_sm : 1) * (num_sms > 0 ? num_sms : 1);
  // at most target / units splits per unit, so that the grid is one wave.
  // Tiles are dealt round-robin to the splits, so the split length need not
  // be a whole number of tiles.
  const long per_unit = target / units > 0 ? target / units : 1;
  long chunk = ceil_div(max_kv_len, per_unit);
  const long lo = tile;
  const long hi = (1024 / tile) * tile;
  if (chunk < lo) chunk = lo;
  bool one_wave = chunk <= hi;  // else several waves of splits of at most hi rows
  if (chunk > hi) chunk = hi;
  // two tiles or fewer: one CTA per head group is faster than a split plus
  // its merge kernel
  if (max_kv_len <= 2L * tile) chunk = ceil_div(max_kv_len, tile) * tile;
  if (const int n = g_decode_splits_override.load(std::memory_order_relaxed); n > 0) {
    chunk = ceil_div(max_kv_len, n);
    one_wave = true;  // (so that a request's splits do not depend on the batch)
  }
  if (chunk < lo) chunk = lo;
  if (ceil_div(max_kv_len, chunk) > 1024) chunk = ceil_div(max_kv_len, 1024);
  p.n_split = int(ceil_div(max_kv_len, chunk));
  // A request of L keys uses min(n_split, ceil(L / chunk)) splits.  In a
  // one-wave grid a request shorter than max_kv_len spreads over all of its
  // splits (at least two tiles each) instead of leaving most of its CTAs
  // idle while the rest carry full-length chunks; in a grid of several waves
  // the splits keep at most `hi` rows each, so that long and short requests
  // balance across the SMs.
  p.chunk = int(one_wave && p.n_split > 1 ? std::min<long>(chunk, 2L * tile) : chunk);
  return p;
}

SplitPlan decode_plan_for(int B, int Hq, int Hkv, int D, int max_kv_len, int dtype, bool paged, int num_sms) {
  const long units = long(B) * Hkv * ((Hq / Hkv + 7) / 8);
  return plan_splits(B, Hq, Hkv, max_kv_len, decode_tile_rows(dtype, D, paged, units, max_kv_len), num_sms,
                     decode_ctas_per_sm(dtype, paged, units, max_kv_len));
}

SplitPlan decode_plan(int B, int Hq, int Hkv, int D, int max_kv_len, int dtype, bool paged) {
  return decode_plan_for(B, Hq, Hkv, D, max_kv_len, dtype, paged, device_sm_count());
}

}  // namespace gqa

using namespace gqa;

namespace {

bool is_device_ptr(const void* p, int dev) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error state of this query
    return false;
  }
  if (attr.type == cudaMemoryTypeDevice) return attr.device == dev;
  if (attr.type == cudaMemoryTypeManaged) return true;
  return false;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Common decode-shape checks; returns GQA_OK or an error code.
int check_decode_shape(int B, int Hq, int Hkv, int D, int S_cap, int max_kv_len, float scale) {
  if (B < 1 || Hq < 1 || Hkv < 1 || S_cap < 1) return GQA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (max_kv_len < 1 || max_kv_len > S_cap) return GQA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return GQA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return GQA_ERR_INVALID_ARG;
  if (B > 65535) return GQA_ERR_INVALID_ARG;
  const int n_hc = (Hq / Hkv + 7) / 8;
  if (long(Hkv) * n_hc > 65535) return GQA_ERR_INVALID_ARG;
  return GQA_OK;
}

int check_ptrs(std::initializer_list<const void*> ptrs, int dev, size_t align) {
  for (const void* p : ptrs) {
    if (p == nullptr) return GQA_ERR_INVALID_ARG;
    if (!aligned(p, align)) return GQA_ERR_INVALID_ARG;
  }
  for (const void* p : ptrs)
    if (!is_device_ptr(p, dev)) return GQA_ERR_NOT_DEVICE_PTR;
  return GQA_OK;
}

size_t decode_ws_size(int B, int Hq, int Hkv, int D, int max_kv_len, int tile, int ctas_per_sm = 2) {
  const SplitPlan p = plan_splits(B, Hq, Hkv, max_kv_len, tile, device_sm_count(), ctas_per_sm);
  return workspace_layout(B, Hq, Hkv, p.n_hc, p.n_split, D).total;
}

}  // namespace

// Shape, dtype and pointer checks of a contiguous-cache decode call, in the
// order gqa_attn_decode applies them (the workspace is checked separately).
int gqa::validate_decode_args(const void* q, const void* k, const void* v, const void* o,
                              const int32_t* kv_lens, int B, int Hq, int Hkv, int D, int S_cap,
                              int max_kv_len, float scale, int dtype) {
  int rc = check_decode_shape(B, Hq, Hkv, D, S_cap, max_kv_len, scale);
  if (rc != GQA_OK) return rc;
  if (dtype != GQA_F32 && dtype != GQA_BF16) return GQA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  rc = check_ptrs({q, k, v, o}, dev, 16);
  if (rc != GQA_OK) return rc;
  if (kv_lens != nullptr) {
    rc = check_ptrs({kv_lens}, dev, 4);
    if (rc != GQA_OK) return rc;
  }
  return GQA_OK;
}

extern "C" {

GQA_ATTN_API int gqa_attn_version(void) { return 100; }

GQA_ATTN_API int gqa_attn_set_plan_override(int decode_splits, int prefill_kv_split) {
  if (decode_splits < 0 || prefill_kv_split < 0 || prefill_kv_split > 8) return GQA_ERR_INVALID_ARG;
  g_decode_splits_override.store(decode_splits, std::memory_order_relaxed);
  g_prefill_kv_split_override.store(prefill_kv_split, std::memory_order_relaxed);
  return GQA_OK;
}

GQA_ATTN_API int gqa_attn_set_prefill_interleave_override(int from_pair) {
  g_prefill_interleave_override.store(from_pair < 0 ? -1 : from_pair, std::memory_order_relaxed);
  return GQA_OK;
}

GQA_ATTN_API int gqa_attn_set_wait_test(uint64_t stall_ns) {
  if (stall_ns > kWaitLimitNs) return GQA_ERR_INVALID_ARG;
  g_wait_test_ns.store(stall_ns, std::memory_order_relaxed);
  return GQA_OK;
}

GQA_ATTN_API const char* gqa_attn_status_string(int status) {
  switch (status) {
    case GQA_OK: return "GQA_OK";
    case GQA_ERR_INVALID_ARG: return "GQA_ERR_INVALID_ARG: invalid shape, length, scale or alignment";
    case GQA_ERR_UNSUPPORTED: return "GQA_ERR_UNSUPPORTED: no kernel for this dtype / head size";
    case GQA_ERR_NOT_DEVICE_PTR: return "GQA_ERR_NOT_DEVICE_PTR: a pointer is not device memory of the current device (there is no CPU path)";
    case GQA_ERR_CUDA: return "GQA_ERR_CUDA: a CUDA call or kernel launch failed";
    case GQA_ERR_WORKSPACE: return "GQA_ERR_WORKSPACE: workspace missing or smaller than *_workspace_size()";
    case GQA_ERR_SCRATCH_LIMIT: return "GQA_ERR_SCRATCH_LIMIT: the problem needs more scratch than the 16 MiB built into gqa_attn_decode_noalloc";
    default: return "unknown gqa_attn status";
  }
}

GQA_ATTN_API size_t gqa_attn_decode_workspace_size(int B, int Hq, int Hkv, int D, int max_kv_len,
                                                   int dtype) {
  if (check_decode_shape(B, Hq, Hkv, D, max_kv_len, max_kv_len, 1.f) != GQA_OK) return 0;
  if (dtype != GQA_F32 && dtype != GQA_BF16) return 0;
  // the same workspace serves gqa_attn_decode_paged, whose kernel may plan
  // more splits: the larger of the two plans
  const SplitPlan c = decode_plan(B, Hq, Hkv, D, max_kv_len, dtype, false);
  const SplitPlan pg = decode_plan(B, Hq, Hkv, D, max_kv_len, dtype, true);
  const size_t contiguous = workspace_layout(B, Hq, Hkv, c.n_hc, c.n_split, D).total;
  const size_t paged = workspace_layout(B, Hq, Hkv, pg.n_hc, pg.n_split, D).total;
  return contiguous > paged ? contiguous : paged;
}

GQA_ATTN_API int gqa_attn_decode_num_splits(int B, int Hq, int Hkv, int D, int max_kv_len,
                                            int dtype) {
  if (check_decode_shape(B, Hq, Hkv, D, max_kv_len, max_kv_len, 1.f) != GQA_OK) return GQA_ERR_INVALID_ARG;
  if (dtype != GQA_F32 && dtype != GQA_BF16) return GQA_ERR_INVALID_ARG;
  return decode_plan(B, Hq, Hkv, D, max_kv_len, dtype, false).n_split;
}

GQA_ATTN_API int gqa_attn_decode_plan_for(int B, int Hq, int Hkv, int D, int max_kv_len, int dtype,
                                          int variant, int num_sms, int32_t* n_split, int32_t* chunk,
                                          int32_t* tile) {
  if (check_decode_shape(B, Hq, Hkv, D, max_kv_len, max_kv_len, 1.f) != GQA_OK) return GQA_ERR_INVALID_ARG;
  if (num_sms < 1 || n_split == nullptr || chunk == nullptr || tile == nullptr) return GQA_ERR_INVALID_ARG;
  if (variant < GQA_PLAN_DECODE || variant > GQA_PLAN_Q4) return GQA_ERR_INVALID_ARG;
  if (variant == GQA_PLAN_Q4 ? dtype != GQA_BF16 : (dtype != GQA_F32 && dtype != GQA_BF16))
    return GQA_ERR_UNSUPPORTED;
  const SplitPlan p =
      variant == GQA_PLAN_Q4
          ? plan_splits(B, Hq, Hkv, max_kv_len, decode_q4_tile_rows(D), num_sms, decode_q4_ctas_per_sm())
          : decode_plan_for(B, Hq, Hkv, D, max_kv_len, dtype, variant == GQA_PLAN_PAGED, num_sms);
  *n_split = p.n_split;
  *chunk = p.chunk;
  *tile = p.tile;
  return GQA_OK;
}

GQA_ATTN_API int gqa_attn_decode(const void* q, const void* k, const void* v, void* o,
                                 const int32_t* kv_lens, int B, int Hq, int Hkv, int D, int S_cap,
                                 int max_kv_len, float scale, int dtype, void* workspace,
                                 size_t ws_bytes, void* stream) {
  int rc = gqa::validate_decode_args(q, k, v, o, kv_lens, B, Hq, Hkv, D, S_cap, max_kv_len, scale, dtype);
  if (rc != GQA_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  if (workspace == nullptr) return GQA_ERR_WORKSPACE;
  rc = check_ptrs({workspace}, dev, 256);
  if (rc == GQA_ERR_INVALID_ARG) return GQA_ERR_WORKSPACE;
  if (rc != GQA_OK) return rc;

  DecodeArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.kv_lens = kv_lens;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.S_cap = S_cap;
  a.max_kv_len = max_kv_len;
  a.scale = scale;
  a.dtype = dtype;
  a.workspace = workspace;
  a.plan = decode_plan(B, Hq, Hkv, D, max_kv_len, dtype, false);
  if (ws_bytes < workspace_layout(B, Hq, Hkv, a.plan.n_hc, a.plan.n_split, D).total)
    return GQA_ERR_WORKSPACE;
  if (launch_decode(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return GQA_ERR_CUDA;
  return GQA_OK;
}

GQA_ATTN_API size_t gqa_attn_decode_layers_workspace_size(int n_layers, int B, int Hq, int Hkv, int D,
                                                          int max_kv_len, int dtype) {
  if (n_layers < 1 || long(n_layers) * B > 65535) return 0;
  if (check_decode_shape(B, Hq, Hkv, D, max_kv_len, max_kv_len, 1.f) != GQA_OK) return 0;
  if (dtype != GQA_F32 && dtype != GQA_BF16) return 0;
  const SplitPlan p = decode_plan(B, Hq, Hkv, D, max_kv_len, dtype, false);
  return workspace_layout(n_layers * B, Hq, Hkv, p.n_hc, p.n_split, D).total;
}

GQA_ATTN_API int gqa_attn_decode_layers(const void* q, const void* k, const void* v, void* o,
                                        const int32_t* kv_lens, int n_layers, int B, int Hq, int Hkv,
                                        int D, int S_cap, int max_kv_len, float scale, int dtype,
                                        void* workspace, size_t ws_bytes, void* stream) {
  if (n_layers < 1 || long(n_layers) * B > 65535) return GQA_ERR_INVALID_ARG;
  int rc = check_decode_shape(B, Hq, Hkv, D, S_cap, max_kv_len, scale);
  if (rc != GQA_OK) return rc;
  if (dtype != GQA_F32 && dtype != GQA_BF16) return GQA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  rc = check_ptrs({q, k, v, o}, dev, 16);
  if (rc != GQA_OK) return rc;
  if (kv_lens != nullptr) {
    rc = check_ptrs({kv_lens}, dev, 4);
    if (rc != GQA_OK) return rc;
  }
  if (workspace == nullptr) return GQA_ERR_WORKSPACE;
  rc = check_ptrs({workspace}, dev, 256);
  if (rc == GQA_ERR_INVALID_ARG) return GQA_ERR_WORKSPACE;
  if (rc != GQA_OK) return rc;
  DecodeArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.kv_lens = kv_lens;
  a.B = n_layers * B;  // layer l, request b is batch index l * B + b of every stacked tensor
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.S_cap = S_cap;
  a.max_kv_len = max_kv_len;
  a.scale = scale;
  a.dtype = dtype;
  a.workspace = workspace;
  a.kv_period = B;
  // the single-layer plan: every (layer, request, head, split) CTA does the
  // work it does in a one-layer call, so the results are bit-identical
  a.plan = decode_plan(B, Hq, Hkv, D, max_kv_len, dtype, false);
  if (ws_bytes < workspace_layout(a.B, Hq, Hkv, a.plan.n_hc, a.plan.n_split, D).total) return GQA_ERR_WORKSPACE;
  if (launch_decode(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return GQA_ERR_CUDA;
  return GQA_OK;
}

GQA_ATTN_API int gqa_attn_decode_paged(const void* q, const void* k_new, const void* v_new,
                                       void* k_pool, void* v_pool, const int32_t* block_table,
                                       const int32_t* kv_lens, void* o, int B, int Hq, int Hkv,
                                       int D, int block_size, int num_blocks, int max_blocks,
                                       int max_kv_len, float scale, int dtype, void* workspace,
                                       size_t ws_bytes, void* stream) {
  if (block_size < 1 || num_blocks < 1 || max_blocks < 1) return GQA_ERR_INVALID_ARG;
  if (long(max_kv_len) > long(max_blocks) * block_size) return GQA_ERR_INVALID_ARG;
  int rc = check_decode_shape(B, Hq, Hkv, D, max_kv_len, max_kv_len, scale);
  if (rc != GQA_OK) return rc;
  if (dtype != GQA_F32 && dtype != GQA_BF16) return GQA_ERR_INVALID_ARG;
  if (block_size % decode_plan(B, Hq, Hkv, D, max_kv_len, dtype, true).tile != 0) return GQA_ERR_UNSUPPORTED;
  // block ids index [num_blocks * Hkv] (block, head) slabs of block_size rows
  if (long(num_blocks) * Hkv > 0x7fffffffL || long(num_blocks) * Hkv * block_size > 0x7fffffffL)
    return GQA_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return GQA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  rc = check_ptrs({q, k_pool, v_pool, o}, dev, 16);
  if (rc != GQA_OK) return rc;
  rc = check_ptrs({block_table, kv_lens}, dev, 4);
  if (rc != GQA_OK) return rc;
  if (k_new != nullptr) {
    rc = check_ptrs({k_new, v_new}, dev, 16);
    if (rc != GQA_OK) return rc;
  }
  if (workspace == nullptr) return GQA_ERR_WORKSPACE;
  rc = check_ptrs({workspace}, dev, 256);
  if (rc == GQA_ERR_INVALID_ARG) return GQA_ERR_WORKSPACE;
  if (rc != GQA_OK) return rc;

  DecodeArgs a;
  a.q = q;
  a.k = k_pool;
  a.v = v_pool;
  a.o = o;
  a.kv_lens = kv_lens;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.S_cap = block_size;
  a.max_kv_len = max_kv_len;
  a.scale = scale;
  a.dtype = dtype;
  a.workspace = workspace;
  a.block_table = block_table;
  a.block_size = block_size;
  a.max_blocks = max_blocks;
  a.num_blocks = num_blocks;
  a.k_new = k_new;
  a.v_new = v_new;
  a.plan = decode_plan(B, Hq, Hkv, D, max_kv_len, dtype, true);
  if (ws_bytes < workspace_layout(B, Hq, Hkv, a.plan.n_hc, a.plan.n_split, D).total)
    return GQA_ERR_WORKSPACE;
  if (launch_decode(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return GQA_ERR_CUDA;
  return GQA_OK;
}

GQA_ATTN_API size_t gqa_attn_decode_q4_workspace_size(int B, int Hq, int Hkv, int D,
                                                      int max_kv_len) {
  if (check_decode_shape(B, Hq, Hkv, D, max_kv_len, max_kv_len, 1.f) != GQA_OK) return 0;
  return decode_ws_size(B, Hq, Hkv, D, max_kv_len, decode_q4_tile_rows(D), decode_q4_ctas_per_sm());
}

GQA_ATTN_API int gqa_attn_decode_q4(const void* q, const uint8_t* k_codes, const uint16_t* k_scale,
                                    const uint16_t* k_bias, const uint8_t* v_codes,
                                    const uint16_t* v_scale, const uint16_t* v_bias, void* o,
                                    const int32_t* kv_lens, int B, int Hq, int Hkv, int D,
                                    int S_cap, int max_kv_len, int group_size, float scale,
                                    void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_decode_shape(B, Hq, Hkv, D, S_cap, max_kv_len, scale);
  if (rc != GQA_OK) return rc;
  if (group_size != 64 || D % group_size != 0) return GQA_ERR_INVALID_ARG;
  if (S_cap % 8 != 0) return GQA_ERR_INVALID_ARG;  // scale/bias tiles are copied in 16-byte pieces
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  rc = check_ptrs({q, k_codes, v_codes, k_scale, k_bias, v_scale, v_bias, o}, dev, 16);
  if (rc != GQA_OK) return rc;
  if (kv_lens != nullptr) {
    rc = check_ptrs({kv_lens}, dev, 4);
    if (rc != GQA_OK) return rc;
  }
  if (workspace == nullptr) return GQA_ERR_WORKSPACE;
  rc = check_ptrs({workspace}, dev, 256);
  if (rc == GQA_ERR_INVALID_ARG) return GQA_ERR_WORKSPACE;
  if (rc != GQA_OK) return rc;

  DecodeQ4Args a;
  a.q = q;
  a.k_codes = k_codes;
  a.k_scale = k_scale;
  a.k_bias = k_bias;
  a.v_codes = v_codes;
  a.v_scale = v_scale;
  a.v_bias = v_bias;
  a.o = o;
  a.kv_lens = kv_lens;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.S_cap = S_cap;
  a.max_kv_len = max_kv_len;
  a.scale = scale;
  a.workspace = workspace;
  a.plan = plan_splits(B, Hq, Hkv, max_kv_len, decode_q4_tile_rows(D), device_sm_count(),
                       decode_q4_ctas_per_sm());
  if (ws_bytes < workspace_layout(B, Hq, Hkv, a.plan.n_hc, a.plan.n_split, D).total)
    return GQA_ERR_WORKSPACE;
  const cudaError_t e = launch_decode_q4(a, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return GQA_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return GQA_ERR_CUDA;
  return GQA_OK;
}

GQA_ATTN_API size_t gqa_attn_decode_q4_residual_workspace_size(int B, int Hq, int Hkv, int D,
                                                               int max_quant) {
  if (check_decode_shape(B, Hq, Hkv, D, max_quant, max_quant, 1.f) != GQA_OK) return 0;
  const SplitPlan p = plan_splits(B, Hq, Hkv, max_quant, decode_q4_tile_rows(D), device_sm_count(),
                                  decode_q4_ctas_per_sm());
  return workspace_layout(B, Hq, Hkv, p.n_hc, p.n_split + 1, D).total;
}

GQA_ATTN_API int gqa_attn_decode_q4_residual(
    const void* q, const uint8_t* k_codes, const uint16_t* k_scale, const uint16_t* k_bias,
    const uint8_t* v_codes, const uint16_t* v_scale, const uint16_t* v_bias, const void* k_res,
    const void* v_res, const int32_t* n_quant, const int32_t* kv_lens, void* o, int B, int Hq, int Hkv,
    int D, int S_cap, int R_cap, int max_quant, int group_size, float scale, void* workspace,
    size_t ws_bytes, void* stream) {
  int rc = check_decode_shape(B, Hq, Hkv, D, S_cap, max_quant, scale);
  if (rc != GQA_OK) return rc;
  if (R_cap < 1 || group_size != 64 || D % group_size != 0) return GQA_ERR_INVALID_ARG;
  if (S_cap % 8 != 0) return GQA_ERR_INVALID_ARG;  // scale/bias tiles are copied in 16-byte pieces
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  rc = check_ptrs({q, k_codes, v_codes, k_scale, k_bias, v_scale, v_bias, o, k_res, v_res}, dev, 16);
  if (rc != GQA_OK) return rc;
  rc = check_ptrs({n_quant, kv_lens}, dev, 4);
  if (rc != GQA_OK) return rc;
  if (workspace == nullptr) return GQA_ERR_WORKSPACE;
  rc = check_ptrs({workspace}, dev, 256);
  if (rc == GQA_ERR_INVALID_ARG) return GQA_ERR_WORKSPACE;
  if (rc != GQA_OK) return rc;

  DecodeQ4Args aq;
  aq.q = q;
  aq.k_codes = k_codes;
  aq.k_scale = k_scale;
  aq.k_bias = k_bias;
  aq.v_codes = v_codes;
  aq.v_scale = v_scale;
  aq.v_bias = v_bias;
  aq.o = o;
  aq.kv_lens = n_quant;
  aq.B = B;
  aq.Hq = Hq;
  aq.Hkv = Hkv;
  aq.D = D;
  aq.S_cap = S_cap;
  aq.max_kv_len = max_quant;
  aq.scale = scale;
  aq.workspace = workspace;
  aq.plan = plan_splits(B, Hq, Hkv, max_quant, decode_q4_tile_rows(D), device_sm_count(),
                        decode_q4_ctas_per_sm());
  if (ws_bytes < workspace_layout(B, Hq, Hkv, aq.plan.n_hc, aq.plan.n_split + 1, D).total)
    return GQA_ERR_WORKSPACE;

  DecodeArgs ar;  // the window: bf16 [B, Hkv, R_cap, D], one split per (request, head chunk)
  ar.q = q;
  ar.k = k_res;
  ar.v = v_res;
  ar.o = o;
  ar.kv_lens = kv_lens;
  ar.B = B;
  ar.Hq = Hq;
  ar.Hkv = Hkv;
  ar.D = D;
  ar.S_cap = R_cap;
  ar.max_kv_len = R_cap;
  ar.scale = scale;
  ar.dtype = GQA_BF16;
  ar.workspace = workspace;
  ar.plan = aq.plan;
  ar.plan.tile = decode_tile_rows(GQA_BF16, D, false, long(B) * Hkv * aq.plan.n_hc, R_cap);
  ar.plan.chunk = ((R_cap + ar.plan.tile - 1) / ar.plan.tile) * ar.plan.tile;
  ar.plan.n_split = 1;
  const cudaError_t e = launch_decode_q4_residual(aq, ar, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return GQA_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return GQA_ERR_CUDA;
  return GQA_OK;
}

GQA_ATTN_API int gqa_attn_prefill(const void* q, const void* k, const void* v, void* o, int B,
                                  int Hq, int Hkv, int D, int q_len, int kv_len, int S_cap,
                                  float scale, int causal, int dtype, void* stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (q_len < 1 || kv_len < 1 || kv_len > S_cap || q_len > kv_len) return GQA_ERR_INVALID_ARG;
  // grid: (B*Hq, pairs of 128-row query tiles), the second extent at most 65535
  if (long(B) * Hq > 0x7fffffffL || (long(q_len) + 255) / 256 > 65535) return GQA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return GQA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return GQA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return GQA_ERR_INVALID_ARG;
  if (dtype != GQA_F32 && dtype != GQA_BF16) return GQA_ERR_INVALID_ARG;
  if (dtype != GQA_BF16) return GQA_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  const int rc = check_ptrs({q, k, v, o}, dev, 16);
  if (rc != GQA_OK) return rc;
  PrefillArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.q_len = q_len;
  a.kv_len = kv_len;
  a.S_cap = S_cap;
  a.scale = scale;
  a.causal = causal;
  const cudaError_t e = launch_prefill(a, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return GQA_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return GQA_ERR_CUDA;
  return GQA_OK;
}

GQA_ATTN_API int gqa_attn_prefill_varlen(const void* q, const void* k, const void* v, void* o,
                                         const int32_t* q_lens, const int32_t* kv_lens, int B, int Hq,
                                         int Hkv, int D, int Tq_cap, int S_cap, float scale, int causal,
                                         int dtype, void* stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (Tq_cap < 1 || S_cap < 1) return GQA_ERR_INVALID_ARG;
  if (long(B) * Hq > 0x7fffffffL || (long(Tq_cap) + 255) / 256 > 65535) return GQA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return GQA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return GQA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return GQA_ERR_INVALID_ARG;
  if (dtype != GQA_F32 && dtype != GQA_BF16) return GQA_ERR_INVALID_ARG;
  if (dtype != GQA_BF16) return GQA_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  int rc = check_ptrs({q, k, v, o}, dev, 16);
  if (rc != GQA_OK) return rc;
  rc = check_ptrs({q_lens, kv_lens}, dev, 4);
  if (rc != GQA_OK) return rc;
  PrefillArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.q_len = Tq_cap;
  a.kv_len = S_cap;
  a.S_cap = S_cap;
  a.scale = scale;
  a.causal = causal;
  a.q_lens = q_lens;
  a.kv_lens = kv_lens;
  const cudaError_t e = launch_prefill(a, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return GQA_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return GQA_ERR_CUDA;
  return GQA_OK;
}

GQA_ATTN_API int gqa_attn_read_device_status(const void* workspace, uint32_t* out, void* stream) {
  if (workspace == nullptr || out == nullptr) return GQA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  if (!is_device_ptr(workspace, dev)) return GQA_ERR_NOT_DEVICE_PTR;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(out, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return GQA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GQA_ERR_CUDA;
  return GQA_OK;
}

GQA_ATTN_API int gqa_attn_clear_device_status(void* workspace, void* stream) {
  if (workspace == nullptr) return GQA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  if (!is_device_ptr(workspace, dev)) return GQA_ERR_NOT_DEVICE_PTR;
  if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GQA_ERR_CUDA;
  return GQA_OK;
}

}  // extern "C"
