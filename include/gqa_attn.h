/*
 * gqa_attn.h -- C ABI of libgqa_attn.so: fused grouped-query attention (GQA)
 * over a KV cache, hand-written for NVIDIA GB300 (sm_103a).
 *
 * The operation (all entry points): for request b, query head h and query
 * row i,
 *     O[b,h,i,:] = softmax_j( scale * Q[b,h,i,:] . K[b,g,j,:] ) V[b,g,j,:],
 *     g = h / (Hq / Hkv),
 * over the visible keys j < kv_len (and, when causal, j <= i + kv_len - q_len).
 * The kernels read the Hkv unexpanded KV heads directly: no repeat_kv copy
 * and no [Hq, q_len, kv_len] score matrix is ever written to memory.
 *   - "2x Faster Qwen2 Decode on Metal in Candle", section "Why It Matters:
 *     7x KV Expansion on Every Decode Step": the fused single-token kernel
 *     indexes the KV heads through the query/KV head ratio in one pass.
 *   - "Fused attention makes a 4,096-token Qwen2 prefill on Metal 4.5x
 *     faster", section "Cause and workaround", items 1-3: K and V are given
 *     before repeat_kv (Hq a multiple of Hkv); the causal mask aligns the
 *     queries to the end of the keys; the rows of each head are contiguous.
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE pointers (cudaMalloc / torch CUDA tensors) on the
 *     current device; the library never copies from host memory and has no
 *     CPU implementation.  A host pointer is rejected with
 *     GQA_ERR_NOT_DEVICE_PTR before anything is launched.
 *   - Layouts are dense, row-major:
 *        Q, O : [B, Hq, q_len, D]      (q_len = 1 for decode)
 *        K, V : [B, Hkv, S_cap, D]     rows of one head contiguous; head
 *                                      stride S_cap*D, batch stride Hkv*S_cap*D
 *     Only rows j < kv_len of K and V are read; rows past kv_len may hold
 *     anything, including NaN.  Every pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on that stream; the library never
 *     synchronises the device.  Kernels are launched with programmatic
 *     stream serialisation: each waits (griddepcontrol.wait) for the work
 *     before it in the stream before touching memory, and lets the next
 *     kernel begin launching early.  Work that follows in the stream sees the
 *     results as usual; a caller's own kernel launched with programmatic
 *     serialisation after a call must itself wait for its predecessor (as
 *     that launch mode always requires) before reading the outputs.
 *   - The library allocates no device memory.  Scratch memory (the split-KV
 *     partials) is a caller-owned `workspace` whose size the matching
 *     *_workspace_size() call returns for the current device.  Only its first
 *     4 bytes (the device status word) need to start at zero; every partial
 *     is written before it is read within a call.  Two calls that may run
 *     concurrently on the GPU must not share a workspace.  A decode call
 *     that splits the keys launches two kernels (splits, then merge).
 *   - Arguments are validated on the host before any launch; on failure the
 *     call returns a negative gqa_status_t and launches nothing.
 *   - The compute entry points may be called from several host threads at
 *     once, each call with its own outputs and workspace; the settings
 *     (plan override, wait limit, wait test) are process-wide and change
 *     only while no other thread is calling.  A calling thread with no
 *     current CUDA context gets the current device's primary context.
 *   - Per-request lengths that are out of range on the device are clamped
 *     and reported through a status word at the start of the workspace
 *     (GQA_DEV_* bits, OR-accumulated until cleared).
 */
#ifndef GQA_ATTN_H_
#define GQA_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GQA_ATTN_API __attribute__((visibility("default")))

typedef enum gqa_status {
  GQA_OK = 0,
  GQA_ERR_INVALID_ARG = -1,    /* bad shape, length, scale or pointer alignment */
  GQA_ERR_UNSUPPORTED = -2,    /* valid, but no kernel for this dtype / D        */
  GQA_ERR_NOT_DEVICE_PTR = -3, /* a pointer is not device memory                 */
  GQA_ERR_CUDA = -4,           /* a CUDA runtime call or launch failed            */
  GQA_ERR_WORKSPACE = -5,      /* workspace missing or too small                  */
  GQA_ERR_SCRATCH_LIMIT = -6   /* problem needs more than the built-in scratch    */
} gqa_status_t;

typedef enum gqa_dtype {
  GQA_F32 = 0,  /* Q, K, V, O in float32; fp32 arithmetic                         */
  GQA_BF16 = 1  /* Q, K, V, O in bfloat16; fp32 accumulation, output rounded RNE */
} gqa_dtype_t;

/* Device status bits (OR-accumulated in the first 4 bytes of a workspace). */
#define GQA_DEV_KVLEN_CLAMPED 1u /* some kv_lens[b] < 0 or > max_kv_len: clamped */
#define GQA_DEV_EMPTY_REQUEST 2u /* some kv_lens[b] == 0: that output is zeros    */
#define GQA_DEV_WAIT_TIMEOUT 4u  /* a bounded wait on a tile copy gave up          */
#define GQA_DEV_BAD_BLOCK 8u     /* a paged-cache block id was outside the pool    */

/* ---------------------------------------------------------------------------
 * Single-token decode (q_len = 1), split-KV with a log-sum-exp combine.
 *
 * Defines: the fused decode attention of "2x Faster Qwen2 Decode on Metal in
 * Candle" ("Why It Matters"; benchmark geometry of sections 2.1 and 2.2),
 * batched across requests with per-request lengths ("Batching Decode
 * Attention Across Requests ...", VeloxQuant-MLX blog, "Part 4": the B axis
 * of the fused decode-attend grid).
 *
 *   q        [B, Hq, 1, D]       dtype
 *   k, v     [B, Hkv, S_cap, D]  dtype
 *   o        [B, Hq, 1, D]       dtype (written)
 *   kv_lens  device int32 [B], number of valid rows per request; NULL means
 *            every request has max_kv_len rows.  A value < 0 or > max_kv_len
 *            is clamped into [0, max_kv_len] and sets GQA_DEV_KVLEN_CLAMPED;
 *            0 writes a zero output row and sets GQA_DEV_EMPTY_REQUEST.
 *   max_kv_len  host upper bound of kv_lens (1 <= max_kv_len <= S_cap); it
 *            sizes the grid and the workspace.
 *   scale    softmax scale, finite and > 0 (usually 1/sqrt(D)).
 *   dtype    GQA_F32 or GQA_BF16.   D in {64, 128}.   Hq % Hkv == 0.
 * Returns GQA_OK or a negative gqa_status_t.
 * ------------------------------------------------------------------------- */
GQA_ATTN_API size_t gqa_attn_decode_workspace_size(int B, int Hq, int Hkv, int D,
                                                   int max_kv_len, int dtype);

GQA_ATTN_API int gqa_attn_decode(const void* q, const void* k, const void* v, void* o,
                                 const int32_t* kv_lens, int B, int Hq, int Hkv, int D,
                                 int S_cap, int max_kv_len, float scale, int dtype,
                                 void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Single-token decode of n_layers layers in one launch (a microbenchmark).
 *
 * "Batching Decode Attention Across Requests Got Us 3.83x Real Throughput --
 * Across Layers Got Us Nothing", results 1 and 2: adding an outermost layer
 * axis to the decode grid replaces 28-80 launches by one and wins at the
 * kernel level, but a real decoder cannot use it, because layer l+1's query
 * needs layer l's complete output.  It is kept for measuring the per-launch
 * cost, not for model decoding.
 *
 * The caller stacks the layers along a leading axis:
 *   q, o  [n_layers, B, Hq, 1, D]     k, v  [n_layers, B, Hkv, S_cap, D]
 * (i.e. the gqa_attn_decode layouts with batch n_layers * B); kv_lens [B]
 * (or NULL) is shared by all layers.  The result equals, bit for bit, n_layers
 * gqa_attn_decode calls on the per-layer slices: every layer uses the split
 * plan of a one-layer call.  Workspace: gqa_attn_decode_layers_workspace_size.
 * n_layers * B <= 65535.  Other arguments and errors as for gqa_attn_decode.
 * ------------------------------------------------------------------------- */
GQA_ATTN_API size_t gqa_attn_decode_layers_workspace_size(int n_layers, int B, int Hq, int Hkv, int D,
                                                          int max_kv_len, int dtype);
GQA_ATTN_API int gqa_attn_decode_layers(const void* q, const void* k, const void* v, void* o,
                                        const int32_t* kv_lens, int n_layers, int B, int Hq, int Hkv,
                                        int D, int S_cap, int max_kv_len, float scale, int dtype,
                                        void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Single-token decode over a PAGED KV cache, with an optional fused append of
 * the new token.
 *
 * The decode kernel reads only the head stride of K and V and needs the rows
 * of a head next to each other; a cache kept in another layout had to be
 * copied first ("Fused attention makes a 4,096-token Qwen2 prefill on Metal
 * 4.5x faster", section "Cause and workaround", item 3).  Paged attention
 * (named in "2x Faster Qwen2 Decode on Metal in Candle", section "Why It
 * Matters", for the author's CPU engine) keeps the cache in fixed-size
 * blocks instead; the pages give no layout, so this one is the library's:
 *
 *   q            [B, Hq, 1, D]                       dtype
 *   k_pool,      [num_blocks, Hkv, block_size, D]    dtype; the rows of one
 *   v_pool                                            (block, KV head) are contiguous
 *   block_table  device int32 [B, max_blocks]: key row j of request b is row
 *                j % block_size of block block_table[b][j / block_size].
 *                Entries past the request's last block are never read.  An
 *                id outside [0, num_blocks) sets GQA_DEV_BAD_BLOCK; that
 *                request's output is then unspecified (no read leaves the pool).
 *   kv_lens      device int32 [B] (required): keys per request, counting the
 *                appended token; clamped like gqa_attn_decode's.
 *   k_new, v_new [B, Hkv, 1, D] dtype, or both NULL.  When given, the token of
 *                request b is written to key row kv_lens[b] - 1 (into the
 *                pools, which the call therefore modifies) and attended to in
 *                the same call.  Requests with kv_lens[b] == 0 write nothing.
 *   o            [B, Hq, 1, D] dtype (written)
 *   block_size   a positive multiple of the decode tile: 64 (bf16, or fp32
 *                with D = 128) or 128 (fp32 with D = 64); else
 *                GQA_ERR_UNSUPPORTED.
 *   max_kv_len   host upper bound of kv_lens, <= max_blocks * block_size.
 *   workspace    as for gqa_attn_decode (gqa_attn_decode_workspace_size with
 *                the same B, Hq, Hkv, D, max_kv_len, dtype).
 * Other arguments and errors as for gqa_attn_decode.
 * ------------------------------------------------------------------------- */
GQA_ATTN_API int gqa_attn_decode_paged(const void* q, const void* k_new, const void* v_new,
                                       void* k_pool, void* v_pool, const int32_t* block_table,
                                       const int32_t* kv_lens, void* o, int B, int Hq, int Hkv,
                                       int D, int block_size, int num_blocks, int max_blocks,
                                       int max_kv_len, float scale, int dtype, void* workspace,
                                       size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Prefill of a batch of requests with their own lengths (varlen, chunked).
 *
 * Serving mixes prefill chunks of many requests, each at its own position in
 * its own cache; gqa_attn_prefill takes one (q_len, kv_len) for the whole
 * batch.  Here request b has q_lens[b] queries aligned to the end of its
 * kv_lens[b] keys ("Fused attention makes a 4,096-token Qwen2 prefill on
 * Metal 4.5x faster", "Cause and workaround", item 2: with the causal mask a
 * chunk at an offset sees all earlier keys).
 *
 *   q, o      bf16 [B, Hq, Tq_cap, D]   rows [0, q_lens[b]) of request b
 *                                       (other rows of o are not written)
 *   k, v      bf16 [B, Hkv, S_cap, D]   rows [0, kv_lens[b]) of request b;
 *                                       rows past it may hold anything
 *   q_lens,   device int32 [B]; kv_lens[b] is clamped into [0, S_cap] and
 *   kv_lens   q_lens[b] into [0, min(Tq_cap, kv_lens[b])]
 *   causal    1: query i of request b sees keys j <= i + kv_lens[b] - q_lens[b];
 *             0: all kv_lens[b] keys
 * D = 64 or 128 (bf16).  Other errors as for gqa_attn_prefill.
 * ------------------------------------------------------------------------- */
GQA_ATTN_API int gqa_attn_prefill_varlen(const void* q, const void* k, const void* v, void* o,
                                         const int32_t* q_lens, const int32_t* kv_lens, int B, int Hq,
                                         int Hkv, int D, int Tq_cap, int S_cap, float scale, int causal,
                                         int dtype, void* stream);

/* ---------------------------------------------------------------------------
 * Decode over a 4-bit cache followed by an unquantized residual window.
 *
 * "Batching Decode Attention Across Requests ...", VeloxQuant-MLX blog,
 * "What this means in practice": the benchmark cache had no fp16 residual
 * window, and a production KIVI cache keeps the most recent tokens
 * unquantized.  Here the window is kept in bf16 (the dtype of q and o):
 * key rows [0, n_quant[b]) of request b come from the 4-bit cache (as in
 * gqa_attn_decode_q4) and key rows [n_quant[b], kv_lens[b]) from rows
 * [0, kv_lens[b] - n_quant[b]) of the window.  A block that ages out of the
 * window is moved into the 4-bit cache with gqa_attn_quantize_q4.
 *
 *   q, o          bf16 [B, Hq, 1, D]
 *   codes, scale, as for gqa_attn_decode_q4, [B, Hkv, S_cap, ...]
 *   bias (K, V)
 *   k_res, v_res  bf16 [B, Hkv, R_cap, D]
 *   n_quant       device int32 [B]: 4-bit rows per request, clamped into
 *                 [0, max_quant] (GQA_DEV_KVLEN_CLAMPED)
 *   kv_lens       device int32 [B]: all keys per request; the window part
 *                 kv_lens[b] - n_quant[b] is clamped into [0, R_cap]
 *   max_quant     host bound of n_quant, 1 <= max_quant <= S_cap
 * A request with no key at all gets a zero row (GQA_DEV_EMPTY_REQUEST).
 * Three kernels run (window, 4-bit splits, merge); the workspace size comes
 * from gqa_attn_decode_q4_residual_workspace_size(B, Hq, Hkv, D, max_quant).
 * Errors as for gqa_attn_decode_q4.
 * ------------------------------------------------------------------------- */
GQA_ATTN_API size_t gqa_attn_decode_q4_residual_workspace_size(int B, int Hq, int Hkv, int D,
                                                               int max_quant);
GQA_ATTN_API int gqa_attn_decode_q4_residual(
    const void* q, const uint8_t* k_codes, const uint16_t* k_scale, const uint16_t* k_bias,
    const uint8_t* v_codes, const uint16_t* v_scale, const uint16_t* v_bias, const void* k_res,
    const void* v_res, const int32_t* n_quant, const int32_t* kv_lens, void* o, int B, int Hq, int Hkv,
    int D, int S_cap, int R_cap, int max_quant, int group_size, float scale, void* workspace,
    size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * 4-bit group-affine quantization of KV rows (the cache format read by
 * gqa_attn_decode_q4).
 *
 * "Batching Decode Attention Across Requests ...", VeloxQuant-MLX blog,
 * "Part 4": quantizing the whole growing history every step cost more than
 * the attention; only the newly aged, group-aligned block of tokens should be
 * quantized each step.  This call quantizes rows [0, rows) of every head of
 * `src` into rows [dst_row0, dst_row0 + rows) of every head of the cache: a
 * whole cache after prefill, or one flushed block per decode step.
 *
 *   src     bf16 [heads, src_head_rows, D]      (heads = B * Hkv)
 *   codes   uint8 [heads, dst_head_rows, D/2]   element 2t in the low nibble
 *                                               of byte t (written)
 *   scale,  fp16 [heads, dst_head_rows, D/64]   (written)
 *   bias
 * Per group of group_size = 64 elements along D: scale = fp16((max - min) /
 * 15), bias = fp16(min), code = clamp(round_half_even((x - bias) / scale), 0,
 * 15), code 0 when scale == 0, where x - bias and the quotient are each the
 * correctly rounded IEEE fp32 result: the codes are a deterministic function
 * of the input, the direct inverse of x = code * scale + bias.  The source is expected to be finite: a NaN element is left out of
 * its group's minimum and maximum and gets code 0.  The pages give the format
 * x = code * scale + bias but no quantizer; this is the library's reading.
 * Rows of the cache outside [dst_row0, dst_row0 + rows) are not touched.
 * D in {64, 128}; src 16-byte and codes 4-byte aligned, scale and bias
 * 2-byte aligned; rows <= src_head_rows, dst_row0 + rows <= dst_head_rows.
 * Errors as for decode.
 * ------------------------------------------------------------------------- */
GQA_ATTN_API int gqa_attn_quantize_q4(const void* src, int64_t src_head_rows, uint8_t* codes,
                                      uint16_t* scale, uint16_t* bias, int64_t dst_head_rows,
                                      int64_t dst_row0, int heads, int rows, int D, int group_size,
                                      void* stream);

/* ---------------------------------------------------------------------------
 * Plan overrides, for tuning and tests only.
 *
 * decode_splits > 0 makes every later decode call (all decode entry points
 * and their *_workspace_size queries) cut each request's keys into that many
 * splits instead of the planner's count (a split still holds at least one
 * tile, and there are at most 1024).  prefill_kv_split in [1, 8] forces the
 * size of the thread-block cluster that shares one query-tile pair's keys in
 * prefill (1 = no split).  0 restores the planner's choice for either.  The
 * setting is process-wide and starts at 0; nothing else (no environment
 * variable) changes a plan.  Change it only while no other thread is calling
 * the library, and size workspaces after changing it.
 * Returns GQA_OK, or GQA_ERR_INVALID_ARG for a negative value or a
 * prefill_kv_split above 8.
 * ------------------------------------------------------------------------- */
GQA_ATTN_API int gqa_attn_set_plan_override(int decode_splits, int prefill_kv_split);

/* Prefill work units, for tuning and tests only.  Prefill runs the 128-row
 * query tiles of a head in pairs (two tiles over the same keys) and, for the
 * longest causal tiles, one tile per CTA whose keys the CTA's two softmax
 * warpgroups take in turn (halving the tile's iterations); the planner picks
 * the first pair run that way.  from_pair >= 0 forces it: pairs from index
 * from_pair on (pair p holds tiles 2p and 2p+1) run as single tiles, so 0
 * makes every tile a single-tile unit and a value past the last pair turns
 * them off.  A negative value restores the planner's choice (the initial
 * setting).  Cluster-split prefill (see above) and per-request lengths
 * always use pairs.  Same threading rules as gqa_attn_set_plan_override.
 * Returns GQA_OK. */
GQA_ATTN_API int gqa_attn_set_prefill_interleave_override(int from_pair);

/* Failure-path test of the kernels, for tests only.  Every wait of a kernel
 * on a copy or a product gives up after 1 s; the CTA then lets the copies it
 * issued land (waiting with the same 1 s limit) and returns, leaving the
 * context usable: a decode CTA writes no partials and sets
 * GQA_DEV_WAIT_TIMEOUT in the workspace status word, a prefill CTA writes its
 * output rows as NaN and sets GQA_DEV_WAIT_TIMEOUT in the prefill status word.
 * With stall_ns > 0 every later launch of gqa_attn_decode, _decode_paged,
 * _decode_layers, _decode_q4, _decode_q4_residual, _prefill and
 * _prefill_varlen makes the thread that issues a CTA's copies, once it has
 * issued its first ones, wait stall_ns on a barrier that nothing arrives on
 * and give up, so that this path runs deterministically: the call reports
 * GQA_DEV_WAIT_TIMEOUT and its outputs are unspecified (a prefill CTA whose
 * copies were all issued before the stall may finish its rows normally).
 * 0 (the initial setting) turns it off.  stall_ns > 10^9 returns GQA_ERR_INVALID_ARG;
 * otherwise GQA_OK.  Same threading rules as gqa_attn_set_plan_override. */
GQA_ATTN_API int gqa_attn_set_wait_test(uint64_t stall_ns);

/* ---------------------------------------------------------------------------
 * Single-token decode without any caller-provided or allocated scratch.
 *
 * There is no counterpart of this entry point in the pages; it exists for
 * callers that cannot allocate device memory (for example a runtime that only
 * hands out the input and output buffers it owns, or code queued while its
 * allocator is unavailable).  It computes exactly what gqa_attn_decode
 * computes, with the same arguments minus the workspace, using a scratch array
 * of GQA_ATTN_NOALLOC_SCRATCH_BYTES compiled into the library: every GPU that
 * loads the library holds that array until the process exits.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.  The address is kept for the life of the
 *     process and belongs to the device's primary context (the one the CUDA
 *     runtime uses): after cudaDeviceReset, or from another driver-API
 *     context, do not call this entry point again in the same process.
 *   - Arguments are checked as gqa_attn_decode checks them, with the same
 *     error codes, before the size limit below.
 *   - Problems whose workspace (gqa_attn_decode_workspace_size) exceeds the
 *     array are rejected with GQA_ERR_SCRATCH_LIMIT before anything runs.
 *   - All calls share the array.  Calls whose GPU work may overlap (other
 *     streams, other host threads) race on it; serialise them.
 *   - It allocates nothing and calls no allocating routine.  The device status
 *     word of gqa_attn_decode is kept in the array and is not reported.
 * ------------------------------------------------------------------------- */
#define GQA_ATTN_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

GQA_ATTN_API int gqa_attn_decode_noalloc(const void* q, const void* k, const void* v, void* o,
                                         const int32_t* kv_lens, int B, int Hq, int Hkv, int D,
                                         int S_cap, int max_kv_len, float scale, int dtype,
                                         void* stream);

/* ---------------------------------------------------------------------------
 * Single-token decode over a 4-bit group-affine quantized KV cache, with the
 * dequantisation done inside the attention loop (no fp16/bf16 copy of the
 * cache is made).
 *
 * Defines: the fused group-affine decode-attend of "Batching Decode Attention
 * Across Requests Got Us 3.83x ..." (VeloxQuant-MLX blog, "The setup" and
 * "Part 4": codes, per-group scales and biases, GROUP_SIZE, a B axis).
 * Element d of a cached row is x = code[d] * scale[d / G] + bias[d / G].
 *
 *   q        bf16 [B, Hq, 1, D];  o bf16 [B, Hq, 1, D] (written)
 *   k_codes, v_codes  uint8 [B, Hkv, S_cap, D/2]: element 2t in the low
 *            nibble of byte t, element 2t+1 in the high nibble
 *   k_scale, k_bias, v_scale, v_bias  fp16 (raw uint16 bits)
 *            [B, Hkv, S_cap, D/G]
 *   group_size  G, must be 64;  D in {64, 128};  S_cap a multiple of 8
 *   kv_lens, max_kv_len, scale, workspace, stream: as gqa_attn_decode.
 * ------------------------------------------------------------------------- */
GQA_ATTN_API size_t gqa_attn_decode_q4_workspace_size(int B, int Hq, int Hkv, int D,
                                                      int max_kv_len);

GQA_ATTN_API int gqa_attn_decode_q4(const void* q, const uint8_t* k_codes,
                                    const uint16_t* k_scale, const uint16_t* k_bias,
                                    const uint8_t* v_codes, const uint16_t* v_scale,
                                    const uint16_t* v_bias, void* o, const int32_t* kv_lens,
                                    int B, int Hq, int Hkv, int D, int S_cap, int max_kv_len,
                                    int group_size, float scale, void* workspace,
                                    size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Prefill (q_len >= 1 query rows per request), causal or not, on the
 * tcgen05 tensor cores with accumulators in tensor memory.
 *
 * Defines: the fused causal prefill of "Fused attention makes a 4,096-token
 * Qwen2 prefill on Metal 4.5x faster" ("Cause and workaround"): one pass
 * over the grouped KV heads, causal mask inside the kernel, queries aligned
 * to the END of the keys, so a chunk of q_len queries at offset
 * kv_len - q_len sees every earlier key (chunked prefill).
 *
 *   q, o     bf16 [B, Hq, q_len, D];  k, v  bf16 [B, Hkv, S_cap, D]
 *   kv_len   keys visible to the last query row (q_len <= kv_len <= S_cap),
 *            the same for every request
 *   causal   1: key j visible to query row i iff j <= i + kv_len - q_len;
 *            0: every key j < kv_len visible
 *   dtype    GQA_BF16 (fp32 accumulation).   D == 64 or 128.
 *   limits   q_len <= 65535 * 256, B * Hq < 2^31 (else GQA_ERR_INVALID_ARG).
 * Errors: as for decode; a dtype / D without a kernel is GQA_ERR_UNSUPPORTED.
 * Nothing is allocated; the call is asynchronous on `stream`.
 * Device-side anomalies of both prefill entry points go to the prefill
 * status word of the device (see gqa_attn_read_prefill_status): a tile copy
 * that does not arrive within the kernel's bounded wait sets
 * GQA_DEV_WAIT_TIMEOUT and the affected output rows are written as NaN
 * (never as plausible values); per-request lengths that had to be clamped
 * (varlen) set GQA_DEV_KVLEN_CLAMPED.
 * ------------------------------------------------------------------------- */
GQA_ATTN_API int gqa_attn_prefill(const void* q, const void* k, const void* v, void* o,
                                  int B, int Hq, int Hkv, int D, int q_len, int kv_len,
                                  int S_cap, float scale, int causal, int dtype,
                                  void* stream);

/* ---------------------------------------------------------------------------
 * Helpers
 * ------------------------------------------------------------------------- */
/* Static, human-readable name of a gqa_status_t. */
GQA_ATTN_API const char* gqa_attn_status_string(int status);

/* Copies the device status word of `workspace` to *out after the work queued
 * on `stream` so far has finished (synchronises that stream). */
GQA_ATTN_API int gqa_attn_read_device_status(const void* workspace, uint32_t* out,
                                             void* stream);

/* Zeroes the device status word of `workspace` (asynchronous on `stream`). */
GQA_ATTN_API int gqa_attn_clear_device_status(void* workspace, void* stream);

/* Prefill has no workspace; its device status lives in the library: one
 * 32-bit word per device (GQA_DEV_* bits, starting at 0), OR-accumulated by
 * every gqa_attn_prefill / gqa_attn_prefill_varlen kernel on that device,
 * whatever its stream, until cleared.  read copies it to *out after the work
 * queued on `stream` so far has finished (synchronises that stream; out must
 * not be NULL); clear zeroes it in stream order and also synchronises.  For
 * flags per call, clear before the call and read after it on the same
 * stream, with no other prefill running on the device in between. */
GQA_ATTN_API int gqa_attn_read_prefill_status(uint32_t* out, void* stream);
GQA_ATTN_API int gqa_attn_clear_prefill_status(void* stream);

/* Number of splits along the keys the decode entry points use for this
 * problem on the current device (the grid's x extent); exposed for tests.
 * A request with fewer keys than max_kv_len may use fewer of them; when the
 * grid is a single wave it spreads its keys over all of them. */
GQA_ATTN_API int gqa_attn_decode_num_splits(int B, int Hq, int Hkv, int D, int max_kv_len,
                                            int dtype);

/* Which decode kernel a plan is for (gqa_attn_decode_plan_for). */
typedef enum gqa_plan_variant {
  GQA_PLAN_DECODE = 0, /* gqa_attn_decode (contiguous cache), dtype GQA_F32 or GQA_BF16  */
  GQA_PLAN_PAGED = 1,  /* gqa_attn_decode_paged, dtype GQA_F32 or GQA_BF16             */
  GQA_PLAN_Q4 = 2      /* gqa_attn_decode_q4 (4-bit cache; bf16 queries), dtype GQA_BF16 */
} gqa_plan_variant_t;

/* The split plan the decode kernel of `variant` would use on a device with
 * num_sms SMs, computed on the host (no GPU needed; for tests of the
 * planner).  Writes the grid's split count, the rows per split that count
 * towards a request's splits, and the kernel's tile height, to host memory:
 * a request of L keys uses min(n_split, ceil(L / chunk)) splits and deals
 * its tiles to them round-robin.  GQA_ERR_INVALID_ARG for a shape the decode
 * entry points reject, an unknown variant, a non-positive num_sms or a null
 * output; GQA_ERR_UNSUPPORTED for a dtype the variant has no kernel for. */
GQA_ATTN_API int gqa_attn_decode_plan_for(int B, int Hq, int Hkv, int D, int max_kv_len, int dtype,
                                          int variant, int num_sms, int32_t* n_split, int32_t* chunk,
                                          int32_t* tile);

/* ABI version (major * 100 + minor). */
GQA_ATTN_API int gqa_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H_ */
