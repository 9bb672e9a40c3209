// decode_q4.cu -- single-token GQA decode over a 4-bit group-affine KV cache.
#include "gqa_attn.h"
#include "internal.h"

namespace gqa {
int decode_q4_tile_rows(int D) { return 64; }
cudaError_t launch_decode_q4(const DecodeQ4Args&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace gqa
