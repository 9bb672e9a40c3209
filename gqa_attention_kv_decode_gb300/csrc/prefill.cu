// prefill.cu -- causal / chunked GQA prefill on tcgen05 tensor cores.
#include "gqa_attn.h"
#include "internal.h"

namespace gqa {
cudaError_t launch_prefill(const PrefillArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace gqa
