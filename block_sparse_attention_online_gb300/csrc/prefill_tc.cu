// bf16 tensor-core prefill (tcgen05 / TMEM / TMA) -- under construction.
#include "internal.h"

namespace attn_skip {
cudaError_t launch_prefill_tc(const PrefillArgs &, cudaStream_t) { return cudaErrorNotYetImplemented; }
}  // namespace attn_skip
