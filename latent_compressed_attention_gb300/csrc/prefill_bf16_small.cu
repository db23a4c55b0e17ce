// bf16 absorbed prefill for small latent ranks (tcgen05).  Under construction.
#include "internal.h"
namespace mla {
bool prefill_bf16_small_supports(int, int, int) { return false; }
cudaError_t launch_prefill_bf16_small(const PrefillArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace mla
