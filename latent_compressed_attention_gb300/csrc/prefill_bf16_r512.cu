// bf16 absorbed prefill for r = 512, d_q = d_v = 128 (tcgen05).  Under construction.
#include "internal.h"
namespace mla {
bool prefill_bf16_r512_supports(int, int, int) { return false; }
cudaError_t launch_prefill_bf16_r512(const PrefillArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace mla
