// bf16 cached-latent decode (tcgen05).  Under construction.
#include "internal.h"
namespace mla {
bool decode_bf16_supports(int, int, int) { return false; }
size_t decode_bf16_workspace_bytes(int, int, int, int, int) { return 0; }
cudaError_t launch_decode_bf16(const DecodeArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace mla
