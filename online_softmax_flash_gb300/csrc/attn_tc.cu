#include "attn_tc.cuh"

namespace osf {
bool attn_tc_supported(const AttnProblem &, const void *, const void *, const void *, const void *) {
    return false;
}
cudaError_t launch_attn_tc(const AttnProblem &, int, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace osf
