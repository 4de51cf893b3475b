#include "decode.cuh"

namespace osf {
bool decode_supported(const AttnProblem &, const void *, const void *, const void *, const void *) {
    return false;
}
int decode_pick_splits(const AttnProblem &, int, int requested) { return requested > 0 ? requested : 1; }
size_t decode_workspace_bytes(const AttnProblem &, int) { return 0; }
cudaError_t launch_decode(AttnProblem &, void *, int, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace osf
