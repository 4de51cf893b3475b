// Split-K decode (Sq == 1) for bfloat16 K/V caches, with a log-sum-exp combine.
#pragma once
#include "osf_internal.cuh"

namespace osf {
bool decode_supported(const AttnProblem &p, const void *Q, const void *K, const void *V, const void *O);
int decode_pick_splits(const AttnProblem &p, int sm_count, int requested);
size_t decode_workspace_bytes(const AttnProblem &p, int splits);
cudaError_t launch_decode(AttnProblem &p, void *workspace, int sm_count, cudaStream_t s);
}  // namespace osf
