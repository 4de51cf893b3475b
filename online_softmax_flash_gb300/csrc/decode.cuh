// Split-K decode (Sq == 1) for bfloat16 K/V caches, with a log-sum-exp combine.
#pragma once
#include "osf_internal.cuh"

namespace osf {
bool decode_supported(const AttnProblem &p, const void *Q, const void *K, const void *V, const void *O);
// Chunks per (batch, kv head): `requested` if > 0, else about four waves of CTAs.
int decode_pick_splits(const AttnProblem &p, int sm_count, int requested);
// Runs the kernel (and the log-sum-exp combine when p.splits > 1; partial pointers set).
cudaError_t launch_decode(const AttnProblem &p, cudaStream_t s);
}  // namespace osf
