// Tensor-core (tcgen05 / TMEM / TMA) attention prefill for bfloat16 Q/K/V.
#pragma once
#include "osf_internal.cuh"

namespace osf {
// True when the problem can run on the tensor-core prefill kernel (bf16, D in {64, 128},
// 16-byte aligned base pointers, Sq > 1).
bool attn_tc_supported(const AttnProblem &p, const void *Q, const void *K, const void *V, const void *O);
// Key-range split count that fills the GPU when there are fewer work items than SMs.
int attn_tc_pick_splits(const AttnProblem &p, int sm_count);
// Runs the kernel (and the log-sum-exp combine when p.splits > 1; partial pointers set).
cudaError_t launch_attn_tc(const AttnProblem &p, int sm_count, cudaStream_t s);
}  // namespace osf
