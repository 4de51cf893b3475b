// Tensor-core (tcgen05 / TMEM / TMA) attention prefill for bfloat16 Q/K/V, and for float32
// Q/K/V with D = 64 through bf16 high / low parts (x3 mode).
#pragma once
#include "osf_internal.cuh"

namespace osf {
// True when the problem can run on the tensor-core prefill kernel: Sq > 1 and either bf16 with
// D in {64, 128} and 16-byte aligned, TMA-addressable tensors, or float32 with D = 64 and an O
// whose rows start on 16-byte boundaries.
bool attn_tc_supported(const AttnProblem &p, const void *Q, const void *K, const void *V, const void *O);
// Workspace bytes the kernel needs beyond the split partial states (the x3 operand parts).
size_t attn_tc_extra_bytes(const AttnProblem &p);
// Key-range split count that fills the GPU when there are fewer work items than SMs.
int attn_tc_pick_splits(const AttnProblem &p, int sm_count);
// Runs the kernel (and the log-sum-exp combine when p.splits > 1; partial pointers set).
cudaError_t launch_attn_tc(const AttnProblem &p, int sm_count, cudaStream_t s);
}  // namespace osf
