// Attention backward on the tcgen05 tensor cores (bf16, D in {64, 128}).
#pragma once
#include "attn_bwd.cuh"

namespace osf {
bool attn_bwd_tc_supported(const BwdProblem &p);
// dK/dV and dQ kernels (the row sums D_i must already be in p.dvec).
cudaError_t launch_attn_bwd_tc(const BwdProblem &p, cudaStream_t s);
}  // namespace osf
