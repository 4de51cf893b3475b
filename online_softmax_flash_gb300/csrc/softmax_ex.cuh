// Scaled, optionally causal row softmax on float32 / bfloat16 strided rows (osf_softmax_rows_ex).
#pragma once
#include "osf_internal.cuh"

namespace osf {
struct SoftmaxExProblem {
    const void *x;
    void *z;
    int x_dtype, z_dtype;   // OSF_F32 / OSF_BF16
    long long rows, T;
    long long xs, zs;       // row strides in elements
    float mult;             // scale * log2(e)
    long long period;       // causal period (0: no mask)
    int sm_count;
    int *status;            // device status word (bounded-wait expiry)
};
void softmax_ex_chunk_geometry(long long rows, long long T, int sm_count, long long &chunk, int &nch);
size_t softmax_ex_workspace_floats(long long rows, long long T, int sm_count);
cudaError_t launch_softmax_ex(const SoftmaxExProblem &q, float *ws, cudaStream_t s);
}  // namespace osf
