// Attention backward (dQ, dK, dV from Q, K, V, O, dO and the saved log-sum-exp).
#pragma once
#include "osf_internal.cuh"

namespace osf {
struct BwdProblem {
    const void *q, *k, *v, *o, *dout;
    const float *lse;      // [B, Hq, Sq] natural-log log-sum-exp of the forward pass
    void *dq, *dk, *dv;
    int dtype;             // OSF_F32 / OSF_BF16
    int B, Hq, Hkv, Sq, Sk, D;
    int causal, causal_off;  // key j visible to row i iff !causal || j <= i + causal_off
    float scale, scale_log2;
    float *dvec;           // workspace [B, Hq, Sq]: rowsum(dO * O)
    // optional workspace (tensor-core path): dS^T as bf16 [128 x 128] tiles, tile (bh, key tile,
    // query tile) at ((bh * ds_rows / 128 + key tile) * ds_ld / 128 + query tile) * 32 KB, each
    // [128 keys][128 queries]; ds_rows and ds_ld the key and query counts rounded up to 128.
    // null: dQ recomputes S and dP instead
    void *ds;
    long long ds_rows, ds_ld;
    int *status;
};
// True when the bf16 tensor-core (mma.sync) kernels handle the problem.
bool attn_bwd_mma_supported(const BwdProblem &p);
cudaError_t launch_attn_bwd(const BwdProblem &p, cudaStream_t s);
}  // namespace osf
