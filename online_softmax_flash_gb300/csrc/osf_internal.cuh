// Internal declarations shared by libosf's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "osf.h"

namespace osf {

// log2(e): scores are kept in base-2 units, s2 = s * scale * log2(e), so every exponential is a
// single ex2 (the "exp(x) = exp2(log2(e) * x)" rewrite of the Triton-Puzzles write-up, Puzzle 8).
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device status word values (match osf_status).
constexpr int kStatusTimeout = OSF_ERR_TIMEOUT;

// ---------------------------------------------------------------- device helpers
// Wait until the grid this kernel was launched as a programmatic dependent of has completed and
// its memory is visible (a no-op for a kernel launched normally).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Merge two (m, l) softmax states (base-2 exponents): the boxed recurrence of
// "Softmax 算子的实现与优化", "Online Softmax", applied to a partial state instead of one block.
__device__ __forceinline__ void merge_ml(float &m, float &l, float m2, float l2) {
    float mn = fmaxf(m, m2);
    if (mn == -INFINITY) return;  // both empty
    l = l * ex2_approx(m - mn) + l2 * ex2_approx(m2 - mn);
    m = mn;
}

// ---------------------------------------------------------------- attention problem
struct AttnProblem {
    const void *q, *k, *v;
    void *o;
    float *lse;          // optional [B, Hq, Sq]
    int dtype;           // OSF_F32 / OSF_BF16
    int B, Hq, Hkv, Sq, Sk, D;
    int causal;          // 1: key j is visible to query row i iff j <= i + causal_off
    int causal_off;      // 0 (top-left) or Sk - Sq (bottom-right)
    float scale_log2;    // scale * log2(e)
    // element strides of the b, h and s dimensions of Q, K, V, O (d is contiguous)
    long long q_sb, q_sh, q_ss, k_sb, k_sh, k_ss, v_sb, v_sh, v_ss, o_sb, o_sh, o_ss;
    // split-K partial state workspace (float): acc [splits][B*Hq*Sq][D], m/l [splits][B*Hq*Sq]
    int splits;
    float *part_acc, *part_m, *part_l;
    void *x3_ws;         // fp32 on the tensor-core path: bf16 high / low parts of Q, K, V
    int *status;         // device status word
};

// Element offsets of row s of head h in batch b.
__host__ __device__ __forceinline__ long long q_at(const AttnProblem &p, int b, int h, long long s) {
    return b * p.q_sb + h * p.q_sh + s * p.q_ss;
}
__host__ __device__ __forceinline__ long long k_at(const AttnProblem &p, int b, int h, long long s) {
    return b * p.k_sb + h * p.k_sh + s * p.k_ss;
}
__host__ __device__ __forceinline__ long long v_at(const AttnProblem &p, int b, int h, long long s) {
    return b * p.v_sb + h * p.v_sh + s * p.v_ss;
}
__host__ __device__ __forceinline__ long long o_at(const AttnProblem &p, int b, int h, long long s) {
    return b * p.o_sb + h * p.o_sh + s * p.o_ss;
}

// SM count of the current device, looked up once per device (the same value every entry point
// sizes its grids and workspaces with).  Returns an osf_status.
int device_sm_count(int *sms);

// Count of kernels launched by the library (diagnostics; see osf_launch_count).
void count_launches(int n);
// Raise `kernel`'s dynamic shared-memory limit to at least `bytes` on the current device.  The
// attribute belongs to the device's context, so every device is configured on its first use
// there; the limit is only ever raised (a smaller request after a larger one keeps the larger
// limit); thread-safe, and a no-op when the limit already suffices.
cudaError_t set_max_dynamic_smem(const void *kernel, int bytes);

// Launch `kernel` as a programmatic dependent of the previous kernel in the stream: it is
// scheduled as soon as every block of that kernel has finished, without the launch gap, and
// must execute griddepcontrol.wait before it reads anything that kernel wrote (the wait returns
// once the previous grid has completed and its memory operations are visible).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Launch in thread-block clusters of shape `cluster` (the grid a multiple of it), as a
// programmatic dependent of the previous kernel when `dependent` (same contract as above).
template <typename... KArgs, typename... Args>
cudaError_t launch_clustered(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             dim3 cluster, bool dependent, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster.x;
    attr[0].val.clusterDim.y = cluster.y;
    attr[0].val.clusterDim.z = cluster.z;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Launchers (return cudaError_t of the launch).
cudaError_t launch_attn_simt(const AttnProblem &p, cudaStream_t s);
cudaError_t launch_attn_combine(const AttnProblem &p, cudaStream_t s);
size_t attn_simt_partial_floats(int splits, long long rows, int D);
int attn_simt_pick_splits(const AttnProblem &p, int sm_count);

cudaError_t launch_softmax_rows(const float *x, float *z, long long rows, long long T,
                                float *ws, int sm_count, cudaStream_t s);
size_t softmax_workspace_floats(long long rows, long long T, int sm_count);

}  // namespace osf
