// Row softmax z = exp(x - m) / l on float32 rows, built on the online (m, l) recurrence.
//
// Sources: Triton-Puzzles write-up (fadingcoder.top/post/105980), "Puzzle 8: Long Softmax"
// (two-loop online form); "Softmax 算子的实现与优化" (blog.euler0525.cn/posts/5db73590),
// "Online Softmax" (the boxed recurrence m' = max(m, m_b), l' = l e^(m - m') + sum e^(x - m'),
// and its invariant l = sum_j e^(x_j - m)) and "CUDA 版本" (warp-shuffle / shared-memory
// two-level reductions).
//
// Two paths:
//  * on-chip rows (T <= 32768, T % 4 == 0, 16-byte aligned): one CTA of up to 1024 threads
//    holds the whole row in registers (up to 8 float4 per thread).  Each thread reduces its
//    values to a local (m, l); the CTA merges the states with the recurrence, and the outputs
//    are produced from the registers: one HBM read and one HBM write per element, instead of
//    the two reads of the pages' single-program loop (the row fits on chip).  Where such a CTA
//    is alone on its SM (by its register use, rows of more than about 13000 elements),
//    persistent CTAs walk the rows and prefetch each next row into L2 while they reduce and
//    write the current one.
//  * chunked rows (longer rows, e.g. the 1-D vector, or unaligned data): kernel 1 splits each
//    row into chunks, one CTA per chunk, and writes each chunk's (m, l); kernel 2 merges a
//    row's chunk states and normalises its chunk -- the pages' two passes (two reads, one
//    write), spread over the whole GPU instead of one program.  Kernel 2 walks its chunk
//    backwards so the part kernel 1 read last is still in L2.
//
// All exponentials are base 2 on x * log2(e).
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "osf_internal.cuh"
#include "sm100_ptx.cuh"

namespace osf {
namespace {

constexpr int kMaxResidentT = 32768;
constexpr int kChunkThreads = 512;

// CTA-wide merge of per-thread (m, l) states; result broadcast to every thread.
__device__ __forceinline__ void block_merge_ml(float &m, float &l, float *sh /* 2*32 */) {
    // warp level: merge with shuffles
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
        merge_ml(m, l, m2, l2);
    }
    const int W = (blockDim.x + 31) >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (W > 1) {
        if (lane == 0) { sh[warp] = m; sh[32 + warp] = l; }
        __syncthreads();
        m = lane < W ? sh[lane] : -INFINITY;
        l = lane < W ? sh[32 + lane] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
            const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
            merge_ml(m, l, m2, l2);
        }
    }
}

// One CTA per row; thread t holds float4 number t + k*blockDim (k < VPT) of the row.
template <int VPT>
__global__ void __launch_bounds__(1024, 1)
softmax_rows_onchip_kernel(const float *__restrict__ x, float *z, int T) {
    __shared__ float sh[64];
    const int nvec = T >> 2;
    const size_t row = blockIdx.x;
    const float4 *xr = reinterpret_cast<const float4 *>(x + row * (size_t)T);
    float4 *zr = reinterpret_cast<float4 *>(z + row * (size_t)T);

    float4 v[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = threadIdx.x + k * blockDim.x;
        v[k] = i < nvec ? __ldcs(xr + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
    // local state: m = max, then e = 2^(x*log2e - m) kept in registers, l = sum e
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        v[k].x *= kLog2e; v[k].y *= kLog2e; v[k].z *= kLog2e; v[k].w *= kLog2e;
        m = fmaxf(m, fmaxf(fmaxf(v[k].x, v[k].y), fmaxf(v[k].z, v[k].w)));
    }
    const float mref = (m == -INFINITY) ? 0.f : m;
    float l = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        v[k].x = ex2_approx(v[k].x - mref); v[k].y = ex2_approx(v[k].y - mref);
        v[k].z = ex2_approx(v[k].z - mref); v[k].w = ex2_approx(v[k].w - mref);
        l += (v[k].x + v[k].y) + (v[k].z + v[k].w);
    }
    float M = m, L = l;
    block_merge_ml(M, L, sh);
    // z = e * 2^(m - M) / L
    const float f = (m == -INFINITY) ? 0.f : ex2_approx(m - M) / L;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = threadIdx.x + k * blockDim.x;
        if (i < nvec) {
            float4 o = v[k];
            o.x *= f; o.y *= f; o.z *= f; o.w *= f;
            __stcs(zr + i, o);
        }
    }
}

// Persistent form of the on-chip kernel: CTA b takes rows b, b + gridDim.x, ...; before it
// reduces a row it asks the bulk-copy engine to prefetch its next row into L2, so the HBM read
// of that row runs while this one is reduced and written (a CTA holding a whole row in
// registers is otherwise alone on its SM and leaves HBM idle between its read and its writes).
template <int VPT>
__global__ void __launch_bounds__(1024, 1)
softmax_rows_resident_kernel(const float *__restrict__ x, float *z, long long rows, int T) {
    __shared__ float sh[2][64];
    const int nvec = T >> 2;
    const uint32_t row_bytes = (uint32_t)T * 4u;
    int par = 0;
    for (long long row = blockIdx.x; row < rows; row += gridDim.x, par ^= 1) {
        const float4 *xr = reinterpret_cast<const float4 *>(x + row * (long long)T);
        float4 *zr = reinterpret_cast<float4 *>(z + row * (long long)T);
        if (threadIdx.x == 0 && row + gridDim.x < rows)
            ptx::prefetch_l2_bulk(x + (row + gridDim.x) * (long long)T, row_bytes);
        float4 v[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int i = threadIdx.x + k * blockDim.x;
            v[k] = i < nvec ? __ldcs(xr + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            v[k].x *= kLog2e; v[k].y *= kLog2e; v[k].z *= kLog2e; v[k].w *= kLog2e;
            m = fmaxf(m, fmaxf(fmaxf(v[k].x, v[k].y), fmaxf(v[k].z, v[k].w)));
        }
        const float mref = (m == -INFINITY) ? 0.f : m;
        float l = 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            v[k].x = ex2_approx(v[k].x - mref); v[k].y = ex2_approx(v[k].y - mref);
            v[k].z = ex2_approx(v[k].z - mref); v[k].w = ex2_approx(v[k].w - mref);
            l += (v[k].x + v[k].y) + (v[k].z + v[k].w);
        }
        float M = m, L = l;
        block_merge_ml(M, L, sh[par]);   // alternate halves: no barrier needed between rows
        const float f = (m == -INFINITY) ? 0.f : ex2_approx(m - M) / L;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int i = threadIdx.x + k * blockDim.x;
            if (i < nvec) {
                float4 o = v[k];
                o.x *= f; o.y *= f; o.z *= f; o.w *= f;
                __stcs(zr + i, o);
            }
        }
    }
}

// (m, l) over x[c0, c1) for this thread's share (stride blockDim.x), merged over the CTA.
template <bool VEC4>
__device__ __forceinline__ void range_state(const float *__restrict__ xr, long long c0, long long c1,
                                            float &m, float &l, float *sh) {
    m = -INFINITY;
    l = 0.f;
    if (VEC4) {
        const float4 *x4 = reinterpret_cast<const float4 *>(xr + c0);
        const long long n4 = (c1 - c0) >> 2;
        for (long long i = threadIdx.x; i < n4; i += blockDim.x) {
            float4 a = __ldg(x4 + i);
            a.x *= kLog2e; a.y *= kLog2e; a.z *= kLog2e; a.w *= kLog2e;
            const float mn = fmaxf(m, fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)));
            const float mr = (mn == -INFINITY) ? 0.f : mn;
            l = l * ex2_approx(m - mr) +
                ((ex2_approx(a.x - mr) + ex2_approx(a.y - mr)) + (ex2_approx(a.z - mr) + ex2_approx(a.w - mr)));
            m = mn;
        }
    } else {
        for (long long i = c0 + threadIdx.x; i < c1; i += blockDim.x) {
            const float a = __ldg(xr + i) * kLog2e;
            const float mn = fmaxf(m, a);
            const float mr = (mn == -INFINITY) ? 0.f : mn;
            l = l * ex2_approx(m - mr) + ex2_approx(a - mr);
            m = mn;
        }
    }
    block_merge_ml(m, l, sh);
}

// z[c0, c1) = 2^(x log2e - m) / l, walking from c1 down to c0.
template <bool VEC4>
__device__ __forceinline__ void range_norm(const float *xr, float *zr, long long c0, long long c1,
                                           float m, float l) {
    const float mref = (m == -INFINITY) ? 0.f : m;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    if (VEC4) {
        const float4 *x4 = reinterpret_cast<const float4 *>(xr + c0);
        float4 *z4 = reinterpret_cast<float4 *>(zr + c0);
        const long long n4 = (c1 - c0) >> 2;
        // four loads in flight per thread, then their four results
        const long long step = (long long)blockDim.x;
        long long i = n4 - 1 - threadIdx.x;
        for (; i - 3 * step >= 0; i -= 4 * step) {
            float4 a[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) a[u] = x4[i - u * step];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float4 o;
                o.x = ex2_approx(a[u].x * kLog2e - mref) * inv;
                o.y = ex2_approx(a[u].y * kLog2e - mref) * inv;
                o.z = ex2_approx(a[u].z * kLog2e - mref) * inv;
                o.w = ex2_approx(a[u].w * kLog2e - mref) * inv;
                __stcs(z4 + i - u * step, o);
            }
        }
        for (; i >= 0; i -= step) {
            const float4 a = x4[i];
            float4 o;
            o.x = ex2_approx(a.x * kLog2e - mref) * inv;
            o.y = ex2_approx(a.y * kLog2e - mref) * inv;
            o.z = ex2_approx(a.z * kLog2e - mref) * inv;
            o.w = ex2_approx(a.w * kLog2e - mref) * inv;
            __stcs(z4 + i, o);
        }
    } else {
        for (long long i = c1 - 1 - threadIdx.x; i >= c0; i -= blockDim.x)
            zr[i] = ex2_approx(xr[i] * kLog2e - mref) * inv;
    }
}

// Rows that are not held on chip but need no workspace: one CTA per row, two passes.
__global__ void __launch_bounds__(kChunkThreads)
softmax_row_stream_kernel(const float *x, float *z, long long T) {
    __shared__ float sh[64];
    const float *xr = x + (long long)blockIdx.x * T;
    float m, l;
    range_state<false>(xr, 0, T, m, l, sh);
    range_norm<false>(xr, z + (long long)blockIdx.x * T, 0, T, m, l);
}

// Chunked path, kernel 1: (m, l) of chunk blockIdx.x of row blockIdx.y.
template <bool VEC4>
__global__ void __launch_bounds__(kChunkThreads)
softmax_chunk_state_kernel(const float *__restrict__ x, long long T, long long chunk, float2 *ws) {
    __shared__ float sh[64];
    const long long row = blockIdx.y;
    const long long c0 = (long long)blockIdx.x * chunk;
    const long long c1 = min(T, c0 + chunk);
    float m, l;
    range_state<VEC4>(x + row * T, c0, c1, m, l, sh);
    if (threadIdx.x == 0) ws[row * gridDim.x + blockIdx.x] = make_float2(m, l);
}

// Chunked path, kernel 2: merge the row's chunk states, then write z for this chunk
// (walking the chunk from its end so the tail kernel 1 read last is served from L2).
template <bool VEC4>
__global__ void __launch_bounds__(kChunkThreads)
softmax_chunk_norm_kernel(const float *x, float *z, long long T, long long chunk,
                          const float2 *__restrict__ ws) {
    griddep_wait();   // launched as a dependent of the chunk-state kernel
    __shared__ float sh[64];
    const long long row = blockIdx.y;
    const int nch = gridDim.x;
    float m = -INFINITY, l = 0.f;
    for (int c = threadIdx.x; c < nch; c += blockDim.x) {
        const float2 st = ws[row * nch + c];
        merge_ml(m, l, st.x, st.y);
    }
    block_merge_ml(m, l, sh);
    const long long c0 = (long long)blockIdx.x * chunk;
    const long long c1 = min(T, c0 + chunk);
    range_norm<VEC4>(x + row * T, z + row * T, c0, c1, m, l);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool onchip_ok(const float *x, const float *z, long long T) {
    return T <= kMaxResidentT && (T & 3) == 0 && aligned16(x) && aligned16(z);
}

// chunk geometry for the chunked path
void chunk_geometry(long long rows, long long T, int sm_count, long long &chunk, int &nch) {
    // aim for ~4 resident CTAs per SM over the whole problem, chunks of >= 8192 elements
    const long long target_ctas = 4LL * sm_count;
    long long per_row = (target_ctas + rows - 1) / rows;
    const long long max_per_row = (T + 8191) / 8192;
    if (per_row > max_per_row) per_row = max_per_row;
    if (per_row < 1) per_row = 1;
    if (per_row > 65535) per_row = 65535;
    chunk = (T + per_row - 1) / per_row;
    chunk = (chunk + 3) & ~3LL;  // keep chunk starts 16-byte aligned
    nch = (int)((T + chunk - 1) / chunk);
}

}  // namespace

size_t softmax_workspace_floats(long long rows, long long T, int sm_count) {
    // rows held on chip or streamed by one CTA need nothing; the chunked path (rows longer
    // than kMaxResidentT) one float2 per chunk
    if (T <= kMaxResidentT) return 0;
    long long chunk;
    int nch;
    chunk_geometry(rows, T, sm_count, chunk, nch);
    return (size_t)rows * nch * 2;
}

// Resident CTAs per SM of `kernel` at `threads` threads (no dynamic shared memory), cached
// per device, kernel and CTA size.
int blocks_per_sm(const void *kernel, int threads) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void *, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_tuple(dev, kernel, threads);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess || n < 1) n = 1;
    cache[key] = n;
    return n;
}

template <int VPT>
cudaError_t launch_rows(const float *x, float *z, long long rows, int T, int threads, int sm_count,
                        cudaStream_t s) {
    if (VPT >= 4 && blocks_per_sm((const void *)softmax_rows_onchip_kernel<VPT>, threads) == 1) {
        // one CTA per row would be alone on its SM: persistent CTAs prefetching their next row
        const int per_sm = blocks_per_sm((const void *)softmax_rows_resident_kernel<VPT>, threads);
        const long long grid = std::min<long long>(rows, (long long)per_sm * sm_count);
        softmax_rows_resident_kernel<VPT><<<(unsigned)grid, threads, 0, s>>>(x, z, rows, T);
    } else {
        softmax_rows_onchip_kernel<VPT><<<(unsigned)rows, threads, 0, s>>>(x, z, T);
    }
    return cudaGetLastError();
}

cudaError_t launch_softmax_rows(const float *x, float *z, long long rows, long long T,
                                float *ws, int sm_count, cudaStream_t s) {
    if (onchip_ok(x, z, T)) {
        const int nvec = (int)(T >> 2);
        int vpt = 1;
        while (vpt < 8 && nvec > 1024 * vpt) vpt *= 2;
        int threads = (nvec + vpt - 1) / vpt;
        threads = ((threads + 31) / 32) * 32;
        cudaError_t e;
        switch (vpt) {
            case 1: e = launch_rows<1>(x, z, rows, (int)T, threads, sm_count, s); break;
            case 2: e = launch_rows<2>(x, z, rows, (int)T, threads, sm_count, s); break;
            case 4: e = launch_rows<4>(x, z, rows, (int)T, threads, sm_count, s); break;
            default: e = launch_rows<8>(x, z, rows, (int)T, threads, sm_count, s); break;
        }
        if (e != cudaSuccess) return e;
        count_launches(1);
        return cudaGetLastError();
    }
    if (T <= kMaxResidentT) {
        softmax_row_stream_kernel<<<(unsigned)rows, kChunkThreads, 0, s>>>(x, z, T);
        count_launches(1);
        return cudaGetLastError();
    }
    long long chunk;
    int nch;
    chunk_geometry(rows, T, sm_count, chunk, nch);
    const bool vec4 = (T & 3) == 0 && aligned16(x) && aligned16(z);
    dim3 grid(nch, (unsigned)rows);
    float2 *w2 = reinterpret_cast<float2 *>(ws);
    cudaError_t e;
    if (vec4) {
        softmax_chunk_state_kernel<true><<<grid, kChunkThreads, 0, s>>>(x, T, chunk, w2);
        e = launch_dependent(softmax_chunk_norm_kernel<true>, grid, dim3(kChunkThreads), 0, s, x, z, T, chunk,
                             (const float2 *)w2);
    } else {
        softmax_chunk_state_kernel<false><<<grid, kChunkThreads, 0, s>>>(x, T, chunk, w2);
        e = launch_dependent(softmax_chunk_norm_kernel<false>, grid, dim3(kChunkThreads), 0, s, x, z, T, chunk,
                             (const float2 *)w2);
    }
    if (e != cudaSuccess) return e;
    count_launches(2);
    return cudaGetLastError();
}

}  // namespace osf
