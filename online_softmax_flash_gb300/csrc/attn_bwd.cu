// Attention backward: dQ, dK, dV of O = softmax(mask(Q K^T * scale)) V for a loss whose gradient
// with respect to O is dO.  The pages describe only the forward pass (the single-pass attention
// of "softmax_attention", section "实现思路", with the GQA mapping and causal mask of
// "从零开始写Qwen3（五-其一）使用Triton实现自注意力", "自注意力原理" and "GQA"); the backward pass is
// the chain rule through that definition:
//     P = softmax(S),  dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  D_i = rowsum(dO_i * O_i),
//     dQ = scale * dS K,  dK = scale * dS^T Q,
// with P rebuilt from the forward's log-sum-exp (P_ij = 2^(S_ij * scale * log2 e - lse_i log2 e)),
// so no [Sq, Sk] matrix is stored.  A kv head's dK and dV sum its G query heads.
//
// Kernels: (1) D_i, one warp per row; (2) dK/dV: one CTA per (b, kv head, 64 keys) walks every
// query head of the group and every query block that sees those keys, so each CTA owns its
// output rows and needs no atomics; (3) dQ: one CTA per (b, q head, 64 rows) walks the key
// blocks its rows see.  bf16 with D in {64, 128} runs (2) and (3) on warp-level tensor cores
// (mma.sync m16n8k16, bf16 in, fp32 accumulate): each warp owns 16 rows, the score
// accumulators are reused in registers as the A operand of the next product (as in the decode
// kernel); other problems run a CUDA-core version with one warp per output row.  bf16 with D in
// {64, 128} and aligned pointers normally takes the tcgen05 kernels of attn_bwd_tc.cu instead;
// the warp-level kernels remain for pointers TMA cannot address.
#include <mutex>
#include <type_traits>

#include "attn_bwd.cuh"
#include "attn_bwd_tc.cuh"
#include "sm100_ptx.cuh"

namespace osf {
namespace {

using namespace ptx;

__device__ __forceinline__ float ldf(const float *p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

__device__ __forceinline__ bool visible(const BwdProblem &p, int i, int j) {
    return i < p.Sq && j < p.Sk && (!p.causal || j <= i + p.causal_off);
}

// ------------------------------------------------------------------ D_i = rowsum(dO_i * O_i)
template <typename T>
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(BwdProblem p) {
    const long long rows = (long long)p.B * p.Hq * p.Sq;
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const T *o = static_cast<const T *>(p.o) + row * p.D;
    const T *g = static_cast<const T *>(p.dout) + row * p.D;
    float acc = 0.f;
    for (int d = lane; d < p.D; d += 32) acc += ldf(o + d) * ldf(g + d);
    acc = warp_sum(acc);
    if (lane == 0) p.dvec[row] = acc;
}

// bf16 with D = 32 * VW (VW = 2 or 4 elements per lane) and rows starting on VW * 2-byte
// boundaries: one warp per four rows, every load of the four rows issued before any arithmetic.
template <int VW>
__global__ void __launch_bounds__(256) bwd_rowdot_vec_kernel(BwdProblem p) {
    using V = typename std::conditional<VW == 4, uint2, uint32_t>::type;
    constexpr int R = 4;
    const long long rows = (long long)p.B * p.Hq * p.Sq;
    const long long row0 = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * R;
    const int lane = threadIdx.x & 31;
    V o[R], g[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const long long row = row0 + r;
        if (row < rows) {
            o[r] = reinterpret_cast<const V *>(static_cast<const __nv_bfloat16 *>(p.o) + row * p.D)[lane];
            g[r] = reinterpret_cast<const V *>(static_cast<const __nv_bfloat16 *>(p.dout) + row * p.D)[lane];
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        float acc = 0.f;
        if (row0 + r < rows) {
            const uint32_t *ow = reinterpret_cast<const uint32_t *>(&o[r]);
            const uint32_t *gw = reinterpret_cast<const uint32_t *>(&g[r]);
#pragma unroll
            for (int w = 0; w < VW / 2; ++w)
                acc += __uint_as_float(ow[w] << 16) * __uint_as_float(gw[w] << 16) +
                       __uint_as_float(ow[w] & 0xffff0000u) * __uint_as_float(gw[w] & 0xffff0000u);
        }
        acc = warp_sum(acc);
        if (lane == r && row0 + r < rows) p.dvec[row0 + r] = acc;
    }
}

// bf16 with D = 8 * LPR and 16-byte aligned rows: LPR lanes per row, one 16-byte load of O and
// of dO per lane and row, four rounds of 32 / LPR rows per warp, every load issued before any
// arithmetic; the partial sums meet within each group of LPR lanes.
template <int LPR>
__global__ void __launch_bounds__(256) bwd_rowdot_v16_kernel(BwdProblem p) {
    constexpr int RPI = 32 / LPR, IT = 4, RPW = RPI * IT;
    const long long rows = (long long)p.B * p.Hq * p.Sq;
    const int lane = threadIdx.x & 31, sub = lane / LPR, c = lane % LPR;
    const long long wrow = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * RPW;
    uint4 o[IT], g[IT];
#pragma unroll
    for (int i = 0; i < IT; ++i) {
        const long long row = wrow + i * RPI + sub;
        if (row < rows) {
            o[i] = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.o) + row * p.D)[c];
            g[i] = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.dout) + row * p.D)[c];
        }
    }
#pragma unroll
    for (int i = 0; i < IT; ++i) {
        const long long row = wrow + i * RPI + sub;
        float acc = 0.f;
        if (row < rows) {
            const uint32_t ow[4] = {o[i].x, o[i].y, o[i].z, o[i].w}, gw[4] = {g[i].x, g[i].y, g[i].z, g[i].w};
#pragma unroll
            for (int w = 0; w < 4; ++w)
                acc += __uint_as_float(ow[w] << 16) * __uint_as_float(gw[w] << 16) +
                       __uint_as_float(ow[w] & 0xffff0000u) * __uint_as_float(gw[w] & 0xffff0000u);
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (c == 0 && row < rows) p.dvec[row] = acc;
    }
}

// ------------------------------------------------------------------ CUDA-core version
// One warp per query row: dQ_i = scale * sum_j dS_ij K_j.
template <typename T>
__global__ void __launch_bounds__(256) bwd_dq_simt_kernel(BwdProblem p) {
    const long long rows = (long long)p.B * p.Hq * p.Sq;
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int i = (int)(row % p.Sq);
    const long long bh = row / p.Sq;
    const int b = (int)(bh / p.Hq), hq = (int)(bh % p.Hq);
    const int kvh = hq / (p.Hq / p.Hkv);
    const int D = p.D;
    const T *q = static_cast<const T *>(p.q) + row * D;
    const T *go = static_cast<const T *>(p.dout) + row * D;
    const T *K = static_cast<const T *>(p.k) + ((long long)b * p.Hkv + kvh) * p.Sk * D;
    const T *V = static_cast<const T *>(p.v) + ((long long)b * p.Hkv + kvh) * p.Sk * D;
    float qr[8], gr[8], acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const int d = lane + 32 * c;
        qr[c] = d < D ? ldf(q + d) : 0.f;
        gr[c] = d < D ? ldf(go + d) : 0.f;
        acc[c] = 0.f;
    }
    const float lse2 = p.lse[row] * kLog2e, dv = p.dvec[row];
    const int j_end = p.causal ? min(p.Sk, max(0, i + p.causal_off + 1)) : p.Sk;
    for (int j = 0; j < j_end; ++j) {
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int d = lane + 32 * c;
            if (d < D) {
                s += qr[c] * ldf(K + (long long)j * D + d);
                dp += gr[c] * ldf(V + (long long)j * D + d);
            }
        }
        s = warp_sum(s);
        dp = warp_sum(dp);
        const float pr = ex2_approx(s * p.scale_log2 - lse2);
        const float ds = pr * (dp - dv);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int d = lane + 32 * c;
            if (d < D) acc[c] += ds * ldf(K + (long long)j * D + d);
        }
    }
    T *dq = static_cast<T *>(p.dq) + row * D;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const int d = lane + 32 * c;
        if (d < D) dq[d] = from_f32<T>(acc[c] * p.scale);
    }
}

// One warp per key row of a kv head: dV_j = sum_i P_ij dO_i, dK_j = scale * sum_i dS_ij Q_i over
// the G query heads of the group.
template <typename T>
__global__ void __launch_bounds__(256) bwd_dkdv_simt_kernel(BwdProblem p) {
    const long long rows = (long long)p.B * p.Hkv * p.Sk;
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int j = (int)(row % p.Sk);
    const long long bk = row / p.Sk;
    const int b = (int)(bk / p.Hkv), kvh = (int)(bk % p.Hkv);
    const int G = p.Hq / p.Hkv, D = p.D;
    const T *k = static_cast<const T *>(p.k) + row * D;
    const T *v = static_cast<const T *>(p.v) + row * D;
    float kr[8], vr[8], dk[8], dv[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const int d = lane + 32 * c;
        kr[c] = d < D ? ldf(k + d) : 0.f;
        vr[c] = d < D ? ldf(v + d) : 0.f;
        dk[c] = dv[c] = 0.f;
    }
    const int i_begin = p.causal ? max(0, j - p.causal_off) : 0;
    for (int g = 0; g < G; ++g) {
        const long long bh = (long long)b * p.Hq + kvh * G + g;
        const T *Q = static_cast<const T *>(p.q) + bh * p.Sq * D;
        const T *GO = static_cast<const T *>(p.dout) + bh * p.Sq * D;
        for (int i = i_begin; i < p.Sq; ++i) {
            float s = 0.f, dp = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int d = lane + 32 * c;
                if (d < D) {
                    s += kr[c] * ldf(Q + (long long)i * D + d);
                    dp += vr[c] * ldf(GO + (long long)i * D + d);
                }
            }
            s = warp_sum(s);
            dp = warp_sum(dp);
            const float pr = ex2_approx(s * p.scale_log2 - p.lse[bh * p.Sq + i] * kLog2e);
            const float ds = pr * (dp - p.dvec[bh * p.Sq + i]);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int d = lane + 32 * c;
                if (d < D) {
                    dv[c] += pr * ldf(GO + (long long)i * D + d);
                    dk[c] += ds * ldf(Q + (long long)i * D + d);
                }
            }
        }
    }
    T *gk = static_cast<T *>(p.dk) + row * D;
    T *gv = static_cast<T *>(p.dv) + row * D;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const int d = lane + 32 * c;
        if (d < D) {
            gk[d] = from_f32<T>(dk[c] * p.scale);
            gv[d] = from_f32<T>(dv[c]);
        }
    }
}

// ------------------------------------------------------------------ tensor-core version (bf16)
// Shared-memory tiles are row-major with rows padded to D + 8 elements, so the 16-byte rows that
// ldmatrix reads for one 8x8 matrix fall in different banks.
template <int D> struct BwdCfg {
    static constexpr int LD = D + 8;
    static constexpr int BQ = D == 64 ? 64 : 32;   // query rows per step of the dK/dV kernel
    static constexpr int BK = D == 64 ? 64 : 32;   // keys per step of the dQ kernel
    static constexpr int NT = D / 8;               // n8 tiles across D
};

// Copy rows [r0, r0 + n) of a [rows_total, D] bf16 matrix into a padded tile (zero past the end).
template <int D>
__device__ __forceinline__ void load_tile(__nv_bfloat16 *dst, const __nv_bfloat16 *src, int r0, int n,
                                          int rows_total) {
    constexpr int LD = D + 8, VPR = D / 8;   // 16-byte vectors per row
    for (int idx = threadIdx.x; idx < n * VPR; idx += blockDim.x) {
        const int r = idx / VPR, c = idx % VPR;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (r0 + r < rows_total) val = *reinterpret_cast<const uint4 *>(src + (long long)(r0 + r) * D + c * 8);
        *reinterpret_cast<uint4 *>(dst + r * LD + c * 8) = val;
    }
}

// A fragment (16 x 16) of rows r0.., cols c0.. of a padded tile.
__device__ __forceinline__ void ld_a(const __nv_bfloat16 *tile, int ld, int r0, int c0, uint32_t (&a)[4]) {
    const int lane = threadIdx.x & 31;
    const int r = r0 + (lane & 7) + ((lane >> 3) & 1) * 8, c = c0 + (lane >> 4) * 8;
    ldmatrix_x4(smem_u32(tile + r * ld + c), a[0], a[1], a[2], a[3]);
}
// B fragments of two n8 tiles where B[k][n] = tile[n][k] (n rows n0..n0+15, k cols k0..k0+15).
__device__ __forceinline__ void ld_b_nt(const __nv_bfloat16 *tile, int ld, int n0, int k0, uint32_t &b0, uint32_t &b1,
                                        uint32_t &b2, uint32_t &b3) {
    const int lane = threadIdx.x & 31, mi = lane >> 3, rr = lane & 7;
    const int r = n0 + ((mi >> 1) << 3) + rr, c = k0 + ((mi & 1) << 3);
    ldmatrix_x4(smem_u32(tile + r * ld + c), b0, b1, b2, b3);
}
// B fragments of two n8 tiles where B[k][n] = tile[k][n] (k rows k0..k0+15, n cols n0..n0+15).
__device__ __forceinline__ void ld_b_t(const __nv_bfloat16 *tile, int ld, int k0, int n0, uint32_t &b0, uint32_t &b1,
                                       uint32_t &b2, uint32_t &b3) {
    const int lane = threadIdx.x & 31, mi = lane >> 3, rr = lane & 7;
    const int r = k0 + ((mi & 1) << 3) + rr, c = n0 + ((mi >> 1) << 3);
    ldmatrix_x4_trans(smem_u32(tile + r * ld + c), b0, b1, b2, b3);
}
// A fragment (16 x 16) from the fp32 accumulators of two n8 tiles (cols 0-7 and 8-15).
__device__ __forceinline__ void acc_to_a(const float (&x)[4], const float (&y)[4], uint32_t (&a)[4]) {
    a[0] = pack_bf16x2(x[0], x[1]);
    a[1] = pack_bf16x2(x[2], x[3]);
    a[2] = pack_bf16x2(y[0], y[1]);
    a[3] = pack_bf16x2(y[2], y[3]);
}

// dK, dV for 64 keys (4 warps x 16) of one (b, kv head).
template <int D>
__global__ void __launch_bounds__(128) bwd_dkdv_mma_kernel(BwdProblem p) {
    using C = BwdCfg<D>;
    constexpr int KB = 64, LD = C::LD, BQ = C::BQ, NT = C::NT;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __nv_bfloat16 *sK = reinterpret_cast<__nv_bfloat16 *>(smem_raw);
    __nv_bfloat16 *sV = sK + KB * LD, *sQ = sV + KB * LD, *sG = sQ + BQ * LD;
    float *sL = reinterpret_cast<float *>(sG + BQ * LD), *sDv = sL + BQ;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int key0 = blockIdx.x * KB;
    const int bk = blockIdx.y, b = bk / p.Hkv, kvh = bk % p.Hkv;
    const int G = p.Hq / p.Hkv;
    const __nv_bfloat16 *Kg = static_cast<const __nv_bfloat16 *>(p.k) + (long long)bk * p.Sk * D;
    const __nv_bfloat16 *Vg = static_cast<const __nv_bfloat16 *>(p.v) + (long long)bk * p.Sk * D;
    load_tile<D>(sK, Kg, key0, KB, p.Sk);
    load_tile<D>(sV, Vg, key0, KB, p.Sk);
    float dk[NT][4], dv[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) dk[t][e] = dv[t][e] = 0.f;
    const int kw = warp * 16;                           // this warp's keys within the block
    const int krow = key0 + kw + (lane >> 2);           // key of accumulator elements 0, 1 (+8: 2, 3)
    // first query row that sees a key of this block
    int q_first = p.causal ? max(0, key0 - p.causal_off) : 0;
    q_first = (q_first / BQ) * BQ;
    for (int g = 0; g < G; ++g) {
        const long long bh = (long long)b * p.Hq + kvh * G + g;
        const __nv_bfloat16 *Qg = static_cast<const __nv_bfloat16 *>(p.q) + bh * p.Sq * D;
        const __nv_bfloat16 *Gg = static_cast<const __nv_bfloat16 *>(p.dout) + bh * p.Sq * D;
        for (int q0 = q_first; q0 < p.Sq; q0 += BQ) {
            __syncthreads();   // previous step's Q, dO done (and K, V stored, first time)
            load_tile<D>(sQ, Qg, q0, BQ, p.Sq);
            load_tile<D>(sG, Gg, q0, BQ, p.Sq);
            for (int r = threadIdx.x; r < BQ; r += blockDim.x) {
                const bool ok = q0 + r < p.Sq;
                sL[r] = ok ? p.lse[bh * p.Sq + q0 + r] * kLog2e : INFINITY;   // P = 0 past Sq
                sDv[r] = ok ? p.dvec[bh * p.Sq + q0 + r] : 0.f;
            }
            __syncthreads();
            // S^T = K_w Q^T  [16 keys x BQ queries]
            float st[BQ / 8][4];
#pragma unroll
            for (int t = 0; t < BQ / 8; ++t) st[t][0] = st[t][1] = st[t][2] = st[t][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t a[4];
                ld_a(sK, LD, kw, kk * 16, a);
#pragma unroll
                for (int j = 0; j < BQ / 16; ++j) {
                    uint32_t b0, b1, b2, b3;
                    ld_b_nt(sQ, LD, j * 16, kk * 16, b0, b1, b2, b3);
                    mma_m16n8k16_bf16(st[2 * j], a, b0, b1);
                    mma_m16n8k16_bf16(st[2 * j + 1], a, b2, b3);
                }
            }
            // P^T (masked), in place
#pragma unroll
            for (int t = 0; t < BQ / 8; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int qi = t * 8 + 2 * (lane & 3) + (e & 1);
                    const int kj = krow + (e >> 1) * 8;
                    st[t][e] = visible(p, q0 + qi, kj) ? ex2_approx(st[t][e] * p.scale_log2 - sL[qi]) : 0.f;
                }
            // dV += P^T dO
#pragma unroll
            for (int j = 0; j < BQ / 16; ++j) {
                uint32_t a[4];
                acc_to_a(st[2 * j], st[2 * j + 1], a);
#pragma unroll
                for (int dt = 0; dt < D / 16; ++dt) {
                    uint32_t b0, b1, b2, b3;
                    ld_b_t(sG, LD, j * 16, dt * 16, b0, b1, b2, b3);
                    mma_m16n8k16_bf16(dv[2 * dt], a, b0, b1);
                    mma_m16n8k16_bf16(dv[2 * dt + 1], a, b2, b3);
                }
            }
            // dP^T = V_w dO^T, then dS^T = P^T * (dP^T - D) in place
            float dpt[BQ / 8][4];
#pragma unroll
            for (int t = 0; t < BQ / 8; ++t) dpt[t][0] = dpt[t][1] = dpt[t][2] = dpt[t][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t a[4];
                ld_a(sV, LD, kw, kk * 16, a);
#pragma unroll
                for (int j = 0; j < BQ / 16; ++j) {
                    uint32_t b0, b1, b2, b3;
                    ld_b_nt(sG, LD, j * 16, kk * 16, b0, b1, b2, b3);
                    mma_m16n8k16_bf16(dpt[2 * j], a, b0, b1);
                    mma_m16n8k16_bf16(dpt[2 * j + 1], a, b2, b3);
                }
            }
#pragma unroll
            for (int t = 0; t < BQ / 8; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int qi = t * 8 + 2 * (lane & 3) + (e & 1);
                    dpt[t][e] = st[t][e] * (dpt[t][e] - sDv[qi]);
                }
            // dK += dS^T Q
#pragma unroll
            for (int j = 0; j < BQ / 16; ++j) {
                uint32_t a[4];
                acc_to_a(dpt[2 * j], dpt[2 * j + 1], a);
#pragma unroll
                for (int dt = 0; dt < D / 16; ++dt) {
                    uint32_t b0, b1, b2, b3;
                    ld_b_t(sQ, LD, j * 16, dt * 16, b0, b1, b2, b3);
                    mma_m16n8k16_bf16(dk[2 * dt], a, b0, b1);
                    mma_m16n8k16_bf16(dk[2 * dt + 1], a, b2, b3);
                }
            }
        }
    }
    // write this warp's 16 keys
    __nv_bfloat16 *dKg = static_cast<__nv_bfloat16 *>(p.dk) + (long long)bk * p.Sk * D;
    __nv_bfloat16 *dVg = static_cast<__nv_bfloat16 *>(p.dv) + (long long)bk * p.Sk * D;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int kj = krow + h * 8;
            if (kj < p.Sk) {
                const int d = t * 8 + 2 * (lane & 3);
                *reinterpret_cast<uint32_t *>(dKg + (long long)kj * D + d) =
                    pack_bf16x2(dk[t][2 * h] * p.scale, dk[t][2 * h + 1] * p.scale);
                *reinterpret_cast<uint32_t *>(dVg + (long long)kj * D + d) = pack_bf16x2(dv[t][2 * h], dv[t][2 * h + 1]);
            }
        }
}

// dQ for 64 query rows (4 warps x 16) of one (b, q head).
template <int D>
__global__ void __launch_bounds__(128) bwd_dq_mma_kernel(BwdProblem p) {
    using C = BwdCfg<D>;
    constexpr int QB = 64, LD = C::LD, BK = C::BK, NT = C::NT;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __nv_bfloat16 *sQ = reinterpret_cast<__nv_bfloat16 *>(smem_raw);
    __nv_bfloat16 *sG = sQ + QB * LD, *sK = sG + QB * LD, *sV = sK + BK * LD;
    float *sL = reinterpret_cast<float *>(sV + BK * LD), *sDv = sL + QB;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q0 = blockIdx.x * QB;
    const long long bh = blockIdx.y;
    const int b = (int)(bh / p.Hq), hq = (int)(bh % p.Hq);
    const int kvh = hq / (p.Hq / p.Hkv);
    const __nv_bfloat16 *Kg = static_cast<const __nv_bfloat16 *>(p.k) + ((long long)b * p.Hkv + kvh) * p.Sk * D;
    const __nv_bfloat16 *Vg = static_cast<const __nv_bfloat16 *>(p.v) + ((long long)b * p.Hkv + kvh) * p.Sk * D;
    load_tile<D>(sQ, static_cast<const __nv_bfloat16 *>(p.q) + bh * p.Sq * D, q0, QB, p.Sq);
    load_tile<D>(sG, static_cast<const __nv_bfloat16 *>(p.dout) + bh * p.Sq * D, q0, QB, p.Sq);
    for (int r = threadIdx.x; r < QB; r += blockDim.x) {
        const bool ok = q0 + r < p.Sq;
        sL[r] = ok ? p.lse[bh * p.Sq + q0 + r] * kLog2e : INFINITY;
        sDv[r] = ok ? p.dvec[bh * p.Sq + q0 + r] : 0.f;
    }
    float dq[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) dq[t][0] = dq[t][1] = dq[t][2] = dq[t][3] = 0.f;
    const int qw = warp * 16;
    const int qrow = q0 + qw + (lane >> 2);   // query row of accumulator elements 0, 1 (+8: 2, 3)
    // last key any row of this block sees
    int k_end = p.Sk;
    if (p.causal) k_end = min(k_end, max(0, min(q0 + QB, p.Sq) - 1 + p.causal_off + 1));
    for (int k0 = 0; k0 < k_end; k0 += BK) {
        __syncthreads();
        load_tile<D>(sK, Kg, k0, BK, p.Sk);
        load_tile<D>(sV, Vg, k0, BK, p.Sk);
        __syncthreads();
        // S = Q_w K^T, dP = dO_w V^T  [16 rows x BK keys]
        float s[BK / 8][4], dp[BK / 8][4];
#pragma unroll
        for (int t = 0; t < BK / 8; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[t][e] = dp[t][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t a[4], g[4];
            ld_a(sQ, LD, qw, kk * 16, a);
            ld_a(sG, LD, qw, kk * 16, g);
#pragma unroll
            for (int j = 0; j < BK / 16; ++j) {
                uint32_t b0, b1, b2, b3;
                ld_b_nt(sK, LD, j * 16, kk * 16, b0, b1, b2, b3);
                mma_m16n8k16_bf16(s[2 * j], a, b0, b1);
                mma_m16n8k16_bf16(s[2 * j + 1], a, b2, b3);
                ld_b_nt(sV, LD, j * 16, kk * 16, b0, b1, b2, b3);
                mma_m16n8k16_bf16(dp[2 * j], g, b0, b1);
                mma_m16n8k16_bf16(dp[2 * j + 1], g, b2, b3);
            }
        }
        // dS = P * (dP - D), P rebuilt from lse
#pragma unroll
        for (int t = 0; t < BK / 8; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int ri = qw + (lane >> 2) + (e >> 1) * 8;
                const int kj = k0 + t * 8 + 2 * (lane & 3) + (e & 1);
                const float pr = visible(p, q0 + ri, kj) ? ex2_approx(s[t][e] * p.scale_log2 - sL[ri]) : 0.f;
                s[t][e] = pr * (dp[t][e] - sDv[ri]);
            }
        // dQ += dS K
#pragma unroll
        for (int j = 0; j < BK / 16; ++j) {
            uint32_t a[4];
            acc_to_a(s[2 * j], s[2 * j + 1], a);
#pragma unroll
            for (int dt = 0; dt < D / 16; ++dt) {
                uint32_t b0, b1, b2, b3;
                ld_b_t(sK, LD, j * 16, dt * 16, b0, b1, b2, b3);
                mma_m16n8k16_bf16(dq[2 * dt], a, b0, b1);
                mma_m16n8k16_bf16(dq[2 * dt + 1], a, b2, b3);
            }
        }
    }
    __nv_bfloat16 *dQg = static_cast<__nv_bfloat16 *>(p.dq) + bh * p.Sq * D;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int qi = qrow + h * 8;
            if (qi < p.Sq)
                *reinterpret_cast<uint32_t *>(dQg + (long long)qi * D + t * 8 + 2 * (lane & 3)) =
                    pack_bf16x2(dq[t][2 * h] * p.scale, dq[t][2 * h + 1] * p.scale);
        }
}

template <int D>
cudaError_t launch_mma(const BwdProblem &p, cudaStream_t s) {
    using C = BwdCfg<D>;
    constexpr int LD = C::LD;
    const size_t smem_kv = (size_t)(2 * 64 + 2 * C::BQ) * LD * 2 + 2 * C::BQ * 4;
    const size_t smem_q = (size_t)(2 * 64 + 2 * C::BK) * LD * 2 + 2 * 64 * 4;
    cudaError_t attr_err = set_max_dynamic_smem((const void *)bwd_dkdv_mma_kernel<D>, (int)smem_kv);
    if (attr_err == cudaSuccess) attr_err = set_max_dynamic_smem((const void *)bwd_dq_mma_kernel<D>, (int)smem_q);
    if (attr_err != cudaSuccess) return attr_err;
    bwd_dkdv_mma_kernel<D><<<dim3((p.Sk + 63) / 64, p.B * p.Hkv), 128, smem_kv, s>>>(p);
    bwd_dq_mma_kernel<D><<<dim3((p.Sq + 63) / 64, p.B * p.Hq), 128, smem_q, s>>>(p);
    count_launches(2);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_simt(const BwdProblem &p, cudaStream_t s) {
    const long long rq = (long long)p.B * p.Hq * p.Sq, rk = (long long)p.B * p.Hkv * p.Sk;
    bwd_dkdv_simt_kernel<T><<<(unsigned)((rk + 7) / 8), 256, 0, s>>>(p);
    bwd_dq_simt_kernel<T><<<(unsigned)((rq + 7) / 8), 256, 0, s>>>(p);
    count_launches(2);
    return cudaGetLastError();
}

}  // namespace

bool attn_bwd_mma_supported(const BwdProblem &p) {
    if (p.dtype != OSF_BF16 || (p.D != 64 && p.D != 128)) return false;
    const uintptr_t a = reinterpret_cast<uintptr_t>(p.q) | reinterpret_cast<uintptr_t>(p.k) |
                        reinterpret_cast<uintptr_t>(p.v) | reinterpret_cast<uintptr_t>(p.dout) |
                        reinterpret_cast<uintptr_t>(p.dq) | reinterpret_cast<uintptr_t>(p.dk) |
                        reinterpret_cast<uintptr_t>(p.dv);
    return (a & 15u) == 0 && (p.Sk + 63) / 64 < 65536 && (long long)p.B * p.Hq < 65536;
}

cudaError_t launch_attn_bwd(const BwdProblem &p, cudaStream_t s) {
    const long long rows = (long long)p.B * p.Hq * p.Sq;
    const unsigned g = (unsigned)((rows + 7) / 8);
    const bool vec_ok = p.dtype == OSF_BF16 && (p.D == 64 || p.D == 128) &&
                        ((reinterpret_cast<uintptr_t>(p.o) | reinterpret_cast<uintptr_t>(p.dout)) & 7u) == 0;
    const bool v16_ok = vec_ok && ((reinterpret_cast<uintptr_t>(p.o) | reinterpret_cast<uintptr_t>(p.dout)) & 15u) == 0;
    if (v16_ok) {
        // 8 warps x (4 rounds of 32 / LPR rows) per CTA
        if (p.D == 128) bwd_rowdot_v16_kernel<16><<<(unsigned)((rows + 63) / 64), 256, 0, s>>>(p);
        else bwd_rowdot_v16_kernel<8><<<(unsigned)((rows + 127) / 128), 256, 0, s>>>(p);
    } else if (vec_ok) {
        const unsigned g4 = (unsigned)((rows + 31) / 32);   // 8 warps x 4 rows per CTA
        if (p.D == 128) bwd_rowdot_vec_kernel<4><<<g4, 256, 0, s>>>(p);
        else bwd_rowdot_vec_kernel<2><<<g4, 256, 0, s>>>(p);
    } else if (p.dtype == OSF_BF16) {
        bwd_rowdot_kernel<__nv_bfloat16><<<g, 256, 0, s>>>(p);
    } else {
        bwd_rowdot_kernel<float><<<g, 256, 0, s>>>(p);
    }
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (attn_bwd_tc_supported(p)) return launch_attn_bwd_tc(p, s);
    if (attn_bwd_mma_supported(p)) return p.D == 64 ? launch_mma<64>(p, s) : launch_mma<128>(p, s);
    return p.dtype == OSF_BF16 ? launch_simt<__nv_bfloat16>(p, s) : launch_simt<float>(p, s);
}

}  // namespace osf
