// General CUDA-core attention forward: any head dim 1..256, float32 or bfloat16 inputs, GQA,
// optional causal mask, optional split over the key range with a log-sum-exp combine.
//
// The recurrence is the one of "softmax_attention" (blog.euler0525.cn/posts/3fb3592b), section
// "实现思路": keys are streamed in blocks; per query row a running max m, a rescale factor
// alpha = exp(m_prev - m), a denominator l and a numerator acc are carried, and the row is
// acc / l at the end, so the [M, N] score matrix never leaves the chip.  Keys past the end of
// the sequence (and, with the causal mask of "从零开始写Qwen3（五-其一）...", "自注意力原理",
// keys after the query) score -inf, never 0.
//
// Unlike the page's one-program-per-query kernel, a CTA owns a tile of BM query rows and
// BN = 64 keys at a time, so every K/V element loaded into shared memory is reused by BM rows;
// S = Q K^T and O += P V are register-tiled 4 x 4 outer products on the FMA pipe.  Scores are
// kept in base 2 (scale * log2 e folded into one multiplier) so each exponential is one ex2.
#include "osf_internal.cuh"

namespace osf {
namespace {

constexpr int BN = 64;  // keys per tile

template <int DP, int BM>
struct SimtCfg {
    static constexpr int THREADS = BM * 4;             // (BM/4) row groups x 16 column groups
    static constexpr int QS = BM + 4;                  // padded length of a transposed Q column
    static constexpr int KS = BN + 4;                  // padded length of a transposed K column
    static constexpr int OC = DP / 16;                 // O columns per thread
    static constexpr int VEC = OC < 4 ? OC : 4;        // contiguous O columns per chunk
    static constexpr int NCH = OC / VEC;               // chunks of VEC columns
    static constexpr int SMEM_FLOATS = DP * QS + DP * KS + BN * DP + BN * QS;
    static constexpr size_t SMEM_BYTES = size_t(SMEM_FLOATS) * sizeof(float);
};

template <typename T>
__device__ __forceinline__ float ld(const T *p) { return to_f32(*p); }

template <typename T, int DP, int BM>
__global__ void __launch_bounds__(BM * 4)
attn_simt_kernel(const AttnProblem p) {
    using C = SimtCfg<DP, BM>;
    extern __shared__ __align__(16) float smem[];
    float *Qs = smem;                    // [DP][QS]  Q tile, transposed
    float *Ks = Qs + DP * C::QS;         // [DP][KS]  K tile, transposed
    float *Vs = Ks + DP * C::KS;         // [BN][DP]  V tile
    float *Ps = Vs + BN * DP;            // [BN][QS]  P tile, transposed

    const int tid = threadIdx.x;
    const int tx = tid & 15;             // key group (S) / column group (O)
    const int ty = tid >> 4;             // row group: rows ty*4 .. ty*4+3

    const int n_qt = (p.Sq + BM - 1) / BM;
    // causal: heaviest (last) query tiles first
    const int qt = p.causal ? (n_qt - 1 - (int)blockIdx.x) : (int)blockIdx.x;
    const int bh = blockIdx.y;           // b * Hq + hq
    const int split = blockIdx.z;
    const int b = bh / p.Hq, hq = bh % p.Hq;
    const int kvh = hq / (p.Hq / p.Hkv);
    const int q0 = qt * BM;
    const int D = p.D;

    const T *Qg = static_cast<const T *>(p.q) + q_at(p, b, hq, q0);
    const T *Kg = static_cast<const T *>(p.k) + k_at(p, b, kvh, 0);
    const T *Vg = static_cast<const T *>(p.v) + v_at(p, b, kvh, 0);

    // key range of this split: a fixed partition of [0, Sk) in whole tiles, clipped by causality
    const int n_kt_all = (p.Sk + BN - 1) / BN;
    const int tps = (n_kt_all + p.splits - 1) / p.splits;
    const int k_begin = split * tps * BN;
    int k_end = min(p.Sk, (split + 1) * tps * BN);
    if (p.causal) k_end = min(k_end, max(k_begin, q0 + BM + p.causal_off));

    for (int idx = tid; idx < BM * DP; idx += C::THREADS) {
        const int r = idx / DP, d = idx % DP;
        Qs[d * C::QS + r] = (q0 + r < p.Sq && d < D) ? ld(Qg + (long long)r * p.q_ss + d) : 0.f;
    }

    float m[4], l[4], acc[4][C::OC];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < C::OC; ++c) acc[i][c] = 0.f;
    }

    for (int kt0 = k_begin; kt0 < k_end; kt0 += BN) {
        __syncthreads();  // previous tile's K/V/P fully consumed (and Q stored, first time)
        for (int idx = tid; idx < BN * DP; idx += C::THREADS) {
            const int c = idx / DP, d = idx % DP;
            const bool ok = (kt0 + c < k_end) && d < D;
            Ks[d * C::KS + c] = ok ? ld(Kg + (long long)(kt0 + c) * p.k_ss + d) : 0.f;
            Vs[c * DP + d] = ok ? ld(Vg + (long long)(kt0 + c) * p.v_ss + d) : 0.f;
        }
        __syncthreads();

        // S = Q K^T for rows ty*4.., keys tx*4..
        float s[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
#pragma unroll 8
        for (int d = 0; d < DP; ++d) {
            const float4 a = *reinterpret_cast<const float4 *>(&Qs[d * C::QS + ty * 4]);
            const float4 k4 = *reinterpret_cast<const float4 *>(&Ks[d * C::KS + tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w};
            const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) s[i][j] = fmaf(av[i], kv[j], s[i][j]);
        }

        // scale (base 2), mask, online max / rescale / denominator
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = q0 + ty * 4 + i;
            float tmax = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int key = kt0 + tx * 4 + j;
                const bool valid = key < k_end && (!p.causal || key <= row + p.causal_off);
                s[i][j] = valid ? s[i][j] * p.scale_log2 : -INFINITY;
                tmax = fmaxf(tmax, s[i][j]);
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
            const float m_new = fmaxf(m[i], tmax);
            const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;   // fully masked so far
            const float alpha = ex2_approx(m[i] - m_ref);
            float rs = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                s[i][j] = ex2_approx(s[i][j] - m_ref);
                rs += s[i][j];
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o);
            l[i] = l[i] * alpha + rs;
            m[i] = m_new;
#pragma unroll
            for (int c = 0; c < C::OC; ++c) acc[i][c] *= alpha;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            *reinterpret_cast<float4 *>(&Ps[(tx * 4 + j) * C::QS + ty * 4]) =
                make_float4(s[0][j], s[1][j], s[2][j], s[3][j]);
        }
        __syncthreads();

        // O += P V
#pragma unroll 4
        for (int kk = 0; kk < BN; ++kk) {
            const float4 a = *reinterpret_cast<const float4 *>(&Ps[kk * C::QS + ty * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int ch = 0; ch < C::NCH; ++ch) {
                const float *vp = &Vs[kk * DP + ch * 16 * C::VEC + tx * C::VEC];
                float vv[C::VEC];
                if constexpr (C::VEC == 4) {
                    const float4 v4 = *reinterpret_cast<const float4 *>(vp);
                    vv[0] = v4.x; vv[1] = v4.y; vv[2] = v4.z; vv[3] = v4.w;
                } else {
#pragma unroll
                    for (int e = 0; e < C::VEC; ++e) vv[e] = vp[e];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int e = 0; e < C::VEC; ++e)
                        acc[i][ch * C::VEC + e] = fmaf(av[i], vv[e], acc[i][ch * C::VEC + e]);
            }
        }
    }

    // epilogue
    const long long rows_total = (long long)p.B * p.Hq * p.Sq;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = q0 + ty * 4 + i;
        if (r >= p.Sq) continue;
        const long long row = (long long)bh * p.Sq + r;
        if (p.splits == 1) {
            const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
            T *Og = static_cast<T *>(p.o) + o_at(p, b, hq, r);
#pragma unroll
            for (int ch = 0; ch < C::NCH; ++ch)
#pragma unroll
                for (int e = 0; e < C::VEC; ++e) {
                    const int col = ch * 16 * C::VEC + tx * C::VEC + e;
                    if (col < D) Og[col] = from_f32<T>(acc[i][ch * C::VEC + e] * inv);
                }
            if (p.lse && tx == 0)
                p.lse[row] = l[i] > 0.f ? (m[i] + __log2f(l[i])) * kLn2 : -INFINITY;
        } else {
            float *A = p.part_acc + ((size_t)split * rows_total + row) * D;
#pragma unroll
            for (int ch = 0; ch < C::NCH; ++ch)
#pragma unroll
                for (int e = 0; e < C::VEC; ++e) {
                    const int col = ch * 16 * C::VEC + tx * C::VEC + e;
                    if (col < D) A[col] = acc[i][ch * C::VEC + e];
                }
            if (tx == 0) {
                p.part_m[(size_t)split * rows_total + row] = m[i];
                p.part_l[(size_t)split * rows_total + row] = l[i];
            }
        }
    }
}

// ---------------------------------------------------------------- few rows, few keys
// float32 problems with few query rows and at most kRowsSk keys per head, D <= 64 (the M = 64,
// N = 100, d = 32 `solve` of "softmax_attention", section "实现思路", is one): a CTA of kRowsW
// warps owns kRowsW consecutive query rows of one (b, q head), one row per warp, as the page runs
// one program per query.  The CTA first copies its kv head's whole K and V into shared memory
// with asynchronous copies that are all issued before the first is waited for, so the kernel
// pays one memory round trip instead of one per key block; each warp then runs the recurrence
// over blocks of 64 keys, lane j scoring keys j and j + 32 of the block.
constexpr int kRowsSk = 256;   // keys a CTA stages (K and V of one kv head)
constexpr int kRowsW = 4;      // warps (query rows) per CTA

template <int DP>
struct RowsCfg {
    static constexpr int KS = DP + 4;   // K row stride in floats: 16-byte aligned, and the 16-byte
                                        // reads of eight consecutive keys hit distinct banks
    static size_t smem_bytes(int sk_pad) { return (size_t)sk_pad * (KS + DP) * sizeof(float); }
};

__device__ __forceinline__ void cp_async16(float *dst, const float *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(float *dst, const float *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// vec: K and V rows start on 16-byte boundaries and D % 4 == 0 (16-byte copies).
template <int DP>
__global__ void __launch_bounds__(kRowsW * 32) attn_rows_kernel(const AttnProblem p, int sk_pad, bool vec) {
    using C = RowsCfg<DP>;
    extern __shared__ __align__(16) float smem[];
    float *Ks = smem;                   // [sk_pad][KS]
    float *Vs = Ks + sk_pad * C::KS;    // [sk_pad][DP]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.y, b = bh / p.Hq, hq = bh % p.Hq;
    const int kvh = hq / (p.Hq / p.Hkv);
    const int D = p.D, Sk = p.Sk;
    const float *Kg = static_cast<const float *>(p.k) + k_at(p, b, kvh, 0);
    const float *Vg = static_cast<const float *>(p.v) + v_at(p, b, kvh, 0);

    // K and V into shared memory; columns past D and keys past Sk are zeros
    if (vec) {
        const int per_row = D >> 2;
        for (int idx = tid; idx < Sk * per_row; idx += kRowsW * 32) {
            const int key = idx / per_row, c = (idx - key * per_row) * 4;
            cp_async16(Ks + key * C::KS + c, Kg + (long long)key * p.k_ss + c);
            cp_async16(Vs + key * DP + c, Vg + (long long)key * p.v_ss + c);
        }
    } else {
        for (int idx = tid; idx < Sk * D; idx += kRowsW * 32) {
            const int key = idx / D, c = idx - key * D;
            cp_async4(Ks + key * C::KS + c, Kg + (long long)key * p.k_ss + c);
            cp_async4(Vs + key * DP + c, Vg + (long long)key * p.v_ss + c);
        }
    }
    for (int idx = tid; idx < sk_pad * DP; idx += kRowsW * 32) {
        const int key = idx / DP, c = idx - key * DP;
        if (key >= Sk || c >= D) {
            Ks[key * C::KS + c] = 0.f;
            Vs[key * DP + c] = 0.f;
        }
    }
    // this warp's query row, in registers (the same addresses in every lane), loaded while the
    // copies are in flight
    const int row = blockIdx.x * kRowsW + warp;
    const bool have_row = row < p.Sq;
    float q[DP];
    if (have_row) {
        const float *Qg = static_cast<const float *>(p.q) + q_at(p, b, hq, row);
#pragma unroll
        for (int d = 0; d < DP; ++d) q[d] = d < D ? Qg[d] : 0.f;
    }
    cp_async_wait_all();
    __syncthreads();
    if (!have_row) return;

    // keys this row sees: [0, lim)
    int lim = Sk;
    if (p.causal) lim = max(0, min(lim, row + p.causal_off + 1));
    float m = -INFINITY, l = 0.f, acc[DP / 32];
#pragma unroll
    for (int c = 0; c < DP / 32; ++c) acc[c] = 0.f;
    for (int kb = 0; kb < lim; kb += 64) {
        float s[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int key = kb + 32 * h + lane;   // < sk_pad: staged (zeros past Sk)
            const float *kr = Ks + key * C::KS;
            float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < DP; c += 4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(kr + c);
                part[0] = fmaf(q[c], k4.x, part[0]);
                part[1] = fmaf(q[c + 1], k4.y, part[1]);
                part[2] = fmaf(q[c + 2], k4.z, part[2]);
                part[3] = fmaf(q[c + 3], k4.w, part[3]);
            }
            const float dot = (part[0] + part[1]) + (part[2] + part[3]);
            s[h] = key < lim ? dot * p.scale_log2 : -INFINITY;   // base 2, scale folded in
        }
        float bmax = fmaxf(s[0], s[1]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
        const float m_new = fmaxf(m, bmax);   // finite: key kb < lim is in the block
        const float alpha = ex2_approx(m - m_new);   // 0 on the first block (m = -inf)
        const float p0 = ex2_approx(s[0] - m_new), p1 = ex2_approx(s[1] - m_new);
        float rs = p0 + p1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o);
        l = l * alpha + rs;
        m = m_new;
#pragma unroll
        for (int c = 0; c < DP / 32; ++c) acc[c] *= alpha;
        // acc[c] (column lane + 32c) += sum over the block's keys of p_key * V[key][column]
        const float *v0 = Vs + kb * DP + lane;
#pragma unroll 8
        for (int j = 0; j < 32; ++j) {
            const float pa = __shfl_sync(0xffffffffu, p0, j), pb = __shfl_sync(0xffffffffu, p1, j);
#pragma unroll
            for (int c = 0; c < DP / 32; ++c)
                acc[c] = fmaf(pb, v0[(32 + j) * DP + 32 * c], fmaf(pa, v0[j * DP + 32 * c], acc[c]));
        }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float *Og = static_cast<float *>(p.o) + o_at(p, b, hq, row);
#pragma unroll
    for (int c = 0; c < DP / 32; ++c)
        if (lane + 32 * c < D) Og[lane + 32 * c] = acc[c] * inv;
    if (p.lse && lane == 0)
        p.lse[(long long)bh * p.Sq + row] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
}

// Log-sum-exp combine of split partial states: M = max_s m_s, w_s = 2^(m_s - M),
// O = sum_s w_s acc_s / sum_s w_s l_s, lse = (M + log2 L) ln 2.  One thread per four columns of
// an output row.  The splits are taken eight at a time with every load of a group issued
// together, and the group folds into running (M, L, O) by the same rescaling rule, so a
// combine over up to eight splits waits for memory once.
template <typename T, bool VEC>
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnProblem p) {
    constexpr int SG = 8;   // splits per load group
    griddep_wait();   // launched as a dependent of the kernel that wrote the partial states
    const long long rows_total = (long long)p.B * p.Hq * p.Sq;
    const int groups = (p.D + 3) >> 2;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long row = idx / groups;
    const int c0 = (int)(idx - row * groups) * 4;
    if (row >= rows_total) return;
    float M = -INFINITY, L = 0.f, a[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s0 = 0; s0 < p.splits; s0 += SG) {
        float ms[SG], ls[SG], acc[SG][4];
#pragma unroll
        for (int i = 0; i < SG; ++i) {
            const int sp = s0 + i;
            ms[i] = -INFINITY;
            ls[i] = 0.f;
            acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
            if (sp < p.splits) {
                const size_t r = (size_t)sp * rows_total + row;
                ms[i] = p.part_m[r];
                ls[i] = p.part_l[r];
                const float *A = p.part_acc + r * p.D + c0;
                if (VEC) {
                    const float4 v = *reinterpret_cast<const float4 *>(A);
                    acc[i][0] = v.x; acc[i][1] = v.y; acc[i][2] = v.z; acc[i][3] = v.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (c0 + e < p.D) acc[i][e] = A[e];
                }
            }
        }
        float mg = M;
#pragma unroll
        for (int i = 0; i < SG; ++i) mg = fmaxf(mg, ms[i]);
        const float mref = mg == -INFINITY ? 0.f : mg;
        const float sc = ex2_approx(M - mref);   // 0 while nothing has been seen
        L *= sc;
#pragma unroll
        for (int e = 0; e < 4; ++e) a[e] *= sc;
#pragma unroll
        for (int i = 0; i < SG; ++i) {
            const float w = ex2_approx(ms[i] - mref);
            L += w * ls[i];
#pragma unroll
            for (int e = 0; e < 4; ++e) a[e] += w * acc[i][e];
        }
        M = mg;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int b = (int)(row / ((long long)p.Hq * p.Sq));
    const int hq = (int)((row / p.Sq) % p.Hq);
    T *Og = static_cast<T *>(p.o) + o_at(p, b, hq, row % p.Sq);
#pragma unroll
    for (int e = 0; e < 4; ++e)
        if (c0 + e < p.D) Og[c0 + e] = from_f32<T>(a[e] * inv);
    if (p.lse && c0 == 0) p.lse[row] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
}

template <typename T, int DP, int BM>
cudaError_t launch_t(const AttnProblem &p, cudaStream_t s) {
    using C = SimtCfg<DP, BM>;
    const cudaError_t e = set_max_dynamic_smem((const void *)attn_simt_kernel<T, DP, BM>, (int)C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid((p.Sq + BM - 1) / BM, p.B * p.Hq, p.splits);
    attn_simt_kernel<T, DP, BM><<<grid, C::THREADS, C::SMEM_BYTES, s>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dp(const AttnProblem &p, cudaStream_t s) {
    if (p.D <= 16) return launch_t<T, 16, 64>(p, s);
    if (p.D <= 32) return launch_t<T, 32, 64>(p, s);
    if (p.D <= 64) return launch_t<T, 64, 64>(p, s);
    if (p.D <= 128) return launch_t<T, 128, 64>(p, s);
    return launch_t<T, 256, 32>(p, s);
}

int block_m(int D) { return D <= 128 ? 64 : 32; }

// Problems the few-rows kernel runs: float32, D <= 64, at most kRowsSk keys, at most 2048 query
// rows in all (512 CTAs, each staging its kv head's K and V).
bool rows_eligible(const AttnProblem &p) {
    return p.dtype == OSF_F32 && p.D <= 64 && p.Sk <= kRowsSk && (long long)p.B * p.Hq * p.Sq <= 2048;
}

template <int DP>
cudaError_t launch_rows_t(const AttnProblem &p, cudaStream_t s) {
    const int sk_pad = (p.Sk + 63) / 64 * 64;
    const size_t smem = RowsCfg<DP>::smem_bytes(sk_pad);
    const cudaError_t e = set_max_dynamic_smem((const void *)attn_rows_kernel<DP>, (int)RowsCfg<DP>::smem_bytes(kRowsSk));
    if (e != cudaSuccess) return e;
    // 16-byte copies when every K and V row starts on a 16-byte boundary
    const bool vec = p.D % 4 == 0 && ((reinterpret_cast<uintptr_t>(p.k) | reinterpret_cast<uintptr_t>(p.v)) & 15) == 0 &&
                     ((p.k_ss | p.k_sh | p.k_sb | p.v_ss | p.v_sh | p.v_sb) & 3) == 0;
    const dim3 grid((unsigned)((p.Sq + kRowsW - 1) / kRowsW), (unsigned)(p.B * p.Hq));
    attn_rows_kernel<DP><<<grid, kRowsW * 32, smem, s>>>(p, sk_pad, vec);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

int attn_simt_pick_splits(const AttnProblem &p, int sm_count) {
    if (rows_eligible(p)) return 1;
    const int BM = block_m(p.D);
    const long long ctas = (long long)((p.Sq + BM - 1) / BM) * p.B * p.Hq;
    const int n_kt = (p.Sk + BN - 1) / BN;
    if (ctas >= 2LL * sm_count || n_kt <= 1) return 1;
    long long want = (2LL * sm_count + ctas - 1) / ctas;
    if (want > n_kt) want = n_kt;
    if (want > 64) want = 64;
    return (int)want;
}

size_t attn_simt_partial_floats(int splits, long long rows, int D) {
    if (splits <= 1) return 0;
    return (size_t)splits * rows * (size_t)(D + 2);
}

cudaError_t launch_attn_simt(const AttnProblem &p, cudaStream_t s) {
    if (p.splits == 1 && rows_eligible(p)) return p.D <= 32 ? launch_rows_t<32>(p, s) : launch_rows_t<64>(p, s);
    return p.dtype == OSF_F32 ? launch_dp<float>(p, s) : launch_dp<__nv_bfloat16>(p, s);
}

cudaError_t launch_attn_combine(const AttnProblem &p, cudaStream_t s) {
    const long long rows_total = (long long)p.B * p.Hq * p.Sq;
    const long long threads = rows_total * ((p.D + 3) / 4);
    const unsigned blocks = (unsigned)((threads + 255) / 256);
    const bool vec = p.D % 4 == 0;   // part_acc rows are then 16-byte aligned
    cudaError_t e;
    if (p.dtype == OSF_F32)
        e = launch_dependent(vec ? attn_combine_kernel<float, true> : attn_combine_kernel<float, false>, dim3(blocks),
                             dim3(256), 0, s, p);
    else
        e = launch_dependent(vec ? attn_combine_kernel<__nv_bfloat16, true> : attn_combine_kernel<__nv_bfloat16, false>,
                             dim3(blocks), dim3(256), 0, s, p);
    if (e != cudaSuccess) return e;
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace osf
