// Row softmax of scale * x with an optional in-row causal mask, for float32 or bfloat16 rows
// addressed through row strides: the softmax of "从零开始写Qwen3（五-其一）使用Triton实现自注意力",
// "softmax的triton实现" (a kernel over attention-weight rows with a row stride, a scale, and the
// causal variant whose load condition keeps column <= row, filling the rest with -inf), built on
// the online (m, l) recurrence of "Softmax 算子的实现与优化", "Online Softmax".
//
// Column j of row r is kept iff j < lim(r) = min(T, r % P + 1) when the causal period P > 0
// (stacked [Sq, Sk] score matrices use P = Sq), else lim = T; dropped columns are written as 0.
// Values are converted to fp32 on load; exponentials are base 2 on x * scale * log2(e).
//
// Paths: a row of at most 72 KB whose start and stride are 16-byte aligned is staged in shared
// memory by bulk copies (up to its causal limit; two pieces beyond 16 KB) for a CTA of 64-256
// threads, so several rows are in flight per SM and one row's load overlaps the others'
// arithmetic; other rows of up to 32768
// elements are held in registers by one CTA of up to 1024 threads (one read, one write per
// element; columns past lim are not read); unaligned short rows stream twice through one CTA;
// longer rows are cut into chunks over the whole GPU (chunk states, then merge + normalise).
#include <mutex>

#include "osf_internal.cuh"
#include "sm100_ptx.cuh"
#include "softmax_ex.cuh"

namespace osf {
namespace {

constexpr int kExMaxResidentT = 32768;
constexpr int kExChunkThreads = 512;

// 16-byte vector loads of E elements, converted to float.
template <typename T> struct Vec;
template <> struct Vec<float> {
    static constexpr int E = 4;
    static constexpr uint32_t SGN = 0x80000000u;   // the sign bit of each element of a 32-bit word
    // 16 raw bytes to E floats, each with its sign flipped by `sgn` (0 or SGN)
    __device__ __forceinline__ static void unpack(uint4 a, uint32_t sgn, float (&f)[4]) {
        f[0] = __uint_as_float(a.x ^ sgn); f[1] = __uint_as_float(a.y ^ sgn);
        f[2] = __uint_as_float(a.z ^ sgn); f[3] = __uint_as_float(a.w ^ sgn);
    }
    __device__ __forceinline__ static void load(const float *p, float (&f)[4]) {
        const float4 a = __ldcs(reinterpret_cast<const float4 *>(p));
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    }
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int E = 8;
    static constexpr uint32_t SGN = 0x80008000u;
    __device__ __forceinline__ static void unpack(uint4 a, uint32_t sgn, float (&f)[8]) {
        const uint32_t w[4] = {a.x ^ sgn, a.y ^ sgn, a.z ^ sgn, a.w ^ sgn};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static void load(const __nv_bfloat16 *p, float (&f)[8]) {
        const uint4 a = __ldcs(reinterpret_cast<const uint4 *>(p));
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

// Store E floats as E output elements (E * sizeof(Tout) bytes, aligned to that size).
template <int E> __device__ __forceinline__ void store_vec(float *p, const float (&f)[E]) {
#pragma unroll
    for (int i = 0; i < E; i += 4) __stcs(reinterpret_cast<float4 *>(p + i), make_float4(f[i], f[i + 1], f[i + 2], f[i + 3]));
}
template <int E> __device__ __forceinline__ void store_vec(__nv_bfloat16 *p, const float (&f)[E]) {
    uint32_t w[E / 2];
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    if constexpr (E == 8)
        __stcs(reinterpret_cast<uint4 *>(p), make_uint4(w[0], w[1], w[2], w[3]));
    else
        __stcs(reinterpret_cast<uint2 *>(p), make_uint2(w[0], w[1]));
}

__device__ __forceinline__ float ld1(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ld1(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// CTA-wide merge of per-thread (m, l) states; result broadcast to every thread.
__device__ __forceinline__ void cta_merge_ml(float &m, float &l, float *sh /* 2*32 */) {
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

__device__ __forceinline__ long long row_limit(long long row, long long T, long long period) {
    return period > 0 ? min(T, row % period + 1) : T;
}

// The staged kernels' arithmetic on one 16-byte vector of E values, columns [col0, col0 + E), in
// base-2 units of x * a with a = |scale| * log2 e (a negative scale is applied by flipping the
// values' signs on load).  Values are paired for f32x2 FMA / add / multiply; columns at or past
// `lim` are dropped (-inf, then 0), and a vector wholly inside the limit takes no per-element test.
template <int E>
__device__ __forceinline__ void fold_vec(float (&f)[E], int col0, int lim, float a, float &m, float &l) {
    static_assert(E == 4 || E == 8, "16-byte vectors of float32 or bfloat16");
    if (col0 + E > lim) {
#pragma unroll
        for (int e = 0; e < E; ++e)
            if (col0 + e >= lim) f[e] = -INFINITY;
    }
    // max of E values: 3-input max over f[0..2], then pairs f[3..4], f[5..6], then f[E - 1]
    float mx = ptx::fmax3(f[0], f[1], f[2]);
#pragma unroll
    for (int e = 3; e + 1 < E; e += 2) mx = ptx::fmax3(mx, f[e], f[e + 1]);
    mx = fmaxf(mx, f[E - 1]);
    const float mn = fmaxf(m, mx * a);
    const float mr = (mn == -INFINITY) ? 0.f : mn;
    const uint64_t a2 = ptx::f2_pack(a, a), n2 = ptx::f2_pack(-mr, -mr);
    uint64_t acc = ptx::f2_pack(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < E / 2; ++k) {
        float p0, p1;
        ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(f[2 * k], f[2 * k + 1]), a2, n2), p0, p1);
        acc = ptx::f2_add(acc, ptx::f2_pack(ex2_approx(p0), ex2_approx(p1)));
    }
    float lo, hi;
    ptx::f2_unpack(acc, lo, hi);
    l = l * ex2_approx(m - mr) + (lo + hi);
    m = mn;
}

// z for one vector: 2^(x a - mref) / l for kept columns (`have`: the vector was loaded), else 0.
template <int E, typename Tout>
__device__ __forceinline__ void emit_vec(const float (&f)[E], int col0, int lim, bool have, float a, float mref,
                                         float inv, Tout *dst) {
    float o[E];
    if (have && col0 + E <= lim) {
        const uint64_t a2 = ptx::f2_pack(a, a), n2 = ptx::f2_pack(-mref, -mref), i2 = ptx::f2_pack(inv, inv);
#pragma unroll
        for (int k = 0; k < E / 2; ++k) {
            float p0, p1;
            ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(f[2 * k], f[2 * k + 1]), a2, n2), p0, p1);
            ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(ex2_approx(p0), ex2_approx(p1)), i2), o[2 * k], o[2 * k + 1]);
        }
    } else if (!have || col0 >= lim) {
        // past the row's limit: zeros, with no exponential evaluated
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = 0.f;
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = (col0 + e < lim) ? ex2_approx(f[e] * a - mref) * inv : 0.f;
    }
    store_vec<E>(dst, o);
}

// One CTA per row; thread t holds vectors t + k * blockDim (k < VPT) of the row in registers.
template <typename Tin, typename Tout, int VPT>
__global__ void __launch_bounds__(1024, 1)
softmax_ex_onchip_kernel(const Tin *__restrict__ x, Tout *z, int T, long long xs, long long zs, float mult,
                         long long period) {
    constexpr int E = Vec<Tin>::E;
    __shared__ float sh[64];
    const long long row = blockIdx.x;
    const Tin *xr = x + row * xs;
    Tout *zr = z + row * zs;
    const int nvec = T / E;
    const int lim = (int)row_limit(row, T, period);
    float v[VPT][E];
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = threadIdx.x + k * blockDim.x;
        if (i < nvec && i * E < lim) {
            Vec<Tin>::load(xr + (long long)i * E, v[k]);
#pragma unroll
            for (int e = 0; e < E; ++e) v[k][e] = (i * E + e < lim) ? v[k][e] * mult : -INFINITY;
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) v[k][e] = -INFINITY;
        }
#pragma unroll
        for (int e = 0; e < E; ++e) m = fmaxf(m, v[k][e]);
    }
    const float mref = (m == -INFINITY) ? 0.f : m;
    float l = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int e = 0; e < E; ++e) {
            v[k][e] = ex2_approx(v[k][e] - mref);
            l += v[k][e];
        }
    float M = m, L = l;
    cta_merge_ml(M, L, sh);
    const float f = (m == -INFINITY) ? 0.f : ex2_approx(m - M) / L;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = threadIdx.x + k * blockDim.x;
        if (i < nvec) {
#pragma unroll
            for (int e = 0; e < E; ++e) v[k][e] *= f;
            store_vec<E>(zr + (long long)i * E, v[k]);
        }
    }
}

// One CTA of NT threads per row (256; 128 for rows of at most 16 KB and 64 for at most 8 KB,
// so more rows are in flight per SM); the row (up to its causal limit, rounded up to 16 bytes) is
// copied into shared memory by NP bulk copies of consecutive pieces, each completing on its own
// mbarrier, then read twice from there: (m, l), folded piece by piece as the pieces land, then z.
// Rows of more than 16 KB take two pieces, so the first half's (m, l) pass overlaps the second
// half's copy (measured on GB300: 64 KB bf16 rows 5826 against 5579 GB/s with one piece; 4 or 8
// pieces, or a 512-thread CTA, were slower; shorter rows gain nothing from pieces).
constexpr uint32_t kSmemRowBytes = 72 * 1024;

template <typename Tin, typename Tout, int NT, int NP>
__global__ void __launch_bounds__(NT)
softmax_ex_smem_kernel(const Tin *__restrict__ x, Tout *z, int T, long long xs, long long zs, float mult,
                       long long period, int *status) {
    constexpr int E = Vec<Tin>::E;
    extern __shared__ __align__(16) uint8_t srow[];
    __shared__ uint64_t bar[NP];
    __shared__ float sh[64];
    const long long row = blockIdx.x;
    const Tin *xr = x + row * xs;
    Tout *zr = z + row * zs;
    const int lim = (int)row_limit(row, T, period);
    const int nload = (lim + E - 1) / E;                 // 16-byte vectors copied
    const int per = (nload + NP - 1) / NP;               // vectors per piece (the last may have fewer)
    const uint32_t sbuf = ptx::smem_u32(srow);
    if (threadIdx.x == 0) {
#pragma unroll
        for (int q = 0; q < NP; ++q) ptx::mbar_init(ptx::smem_u32(&bar[q]), 1);
        ptx::mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            const int v0 = q * per, n = min(per, nload - v0);
            if (n > 0) {
                ptx::mbar_expect_tx(ptx::smem_u32(&bar[q]), (uint32_t)n * 16u);
                ptx::bulk_load(sbuf + (uint32_t)v0 * 16u, xr + (long long)v0 * E, (uint32_t)n * 16u,
                               ptx::smem_u32(&bar[q]));
            }
        }
    }
    const Tin *sx = reinterpret_cast<const Tin *>(srow);
    const float a = fabsf(mult);
    const uint32_t sgn = mult < 0.f ? Vec<Tin>::SGN : 0u;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
#pragma unroll 1
    for (int q = 0; q < NP; ++q) {
        const int v0 = q * per, v1 = min(nload, v0 + per);
        if (v1 <= v0) break;
        ok = ok && ptx::mbar_wait(ptx::smem_u32(&bar[q]), 0, nullptr);
        if (!ok) break;
        for (int i = v0 + threadIdx.x; i < v1; i += NT) {
            float f[E];
            Vec<Tin>::unpack(*reinterpret_cast<const uint4 *>(sx + i * E), sgn, f);
            fold_vec<E>(f, i * E, lim, a, m, l);
        }
    }
    if (!__syncthreads_and(ok)) {
        // a copy never completed: record it, give the copies a bounded chance to land, leave
        if (threadIdx.x == 0) {
            atomicExch(status, kStatusTimeout);
            for (int q = 0; q < NP; ++q) ptx::mbar_wait(ptx::smem_u32(&bar[q]), 0, nullptr, 20000000ull);
        }
        __syncthreads();
        return;
    }
    cta_merge_ml(m, l, sh);
    const float mref = (m == -INFINITY) ? 0.f : m;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int nvec = T / E;
    for (int i = threadIdx.x; i < nvec; i += NT) {
        float f[E];
        if (i < nload) Vec<Tin>::unpack(*reinterpret_cast<const uint4 *>(sx + i * E), sgn, f);
        emit_vec<E, Tout>(f, i * E, lim, i < nload, a, mref, inv, zr + (long long)i * E);
    }
}

// Rows of 32-64 KB, one CTA of NT threads per row: the first h vectors of the row are copied into
// shared memory by one bulk copy, the rest are loaded into registers (VPT 16-byte vectors per
// thread, kept packed), so a CTA needs half a row of shared memory and four rows are in flight
// per SM instead of three.  (m, l) over the register half while the copy lands, then over the
// shared half; z from both.
template <typename Tin, typename Tout, int NT, int VPT>
__global__ void __launch_bounds__(NT)
softmax_ex_split_kernel(const Tin *__restrict__ x, Tout *z, int T, long long xs, long long zs, float mult,
                        long long period, int *status) {
    constexpr int E = Vec<Tin>::E;
    extern __shared__ __align__(16) uint8_t srow[];
    __shared__ uint64_t bar;
    __shared__ float sh[64];
    const long long row = blockIdx.x;
    const Tin *xr = x + row * xs;
    Tout *zr = z + row * zs;
    const int lim = (int)row_limit(row, T, period);
    const int nvec = T / E, h = nvec - VPT * NT;           // vectors [0, h) in shared memory
    const int nload = (lim + E - 1) / E;                   // vectors that hold kept columns
    const int ns = min(h, nload);                          // of them, copied
    const uint32_t sbuf = ptx::smem_u32(srow);
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        ptx::mbar_init_fence();
        if (ns > 0) {
            ptx::mbar_expect_tx(ptx::smem_u32(&bar), (uint32_t)ns * 16u);
            ptx::bulk_load(sbuf, xr, (uint32_t)ns * 16u, ptx::smem_u32(&bar));
        }
    }
    // the register half: vector h + k * NT + threadIdx.x
    uint4 rv[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = h + k * NT + (int)threadIdx.x;
        rv[k] = (i < nload) ? __ldcs(reinterpret_cast<const uint4 *>(xr + (long long)i * E)) : make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    const float a = fabsf(mult);
    const uint32_t sgn = mult < 0.f ? Vec<Tin>::SGN : 0u;
    float m = -INFINITY, l = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = h + k * NT + (int)threadIdx.x;
        if (i < nload) {
            float f[E];
            Vec<Tin>::unpack(rv[k], sgn, f);
            fold_vec<E>(f, i * E, lim, a, m, l);
        }
    }
    const bool ok = ns <= 0 || ptx::mbar_wait(ptx::smem_u32(&bar), 0, nullptr);
    if (!__syncthreads_and(ok)) {
        // the copy never completed: record it, give it a bounded chance to land, leave
        if (threadIdx.x == 0) {
            atomicExch(status, kStatusTimeout);
            ptx::mbar_wait(ptx::smem_u32(&bar), 0, nullptr, 20000000ull);
        }
        __syncthreads();
        return;
    }
    const Tin *sx = reinterpret_cast<const Tin *>(srow);
    for (int i = threadIdx.x; i < ns; i += NT) {
        float f[E];
        Vec<Tin>::unpack(*reinterpret_cast<const uint4 *>(sx + i * E), sgn, f);
        fold_vec<E>(f, i * E, lim, a, m, l);
    }
    cta_merge_ml(m, l, sh);
    const float mref = (m == -INFINITY) ? 0.f : m;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    for (int i = threadIdx.x; i < h; i += NT) {
        float f[E];
        if (i < ns) Vec<Tin>::unpack(*reinterpret_cast<const uint4 *>(sx + i * E), sgn, f);
        emit_vec<E, Tout>(f, i * E, lim, i < ns, a, mref, inv, zr + (long long)i * E);
    }
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = h + k * NT + (int)threadIdx.x;
        if (i < nvec) {
            float f[E];
            Vec<Tin>::unpack(rv[k], sgn, f);
            emit_vec<E, Tout>(f, i * E, lim, i < nload, a, mref, inv, zr + (long long)i * E);
        }
    }
}

// Causal rows, two per CTA: rows i and P - 1 - i of one [P, T] score matrix (P <= T) keep
// i + 1 and P - i columns, P + 1 together, so both kept parts fit one row-sized buffer.  They
// are staged by two bulk copies (row A's vectors, then row B's) and each thread folds the
// vectors it reads into the state of the row they belong to; the two (m, l) states are merged
// over the CTA together; then both rows are written (0 past each row's limit).  Half the CTAs of
// one row per CTA, each with twice the bytes in flight.
template <typename Tin, typename Tout, int NT>
__global__ void __launch_bounds__(NT)
softmax_ex_pair_kernel(const Tin *__restrict__ x, Tout *z, long long rows, int T, long long xs, long long zs,
                       float mult, long long period, int *status) {
    constexpr int E = Vec<Tin>::E;
    extern __shared__ __align__(16) uint8_t srow[];
    __shared__ uint64_t bar;
    __shared__ float sh[2][64];
    const long long half = (period + 1) / 2;                  // CTAs per score matrix
    const long long blk = blockIdx.x / half, i = blockIdx.x % half;
    const long long ra = blk * period + i, rb = blk * period + (period - 1 - i);
    if (ra >= rows) return;                                   // past a last, partial matrix (rb > ra)
    const bool has_b = rb != ra && rb < rows;                 // the middle row of an odd P is alone
    const int la = (int)min((long long)T, i + 1), lb = has_b ? (int)min((long long)T, period - i) : 0;
    const int na = (la + E - 1) / E, nb = (lb + E - 1) / E;   // 16-byte vectors copied per row
    const Tin *xa = x + ra * xs, *xb = x + rb * xs;
    const uint32_t sbuf = ptx::smem_u32(srow);
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        ptx::mbar_init_fence();
        ptx::mbar_expect_tx(ptx::smem_u32(&bar), (uint32_t)(na + nb) * 16u);
        ptx::bulk_load(sbuf, xa, (uint32_t)na * 16u, ptx::smem_u32(&bar));
        if (nb > 0) ptx::bulk_load(sbuf + (uint32_t)na * 16u, xb, (uint32_t)nb * 16u, ptx::smem_u32(&bar));
    }
    __syncthreads();
    const bool ok = ptx::mbar_wait(ptx::smem_u32(&bar), 0, nullptr);
    if (!__syncthreads_and(ok)) {
        // the copies never completed: record it, give them a bounded chance to land, leave
        if (threadIdx.x == 0) {
            atomicExch(status, kStatusTimeout);
            ptx::mbar_wait(ptx::smem_u32(&bar), 0, nullptr, 20000000ull);
        }
        __syncthreads();
        return;
    }
    const Tin *sx = reinterpret_cast<const Tin *>(srow);
    const float a = fabsf(mult);
    const uint32_t sgn = mult < 0.f ? Vec<Tin>::SGN : 0u;
    float ma = -INFINITY, lA = 0.f, mb = -INFINITY, lB = 0.f;
    for (int v = threadIdx.x; v < na + nb; v += NT) {
        const bool in_b = v >= na;                            // row A or B
        float f[E];
        Vec<Tin>::unpack(*reinterpret_cast<const uint4 *>(sx + v * E), sgn, f);
        if (in_b) fold_vec<E>(f, (v - na) * E, lb, a, mb, lB);
        else fold_vec<E>(f, v * E, la, a, ma, lA);
    }
    cta_merge_ml(ma, lA, sh[0]);
    cta_merge_ml(mb, lB, sh[1]);
    const int nvec = T / E;
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        if (w == 1 && !has_b) break;
        const float mw = w ? mb : ma, lw = w ? lB : lA;
        const float mref = (mw == -INFINITY) ? 0.f : mw;
        const float inv = lw > 0.f ? 1.f / lw : 0.f;
        const int n = w ? nb : na, lim = w ? lb : la;
        const Tin *sw = sx + (w ? na : 0) * E;
        Tout *zr = z + (w ? rb : ra) * zs;
        for (int v = threadIdx.x; v < nvec; v += NT) {
            float f[E];
            if (v < n) Vec<Tin>::unpack(*reinterpret_cast<const uint4 *>(sw + v * E), sgn, f);
            emit_vec<E, Tout>(f, v * E, lim, v < n, a, mref, inv, zr + (long long)v * E);
        }
    }
}

// (m, l) of the kept columns of x[c0, c1) (values * mult), merged over the CTA.
template <typename Tin>
__device__ __forceinline__ void ex_range_state(const Tin *xr, long long c0, long long c1, float mult, float &m,
                                               float &l, float *sh) {
    m = -INFINITY;
    l = 0.f;
    for (long long i = c0 + threadIdx.x; i < c1; i += blockDim.x) {
        const float a = ld1(xr + i) * mult;
        const float mn = fmaxf(m, a);
        const float mr = (mn == -INFINITY) ? 0.f : mn;
        l = l * ex2_approx(m - mr) + ex2_approx(a - mr);
        m = mn;
    }
    cta_merge_ml(m, l, sh);
}

// z[c0, c1) = 2^(x * mult - m) / l for kept columns (j < lim), 0 after; from c1 down to c0.
template <typename Tin, typename Tout>
__device__ __forceinline__ void ex_range_norm(const Tin *xr, Tout *zr, long long c0, long long c1, long long lim,
                                              float mult, float m, float l) {
    const float mref = (m == -INFINITY) ? 0.f : m;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    for (long long i = c1 - 1 - threadIdx.x; i >= c0; i -= blockDim.x)
        zr[i] = from_f32<Tout>(i < lim ? ex2_approx(ld1(xr + i) * mult - mref) * inv : 0.f);
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kExChunkThreads)
softmax_ex_stream_kernel(const Tin *x, Tout *z, long long T, long long xs, long long zs, float mult,
                         long long period) {
    __shared__ float sh[64];
    const long long row = blockIdx.x;
    const long long lim = row_limit(row, T, period);
    float m, l;
    ex_range_state(x + row * xs, 0, lim, mult, m, l, sh);
    ex_range_norm(x + row * xs, z + row * zs, 0, T, lim, mult, m, l);
}

template <typename Tin>
__global__ void __launch_bounds__(kExChunkThreads)
softmax_ex_chunk_state_kernel(const Tin *x, long long T, long long xs, float mult, long long period,
                              long long chunk, float2 *ws) {
    __shared__ float sh[64];
    const long long row = blockIdx.y;
    const long long lim = row_limit(row, T, period);
    const long long c0 = (long long)blockIdx.x * chunk;
    const long long c1 = min(lim, c0 + chunk);
    float m, l;
    ex_range_state(x + row * xs, c0, c1, mult, m, l, sh);
    if (threadIdx.x == 0) ws[row * gridDim.x + blockIdx.x] = make_float2(m, l);
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kExChunkThreads)
softmax_ex_chunk_norm_kernel(const Tin *x, Tout *z, long long T, long long xs, long long zs, float mult,
                             long long period, long long chunk, const float2 *__restrict__ ws) {
    griddep_wait();   // launched as a dependent of the chunk-state kernel
    __shared__ float sh[64];
    const long long row = blockIdx.y;
    const int nch = gridDim.x;
    float m = -INFINITY, l = 0.f;
    for (int c = threadIdx.x; c < nch; c += blockDim.x) {
        const float2 st = ws[row * nch + c];
        merge_ml(m, l, st.x, st.y);
    }
    cta_merge_ml(m, l, sh);
    const long long c0 = (long long)blockIdx.x * chunk;
    const long long c1 = min(T, c0 + chunk);
    ex_range_norm(x + row * xs, z + row * zs, c0, c1, row_limit(row, T, period), mult, m, l);
}

bool al16(const void *p, long long stride_bytes) {
    return ((reinterpret_cast<uintptr_t>(p) | (uintptr_t)stride_bytes) & 15u) == 0;
}

template <typename Tin, typename Tout>
cudaError_t launch_typed(const SoftmaxExProblem &q, float *ws, cudaStream_t s) {
    const Tin *x = static_cast<const Tin *>(q.x);
    Tout *z = static_cast<Tout *>(q.z);
    constexpr int E = Vec<Tin>::E;
    const unsigned rows = (unsigned)q.rows;
    const bool aligned = q.T % E == 0 && al16(x, q.xs * (long long)sizeof(Tin)) &&
                         al16(z, q.zs * (long long)sizeof(Tout));
    if (aligned && q.period > 0 && q.period <= q.T && (uint64_t)q.T * sizeof(Tin) <= 8 * 1024) {
        // short causal rows: two complementary rows per CTA (buffer: P + 1 columns and the
        // rounding of two rows to whole vectors)
        const size_t smem = ((size_t)q.T / E + 2) * 16;
        const long long half = (q.period + 1) / 2;
        const long long ctas = (q.rows + q.period - 1) / q.period * half;
        if (ctas < (1LL << 31)) {
            softmax_ex_pair_kernel<Tin, Tout, 64><<<(unsigned)ctas, 64, smem, s>>>(x, z, q.rows, (int)q.T, q.xs, q.zs,
                                                                                  q.mult, q.period, q.status);
            count_launches(1);
            return cudaGetLastError();
        }
    }
    if (aligned && (uint64_t)q.T * sizeof(Tin) <= kSmemRowBytes) {
        const size_t smem = (size_t)q.T * sizeof(Tin);
        if (smem <= 8 * 1024) {
            softmax_ex_smem_kernel<Tin, Tout, 64, 1><<<rows, 64, smem, s>>>(x, z, (int)q.T, q.xs, q.zs, q.mult,
                                                                                  q.period, q.status);
        } else if (smem <= 16 * 1024) {
            softmax_ex_smem_kernel<Tin, Tout, 128, 1><<<rows, 128, smem, s>>>(x, z, (int)q.T, q.xs, q.zs,
                                                                                    q.mult, q.period, q.status);
        } else if (q.T / E > 8 * 256 && q.T / E <= 2 * 8 * 256) {
            // 32-64 KB rows: half in shared memory, 8 vectors per thread in registers
            const size_t hsmem = (size_t)(q.T / E - 8 * 256) * 16;
            softmax_ex_split_kernel<Tin, Tout, 256, 8><<<rows, 256, hsmem, s>>>(x, z, (int)q.T, q.xs, q.zs, q.mult,
                                                                                 q.period, q.status);
        } else {
            const cudaError_t attr_err = set_max_dynamic_smem(
                (const void *)softmax_ex_smem_kernel<Tin, Tout, 256, 2>, (int)kSmemRowBytes);
            if (attr_err != cudaSuccess) return attr_err;
            softmax_ex_smem_kernel<Tin, Tout, 256, 2><<<rows, 256, smem, s>>>(x, z, (int)q.T, q.xs, q.zs,
                                                                                        q.mult, q.period, q.status);
        }
        count_launches(1);
        return cudaGetLastError();
    }
    if (q.T <= kExMaxResidentT && aligned) {
        const int nvec = (int)(q.T / E);
        int vpt = 1;
        while (vpt < 32 / E && nvec > 1024 * vpt) vpt *= 2;
        int threads = (nvec + vpt - 1) / vpt;
        threads = ((threads + 31) / 32) * 32;
        const int T = (int)q.T;
        switch (vpt) {
            case 1: softmax_ex_onchip_kernel<Tin, Tout, 1><<<rows, threads, 0, s>>>(x, z, T, q.xs, q.zs, q.mult, q.period); break;
            case 2: softmax_ex_onchip_kernel<Tin, Tout, 2><<<rows, threads, 0, s>>>(x, z, T, q.xs, q.zs, q.mult, q.period); break;
            case 4: softmax_ex_onchip_kernel<Tin, Tout, 4><<<rows, threads, 0, s>>>(x, z, T, q.xs, q.zs, q.mult, q.period); break;
            default:
                if constexpr (E == 4)
                    softmax_ex_onchip_kernel<Tin, Tout, 8><<<rows, threads, 0, s>>>(x, z, T, q.xs, q.zs, q.mult, q.period);
                break;
        }
        count_launches(1);
        return cudaGetLastError();
    }
    if (q.T <= kExMaxResidentT) {
        softmax_ex_stream_kernel<Tin, Tout><<<rows, kExChunkThreads, 0, s>>>(x, z, q.T, q.xs, q.zs, q.mult, q.period);
        count_launches(1);
        return cudaGetLastError();
    }
    long long chunk;
    int nch;
    softmax_ex_chunk_geometry(q.rows, q.T, q.sm_count, chunk, nch);
    dim3 grid(nch, rows);
    float2 *w2 = reinterpret_cast<float2 *>(ws);
    softmax_ex_chunk_state_kernel<Tin><<<grid, kExChunkThreads, 0, s>>>(x, q.T, q.xs, q.mult, q.period, chunk, w2);
    cudaError_t e = launch_dependent(softmax_ex_chunk_norm_kernel<Tin, Tout>, grid, dim3(kExChunkThreads), 0, s, x, z,
                                     q.T, q.xs, q.zs, q.mult, q.period, chunk, (const float2 *)w2);
    if (e != cudaSuccess) return e;
    count_launches(2);
    return cudaGetLastError();
}

}  // namespace

void softmax_ex_chunk_geometry(long long rows, long long T, int sm_count, long long &chunk, int &nch) {
    // about four resident CTAs per SM over the whole problem, chunks of at least 8192 elements
    const long long target_ctas = 4LL * sm_count;
    long long per_row = (target_ctas + rows - 1) / rows;
    const long long max_per_row = (T + 8191) / 8192;
    if (per_row > max_per_row) per_row = max_per_row;
    if (per_row < 1) per_row = 1;
    if (per_row > 65535) per_row = 65535;
    chunk = (T + per_row - 1) / per_row;
    nch = (int)((T + chunk - 1) / chunk);
}

size_t softmax_ex_workspace_floats(long long rows, long long T, int sm_count) {
    if (T <= kExMaxResidentT) return 0;
    long long chunk;
    int nch;
    softmax_ex_chunk_geometry(rows, T, sm_count, chunk, nch);
    return (size_t)rows * nch * 2;
}

cudaError_t launch_softmax_ex(const SoftmaxExProblem &q, float *ws, cudaStream_t s) {
    if (q.x_dtype == OSF_F32 && q.z_dtype == OSF_F32) return launch_typed<float, float>(q, ws, s);
    if (q.x_dtype == OSF_F32) return launch_typed<float, __nv_bfloat16>(q, ws, s);
    if (q.z_dtype == OSF_F32) return launch_typed<__nv_bfloat16, float>(q, ws, s);
    return launch_typed<__nv_bfloat16, __nv_bfloat16>(q, ws, s);
}

}  // namespace osf
