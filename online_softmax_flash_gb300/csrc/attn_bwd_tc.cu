// Attention backward on the tcgen05 tensor cores (bf16, D in {64, 128}): the same chain rule as
// attn_bwd.cu (dV = P^T dO, dS = P * (dO V^T - D), dQ = scale dS K, dK = scale dS^T Q, P rebuilt
// from the forward's log-sum-exp), with every product a tcgen05.mma into TMEM and the operand
// tiles streamed by TMA, as in the forward kernel.
//
// dQ kernel: one CTA per (b, q head, 128 query rows).  Warp 0 loads Q and dO once and streams
// K, V tiles (128 keys) through a ring; warp 1 issues S = Q K^T and dP = dO V^T (both operands in
// shared memory) into TMEM, then dQ += dS K with dS read from TMEM; warps 4-7 (thread r = row r)
// rebuild P, form dS = P (dP - D_r) and write it as bf16 over S.
//
// dK/dV kernel: one CTA per (b, kv head, 128 keys) walks every query head of the group and every
// query tile that sees these keys: S^T = K Q^T, dP^T = V dO^T, then dV += P^T dO and
// dK += dS^T Q with P^T and dS^T read from TMEM; thread r owns key r, so each column (query) of
// P^T needs that query's lse and D, read from a small shared-memory table per tile.
//
// TMEM (dQ): S [0,128), dP [128,256), dQ [256,256+D).  (dK/dV): S^T [0,128), dP^T [128,256),
// dK [256,256+D), dV [256+D,256+2D).  bf16 P / dS overwrite the first 64 columns of their region.
// Every wait is bounded (2 s): on expiry the CTA records OSF_ERR_TIMEOUT, drains, frees TMEM.
#include <mutex>

#include "attn_bwd.cuh"
#include "attn_bwd_tc.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.cuh"

namespace osf {
namespace {

using namespace ptx;

constexpr int TB = 128;                 // rows (queries or keys) per tile
constexpr int NT_THREADS = 256;         // warp 0 TMA, warp 1 MMA, warps 4-7 compute
constexpr int MAX_RING = 8;
constexpr uint32_t TMEM_COLS = 512;

template <int D>
struct BtCfg {
    // ring stages of one [128 x D] bf16 tile each; at D = 64 the deeper ring also keeps one CTA
    // per SM, so the CTAs do not queue for TMEM (each takes all 512 columns)
    static constexpr int RING = D == 64 ? 8 : 4;
    static constexpr uint32_t TILE = TB * D * 2;
    static constexpr uint32_t DBLK = TB * 128;                  // bytes between 64-column blocks
    static constexpr uint32_t A_OFF = 0;                        // two resident tiles (Q, dO) or (K, V)
    static constexpr uint32_t RING_OFF = 2 * TILE;
    static constexpr uint32_t TAB_OFF = RING_OFF + RING * TILE;  // lse / D tables (dK/dV kernel)
    static constexpr uint32_t SMEM_BYTES = TAB_OFF + 4 * TB * 4 + 1024;
    static constexpr uint32_t IDESC_SS = idesc_bf16_f32(TB, TB, 0, 0);   // [128 x 128] scores
    static constexpr uint32_t IDESC_TS = idesc_bf16_f32(TB, D, 0, 1);    // [128 x D] += P [128 x 128] X
};

struct BtBars {
    uint64_t a_full;
    uint64_t full[MAX_RING], empty[MAX_RING];
    uint64_t s_full, p_full, done, drain;
};

__device__ __forceinline__ void bt_timeout(volatile int *abort, int *status) {
    *abort = 1;
    if (status) atomicExch(status, kStatusTimeout);
}
__device__ __forceinline__ void bt_settle() {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000ull) {
    }
}

// X (+)= A(tmem, bf16 [128 x 128]) * B(smem tile [128 x D], MN-major): 8 k-steps of 16 rows.
template <int D>
__device__ __forceinline__ void issue_ts(uint32_t dst, uint32_t a_tmem, uint32_t b_tile, bool acc) {
    using C = BtCfg<D>;
    const uint64_t bd = sdesc_sw128(b_tile, C::DBLK, 1024);
#pragma unroll
    for (int k = 0; k < TB / 16; ++k) mma_ts(dst, a_tmem + k * 8, bd + ((k * 2048) >> 4), C::IDESC_TS, acc || k > 0);
}
// X = A(smem tile [128 x D]) * B(smem tile [128 x D])^T: D/16 k-steps.
template <int D>
__device__ __forceinline__ void issue_ss(uint32_t dst, uint32_t a_tile, uint32_t b_tile) {
    using C = BtCfg<D>;
    const uint64_t ad = sdesc_sw128(a_tile, 16, 1024), bd = sdesc_sw128(b_tile, 16, 1024);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = ((k >> 2) * C::DBLK + (k & 3) * 32) >> 4;
        mma_ss(dst, ad + off, bd + off, C::IDESC_SS, k > 0);
    }
}

// ====================================================================== dQ
template <int D>
__global__ void __launch_bounds__(NT_THREADS, 1)
bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mg,
                 const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv, const BwdProblem p) {
    using C = BtCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ BtBars bars;
    __shared__ uint32_t tmem_sh;
    __shared__ volatile int abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = sbase + C::A_OFF, sG = sQ + C::TILE, sRing = sbase + C::RING_OFF;
    const int q0 = blockIdx.x * TB;
    const int bh = blockIdx.y, b = bh / p.Hq, hq = bh % p.Hq;
    const int kvh = hq / (p.Hq / p.Hkv);
    int n = (p.Sk + TB - 1) / TB;   // key tiles these rows see
    if (p.causal) {
        const int last = min(q0 + TB - 1, p.Sq - 1) + p.causal_off;
        n = min(n, last < 0 ? 0 : last / TB + 1);
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_sh), TMEM_COLS);
    if (tid == 32) {
        mbar_init(smem_u32(&bars.a_full), 1);
        for (int s = 0; s < C::RING; ++s) {
            mbar_init(smem_u32(&bars.full[s]), 1);
            mbar_init(smem_u32(&bars.empty[s]), 1);
        }
        mbar_init(smem_u32(&bars.s_full), 1);
        mbar_init(smem_u32(&bars.p_full), 4);
        mbar_init(smem_u32(&bars.done), 1);
        mbar_init(smem_u32(&bars.drain), 1);
        abort_flag = 0;
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_sh;
    const uint32_t tS = tmem, tP = tmem + 128, tQ = tmem + 256;

    if (warp == 0 && lane == 0 && n > 0) {
        // ------------------------------------------------------------ TMA: Q, dO; then K_j V_j
        bool ok = true;
        mbar_expect_tx(smem_u32(&bars.a_full), 2 * C::TILE);
        tma_load_5d(sQ, &mq, smem_u32(&bars.a_full), 0, q0, 0, hq, b);
        tma_load_5d(sG, &mg, smem_u32(&bars.a_full), 0, q0, 0, hq, b);
        for (int m = 0; m < 2 * n && ok; ++m) {
            const int st = m % C::RING;
            ok = mbar_wait(smem_u32(&bars.empty[st]), ((m / C::RING) & 1) ^ 1, &abort_flag);
            if (!ok) break;
            mbar_expect_tx(smem_u32(&bars.full[st]), C::TILE);
            tma_load_5d(sRing + st * C::TILE, (m & 1) ? &mv : &mk, smem_u32(&bars.full[st]), 0, (m >> 1) * TB, 0, kvh,
                        b);
        }
        if (!ok) {
            bt_timeout(&abort_flag, p.status);
            bt_settle();
        }
    } else if (warp == 1 && lane == 0 && n > 0) {
        // ------------------------------------------------------------ MMA issue
        auto wait_full = [&](int m) {
            return mbar_wait_spin(smem_u32(&bars.full[m % C::RING]), (m / C::RING) & 1, &abort_flag);
        };
        bool ok = mbar_wait_spin(smem_u32(&bars.a_full), 0, &abort_flag);
        if (ok) ok = wait_full(0) && wait_full(1);
        if (ok) {
            tc_fence_after();
            issue_ss<D>(tS, sQ, sRing + 0 * C::TILE);          // S = Q K_0^T
            issue_ss<D>(tP, sG, sRing + 1 * C::TILE);          // dP = dO V_0^T
            mma_commit(smem_u32(&bars.s_full));
            mma_commit(smem_u32(&bars.empty[1 % C::RING]));       // V_0 is done
        }
        for (int j = 0; j < n && ok; ++j) {
            const int mk_ = 2 * j;
            ok = mbar_wait_spin(smem_u32(&bars.p_full), j & 1, &abort_flag);
            if (!ok) break;
            tc_fence_after();
            issue_ts<D>(tQ, tS, sRing + (mk_ % C::RING) * C::TILE, j > 0);   // dQ += dS K_j
            mma_commit(smem_u32(&bars.empty[mk_ % C::RING]));                // K_j is done
            if (j + 1 < n) {
                ok = wait_full(mk_ + 2) && wait_full(mk_ + 3);
                if (!ok) break;
                tc_fence_after();
                issue_ss<D>(tS, sQ, sRing + ((mk_ + 2) % C::RING) * C::TILE);
                issue_ss<D>(tP, sG, sRing + ((mk_ + 3) % C::RING) * C::TILE);
                mma_commit(smem_u32(&bars.s_full));
                mma_commit(smem_u32(&bars.empty[(mk_ + 3) % C::RING]));
            }
        }
        if (ok) mma_commit(smem_u32(&bars.done));
        else bt_timeout(&abort_flag, p.status);
        mma_commit(smem_u32(&bars.drain));
        mbar_wait(smem_u32(&bars.drain), 0, nullptr, 20000000ull);
    } else if (warp >= 4) {
        // ------------------------------------------------------------ compute: dS, then dQ out
        const int r = tid - 128, row = q0 + r;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const bool row_ok = row < p.Sq;
        const long long grow = (long long)bh * p.Sq + row;
        const float lse2 = row_ok ? p.lse[grow] * kLog2e : INFINITY;
        const float dvr = row_ok ? p.dvec[grow] : 0.f;
        const float c2 = p.scale_log2;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            ok = mbar_wait(smem_u32(&bars.s_full), j & 1, &abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const int key0 = j * TB;
            int lim = p.Sk - key0;
            if (p.causal) lim = min(lim, row + p.causal_off - key0 + 1);
            if (!row_ok) lim = 0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t s[32], dp[32];
                tmem_ld32(tS + lane_off + c * 32, s);
                tmem_ld32(tP + lane_off + c * 32, dp);
                tmem_ld_wait();
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    float d0 = 0.f, d1 = 0.f;
                    const int col = c * 32 + 2 * k;
                    if (col < lim)
                        d0 = ex2_approx(__uint_as_float(s[2 * k]) * c2 - lse2) * (__uint_as_float(dp[2 * k]) - dvr);
                    if (col + 1 < lim)
                        d1 = ex2_approx(__uint_as_float(s[2 * k + 1]) * c2 - lse2) * (__uint_as_float(dp[2 * k + 1]) - dvr);
                    pk[k] = pack_bf16x2(d0, d1);
                }
                // columns 16c .. 16c+15 hold S chunk c/2, already read
                tmem_st16(tS + lane_off + c * 16, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7], pk[8], pk[9],
                          pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars.p_full));
        }
        if (!ok) bt_timeout(&abort_flag, p.status);
        // epilogue: dQ = scale * (dS K summed over key tiles); rows with no key get 0
        bool have = false;
        if (ok && n > 0) {
            have = mbar_wait(smem_u32(&bars.done), 0, &abort_flag);
            have = __all_sync(0xffffffffu, have);
            if (!have) bt_timeout(&abort_flag, p.status);
            tc_fence_after();
        }
        __nv_bfloat16 *dq = static_cast<__nv_bfloat16 *>(p.dq) + grow * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            if (have) {
                tmem_ld32(tQ + lane_off + c * 32, o);
                tmem_ld_wait();
            }
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
                pk[k] = have ? pack_bf16x2(__uint_as_float(o[2 * k]) * p.scale, __uint_as_float(o[2 * k + 1]) * p.scale) : 0u;
            if (row_ok) {
                uint4 *dst = reinterpret_cast<uint4 *>(dq + c * 32);
#pragma unroll
                for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
            }
        }
    }
    tc_fence_before();
    __syncwarp();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ====================================================================== dK, dV
template <int D>
__global__ void __launch_bounds__(NT_THREADS, 1)
bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mg,
                   const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv, const BwdProblem p) {
    using C = BtCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ BtBars bars;
    __shared__ uint32_t tmem_sh;
    __shared__ volatile int abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sK = sbase + C::A_OFF, sV = sK + C::TILE, sRing = sbase + C::RING_OFF;
    float *tab = reinterpret_cast<float *>(smem_raw + (sbase - smem_u32(smem_raw)) + C::TAB_OFF);   // [2][2][128]
    const int key0 = blockIdx.x * TB;
    const int bk = blockIdx.y, b = bk / p.Hkv, kvh = bk % p.Hkv;
    const int G = p.Hq / p.Hkv;
    // query tiles that see a key of this block: from the first row that sees key0
    int q_first = p.causal ? max(0, key0 - p.causal_off) : 0;
    q_first /= TB;
    const int n_qt = (p.Sq + TB - 1) / TB;
    const int per_head = max(0, n_qt - q_first);
    const int n = G * per_head;   // steps: (head g, query tile) pairs
    if (warp == 0) tmem_alloc(smem_u32(&tmem_sh), TMEM_COLS);
    if (tid == 32) {
        mbar_init(smem_u32(&bars.a_full), 1);
        for (int s = 0; s < C::RING; ++s) {
            mbar_init(smem_u32(&bars.full[s]), 1);
            mbar_init(smem_u32(&bars.empty[s]), 1);
        }
        mbar_init(smem_u32(&bars.s_full), 1);
        mbar_init(smem_u32(&bars.p_full), 4);
        mbar_init(smem_u32(&bars.done), 1);
        mbar_init(smem_u32(&bars.drain), 1);
        abort_flag = 0;
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_sh;
    const uint32_t tS = tmem, tP = tmem + 128, tK = tmem + 256, tV = tmem + 256 + D;
    auto step_at = [&](int m, int &hq, int &qt) {
        hq = kvh * G + m / per_head;
        qt = q_first + m % per_head;
    };

    if (warp == 0 && lane == 0 && n > 0) {
        // ------------------------------------------------------------ TMA: K, V; then Q_m dO_m
        bool ok = true;
        mbar_expect_tx(smem_u32(&bars.a_full), 2 * C::TILE);
        tma_load_5d(sK, &mk, smem_u32(&bars.a_full), 0, key0, 0, kvh, b);
        tma_load_5d(sV, &mv, smem_u32(&bars.a_full), 0, key0, 0, kvh, b);
        for (int m = 0; m < 2 * n && ok; ++m) {
            const int st = m % C::RING;
            ok = mbar_wait(smem_u32(&bars.empty[st]), ((m / C::RING) & 1) ^ 1, &abort_flag);
            if (!ok) break;
            int hq, qt;
            step_at(m >> 1, hq, qt);
            mbar_expect_tx(smem_u32(&bars.full[st]), C::TILE);
            tma_load_5d(sRing + st * C::TILE, (m & 1) ? &mg : &mq, smem_u32(&bars.full[st]), 0, qt * TB, 0, hq, b);
        }
        if (!ok) {
            bt_timeout(&abort_flag, p.status);
            bt_settle();
        }
    } else if (warp == 1 && lane == 0 && n > 0) {
        // ------------------------------------------------------------ MMA issue
        auto wait_full = [&](int m) {
            return mbar_wait_spin(smem_u32(&bars.full[m % C::RING]), (m / C::RING) & 1, &abort_flag);
        };
        bool ok = mbar_wait_spin(smem_u32(&bars.a_full), 0, &abort_flag);
        if (ok) ok = wait_full(0) && wait_full(1);
        if (ok) {
            tc_fence_after();
            issue_ss<D>(tS, sK, sRing + 0 * C::TILE);          // S^T = K Q_0^T
            issue_ss<D>(tP, sV, sRing + 1 * C::TILE);          // dP^T = V dO_0^T
            mma_commit(smem_u32(&bars.s_full));
        }
        for (int j = 0; j < n && ok; ++j) {
            const int mq_ = 2 * j, mg_ = 2 * j + 1;
            ok = mbar_wait_spin(smem_u32(&bars.p_full), j & 1, &abort_flag);
            if (!ok) break;
            tc_fence_after();
            issue_ts<D>(tV, tS, sRing + (mg_ % C::RING) * C::TILE, j > 0);   // dV += P^T dO
            issue_ts<D>(tK, tP, sRing + (mq_ % C::RING) * C::TILE, j > 0);   // dK += dS^T Q
            mma_commit(smem_u32(&bars.empty[mq_ % C::RING]));
            mma_commit(smem_u32(&bars.empty[mg_ % C::RING]));
            if (j + 1 < n) {
                ok = wait_full(mq_ + 2) && wait_full(mg_ + 2);
                if (!ok) break;
                tc_fence_after();
                issue_ss<D>(tS, sK, sRing + ((mq_ + 2) % C::RING) * C::TILE);
                issue_ss<D>(tP, sV, sRing + ((mg_ + 2) % C::RING) * C::TILE);
                mma_commit(smem_u32(&bars.s_full));
            }
        }
        if (ok) mma_commit(smem_u32(&bars.done));
        else bt_timeout(&abort_flag, p.status);
        mma_commit(smem_u32(&bars.drain));
        mbar_wait(smem_u32(&bars.drain), 0, nullptr, 20000000ull);
    } else if (warp >= 4) {
        // ------------------------------------------------------------ compute: P^T, dS^T
        const int r = tid - 128, key = key0 + r;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const float c2 = p.scale_log2;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            int hq, qt;
            step_at(j, hq, qt);
            const int qbase = qt * TB;
            // this step's per-query lse (base 2) and D, double-buffered between steps
            float *tl = tab + (j & 1) * 2 * TB, *td = tl + TB;
            {
                const int q = qbase + r;
                const long long gq = ((long long)b * p.Hq + hq) * p.Sq + q;
                tl[r] = q < p.Sq ? p.lse[gq] * kLog2e : INFINITY;
                td[r] = q < p.Sq ? p.dvec[gq] : 0.f;
            }
            // every warp passes this barrier once per step, even after a failed wait (then it
            // skips the work), so no warp can wait here for one that has left the loop
            named_barrier(1, 128);
            if (!ok) continue;
            ok = mbar_wait(smem_u32(&bars.s_full), j & 1, &abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) continue;
            tc_fence_after();
            // query column q is visible to this key iff q < Sq, key < Sk and (causal) key <= q + off
            int qmin = 0;   // first visible column of the tile
            if (p.causal) qmin = key - p.causal_off - qbase;
            const int qmax = min(TB, p.Sq - qbase);   // columns past the sequence are out
            const bool key_ok = key < p.Sk;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t s[32], dp[32];
                tmem_ld32(tS + lane_off + c * 32, s);
                tmem_ld32(tP + lane_off + c * 32, dp);
                tmem_ld_wait();
                uint32_t pp[16], pd[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    float p0 = 0.f, p1 = 0.f, d0 = 0.f, d1 = 0.f;
                    const int col = c * 32 + 2 * k;
                    if (key_ok && col >= qmin && col < qmax) {
                        p0 = ex2_approx(__uint_as_float(s[2 * k]) * c2 - tl[col]);
                        d0 = p0 * (__uint_as_float(dp[2 * k]) - td[col]);
                    }
                    if (key_ok && col + 1 >= qmin && col + 1 < qmax) {
                        p1 = ex2_approx(__uint_as_float(s[2 * k + 1]) * c2 - tl[col + 1]);
                        d1 = p1 * (__uint_as_float(dp[2 * k + 1]) - td[col + 1]);
                    }
                    pp[k] = pack_bf16x2(p0, p1);
                    pd[k] = pack_bf16x2(d0, d1);
                }
                tmem_st16(tS + lane_off + c * 16, pp[0], pp[1], pp[2], pp[3], pp[4], pp[5], pp[6], pp[7], pp[8], pp[9],
                          pp[10], pp[11], pp[12], pp[13], pp[14], pp[15]);
                tmem_st16(tP + lane_off + c * 16, pd[0], pd[1], pd[2], pd[3], pd[4], pd[5], pd[6], pd[7], pd[8], pd[9],
                          pd[10], pd[11], pd[12], pd[13], pd[14], pd[15]);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars.p_full));
        }
        if (!ok) bt_timeout(&abort_flag, p.status);
        // epilogue: dK = scale * dS^T Q, dV = P^T dO (zero when no query sees this key)
        bool have = false;
        if (ok && n > 0) {
            have = mbar_wait(smem_u32(&bars.done), 0, &abort_flag);
            have = __all_sync(0xffffffffu, have);
            if (!have) bt_timeout(&abort_flag, p.status);
            tc_fence_after();
        }
        // the TMEM loads are warp-collective (.sync.aligned): every lane issues them, and only
        // the stores of keys past Sk are skipped
        const bool key_ok = key < p.Sk;
        const long long gk = (long long)bk * p.Sk + (key_ok ? key : 0);
        __nv_bfloat16 *dk = static_cast<__nv_bfloat16 *>(p.dk) + gk * D;
        __nv_bfloat16 *dv = static_cast<__nv_bfloat16 *>(p.dv) + gk * D;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t src = (h ? tV : tK) + lane_off;
            const float sc = h ? 1.f : p.scale;
            __nv_bfloat16 *out = h ? dv : dk;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                if (have) {
                    tmem_ld32(src + c * 32, o);
                    tmem_ld_wait();
                }
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    pk[k] = have ? pack_bf16x2(__uint_as_float(o[2 * k]) * sc, __uint_as_float(o[2 * k + 1]) * sc) : 0u;
                if (key_ok) {
                    uint4 *dst = reinterpret_cast<uint4 *>(out + c * 32);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncwarp();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

template <int D>
cudaError_t launch_t(const BwdProblem &p, cudaStream_t s) {
    using C = BtCfg<D>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(bwd_dq_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)C::SMEM_BYTES);
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(bwd_dkdv_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)C::SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const long long qs = (long long)p.Sq * D, ks = (long long)p.Sk * D;
    CUtensorMap mq, mg, mk, mv;
    if (!make_bf16_tile_map_strided(&mq, p.q, D, p.Sq, p.Hq, p.B, D, qs, qs * p.Hq, TB) ||
        !make_bf16_tile_map_strided(&mg, p.dout, D, p.Sq, p.Hq, p.B, D, qs, qs * p.Hq, TB) ||
        !make_bf16_tile_map_strided(&mk, p.k, D, p.Sk, p.Hkv, p.B, D, ks, ks * p.Hkv, TB) ||
        !make_bf16_tile_map_strided(&mv, p.v, D, p.Sk, p.Hkv, p.B, D, ks, ks * p.Hkv, TB))
        return cudaErrorInvalidValue;
    bwd_dkdv_tc_kernel<D><<<dim3((p.Sk + TB - 1) / TB, p.B * p.Hkv), NT_THREADS, C::SMEM_BYTES, s>>>(mq, mg, mk, mv, p);
    bwd_dq_tc_kernel<D><<<dim3((p.Sq + TB - 1) / TB, p.B * p.Hq), NT_THREADS, C::SMEM_BYTES, s>>>(mq, mg, mk, mv, p);
    count_launches(2);
    return cudaGetLastError();
}

}  // namespace

bool attn_bwd_tc_supported(const BwdProblem &p) {
    if (p.dtype != OSF_BF16 || (p.D != 64 && p.D != 128)) return false;
    const uintptr_t a = reinterpret_cast<uintptr_t>(p.q) | reinterpret_cast<uintptr_t>(p.k) |
                        reinterpret_cast<uintptr_t>(p.v) | reinterpret_cast<uintptr_t>(p.dout) |
                        reinterpret_cast<uintptr_t>(p.dq) | reinterpret_cast<uintptr_t>(p.dk) |
                        reinterpret_cast<uintptr_t>(p.dv);
    if ((a & 15u) != 0) return false;
    if ((p.Sk + TB - 1) / TB >= 65536 * 32 || (long long)p.B * p.Hq >= 65536) return false;
    return tensor_map_encoder() != nullptr;
}

cudaError_t launch_attn_bwd_tc(const BwdProblem &p, cudaStream_t s) {
    return p.D == 64 ? launch_t<64>(p, s) : launch_t<128>(p, s);
}

}  // namespace osf
