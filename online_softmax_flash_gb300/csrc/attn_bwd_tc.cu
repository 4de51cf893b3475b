// Attention backward on the tcgen05 tensor cores (bf16, D in {64, 128}): the same chain rule as
// attn_bwd.cu (dV = P^T dO, dS = P * (dO V^T - D), dQ = scale dS K, dK = scale dS^T Q, P rebuilt
// from the forward's log-sum-exp), with every product a tcgen05.mma into TMEM and the operand
// tiles streamed by TMA, as in the forward kernel.
//
// Warp roles (384 threads): warp 0 issues the TMA loads, warps 1 and 3 the MMAs (one thread each,
// two independent instruction streams: one thread cannot issue tcgen05.mma as fast as the tensor
// pipe runs M128 N128 products), warp 2 (dK/dV kernel) fills a small ring of per-query lse / D
// tables, warps 4-11 compute.  Compute warp w owns the
// TMEM lanes 32 (w % 4) .. +31 (one row of the tile per thread) and one half of the 128 columns,
// h = (w - 4) / 4, so two warps share each sub-partition.
//
// Each step works in two phases that let the tensor pipe run ahead of the compute warps:
//   phase A reads the scores, rebuilds P (kept in fp32 registers) and releases the score
//   columns; phase B reads dP and forms dS = P (dP - D).
//
// dK/dV kernel: one CTA per (b, kv head, 128 keys), K and V resident, walking every query tile
// of every query head of the group that sees these keys.  Per step j (query tile Q_j, dO_j):
//   S^T = K Q_j^T, dP^T = V dO_j^T;  A: P^T as bf16 over the first half of each warp's S^T
//   columns, then dV += P^T dO_j;  B: dS^T over dP^T, then dK += dS^T Q_j.
//   Issuer A: dV_j then S^T_{j+1} (while phase B runs); issuer B: dK_j then dP^T_{j+1} (while
//   phase A of step j+1 runs).
// dQ, two ways.  With a dS workspace (the default) the dK/dV CTAs also store dS^T and a separate
// persistent product computes dQ = scale * dS K over it (bwd_dq_gemm_kernel, below).  Without
// one, dQ CTAs run in the dK/dV grid: one CTA per (b, q head, 128 query rows), Q and dO
// resident, K_j, V_j streamed: S = Q K_j^T, dP = dO V_j^T;  phase A releases S (issuer A issues
// S_{j+1} at once);  phase B writes dS as bf16 into its own columns, then issuer B issues
// dQ += dS K_j and dP_{j+1}.
//
// TMEM (512 columns).  dK/dV: S^T [0,128), dP^T [128,256), dK [256,256+D), dV [256+D,256+2D).
// dQ: S [0,128), dP [128,256), dQ [256,256+D), dS (bf16) [256+D,256+D+64).
// Every wait is bounded (2 s): on expiry the CTA records OSF_ERR_TIMEOUT, drains, frees TMEM.
// TMEM loads and stores are warp-collective: every lane of a warp issues them, and only the
// global stores of rows outside the problem are skipped.
#include <climits>
#include <mutex>

#include "attn_bwd.cuh"
#include "attn_bwd_tc.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.cuh"

namespace osf {
namespace {

using namespace ptx;

constexpr int TB = 128;                 // rows (queries or keys) per tile
constexpr int NT_THREADS = 384;         // warps 0-3 control, 4-11 compute
constexpr int NCW = 8;                  // compute warps
constexpr int MAX_RING = 8;
constexpr int TSTAGES = 4;              // lse / D table stages (dK/dV kernel)
constexpr uint32_t TMEM_COLS = 512;

template <int D>
struct BtCfg {
    // ring stages of one [128 x D] bf16 tile each
    static constexpr int RING = D == 64 ? 8 : 4;
    static constexpr uint32_t TILE = TB * D * 2;
    static constexpr uint32_t DBLK = TB * 128;                  // bytes between 64-column blocks
    static constexpr uint32_t A_OFF = 0;                        // two resident tiles (Q, dO) or (K, V)
    static constexpr uint32_t RING_OFF = 2 * TILE;
    static constexpr uint32_t TAB_OFF = RING_OFF + RING * TILE;  // [TSTAGES][2][128] floats
    // dK/dV with a dS workspace: a 2 KB staging tile per compute warp for the TMA stores of dS^T
    static constexpr uint32_t STG_OFF = TAB_OFF + TSTAGES * 2 * TB * 4;
    static constexpr uint32_t SMEM_BYTES = STG_OFF + NCW * 2048 + 1024;
    static constexpr uint32_t IDESC_SS = idesc_bf16_f32(TB, TB, 0, 0);   // [128 x 128] scores
    static constexpr uint32_t IDESC_TS = idesc_bf16_f32(TB, D, 0, 1);    // [128 x D] += P [128 x 128] X
};

struct BtBars {
    uint64_t a_full;
    uint64_t full[MAX_RING], empty[MAX_RING];
    uint64_t t_full[TSTAGES], t_empty[TSTAGES];
    uint64_t s_full, dp_full, pa, pb, done, drain[2];
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
// A's k-steps 0-3 start at column `a_lo`, 4-7 at `a_hi` (two warps write the two halves).
template <int D>
__device__ __forceinline__ void issue_ts(uint32_t dst, uint32_t a_lo, uint32_t a_hi, uint32_t b_tile, bool acc) {
    using C = BtCfg<D>;
    const uint64_t bd = sdesc_sw128(b_tile, C::DBLK, 1024);
#pragma unroll
    for (int k = 0; k < TB / 16; ++k)
        mma_ts(dst, (k < 4 ? a_lo : a_hi - 32) + k * 8, bd + ((k * 2048) >> 4), C::IDESC_TS, acc || k > 0);
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

// 32 floats as bf16 pairs `pk` into 16 TMEM columns.
__device__ __forceinline__ void pack_store16(uint32_t taddr, const float (&v)[32], uint32_t (&pk)[16]) {
#pragma unroll
    for (int k = 0; k < 16; ++k) pk[k] = pack_bf16x2(v[2 * k], v[2 * k + 1]);
    tmem_st16(taddr, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7], pk[8], pk[9], pk[10], pk[11], pk[12],
              pk[13], pk[14], pk[15]);
}
__device__ __forceinline__ void pack_store16(uint32_t taddr, const float (&v)[32]) {
    uint32_t pk[16];
    pack_store16(taddr, v, pk);
}

// 32 columns of TMEM (fp32) times `sc`, as bf16, to global memory when `store`.
__device__ __forceinline__ void tmem_to_bf16(uint32_t taddr, bool have, float sc, bool store, __nv_bfloat16 *dst) {
    uint32_t o[32];
    if (have) {
        tmem_ld32(taddr, o);
        tmem_ld_wait();
    }
    uint32_t pk[16];
#pragma unroll
    for (int k = 0; k < 16; ++k)
        pk[k] = have ? pack_bf16x2(__uint_as_float(o[2 * k]) * sc, __uint_as_float(o[2 * k + 1]) * sc) : 0u;
    if (store) {
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int k = 0; k < 4; ++k) d4[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
    }
}

template <int D>
__device__ __forceinline__ void init_bars(BtBars &bars, volatile int &abort_flag) {
    using C = BtCfg<D>;
    mbar_init(smem_u32(&bars.a_full), 1);
    for (int s = 0; s < C::RING; ++s) {
        mbar_init(smem_u32(&bars.full[s]), 1);
        mbar_init(smem_u32(&bars.empty[s]), 2);   // one release from each issuer
    }
    for (int s = 0; s < TSTAGES; ++s) {
        mbar_init(smem_u32(&bars.t_full[s]), 32);
        mbar_init(smem_u32(&bars.t_empty[s]), NCW);
    }
    mbar_init(smem_u32(&bars.s_full), 1);
    mbar_init(smem_u32(&bars.dp_full), 1);
    mbar_init(smem_u32(&bars.pa), NCW);
    mbar_init(smem_u32(&bars.pb), NCW);
    mbar_init(smem_u32(&bars.done), 2);
    mbar_init(smem_u32(&bars.drain[0]), 1);
    mbar_init(smem_u32(&bars.drain[1]), 1);
    abort_flag = 0;
    mbar_init_fence();
}

// ====================================================================== dQ
// The two bodies below run as one grid (bwd_tc_kernel): CTA `bid` of each.  The tensor maps are
// the kernel's __grid_constant__ parameters, passed by reference so TMA sees their addresses.
template <int D>
__device__ __forceinline__ void bwd_dq_body(const CUtensorMap &mq, const CUtensorMap &mg, const CUtensorMap &mk,
                                            const CUtensorMap &mv, const BwdProblem &p, unsigned bid) {
    using C = BtCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ BtBars bars;
    __shared__ uint32_t tmem_sh;
    __shared__ volatile int abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = sbase + C::A_OFF, sG = sQ + C::TILE, sRing = sbase + C::RING_OFF;
    // the query tiles that see the most key tiles (the last ones, under a causal mask) go first
    const int BH = p.B * p.Hq, nqt = (p.Sq + TB - 1) / TB;
    const int q0 = (nqt - 1 - (int)(bid / BH)) * TB;
    const int bh = (int)(bid % BH), b = bh / p.Hq, hq = bh % p.Hq;
    const int kvh = hq / (p.Hq / p.Hkv);
    int n = (p.Sk + TB - 1) / TB;   // key tiles these rows see
    if (p.causal) {
        const int last = min(q0 + TB - 1, p.Sq - 1) + p.causal_off;
        n = min(n, last < 0 ? 0 : last / TB + 1);
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_sh), TMEM_COLS);
    if (tid == 32) init_bars<D>(bars, abort_flag);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_sh;
    const uint32_t tS = tmem, tP = tmem + 128, tQ = tmem + 256, tdS = tmem + 256 + D;

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
    } else if ((warp == 1 || warp == 3) && lane == 0 && n > 0) {
        // ------------------------------------------------------------ MMA issue, two threads
        // Issuer A (warp 1): S = Q K_j^T.  Issuer B (warp 3): dP = dO V_j^T and dQ += dS K_j.
        // Neither touches the other's TMEM columns; a ring slot is free once both have released
        // it (B releases the V slots twice).  B's commit after dP_{j+1} covers dQ_j, so phase B
        // of step j+1 may overwrite dS.
        const bool is_a = warp == 1;
        auto wait_full = [&](int m) {
            return mbar_wait_spin(smem_u32(&bars.full[m % C::RING]), (m / C::RING) & 1, &abort_flag);
        };
        auto ring = [&](int m) { return sRing + (m % C::RING) * C::TILE; };
        auto release = [&](int m) { mma_commit(smem_u32(&bars.empty[m % C::RING])); };
        bool ok = mbar_wait_spin(smem_u32(&bars.a_full), 0, &abort_flag) && wait_full(is_a ? 0 : 1);
        if (ok) {
            tc_fence_after();
            if (is_a) {
                issue_ss<D>(tS, sQ, ring(0));                  // S = Q K_0^T
                mma_commit(smem_u32(&bars.s_full));
                release(0);
            } else {
                issue_ss<D>(tP, sG, ring(1));                  // dP = dO V_0^T
                mma_commit(smem_u32(&bars.dp_full));
                release(1);
                release(1);
            }
        }
        for (int j = 0; j < n && ok; ++j) {
            const int mk_ = 2 * j;
            if (is_a) {
                // phase A of step j has read S: the next S may overwrite it
                ok = mbar_wait_spin(smem_u32(&bars.pa), j & 1, &abort_flag);
                if (!ok || j + 1 >= n) continue;
                ok = wait_full(mk_ + 2);
                if (!ok) break;
                tc_fence_after();
                issue_ss<D>(tS, sQ, ring(mk_ + 2));
                mma_commit(smem_u32(&bars.s_full));
                release(mk_ + 2);
            } else {
                // phase B has read dP and written dS
                ok = mbar_wait_spin(smem_u32(&bars.pb), j & 1, &abort_flag) && wait_full(mk_);
                if (!ok) break;
                tc_fence_after();
                issue_ts<D>(tQ, tdS, tdS + 32, ring(mk_), j > 0);   // dQ += dS K_j
                release(mk_);
                if (j + 1 < n) {
                    ok = wait_full(mk_ + 3);
                    if (!ok) break;
                    tc_fence_after();
                    issue_ss<D>(tP, sG, ring(mk_ + 3));
                    mma_commit(smem_u32(&bars.dp_full));
                    release(mk_ + 3);
                    release(mk_ + 3);
                }
            }
        }
        if (ok) mma_commit(smem_u32(&bars.done));
        else bt_timeout(&abort_flag, p.status);
        const uint32_t dr = smem_u32(&bars.drain[is_a ? 0 : 1]);
        mma_commit(dr);
        mbar_wait(dr, 0, nullptr, 20000000ull);
    } else if (warp >= 4) {
        // ------------------------------------------------------------ compute: dS, then dQ out
        griddep_wait();   // the grid is a programmatic dependent of the row-sum kernel (D_i)
        const int q4 = warp & 3, h = (warp - 4) >> 2;
        const int r = q4 * 32 + lane, row = q0 + r;
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const bool row_ok = row < p.Sq;
        const long long grow = (long long)bh * p.Sq + row;
        const float lse2 = row_ok ? p.lse[grow] * kLog2e : INFINITY;
        const float dvr = row_ok ? p.dvec[grow] : 0.f;
        const float c2 = p.scale_log2;
        // packed pairs: scale, -lse and -D of this row
        const uint64_t c22 = f2_pack(c2, c2), nl2 = f2_pack(-lse2, -lse2), nd2 = f2_pack(-dvr, -dvr);
        const int col0 = h * 64;   // this warp's score columns
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            ok = mbar_wait(smem_u32(&bars.s_full), j & 1, &abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const int key0 = j * TB;
            // a full tile: every key exists and every row of the tile sees all of them
            const bool full = key0 + TB <= p.Sk && (!p.causal || key0 + TB - 1 <= q0 + p.causal_off);
            int lim = p.Sk - key0 - col0;
            if (p.causal) lim = min(lim, row + p.causal_off - key0 + 1 - col0);
            if (!row_ok) lim = 0;
            // phase A: P for this warp's 64 columns, kept in registers
            float pv[64];
            {
                uint32_t s[64];
                tmem_ld32(tS + lane_off + col0, *reinterpret_cast<uint32_t(*)[32]>(s));
                tmem_ld32(tS + lane_off + col0 + 32, *reinterpret_cast<uint32_t(*)[32]>(s + 32));
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 64; k += 2) {
                    float a0, a1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(s[k]), __uint_as_float(s[k + 1])), c22, nl2), a0, a1);
                    const float e0 = ex2_approx(a0), e1 = ex2_approx(a1);
                    pv[k] = (full || k < lim) ? e0 : 0.f;
                    pv[k + 1] = (full || k + 1 < lim) ? e1 : 0.f;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars.pa));
            // phase B: dS = P (dP - D_r), as bf16 into this warp's 32 columns of the dS region
            ok = mbar_wait(smem_u32(&bars.dp_full), j & 1, &abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t d[32];
                tmem_ld32(tP + lane_off + col0 + 32 * c, d);
                tmem_ld_wait();
                float ds[32];
#pragma unroll
                for (int k = 0; k < 32; k += 2)
                    f2_unpack(f2_mul(f2_pack(pv[32 * c + k], pv[32 * c + k + 1]),
                                     f2_add(f2_pack(__uint_as_float(d[k]), __uint_as_float(d[k + 1])), nd2)),
                              ds[k], ds[k + 1]);
                pack_store16(tdS + lane_off + h * 32 + 16 * c, ds);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars.pb));
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
        __nv_bfloat16 *dq = static_cast<__nv_bfloat16 *>(p.dq) + (row_ok ? grow : 0) * D;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            const int cc = h * (D / 64) + c;   // 32-column chunk of dQ
            tmem_to_bf16(tQ + lane_off + cc * 32, have, p.scale, row_ok, dq + cc * 32);
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
__device__ __forceinline__ void bwd_dkdv_body(const CUtensorMap &mq, const CUtensorMap &mg, const CUtensorMap &mk,
                                              const CUtensorMap &mv, const CUtensorMap &mdst, const BwdProblem &p,
                                              unsigned bid) {
    using C = BtCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ BtBars bars;
    __shared__ uint32_t tmem_sh;
    __shared__ volatile int abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sK = sbase + C::A_OFF, sV = sK + C::TILE, sRing = sbase + C::RING_OFF;
    float *tab = reinterpret_cast<float *>(smem_raw + (sbase - smem_u32(smem_raw)) + C::TAB_OFF);
    // the key tiles seen by the most query tiles (the first ones, under a causal mask) go first
    const int BK = p.B * p.Hkv;
    const int key0 = (int)(bid / BK) * TB;
    const int bk = (int)(bid % BK), b = bk / p.Hkv, kvh = bk % p.Hkv;
    const int G = p.Hq / p.Hkv;
    // query tiles that see a key of this block: from the first row that sees key0
    int q_first = p.causal ? max(0, key0 - p.causal_off) : 0;
    q_first /= TB;
    const int n_qt = (p.Sq + TB - 1) / TB;
    const int per_head = max(0, n_qt - q_first);
    const int n = G * per_head;   // steps: (head g, query tile) pairs
    if (warp == 0) tmem_alloc(smem_u32(&tmem_sh), TMEM_COLS);
    if (tid == 32) init_bars<D>(bars, abort_flag);
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
            // Q and dO tiles are read again by the CTAs of the other key tiles: keep them in L2
            tma_load_5d_hint(sRing + st * C::TILE, (m & 1) ? &mg : &mq, smem_u32(&bars.full[st]), 0, qt * TB, 0, hq, b,
                             l2_policy_evict_last());
        }
        if (!ok) {
            bt_timeout(&abort_flag, p.status);
            bt_settle();
        }
    } else if ((warp == 1 || warp == 3) && lane == 0 && n > 0) {
        // ------------------------------------------------------------ MMA issue, two threads
        // Issuer A (warp 1): S^T = K Q_j^T and dV += P^T dO_j.  Issuer B (warp 3):
        // dP^T = V dO_j^T and dK += dS^T Q_j.  A only touches S^T and dV, B only dP^T and dK;
        // Q_j and dO_j each feed one product of each side, so each side releases every slot once.
        const bool is_a = warp == 1;
        auto wait_full = [&](int m) {
            return mbar_wait_spin(smem_u32(&bars.full[m % C::RING]), (m / C::RING) & 1, &abort_flag);
        };
        auto ring = [&](int m) { return sRing + (m % C::RING) * C::TILE; };
        auto release = [&](int m) { mma_commit(smem_u32(&bars.empty[m % C::RING])); };
        const int own = is_a ? 0 : 1;              // stream offset of this side's score operand
        const uint32_t tX = is_a ? tS : tP, sX = is_a ? sK : sV;
        bool ok = mbar_wait_spin(smem_u32(&bars.a_full), 0, &abort_flag) && wait_full(own);
        if (ok) {
            tc_fence_after();
            issue_ss<D>(tX, sX, ring(own));        // S^T = K Q_0^T  /  dP^T = V dO_0^T
            mma_commit(smem_u32(is_a ? &bars.s_full : &bars.dp_full));
            release(own);
        }
        for (int j = 0; j < n && ok; ++j) {
            // A: P^T is in TMEM, dV += P^T dO_j.  B: dS^T is in TMEM, dK += dS^T Q_j.
            const int other = 2 * j + 1 - own;     // dO_j for A, Q_j for B
            ok = mbar_wait_spin(smem_u32(is_a ? &bars.pa : &bars.pb), j & 1, &abort_flag) && wait_full(other);
            if (!ok) break;
            tc_fence_after();
            if (is_a) issue_ts<D>(tV, tS, tS + 64, ring(other), j > 0);
            else issue_ts<D>(tK, tP, tP + 64, ring(other), j > 0);
            release(other);
            if (j + 1 < n) {
                const int next = 2 * j + 2 + own;  // Q_{j+1} for A, dO_{j+1} for B
                ok = wait_full(next);
                if (!ok) break;
                tc_fence_after();
                issue_ss<D>(tX, sX, ring(next));
                mma_commit(smem_u32(is_a ? &bars.s_full : &bars.dp_full));
                release(next);
            }
        }
        if (ok) mma_commit(smem_u32(&bars.done));
        else bt_timeout(&abort_flag, p.status);
        const uint32_t dr = smem_u32(&bars.drain[own]);
        mma_commit(dr);
        mbar_wait(dr, 0, nullptr, 20000000ull);
    } else if (warp == 2 && n > 0) {
        // ------------------------------------------------------------ per-query lse (base 2), D
        // the kernel is a programmatic dependent of the row-sum kernel that writes D
        griddep_wait();
        bool ok = true;
        for (int m = 0; m < n; ++m) {
            const int st = m % TSTAGES;
            ok = mbar_wait(smem_u32(&bars.t_empty[st]), ((m / TSTAGES) & 1) ^ 1, &abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            int hq, qt;
            step_at(m, hq, qt);
            float *tl = tab + st * 2 * TB, *td = tl + TB;
            const long long row0 = ((long long)b * p.Hq + hq) * p.Sq;
#pragma unroll
            for (int i = 0; i < TB / 32; ++i) {
                const int c = lane + 32 * i, q = qt * TB + c;
                // negated, the addends of the compute warps' packed FMA and add
                tl[c] = q < p.Sq ? -p.lse[row0 + q] * kLog2e : -INFINITY;
                td[c] = q < p.Sq ? -p.dvec[row0 + q] : 0.f;
            }
            mbar_arrive(smem_u32(&bars.t_full[st]));
        }
        if (!ok) bt_timeout(&abort_flag, p.status);
    } else if (warp >= 4) {
        // ------------------------------------------------------------ compute: P^T, dS^T
        const int q4 = warp & 3, h = (warp - 4) >> 2;
        const int r = q4 * 32 + lane, key = key0 + r;
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const uint64_t c22 = f2_pack(p.scale_log2, p.scale_log2);
        const int col0 = h * 64;   // this warp's query columns
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            int hq, qt;
            step_at(j, hq, qt);
            const int qbase = qt * TB, st = j % TSTAGES;
            ok = mbar_wait(smem_u32(&bars.s_full), j & 1, &abort_flag) &&
                 mbar_wait(smem_u32(&bars.t_full[st]), (j / TSTAGES) & 1, &abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const float4 *tl4 = reinterpret_cast<const float4 *>(tab + st * 2 * TB + col0);
            const float4 *td4 = reinterpret_cast<const float4 *>(tab + st * 2 * TB + TB + col0);
            // query column q is visible to this key iff (causal) key <= q + off; columns past
            // Sq have lse = +inf (P = 0) and zero Q, dO rows; keys past Sk are never stored
            const bool full = !p.causal || key0 + TB - 1 - p.causal_off <= qbase;
            const int qmin = p.causal ? key - p.causal_off - qbase - col0 : INT_MIN;
            // phase A: P^T for this warp's 64 columns (fp32 in registers, bf16 into TMEM)
            float pv[64];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t s[32];
                tmem_ld32(tS + lane_off + col0 + 32 * c, s);
                tmem_ld_wait();
#pragma unroll
                for (int k4 = 0; k4 < 8; ++k4) {
                    const float4 l = tl4[8 * c + k4];   // -lse (base 2) of four query columns
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const int k = 4 * k4 + e;
                        float a0, a1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(s[k]), __uint_as_float(s[k + 1])), c22,
                                         e ? f2_pack(l.z, l.w) : f2_pack(l.x, l.y)),
                                  a0, a1);
                        const float x0 = ex2_approx(a0), x1 = ex2_approx(a1);
                        pv[32 * c + k] = (full || 32 * c + k >= qmin) ? x0 : 0.f;
                        pv[32 * c + k + 1] = (full || 32 * c + k + 1 >= qmin) ? x1 : 0.f;
                    }
                }
                pack_store16(tS + lane_off + col0 + 16 * c, *reinterpret_cast<const float(*)[32]>(pv + 32 * c));
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars.pa));
            // phase B: dS^T = P^T (dP^T - D_q), bf16 into TMEM (and to the workspace when dQ runs
            // as a separate product)
            uint32_t dpk[2][16];   // this key's 64 values of dS^T as bf16 pairs
            ok = mbar_wait(smem_u32(&bars.dp_full), j & 1, &abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t d[32];
                tmem_ld32(tP + lane_off + col0 + 32 * c, d);
                tmem_ld_wait();
                float ds[32];
#pragma unroll
                for (int k4 = 0; k4 < 8; ++k4) {
                    const float4 dd = td4[8 * c + k4];   // -D of four query columns
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const int k = 4 * k4 + e;
                        f2_unpack(f2_mul(f2_pack(pv[32 * c + k], pv[32 * c + k + 1]),
                                         f2_add(f2_pack(__uint_as_float(d[k]), __uint_as_float(d[k + 1])),
                                                e ? f2_pack(dd.z, dd.w) : f2_pack(dd.x, dd.y))),
                                  ds[k], ds[k + 1]);
                    }
                }
                pack_store16(tP + lane_off + col0 + 16 * c, ds, dpk[c]);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&bars.pb));
                mbar_arrive(smem_u32(&bars.t_empty[st]));
            }
            // The workspace copy of dS^T leaves after the hand-off: this warp's [32 keys x 64
            // queries] through its 2 KB staging tile ([32 rows][64 B], 64-byte swizzle) as two TMA
            // stores of [32 x 32], so the copy engine, not the load/store unit, writes the rows.
            if (p.ds) {
                const uint32_t stg = sbase + C::STG_OFF + (uint32_t)(warp - 4) * 2048u;
                // rows of keys past Sk are zero: their K rows are zero-filled, so P^T there is
                // 2^-lse, which overflows for rows whose scores are all far below zero, and the
                // dQ product must not meet inf * 0
                const uint32_t keep = key < p.Sk ? 0xffffffffu : 0u;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (lane == 0) bulk_wait_read();   // the previous store has read the tile
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        st_shared_v4(stg + (uint32_t)lane * 64 + ((uint32_t)(k ^ ((lane >> 1) & 3)) << 4),
                                     dpk[c][4 * k] & keep, dpk[c][4 * k + 1] & keep, dpk[c][4 * k + 2] & keep,
                                     dpk[c][4 * k + 3] & keep);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int nkt = (int)(p.ds_rows / TB), nqt = (int)(p.ds_ld / TB);
                        const int tile = (((b * p.Hq + hq) * nkt) + key0 / TB) * nqt + qbase / TB;
                        // dS^T is read once, by the dQ product: it gives way in L2 first
                        tma_store_3d_hint(&mdst, stg, col0 + 32 * c, q4 * 32, tile, l2_policy_evict_first());
                        bulk_commit();
                    }
                }
            }
        }
        if (!ok) bt_timeout(&abort_flag, p.status);
        if (p.ds && lane == 0) bulk_wait_all();   // the dS^T stores have landed
        // epilogue: dK = scale * dS^T Q (warps of half 0), dV = P^T dO (half 1); zero when no
        // query sees this key
        bool have = false;
        if (ok && n > 0) {
            have = mbar_wait(smem_u32(&bars.done), 0, &abort_flag);
            have = __all_sync(0xffffffffu, have);
            if (!have) bt_timeout(&abort_flag, p.status);
            tc_fence_after();
        }
        const bool key_ok = key < p.Sk;
        const long long gk = (long long)bk * p.Sk + (key_ok ? key : 0);
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(h ? p.dv : p.dk) + gk * D;
        const uint32_t src = (h ? tV : tK) + lane_off;
        const float sc = h ? 1.f : p.scale;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_to_bf16(src + c * 32, have, sc, key_ok, out + c * 32);
    }
    tc_fence_before();
    __syncwarp();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// One grid: CTAs [0, n_dkdv) are dK/dV CTAs, the rest dQ CTAs, each group heaviest first, so
// dQ work fills the SMs the dK/dV tail leaves idle.
template <int D>
__global__ void __launch_bounds__(NT_THREADS, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mg,
              const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
              const __grid_constant__ CUtensorMap mdst, const BwdProblem p, unsigned n_dkdv) {
    if (blockIdx.x < n_dkdv) bwd_dkdv_body<D>(mq, mg, mk, mv, mdst, p, blockIdx.x);
    else bwd_dq_body<D>(mq, mg, mk, mv, p, blockIdx.x - n_dkdv);
}

// ====================================================================== dQ as one product
// With a dS workspace the dK/dV CTAs also store dS^T (bf16, one contiguous 32 KB [128 keys][128
// queries] tile per (b, q head, key tile, query tile), so a tile load reads one run of HBM), and
// dQ = scale * dS K becomes a plain product over the key tiles a query tile sees: S and dP are
// not recomputed, so a (query tile, key tile) pair costs five products in all instead of seven.  An item is one query tile of `hp` query heads of one kv group (two when the
// group size is even, so each K tile feeds two heads' products); persistent CTAs (one per SM)
// walk the items heaviest first, in snake order.  Warp 0 streams the dS^T tiles and warp 6 the K
// tiles by TMA, each through its own ring (a load takes a couple of microseconds under load, so
// several of each must be in flight per SM).  Warp 1 issues the MMAs into one of two sets of
// TMEM accumulators, and warps 2-5 scale and store one set while the next item's products run.
// Both operands are MN-major in shared memory: a dS^T tile is [128 keys][128 queries] (queries
// contiguous, two 64-column blocks) and serves as dS, and a K tile is [128 keys][D].
template <int D>
struct DqCfg {
    static constexpr uint32_t A_TILE = TB * TB * 2;
    static constexpr uint32_t B_TILE = TB * D * 2;
    static constexpr int K_STAGES = 3;
    static constexpr int FIT = (int)((232448u - 1024u - K_STAGES * B_TILE) / A_TILE);
    static constexpr int DS_STAGES = FIT < 6 ? FIT : 6;          // 4 at D = 128, 5 at D = 64
    static constexpr uint32_t K_OFF = DS_STAGES * A_TILE;
    static constexpr uint32_t SMEM_BYTES = K_OFF + K_STAGES * B_TILE + 1024;
    static constexpr uint32_t DBLK = TB * 128;                  // bytes between 64-column blocks
    static constexpr uint32_t IDESC = idesc_bf16_f32(TB, D, 1, 1);
    static constexpr uint32_t TMEM_COLS = 4 * D;                // 2 sets x up to 2 heads
    static_assert(DS_STAGES >= 2 && DS_STAGES <= 6 && K_STAGES <= 4, "ring barriers");
};
constexpr int DQ_THREADS = 224;   // warp 0 dS^T loads, 1 MMA, 2-5 epilogue, 6 K loads

struct DqBars {
    uint64_t ds_full[6], ds_empty[6], k_full[4], k_empty[4], acc_full[2], acc_empty[2], drain;
};

// Item `it`, heaviest first: its first query row, first (b, q head) index and key-tile count.
__device__ __forceinline__ void dq_item(const BwdProblem &p, int hp, int it, int &q0, int &bh, int &n) {
    const int BHP = p.B * p.Hq / hp, nqt = (p.Sq + TB - 1) / TB;
    q0 = (nqt - 1 - it / BHP) * TB;
    bh = (it % BHP) * hp;
    n = (p.Sk + TB - 1) / TB;
    if (p.causal) {
        const int last = min(q0 + TB - 1, p.Sq - 1) + p.causal_off;
        n = min(n, last < 0 ? 0 : last / TB + 1);
    }
}
// This CTA's item of round r (forward on even rounds, backward on odd ones), or -1.
__device__ __forceinline__ int dq_item_of(int r, int n_items) {
    const int g = (int)gridDim.x, c = (r & 1) ? g - 1 - (int)blockIdx.x : (int)blockIdx.x;
    const long long it = (long long)r * g + c;
    return it < n_items ? (int)it : -1;
}

template <int D>
__global__ void __launch_bounds__(DQ_THREADS, 1)
bwd_dq_gemm_kernel(const __grid_constant__ CUtensorMap mds, const __grid_constant__ CUtensorMap mk, const BwdProblem p,
                   int hp, int n_items) {
    using C = DqCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ DqBars bars;
    __shared__ uint32_t tmem_sh;
    __shared__ volatile int abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u, sK = sbase + C::K_OFF;
    if (warp == 0) tmem_alloc(smem_u32(&tmem_sh), C::TMEM_COLS);
    if (tid == 32) {
        for (int s = 0; s < C::DS_STAGES; ++s) {
            mbar_init(smem_u32(&bars.ds_full[s]), 1);
            mbar_init(smem_u32(&bars.ds_empty[s]), 1);
        }
        for (int s = 0; s < C::K_STAGES; ++s) {
            mbar_init(smem_u32(&bars.k_full[s]), 1);
            mbar_init(smem_u32(&bars.k_empty[s]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bars.acc_full[i]), 1);
            mbar_init(smem_u32(&bars.acc_empty[i]), 4);   // one arrival per epilogue warp
        }
        mbar_init(smem_u32(&bars.drain), 1);
        abort_flag = 0;
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_sh;
    // dS^T is written by the dK/dV grid this kernel depends on; every role waits for it here, so
    // no bounded wait below starts counting before that grid has finished
    griddep_wait();

    if ((warp == 0 || warp == 6) && lane == 0) {
        // ------------------------------------------------------------ TMA: dS^T (warp 0), K (warp 6)
        const bool is_ds = warp == 0;
        const int stages = is_ds ? C::DS_STAGES : C::K_STAGES, per = is_ds ? hp : 1;
        const uint32_t tile = is_ds ? C::A_TILE : C::B_TILE, ring = is_ds ? sbase : sK;
        uint64_t *full = is_ds ? bars.ds_full : bars.k_full, *empty = is_ds ? bars.ds_empty : bars.k_empty;
        tma_prefetch_desc(is_ds ? &mds : &mk);
        const int G = p.Hq / p.Hkv;
        bool ok = true;
        int g = 0;   // tiles streamed so far
        for (int r = 0; ok; ++r) {
            const int it = dq_item_of(r, n_items);
            if (it < 0) break;
            int q0, bh, n;
            dq_item(p, hp, it, q0, bh, n);
            const int b = bh / p.Hq, kvh = (bh % p.Hq) / G;
            for (int j = 0; j < n && ok; ++j) {
                for (int h = 0; h < per; ++h, ++g) {
                    const int st = g % stages;
                    ok = mbar_wait(smem_u32(&empty[st]), ((g / stages) & 1) ^ 1, &abort_flag);
                    if (!ok) break;
                    const uint32_t dst = ring + st * tile;
                    mbar_expect_tx(smem_u32(&full[st]), tile);
                    if (is_ds)   // read once: evict first, so the K tiles and dQ rows stay in L2
                        tma_load_4d_hint(dst, &mds, smem_u32(&full[st]), 0, 0, 0,
                                         (int)(((long long)(bh + h) * (p.ds_rows / TB) + j) * (p.ds_ld / TB) + q0 / TB),
                                         l2_policy_evict_first());
                    else tma_load_5d(dst, &mk, smem_u32(&full[st]), 0, j * TB, 0, kvh, b);
                }
            }
        }
        if (!ok) {
            bt_timeout(&abort_flag, p.status);
            bt_settle();
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issue
        bool ok = true;
        int gd = 0, gk = 0, a = 0;   // dS^T and K tiles consumed, accumulator sets filled
        for (int r = 0; ok; ++r) {
            const int it = dq_item_of(r, n_items);
            if (it < 0) break;
            int q0, bh, n;
            dq_item(p, hp, it, q0, bh, n);
            if (n == 0) continue;
            const int buf = a & 1;
            // the epilogue has read this set's previous item
            if (a >= 2 && !(ok = mbar_wait_spin(smem_u32(&bars.acc_empty[buf]), ((a >> 1) - 1) & 1, &abort_flag)))
                break;
            for (int j = 0; j < n && ok; ++j, ++gk) {
                const int sk = gk % C::K_STAGES;
                ok = mbar_wait_spin(smem_u32(&bars.k_full[sk]), (gk / C::K_STAGES) & 1, &abort_flag);
                const uint64_t bd = sdesc_sw128(sK + sk * C::B_TILE, C::DBLK, 1024);
                for (int h = 0; h < hp && ok; ++h, ++gd) {
                    const int sd = gd % C::DS_STAGES;
                    ok = mbar_wait_spin(smem_u32(&bars.ds_full[sd]), (gd / C::DS_STAGES) & 1, &abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t ad = sdesc_sw128(sbase + sd * C::A_TILE, C::DBLK, 1024);
                    const uint32_t dst = tmem + (uint32_t)((buf * 2 + h) * D);
#pragma unroll
                    for (int k = 0; k < TB / 16; ++k)   // 16 keys per k-step: 16 rows of both tiles
                        mma_ss(dst, ad + ((k * 2048) >> 4), bd + ((k * 2048) >> 4), C::IDESC, j > 0 || k > 0);
                    mma_commit(smem_u32(&bars.ds_empty[sd]));
                }
                if (ok) mma_commit(smem_u32(&bars.k_empty[sk]));
            }
            if (!ok) break;
            mma_commit(smem_u32(&bars.acc_full[buf]));
            ++a;
        }
        if (!ok) bt_timeout(&abort_flag, p.status);
        mma_commit(smem_u32(&bars.drain));
        mbar_wait(smem_u32(&bars.drain), 0, nullptr, 20000000ull);
    } else if (warp >= 2 && warp <= 5) {
        // ------------------------------------------------------------ epilogue: dQ = scale * acc
        const int q4 = warp & 3;   // warps 2-5 cover the four TMEM lane quarters
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        bool ok = true;
        int a = 0;
        for (int r = 0;; ++r) {
            const int it = dq_item_of(r, n_items);
            if (it < 0) break;
            int q0, bh, n;
            dq_item(p, hp, it, q0, bh, n);
            const int row = q0 + q4 * 32 + lane;
            const bool row_ok = row < p.Sq;
            const int buf = a & 1;
            bool have = false;   // rows that see no key get dQ = 0
            if (n > 0 && ok) {
                have = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.acc_full[buf]), (a >> 1) & 1, &abort_flag));
                if (!have) {
                    ok = false;
                    bt_timeout(&abort_flag, p.status);
                }
                tc_fence_after();
            }
            for (int h = 0; h < hp; ++h) {
                __nv_bfloat16 *dq =
                    static_cast<__nv_bfloat16 *>(p.dq) + ((long long)(bh + h) * p.Sq + (row_ok ? row : 0)) * D;
                const uint32_t src = tmem + (uint32_t)((buf * 2 + h) * D) + lane_off;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) tmem_to_bf16(src + c * 32, have, p.scale, row_ok, dq + c * 32);
            }
            if (n > 0) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars.acc_empty[buf]));
                ++a;
            }
        }
    }
    tc_fence_before();
    __syncwarp();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D>
cudaError_t launch_t(const BwdProblem &p, cudaStream_t s) {
    using C = BtCfg<D>;
    const cudaError_t attr_err = set_max_dynamic_smem((const void *)bwd_tc_kernel<D>, (int)C::SMEM_BYTES);
    if (attr_err != cudaSuccess) return attr_err;
    const long long qs = (long long)p.Sq * D, ks = (long long)p.Sk * D;
    CUtensorMap mq, mg, mk, mv;
    if (!make_bf16_tile_map_strided(&mq, p.q, D, p.Sq, p.Hq, p.B, D, qs, qs * p.Hq, TB) ||
        !make_bf16_tile_map_strided(&mg, p.dout, D, p.Sq, p.Hq, p.B, D, qs, qs * p.Hq, TB) ||
        !make_bf16_tile_map_strided(&mk, p.k, D, p.Sk, p.Hkv, p.B, D, ks, ks * p.Hkv, TB) ||
        !make_bf16_tile_map_strided(&mv, p.v, D, p.Sk, p.Hkv, p.B, D, ks, ks * p.Hkv, TB))
        return cudaErrorInvalidValue;
    const unsigned nkv = (unsigned)((p.Sk + TB - 1) / TB) * (unsigned)(p.B * p.Hkv);
    const unsigned nq = (unsigned)((p.Sq + TB - 1) / TB) * (unsigned)(p.B * p.Hq);
    if ((unsigned long long)nkv + nq >= (1ull << 31)) return cudaErrorInvalidValue;
    if (!p.ds) {
        // dK/dV and dQ CTAs in one grid
        cudaError_t e = launch_dependent(bwd_tc_kernel<D>, dim3(nkv + nq), dim3(NT_THREADS), C::SMEM_BYTES, s, mq, mg,
                                         mk, mv, mq, p, nkv);   // (no dS stores: the fifth map is unused)
        if (e != cudaSuccess) return e;
        count_launches(1);
        return cudaGetLastError();
    }
    // dK/dV CTAs (they also store dS^T), then dQ = scale * dS K as a dependent grid
    using Q = DqCfg<D>;
    CUtensorMap mds, mdst;
    const long long n_tiles = (long long)p.B * p.Hq * (p.ds_rows / TB) * (p.ds_ld / TB);
    if (!make_bf16_tile_map(&mds, p.ds, TB, TB, n_tiles, TB, 2) ||
        !make_bf16_store_map_32x32(&mdst, p.ds, TB, TB, n_tiles))
        return cudaErrorInvalidValue;
    cudaError_t e = set_max_dynamic_smem((const void *)bwd_dq_gemm_kernel<D>, (int)Q::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    int sms = 0;
    if (device_sm_count(&sms) != OSF_OK || sms <= 0) return cudaErrorInvalidValue;
    e = launch_dependent(bwd_tc_kernel<D>, dim3(nkv), dim3(NT_THREADS), C::SMEM_BYTES, s, mq, mg, mk, mv, mdst, p,
                         nkv);
    if (e != cudaSuccess) return e;
    const int hp = (p.Hq / p.Hkv) % 2 == 0 ? 2 : 1;   // query heads per item: two of one kv group
    const int n_items = (int)nq / hp;
    e = launch_dependent(bwd_dq_gemm_kernel<D>, dim3((unsigned)min(sms, n_items)), dim3(DQ_THREADS), Q::SMEM_BYTES, s,
                         mds, mk, p, hp, n_items);
    if (e != cudaSuccess) return e;
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
    // one-dimensional grids of (row tile, batch x head) CTAs
    const long long nkv = (long long)((p.Sk + TB - 1) / TB) * p.B * p.Hkv;
    const long long nq = (long long)((p.Sq + TB - 1) / TB) * p.B * p.Hq;
    if (nkv >= (1LL << 31) || nq >= (1LL << 31)) return false;
    return tensor_map_encoder() != nullptr;
}

cudaError_t launch_attn_bwd_tc(const BwdProblem &p, cudaStream_t s) {
    return p.D == 64 ? launch_t<64>(p, s) : launch_t<128>(p, s);
}

}  // namespace osf
