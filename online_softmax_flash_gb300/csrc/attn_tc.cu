// Tensor-core attention prefill for bfloat16 Q/K/V on sm_103a: tcgen05 MMAs with fp32
// accumulators in tensor memory (TMEM), K/V tiles streamed by TMA into shared-memory rings,
// and the online-softmax recurrence run by threads that each own one query row.
//
// The method is the single-pass attention of "softmax_attention" (blog.euler0525.cn/posts/
// 3fb3592b), section "实现思路": per query row a running max, a rescale factor, a running
// denominator and numerator, keys past the sequence end scored -inf; with the GQA mapping and
// top-left causal mask of "从零开始写Qwen3（五-其一）使用Triton实现自注意力", sections "自注意力原理"
// and "GQA".  The page runs one program per query on CUDA cores; here a CTA owns 2 x 128 query
// rows and both matrix products run on the tensor cores.
//
// CG = 2 (head dim 128): the kernel runs on pairs of CTAs (a cluster of two SMs) with
// cta_group::2 MMAs of M = 256.  Each CTA keeps its own 2 x 128 query rows, but holds only half
// of every key tile (64 of its 128 keys for S = Q K^T, 64 of the 128 value columns for
// O += P V); one thread of the pair issues every MMA for both SMs.  A single SM running
// M = 128 MMAs with both operands in shared memory reads 128 B/clk -- all of its shared-memory
// bandwidth -- and starves the TMA writes that refill the K/V ring; splitting B across the pair
// cuts each SM's shared-memory traffic per key tile from 256 KB to 160 KB.  The pair is two query
// heads of one kv head (same rows, same causal range) when the GQA group is even, otherwise two
// consecutive 256-row blocks of one head.  CG = 1 (head dim 64) is the same kernel on one SM.
//
// Roles (12 warps per CTA):
//   warp 0      TMA: this CTA's Q tiles once, then its part of every K tile
//   warp 2      TMA: its part of every V tile
//   warp 1      MMA issue (one thread; on the leader CTA only when CG = 2):
//               S_t = Q_t K^T (both operands in shared memory), O_t += P_t V (P read from TMEM)
//   warps 4-7   softmax for Q tile 0, warps 8-11 for Q tile 1: thread r owns TMEM lane r, i.e.
//               query row r of its tile, so row max and row sum need no cross-thread traffic.
//
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 [256+D,256+2D).  P_t (bf16,
// two per column) overwrites the first 64 columns of S_t and is read from there by the PV MMA.
// The two Q tiles are ping-ponged so one tile's softmax overlaps the other tile's MMAs.
//
// Scores are kept in base 2 (scale * log2 e folded into one multiplier).  The rescale of O is
// lazy: a row keeps its reference maximum until a tile raises the maximum by more than 8
// (a factor 256), so O is rarely touched; the result O / l is the same for any reference.
//
// Every mbarrier wait is bounded (2 s); on expiry the CTA records OSF_ERR_TIMEOUT in the
// device status word, drains its own MMAs, lets its copies land, frees TMEM and exits.
#include <mutex>

#include "attn_tc.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.cuh"

namespace osf {
namespace {

using namespace ptx;

constexpr int BM = 128;             // query rows per Q tile (per CTA)
constexpr int BN = 128;             // keys per key tile (per pair)
constexpr int NTHREADS = 384;       // 12 warps: 0-3 control, 4-7 softmax tile 0, 8-11 tile 1
constexpr uint32_t TMEM_COLS = 512;
// Register split after set-up: the control warpgroup (TMA + MMA issue) needs few registers, the
// two softmax warpgroups hold a whole 128-column score row each.  128*56 + 256*224 = 384*168,
// the registers the CTA is launched with (168 per thread).
constexpr int kCtrlRegs = 56, kSoftmaxRegs = 224;
constexpr float kRescaleThreshold = 8.0f;   // base-2 units

template <int D, int CG>
struct TcCfg {
    static_assert(CG == 1 || (CG == 2 && D == 128), "pair kernel is for head dim 128");
    static constexpr int KV_STAGES = (CG == 2 || D == 64) ? 4 : 2;
    static constexpr int K_ROWS = BN / CG;                       // keys of a K tile held here
    static constexpr int V_COLS = D / CG;                        // value columns held here
    static constexpr uint32_t Q_TILE = BM * D * 2;
    static constexpr uint32_t K_PART = K_ROWS * D * 2;
    static constexpr uint32_t V_PART = BN * V_COLS * 2;
    static constexpr uint32_t Q_DBLK = BM * 128;                 // bytes between 64-column blocks
    static constexpr uint32_t K_DBLK = K_ROWS * 128;
    static constexpr uint32_t V_DBLK = BN * 128;
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t K_OFF = 2 * Q_TILE;
    static constexpr uint32_t V_OFF = K_OFF + KV_STAGES * K_PART;
    static constexpr uint32_t SMEM_BYTES = V_OFF + KV_STAGES * V_PART + 1024;  // + alignment slack
    static constexpr uint32_t S_COL0 = 0, S_COL1 = 128, O_COL0 = 256, O_COL1 = 256 + D;
    static constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM * CG, BN, 0, 0);
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM * CG, D, 0, 1);
};

struct Barriers {
    uint64_t q;
    uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
    uint64_t s_full[2], p_full[2], o_final[2];
    uint64_t drain;
};

__device__ __forceinline__ void raise_timeout(volatile int *abort, int *status) {
    *abort = 1;
    if (status) atomicExch(status, kStatusTimeout);
}

// Give copies already issued by this CTA time to land before it releases its shared memory
// (only on the timeout path; the copies complete on a barrier this thread may not own).
__device__ __forceinline__ void settle_copies() {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000ull) {
    }
}

template <int D, int CG>
__global__ void __launch_bounds__(NTHREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, const AttnProblem p, int n_qb) {
    using C = TcCfg<D, CG>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ Barriers bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = sbase + C::Q_OFF, sK = sbase + C::K_OFF, sV = sbase + C::V_OFF;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0;
    const bool leader = rank == 0;

    // ------------------------------------------------------------------ work item
    // A pair item is (head unit, block of query rows).  Pair of heads: both CTAs take the same
    // 256 rows of heads 2u, 2u+1; otherwise the CTAs take rows [q0, q0+256) and [q0+256, q0+512).
    const int G = p.Hq / p.Hkv;
    const bool pair_heads = CG == 2 && (G % 2) == 0;
    const int units = pair_heads ? p.B * p.Hq / 2 : p.B * p.Hq;
    const int item = blockIdx.x / CG;
    const int qb_rank = item / units;
    const int u = item % units;
    const int qb = p.causal ? (n_qb - 1 - qb_rank) : qb_rank;   // heaviest blocks first
    const int rows_per_item = (CG == 2 && !pair_heads) ? 4 * BM : 2 * BM;
    const int q0 = qb * rows_per_item;                          // first row of the item
    const int bh = pair_heads ? 2 * u + (int)rank : u;          // b * Hq + hq of this CTA
    const int rb = q0 + ((CG == 2 && !pair_heads) ? (int)rank * 2 * BM : 0);   // this CTA's first row
    const int rb_hi = q0 + ((CG == 2 && !pair_heads) ? 2 * BM : 0);            // highest CTA's first row
    const int b = bh / p.Hq, hq = bh % p.Hq;
    const int kvbh = b * p.Hkv + hq / G;
    const int ntiles = (q0 + BM < p.Sq) ? 2 : 1;                // tile 1 of the leader's rows exists
    const int n_kt_all = (p.Sk + BN - 1) / BN;
    const int tps = (n_kt_all + p.splits - 1) / p.splits;
    const int kt_begin = blockIdx.y * tps;
    const int kt_end = min(n_kt_all, kt_begin + tps);
    // key tiles each pair-tile visits (causal: up to the last row of either CTA's tile)
    int e0 = kt_end, e1 = kt_end;
    if (p.causal) {
        e0 = min(e0, min(rb_hi + BM - 1, p.Sq - 1) / BN + 1);
        e1 = min(e1, min(rb_hi + 2 * BM - 1, p.Sq - 1) / BN + 1);
    }
    const int n0 = max(0, e0 - kt_begin);
    const int n1 = ntiles == 2 ? max(0, e1 - kt_begin) : 0;
    const int n_kv = max(n0, n1);

    // ------------------------------------------------------------------ set-up
    if (warp == 0) {
        if constexpr (CG == 2)
            tmem_alloc_pair(smem_u32(&tmem_base_sh), TMEM_COLS);
        else
            tmem_alloc(smem_u32(&tmem_base_sh), TMEM_COLS);
    }
    if (tid == 32) {
        mbar_init(smem_u32(&bars.q), 1);
        for (int s = 0; s < C::KV_STAGES; ++s) {
            mbar_init(smem_u32(&bars.k_full[s]), 1);
            mbar_init(smem_u32(&bars.k_empty[s]), 1);
            mbar_init(smem_u32(&bars.v_full[s]), 1);
            mbar_init(smem_u32(&bars.v_empty[s]), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_u32(&bars.s_full[t]), 1);
            mbar_init(smem_u32(&bars.p_full[t]), CG);       // one arrival per CTA of the pair
            mbar_init(smem_u32(&bars.o_final[t]), 1);
        }
        mbar_init(smem_u32(&bars.drain), 1);
        abort_flag = 0;
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync();   // the leader's barriers exist before the peer signals them
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    // Barrier that completes a pair-wide event: the leader's copy (this CTA's own when CG = 1).
    auto lead = [&](uint64_t &bar) -> uint32_t {
        return CG == 2 ? mapa_shared(smem_u32(&bar), 0) : smem_u32(&bar);
    };
    auto commit = [&](uint64_t &bar) {
        if constexpr (CG == 2)
            mma_commit_pair(smem_u32(&bar), 3);
        else
            mma_commit(smem_u32(&bar));
    };

    if (warp < 4) {
      setmaxnreg_dec<kCtrlRegs>();
      if ((warp == 0 || warp == 2) && lane == 0 && n_kv > 0) {
        // ============================================================== TMA producers
        // warp 0 streams Q and K, warp 2 streams V: each tile part is one TMA instruction, and
        // the two streams are issued by different threads so neither waits behind the other.
        // Copies complete on the leader's barriers; the leader arms them for both CTAs' bytes.
        const bool is_k = warp == 0;
        const CUtensorMap *map = is_k ? &mk : &mv;
        tma_prefetch_desc(map);
        if (is_k) {
            tma_prefetch_desc(&mq);
            if (leader) mbar_expect_tx(smem_u32(&bars.q), CG * ntiles * C::Q_TILE);
            for (int t = 0; t < ntiles; ++t)
                tma_load_4d<CG == 2>(sQ + t * C::Q_TILE, &mq, lead(bars.q), 0, rb + t * BM, 0, bh);
        }
        const uint32_t ring = is_k ? sK : sV;
        const uint32_t part = is_k ? C::K_PART : C::V_PART;
        uint64_t *full = is_k ? bars.k_full : bars.v_full;
        uint64_t *empty = is_k ? bars.k_empty : bars.v_empty;
        bool ok = true;
        for (int i = 0; i < n_kv; ++i) {
            const int st = i % C::KV_STAGES;
            ok = mbar_wait(smem_u32(&empty[st]), ((i / C::KV_STAGES) & 1) ^ 1, &abort_flag);
            if (!ok) break;
            if (leader) mbar_expect_tx(smem_u32(&full[st]), CG * part);
            const int key0 = (kt_begin + i) * BN;
            if (is_k)   // this CTA's K rows: keys [key0 + rank * K_ROWS, + K_ROWS), all columns
                tma_load_4d<CG == 2>(ring + st * part, map, lead(full[st]), 0, key0 + (int)rank * C::K_ROWS, 0, kvbh);
            else        // this CTA's V columns: all BN keys, column block `rank` (CG = 2)
                tma_load_4d<CG == 2>(ring + st * part, map, lead(full[st]), 0, key0, (int)rank, kvbh);
        }
        if (!ok) {
            raise_timeout(&abort_flag, p.status);
            settle_copies();
        }
      } else if (warp == 1 && lane == 0 && n_kv > 0 && leader) {
        // ============================================================== MMA issuer
        // Descriptors are built once per operand tile; stepping along K adds the byte offset
        // (>> 4) to the start-address field, which cannot carry out of its 14 bits because
        // shared-memory addresses stay below 256 KiB.
        auto issue_s = [&](int t, int st) {
            const uint64_t qd = sdesc_sw128(sQ + t * C::Q_TILE, 16, 1024);
            const uint64_t kd = sdesc_sw128(sK + st * C::K_PART, 16, 1024);
            const uint32_t dst = tmem + (t ? C::S_COL1 : C::S_COL0);
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t aoff = ((k >> 2) * C::Q_DBLK + (k & 3) * 32) >> 4;
                const uint32_t boff = ((k >> 2) * C::K_DBLK + (k & 3) * 32) >> 4;
                if constexpr (CG == 2)
                    mma_ss_pair(dst, qd + aoff, kd + boff, C::IDESC_QK, k > 0);
                else
                    mma_ss(dst, qd + aoff, kd + boff, C::IDESC_QK, k > 0);
            }
        };
        auto issue_pv = [&](int t, int st, bool acc) {
            const uint64_t vd = sdesc_sw128(sV + st * C::V_PART, C::V_DBLK, 1024);
            const uint32_t dst = tmem + (t ? C::O_COL1 : C::O_COL0);
            const uint32_t pa = tmem + (t ? C::S_COL1 : C::S_COL0);
#pragma unroll
            for (int k = 0; k < BN / 16; ++k) {
                if constexpr (CG == 2)
                    mma_ts_pair(dst, pa + k * 8, vd + ((k * 2048) >> 4), C::IDESC_PV, acc || k > 0);
                else
                    mma_ts(dst, pa + k * 8, vd + ((k * 2048) >> 4), C::IDESC_PV, acc || k > 0);
            }
        };
        bool ok = mbar_wait_spin(smem_u32(&bars.q), 0, &abort_flag);
        if (ok) ok = mbar_wait_spin(smem_u32(&bars.k_full[0]), 0, &abort_flag);
        if (ok) {
            tc_fence_after();
            if (n0 > 0) {
                issue_s(0, 0);
                commit(bars.s_full[0]);
            }
            if (n1 > 0) {
                issue_s(1, 0);
                commit(bars.s_full[1]);
            }
            commit(bars.k_empty[0]);
        }
        for (int i = 0; i < n_kv && ok; ++i) {
            const int st = i % C::KV_STAGES;
            const int nx = i + 1;
            const int st2 = nx % C::KV_STAGES;
            ok = mbar_wait_spin(smem_u32(&bars.v_full[st]), (i / C::KV_STAGES) & 1, &abort_flag);
            if (!ok) break;
            if (i < n0) {
                ok = mbar_wait_spin(smem_u32(&bars.p_full[0]), i & 1, &abort_flag);
                if (!ok) break;
                tc_fence_after();
                issue_pv(0, st, i > 0);
                if (i == n0 - 1) commit(bars.o_final[0]);
            }
            if (nx < n_kv) {
                ok = mbar_wait_spin(smem_u32(&bars.k_full[st2]), (nx / C::KV_STAGES) & 1, &abort_flag);
                if (!ok) break;
                tc_fence_after();
                if (nx < n0) {
                    issue_s(0, st2);
                    commit(bars.s_full[0]);
                }
            }
            if (i < n1) {
                ok = mbar_wait_spin(smem_u32(&bars.p_full[1]), i & 1, &abort_flag);
                if (!ok) break;
                tc_fence_after();
                issue_pv(1, st, i > 0);
                if (i == n1 - 1) commit(bars.o_final[1]);
            }
            commit(bars.v_empty[st]);
            if (nx < n_kv) {
                if (nx < n1) {
                    issue_s(1, st2);
                    commit(bars.s_full[1]);
                }
                commit(bars.k_empty[st2]);
            }
        }
        if (!ok) raise_timeout(&abort_flag, p.status);
        // every MMA issued above completes before TMEM is released
        if constexpr (CG == 2)
            mma_commit_pair(smem_u32(&bars.drain), 1);
        else
            mma_commit(smem_u32(&bars.drain));
        mbar_wait(smem_u32(&bars.drain), 0, nullptr, 20000000ull);
      }
    } else {
        setmaxnreg_inc<kSoftmaxRegs>();
        // ============================================================== softmax
        const int t = (warp - 4) >> 2;           // Q tile
        const int r = tid - 128 * (t + 1);       // row within the tile == TMEM lane
        const int row = rb + t * BM + r;
        const int row_first = rb + t * BM;       // first row of this CTA's tile
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t s_addr = lane_base + (t ? C::S_COL1 : C::S_COL0);
        const uint32_t o_addr = lane_base + (t ? C::O_COL1 : C::O_COL0);
        const uint32_t p_full_lead = lead(bars.p_full[t]);
        const int nt = t ? n1 : n0;
        const float sl2 = p.scale_log2;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int i = 0; i < nt; ++i) {
            ok = mbar_wait(smem_u32(&bars.s_full[t]), i & 1, &abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + c * 32, sr[c]);
            tmem_ld_wait();
            const int key0 = (kt_begin + i) * BN;
            const bool need_mask = (key0 + BN > p.Sk) || (p.causal && key0 + BN - 1 > row_first);
            if (need_mask) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const int key = key0 + c * 32 + k;
                        const bool valid = key < p.Sk && (!p.causal || key <= row);
                        if (!valid) sr[c][k] = __float_as_uint(-INFINITY);
                    }
            }
            // row max: eight independent chains of 3-input max, then a short tree
            float mm[8];
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const int c = g >> 1, k0 = (g & 1) * 16;
                mm[g] = fmaxf(__uint_as_float(sr[c][k0]), __uint_as_float(sr[c][k0 + 1]));
#pragma unroll
                for (int v = 1; v < 8; ++v)
                    mm[g] = fmax3(mm[g], __uint_as_float(sr[c][k0 + 2 * v]), __uint_as_float(sr[c][k0 + 2 * v + 1]));
            }
            const float mx = fmax3(fmax3(mm[0], mm[1], mm[2]), fmax3(mm[3], mm[4], mm[5]), fmaxf(mm[6], mm[7]));
            const float m_tile = mx * sl2;   // -inf stays -inf (sl2 > 0)
            const float m_new = fmaxf(m_ref, m_tile);
            const bool rescale = __any_sync(0xffffffffu, m_new > m_ref + kRescaleThreshold);
            float alpha = 1.f;
            if (rescale) {
                alpha = ex2_approx(m_ref - m_new);   // m_ref == -inf -> 0
                l *= alpha;
                m_ref = m_new;
            }
            const float mr = (m_ref == -INFINITY) ? 0.f : m_ref;
            const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(-mr, -mr);
            uint64_t acc[4];
            // p = 2^(s * scale * log2e - m): pairs through one f32x2 FMA, sums in four
            // independent f32x2 accumulators; P packed to bf16 over the first half of S.
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                acc[c] = f2_pack(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    float p0, p1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c][2 * k]), __uint_as_float(sr[c][2 * k + 1])), sc2, nm2),
                              p0, p1);
                    p0 = ex2_approx(p0);
                    p1 = ex2_approx(p1);
                    acc[c] = f2_add(acc[c], f2_pack(p0, p1));
                    sr[c][k] = pack_bf16x2(p0, p1);
                }
                tmem_st16(s_addr + c * 16, sr[c][0], sr[c][1], sr[c][2], sr[c][3], sr[c][4], sr[c][5], sr[c][6],
                          sr[c][7], sr[c][8], sr[c][9], sr[c][10], sr[c][11], sr[c][12], sr[c][13], sr[c][14],
                          sr[c][15]);
            }
            float rs;
            {
                const uint64_t a2 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
                float lo, hi;
                f2_unpack(a2, lo, hi);
                rs = lo + hi;
            }
            if (rescale && i > 0) {
                // O_t += P V of earlier tiles has completed: the commit that signalled s_full
                // for this tile covers every MMA issued before it.  The PV MMA of this tile
                // waits for p_full, signalled below, after the rescaled O is stored.
                const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(o_addr + c * 32, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        float a, bb;
                        f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * k]), __uint_as_float(o[2 * k + 1])), al2), a, bb);
                        o[2 * k] = __float_as_uint(a);
                        o[2 * k + 1] = __float_as_uint(bb);
                    }
                    tmem_st32(o_addr + c * 32, o);
                }
            }
            l += rs;
            // P (and any rescaled O) of all 128 rows are in TMEM: one arrival per CTA.
            tmem_st_wait();
            tc_fence_before();
            named_barrier(1 + t, 128);
            if (r == 0) {
                if (CG == 2 && !leader)
                    mbar_arrive_cluster_relaxed(p_full_lead);
                else
                    mbar_arrive(smem_u32(&bars.p_full[t]));
            }
        }
        if (!ok) raise_timeout(&abort_flag, p.status);
        // ---------------------------------------------------------- epilogue
        if (t < ntiles) {
            bool have_o = false;
            if (ok && nt > 0) {
                ok = mbar_wait(smem_u32(&bars.o_final[t]), 0, &abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) raise_timeout(&abort_flag, p.status);
                have_o = ok;
                tc_fence_after();
            }
            const long long rows_total = (long long)p.B * p.Hq * p.Sq;
            const long long grow = (long long)bh * p.Sq + row;
            const bool row_ok = row < p.Sq;
            if (p.splits == 1) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
                __nv_bfloat16 *Og = static_cast<__nv_bfloat16 *>(p.o) + grow * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    if (have_o) {
                        tmem_ld32(o_addr + c * 32, o);
                        tmem_ld_wait();
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        pk[k] = have_o ? pack_bf16x2(__uint_as_float(o[2 * k]) * inv, __uint_as_float(o[2 * k + 1]) * inv)
                                       : 0u;
                    if (row_ok) {
                        uint4 *dst = reinterpret_cast<uint4 *>(Og + c * 32);
#pragma unroll
                        for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                    }
                }
                if (p.lse && row_ok) p.lse[grow] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
            } else {
                float *A = p.part_acc + ((size_t)blockIdx.y * rows_total + grow) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    if (have_o) {
                        tmem_ld32(o_addr + c * 32, o);
                        tmem_ld_wait();
                    }
                    if (row_ok) {
                        float4 *dst = reinterpret_cast<float4 *>(A + c * 32);
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            dst[k] = have_o ? make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                                          __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]))
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                if (row_ok) {
                    p.part_m[(size_t)blockIdx.y * rows_total + grow] = have_o ? m_ref : -INFINITY;
                    p.part_l[(size_t)blockIdx.y * rows_total + grow] = have_o ? l : 0.f;
                }
            }
        }
    }

    tc_fence_before();
    __syncwarp();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync();   // the peer may still be read by the pair's MMAs until here
    if (warp == 0) {
        tc_fence_after();
        if constexpr (CG == 2)
            tmem_dealloc_pair(tmem, TMEM_COLS);
        else
            tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------------- host side
template <int D, int CG>
cudaError_t launch_t(const AttnProblem &p, cudaStream_t s) {
    using C = TcCfg<D, CG>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(attn_tc_kernel<D, CG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)C::SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap mq, mk, mv;
    if (!make_bf16_tile_map(&mq, p.q, D, p.Sq, (long long)p.B * p.Hq, BM) ||
        !make_bf16_tile_map(&mk, p.k, D, p.Sk, (long long)p.B * p.Hkv, C::K_ROWS) ||
        !make_bf16_tile_map(&mv, p.v, D, p.Sk, (long long)p.B * p.Hkv, BN, C::V_COLS / 64))
        return cudaErrorInvalidValue;
    const int G = p.Hq / p.Hkv;
    const bool pair_heads = CG == 2 && (G % 2) == 0;
    const int rows_per_item = (CG == 2 && !pair_heads) ? 4 * BM : 2 * BM;
    const int n_qb = (p.Sq + rows_per_item - 1) / rows_per_item;
    const int units = pair_heads ? p.B * p.Hq / 2 : p.B * p.Hq;
    const long long ctas = (long long)n_qb * units * CG;
    if (ctas >= (1LL << 31)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)ctas, (unsigned)p.splits);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    if (CG == 2) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, attn_tc_kernel<D, CG>, mq, mk, mv, p, n_qb);
    count_launches(1);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

// CTAs the kernel runs for a problem (before any key split).
long long tc_ctas(const AttnProblem &p) {
    const int CG = p.D == 128 ? 2 : 1;
    const int G = p.Hq / p.Hkv;
    const bool pair_heads = CG == 2 && (G % 2) == 0;
    const int rows_per_item = (CG == 2 && !pair_heads) ? 4 * BM : 2 * BM;
    const long long n_qb = (p.Sq + rows_per_item - 1) / rows_per_item;
    return n_qb * (pair_heads ? (long long)p.B * p.Hq / 2 : (long long)p.B * p.Hq) * CG;
}

}  // namespace

bool attn_tc_supported(const AttnProblem &p, const void *Q, const void *K, const void *V, const void *O) {
    if (p.dtype != OSF_BF16 || p.Sq < 2 || (p.D != 64 && p.D != 128)) return false;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return false;
    if (tc_ctas(p) >= (1LL << 31)) return false;
    return tensor_map_encoder() != nullptr;
}

int attn_tc_pick_splits(const AttnProblem &p, int sm_count) {
    const long long ctas = tc_ctas(p);
    const int n_kt = (p.Sk + BN - 1) / BN;
    if (ctas >= sm_count || n_kt <= 1) return 1;
    int want = (int)((sm_count + ctas - 1) / ctas);
    if (want > n_kt) want = n_kt;
    const int tps = (n_kt + want - 1) / want;
    return (n_kt + tps - 1) / tps;   // no empty split
}

cudaError_t launch_attn_tc(const AttnProblem &p, int sm_count, cudaStream_t s) {
    (void)sm_count;
    cudaError_t e = p.D == 64 ? launch_t<64, 1>(p, s) : launch_t<128, 2>(p, s);
    if (e == cudaSuccess && p.splits > 1) e = launch_attn_combine(p, s);
    return e;
}

}  // namespace osf
