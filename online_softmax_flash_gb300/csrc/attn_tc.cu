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
// Roles (12 warps per CTA):
//   warps 0, 2  TMA: the Q tiles once, then K (warp 0) and V (warp 2) tiles through one
//               shared ring, one instruction per tile
//   warp 1      MMA issue (one thread): S_t = Q_t K^T (both operands in shared memory),
//               O_t += P_t V (P read from TMEM; bf16 with D = 64: from shared memory)
//   warps 4-7   softmax for Q tile 0, warps 8-11 for Q tile 1: thread r owns TMEM lane r, i.e.
//               query row r of its tile, so row max and row sum need no cross-thread traffic.
//
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+DO), O_1 [256+DO,256+2DO), DO = D
// (float32 mode: 2D).  P_t (bf16, two per column) overwrites the first 64 columns of S_t and is
// read from there by the PV MMA; bf16 with D = 64 writes P_t to a shared-memory operand tile
// instead; float32 mode keeps P's two parts in each 32-column chunk of S_t.  The two Q tiles are
// ping-ponged so one tile's softmax overlaps the other tile's MMAs.
//
// Scores are kept in base 2 (scale * log2 e folded into one multiplier).  The rescale of O is
// lazy: a row keeps its reference maximum until a tile raises the maximum by more than 8
// (a factor 256), so O is rarely touched; the result O / l is the same for any reference.
//
// Every mbarrier wait is bounded (2 s); on expiry the CTA records OSF_ERR_TIMEOUT in the
// device status word, drains its own MMAs, lets its copies land, frees TMEM and exits.
#include <map>
#include <mutex>
#include <utility>

#include "attn_tc.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.cuh"

namespace osf {
namespace {

using namespace ptx;

constexpr int BM = 128;             // query rows per Q tile
constexpr int BN = 128;             // keys per key tile
constexpr int NTHREADS = 384;       // 12 warps: 0-3 control, 4-7 softmax tile 0, 8-11 tile 1
constexpr uint32_t TMEM_COLS = 512;
// Register split after set-up: the two softmax warpgroups hold a whole 128-column score row
// each; the control warpgroup (TMA + MMA issue) keeps 88.  Issuing one tcgen05.mma costs the
// issuing thread about 46 cycles against 64 cycles of tensor work, so any spill or recomputation
// in the issue loop starves the tensor pipe (its queue holds only a few instructions); below
// about 88 registers that happened.  128*88 + 256*208 = 384*168, the registers the CTA is
// launched with (168 per thread).
constexpr int kCtrlRegs = 88, kSoftmaxRegs = 208;
// x3 mode: the issuer carries six score products per tile and the softmax holds one chunk at a
// time: 128*120 + 256*192 = 384*168 as well
constexpr int kCtrlRegsX3 = 120, kSoftmaxRegsX3 = 192;
constexpr float kRescaleThreshold = 8.0f;   // base-2 units

constexpr uint32_t kSmemLimit = 232448;   // dynamic shared memory per CTA (227 KiB)
constexpr int kMaxStages = 12;

// X3 (float32 Q, K, V, D = 64): every operand is a sum of bf16 parts and every product a sum
// of bf16 products with fp32 accumulation.  Q and K have three parts, x = h + m + l with
// h = bf16(x), m = bf16(x - h), l = bf16(x - h - m) (x to about 2^-26 relative), and
//   S = Qh Kh^T + Qh Km^T + Qm Kh^T + Qh Kl^T + Ql Kh^T + Qm Km^T
// drops only terms of about 2^-24 relative: the exponent turns an absolute error of S into a
// relative error of P, so S must be as good as float32.  V and P (in [0, 1]) have two parts,
// h and l = bf16(x - h) (about 2^-17 relative), and O += Ph [Vh | Vl] + Pl [Vh | Vl] (Pl Vh alone
// when Vh and Vl are not in adjacent ring stages), with O = O[:, :D] + O[:, D:] at the end.
template <int D, bool X3>
struct TcCfg {
    static constexpr uint32_t TILE = BN * D * 2;                 // one [128 x D] bf16 tile (Q, K or V)
    static constexpr uint32_t DBLK = BN * 128;                   // bytes between 64-column blocks
    static constexpr int QP = X3 ? 3 : 1, KP = X3 ? 3 : 1, VP = X3 ? 2 : 1;   // parts per operand
    static constexpr int QT = 2 * QP;                            // resident Q tiles: part p of tile t at 2p + t
    static constexpr int NPOS = KP + VP;                         // ring positions per key tile
    // K and V tiles share one ring, filled in the order they are consumed (K0 V0 K1 V1 ..., in
    // x3 mode K0h K0m K0l V0h V0l ...); the ring takes what the Q tiles leave of shared memory
    // (5 stages at D = 128, 8 in x3 mode).
    // bf16 with D = 64: P goes to the MMA through shared memory (a K-major [128 x 128] tile per Q
    // tile), so PV reads both operands from shared memory rather than P from TMEM
    static constexpr bool PSMEM = !X3 && D == 64;
    static constexpr uint32_t P_TILE = BM * BN * 2;
    static constexpr uint32_t P_BYTES = PSMEM ? 2 * P_TILE : 0;
    static constexpr int FIT = (int)((kSmemLimit - 2048 - QT * TILE - P_BYTES) / TILE);
    static constexpr int STAGES = FIT < kMaxStages ? FIT : kMaxStages;
    static_assert(!X3 || (D == 64 && STAGES >= 2 * NPOS - 2 && TILE == DBLK), "x3 mode is built for D = 64");
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t RING_OFF = QT * TILE;
    static constexpr uint32_t P_OFF = RING_OFF + STAGES * TILE;
    static constexpr uint32_t SMEM_BYTES = P_OFF + P_BYTES + 1024;  // + alignment slack
    static constexpr int DO = X3 ? 2 * D : D;                    // TMEM columns of one O accumulator
    static constexpr uint32_t S_COL0 = 0, S_COL1 = 128, O_COL0 = 256, O_COL1 = 256 + DO;
    static constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, 0, 0);
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, 0, 1);
    static constexpr uint32_t IDESC_PV2 = idesc_bf16_f32(BM, 2 * D, 0, 1);
};

struct Barriers {
    uint64_t q_full, q_empty;
    uint64_t full[kMaxStages], empty[kMaxStages];
    uint64_t s_full[2], p_full[2], o_final[2], o_empty[2];
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

// One work item: 2 x 128 query rows of one (b, q-head), over the key tiles of this CTA's split.
struct Item {
    int q0, bh, b, hq, kvh, ntiles, n0, n1, n_kv, kt_begin;
};

// Item of round r for this CTA: rounds walk the item list in snake order (forward on even
// rounds, backward on odd ones), which pairs heavy causal blocks with light ones.
__device__ __forceinline__ bool item_at(const AttnProblem &p, int n_qb, int n_items, int r, Item &w) {
    const int g = (int)gridDim.x;
    const int c = (r & 1) ? g - 1 - (int)blockIdx.x : (int)blockIdx.x;
    const long long it = (long long)r * g + c;
    if (it >= n_items) return false;
    const int units = p.B * p.Hq;
    const int qb_rank = (int)(it / units);
    w.bh = (int)(it % units);
    const int qb = p.causal ? (n_qb - 1 - qb_rank) : qb_rank;   // heaviest blocks first
    w.q0 = qb * 2 * BM;
    w.b = w.bh / p.Hq;
    w.hq = w.bh % p.Hq;
    w.kvh = w.hq / (p.Hq / p.Hkv);
    w.ntiles = (w.q0 + BM < p.Sq) ? 2 : 1;
    const int n_kt_all = (p.Sk + BN - 1) / BN;
    const int tps = (n_kt_all + p.splits - 1) / p.splits;
    w.kt_begin = blockIdx.y * tps;
    const int kt_end = min(n_kt_all, w.kt_begin + tps);
    // key tiles each Q tile visits (causal: up to the last key its last row sees)
    int e0 = kt_end, e1 = kt_end;
    if (p.causal) {
        const int last0 = min(w.q0 + BM - 1, p.Sq - 1) + p.causal_off;
        const int last1 = min(w.q0 + 2 * BM - 1, p.Sq - 1) + p.causal_off;
        e0 = min(e0, last0 < 0 ? 0 : last0 / BN + 1);
        e1 = min(e1, last1 < 0 ? 0 : last1 / BN + 1);
    }
    w.n0 = max(0, e0 - w.kt_begin);
    w.n1 = w.ntiles == 2 ? max(0, e1 - w.kt_begin) : 0;
    w.n_kv = max(w.n0, w.n1);
    return true;
}

// Persistent: each CTA walks its work items (item_at) with one pipeline whose state -- ring
// position, barrier phases -- carries from item to item, so an item's Q tiles and first K/V
// tiles load while the previous item finishes.
//
// MERGE (key splits, one item per CTA): the CTAs of a thread-block cluster run the splits of one
// item and merge their results through distributed shared memory at the end, instead of writing
// partial states for a separate combine kernel.
template <int D, bool X3, bool MERGE>
__global__ void __launch_bounds__(NTHREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mqm,
               const __grid_constant__ CUtensorMap mkm, const __grid_constant__ CUtensorMap mql,
               const __grid_constant__ CUtensorMap mkl, const __grid_constant__ CUtensorMap mvl,
               const AttnProblem p, int n_qb, int n_items) {
    using C = TcCfg<D, X3>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ Barriers bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = sbase + C::Q_OFF, sRing = sbase + C::RING_OFF;
    // ring position of the n-th tile of the stream K V K V ...: stage and phase parity
    auto stage_of = [](int n) { return n % C::STAGES; };
    auto parity_of = [](int n) { return (n / C::STAGES) & 1; };

    // ------------------------------------------------------------------ set-up
    if (warp == 0) tmem_alloc(smem_u32(&tmem_base_sh), TMEM_COLS);
    if (tid == 32) {
        mbar_init(smem_u32(&bars.q_full), 1);
        mbar_init(smem_u32(&bars.q_empty), 1);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&bars.full[s]), 1);
            mbar_init(smem_u32(&bars.empty[s]), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_u32(&bars.s_full[t]), 1);
            mbar_init(smem_u32(&bars.p_full[t]), 4);     // one arrival per softmax warp
            mbar_init(smem_u32(&bars.o_final[t]), 1);
            mbar_init(smem_u32(&bars.o_empty[t]), 4);
        }
        mbar_init(smem_u32(&bars.drain), 1);
        abort_flag = 0;
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    // MERGE: a softmax thread's final row state, kept for the cluster merge at the end
    float fin_m = -INFINITY, fin_l = 0.f;
    bool fin_have = false;

    if (warp < 4) {
      setmaxnreg_dec<X3 ? kCtrlRegsX3 : kCtrlRegs>();
      if ((warp == 0 || warp == 2) && lane == 0) {
        // float32 mode runs as a dependent of the split pre-pass: its parts are read by TMA only
        if (X3) griddep_wait();
        // ============================================================== TMA producers
        // The ring receives K V K V ... in consumption order; warp 0 issues the Q tiles and the
        // K tiles (even stream positions), warp 2 the V tiles (odd positions), one TMA
        // instruction per tile, so neither stream waits behind the other's instruction issue.
        // An item's Q tiles load once the previous item's last Q K^T products have completed.
        const int odd = warp == 2;
        const CUtensorMap *map = odd ? &mv : &mk, *map_lo = odd ? &mvl : &mkl;
        tma_prefetch_desc(map);
        if (X3) {
            tma_prefetch_desc(map_lo);
            if (!odd) tma_prefetch_desc(&mkm);
        }
        if (!odd) {
            tma_prefetch_desc(&mq);
            if (X3) {
                tma_prefetch_desc(&mqm);
                tma_prefetch_desc(&mql);
            }
        }
        bool ok = true;
        int gt = 0, qc = 0;   // key tiles streamed so far, Q loads so far
        Item w;
        for (int r = 0; ok && item_at(p, n_qb, n_items, r, w); ++r) {
            if (w.n_kv == 0) continue;
            if (!odd) {
                ok = mbar_wait(smem_u32(&bars.q_empty), (qc & 1) ^ 1, &abort_flag);
                if (!ok) break;
                ++qc;
                mbar_expect_tx(smem_u32(&bars.q_full), w.ntiles * C::TILE * C::QP);
#pragma unroll
                for (int part = 0; part < C::QP; ++part)
                    for (int t = 0; t < w.ntiles; ++t)
                        tma_load_5d(sQ + (2 * part + t) * C::TILE, part == 0 ? &mq : part == 1 ? &mqm : &mql,
                                    smem_u32(&bars.q_full), 0, w.q0 + t * BM, 0, w.hq, w.b);
            }
            for (int j = 0; j < w.n_kv && ok; ++j) {
#pragma unroll
                for (int part = 0; part < (odd ? C::VP : C::KP); ++part) {
                    const int n = C::NPOS * (gt + j) + (odd ? C::KP : 0) + part;
                    const int st = stage_of(n);
                    ok = mbar_wait(smem_u32(&bars.empty[st]), parity_of(n) ^ 1, &abort_flag);
                    if (!ok) break;
                    mbar_expect_tx(smem_u32(&bars.full[st]), C::TILE);
                    const CUtensorMap *mp = part == 0 ? map : (part == 2 || odd) ? map_lo : &mkm;
                    tma_load_5d(sRing + st * C::TILE, mp, smem_u32(&bars.full[st]), 0, (w.kt_begin + j) * BN, 0,
                                w.kvh, w.b);
                }
            }
            gt += w.n_kv;
        }
        if (!ok) {
            raise_timeout(&abort_flag, p.status);
            settle_copies();
        }
      } else if (warp == 1 && lane == 0) {
        // ============================================================== MMA issuer
        // Issue order per key tile i:  O_0 += P_0 V_i;  S_0 = Q_0 K_{i+1}^T;  O_1 += P_1 V_i;
        // S_1 = Q_1 K_{i+1}^T, so one tile's softmax runs while the other tile's products do.
        // Each PV waits for its tile's P; the commit after a tile's S covers the PV before it,
        // which the softmax relies on when it rescales O.  An item's first PV of a tile also
        // waits until the softmax has read that tile's O of the previous item.
        //
        // Descriptors are built once per operand tile; stepping along K adds the byte offset
        // (>> 4) to the start-address field, which cannot carry out of its 14 bits because
        // shared-memory addresses stay below 256 KiB.
        // Stream positions of key tile g: K parts from NPOS*g, V parts from NPOS*g + KP.  An
        // operand's parts (consecutive positions from stage st, parity ph) are waited for and
        // released together.  Stages and parities are computed before the waits: anything
        // between a wait and the MMAs it releases lengthens the P hand-off chain.
        // the stage after stage s (the parity flips when the ring wraps)
        auto next_stage = [](int s) { return s + 1 == C::STAGES ? 0 : s + 1; };
        auto wait_parts = [&](int st, uint32_t ph, int parts) {
            bool r = mbar_wait_spin(smem_u32(&bars.full[st]), ph, &abort_flag);
            for (int q = 1; q < parts && r; ++q) {
                st = next_stage(st);
                if (st == 0) ph ^= 1;
                r = mbar_wait_spin(smem_u32(&bars.full[st]), ph, &abort_flag);
            }
            return r;
        };
        auto release_parts = [&](int st, int parts) {
            mma_commit(smem_u32(&bars.empty[st]));
            for (int q = 1; q < parts; ++q) {
                st = next_stage(st);
                mma_commit(smem_u32(&bars.empty[st]));
            }
        };
        // D/16 k-steps of S (+)= A B^T with both operands [128 x D] tiles in shared memory
        auto qk = [&](uint32_t dst, uint32_t a_tile, uint32_t b_tile, bool acc) {
            const uint64_t ad = sdesc_sw128(a_tile, 16, 1024), bd = sdesc_sw128(b_tile, 16, 1024);
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t off = ((k >> 2) * C::DBLK + (k & 3) * 32) >> 4;
                mma_ss(dst, ad + off, bd + off, C::IDESC_QK, acc || k > 0);
            }
        };
        // S_t = Q_t K^T for the K tile (first part) in stage k0 (x3: six part products)
        auto issue_s = [&](int t, int k0) {
            const uint32_t dst = tmem + (t ? C::S_COL1 : C::S_COL0);
            auto qp = [&](int part) { return sQ + (2 * part + t) * C::TILE; };
            qk(dst, qp(0), sRing + k0 * C::TILE, false);
            if constexpr (X3) {
                const int k1 = next_stage(k0), k2 = next_stage(k1);
                const uint32_t kh = sRing + k0 * C::TILE, km = sRing + k1 * C::TILE, kl = sRing + k2 * C::TILE;
                qk(dst, qp(0), km, true);
                qk(dst, qp(1), kh, true);
                qk(dst, qp(0), kl, true);
                qk(dst, qp(2), kh, true);
                qk(dst, qp(1), km, true);
            }
        };
        // k-steps of O (+)= P V: P (bf16) in TMEM from column pa, V tile at vd, N per idesc
        auto pv = [&](uint32_t dst, uint32_t pa, uint64_t vd, uint32_t idesc, bool acc) {
#pragma unroll
            for (int k = 0; k < BN / 16; ++k) mma_ts(dst, pa + k * 8, vd + ((k * 2048) >> 4), idesc, acc || k > 0);
        };
        // x3 layout: keys 32c..32c+31 of a P part sit in columns 32c + [0, 16) (hi) or + [16, 32)
        // (lo); k-step k (16 keys) starts at column 32 (k / 2) + 8 (k % 2) from the part's base
        auto pv_x3 = [&](uint32_t dst, uint32_t pa, uint64_t vd, uint32_t idesc, bool acc) {
#pragma unroll
            for (int k = 0; k < BN / 16; ++k)
                mma_ts(dst, pa + 32 * (k >> 1) + 8 * (k & 1), vd + ((k * 2048) >> 4), idesc, acc || k > 0);
        };
        // O_t (+)= P_t V for the V tile (first part) in stage sv; P_t is the bf16 copy over S_t's
        // first 64 columns (x3: P hi there, P lo over the next 64)
        auto issue_pv = [&](int t, int sv, bool acc) {
            const uint32_t dst = tmem + (t ? C::O_COL1 : C::O_COL0);
            const uint32_t pa = tmem + (t ? C::S_COL1 : C::S_COL0);
            const uint64_t vd = sdesc_sw128(sRing + sv * C::TILE, C::DBLK, 1024);
            if constexpr (C::PSMEM) {
                (void)pa;
                const uint64_t pd = sdesc_sw128(sbase + C::P_OFF + t * C::P_TILE, 16, 1024);
#pragma unroll
                for (int k = 0; k < BN / 16; ++k) {
                    const uint32_t offa = ((k >> 2) * C::DBLK + (k & 3) * 32) >> 4;
                    mma_ss(dst, pd + offa, vd + ((k * 2048) >> 4), C::IDESC_PV, acc || k > 0);
                }
            } else if constexpr (!X3) {
                pv(dst, pa, vd, C::IDESC_PV, acc);
            } else {
                const int sl = next_stage(sv);
                if (sl == sv + 1) {
                    // Ph [Vh | Vl] and Pl [Vh | Vl]: V lo is the next stage, one 64-column block
                    // on, so both are N = 2D products (Pl Vl, about 2^-18 of P V, comes for free)
                    pv_x3(dst, pa, vd, C::IDESC_PV2, acc);
                    pv_x3(dst, pa + 16, vd, C::IDESC_PV2, true);
                } else {
                    pv_x3(dst, pa, vd, C::IDESC_PV, acc);
                    pv_x3(dst + D, pa, sdesc_sw128(sRing + sl * C::TILE, C::DBLK, 1024), C::IDESC_PV, acc);
                    pv_x3(dst, pa + 16, vd, C::IDESC_PV, true);   // + Pl Vh into the first D columns
                }
            }
        };
        // PV for Q tile t at key tile i of an item; pc[t] counts P handshakes, oe[t] the O
        // hand-backs owed by earlier items
        int pc[2] = {0, 0}, oe[2] = {0, 0};
        auto pv_step = [&](int t, int i, int nt, int sv) -> bool {
            if (i == 0 && oe[t] > 0 &&
                !mbar_wait_spin(smem_u32(&bars.o_empty[t]), (oe[t] - 1) & 1, &abort_flag))
                return false;
            if (!mbar_wait_spin(smem_u32(&bars.p_full[t]), pc[t] & 1, &abort_flag)) return false;
            ++pc[t];
            tc_fence_after();
            issue_pv(t, sv, i > 0);
            if (i == nt - 1) mma_commit(smem_u32(&bars.o_final[t]));
            return true;
        };
        bool ok = true;
        int gt = 0, qc = 0;
        Item w;
        for (int r = 0; ok && item_at(p, n_qb, n_items, r, w); ++r) {
            if (w.n_kv == 0) continue;
            const int n0 = w.n0, n1 = w.n1, n_kv = w.n_kv;
            ok = mbar_wait_spin(smem_u32(&bars.q_full), qc & 1, &abort_flag);
            ++qc;
            const int sk0 = stage_of(C::NPOS * gt);
            if (ok) ok = wait_parts(sk0, parity_of(C::NPOS * gt), C::KP);
            if (!ok) break;
            tc_fence_after();
            if (n0 > 0) {
                issue_s(0, sk0);
                mma_commit(smem_u32(&bars.s_full[0]));
            }
            if (n1 > 0) {
                issue_s(1, sk0);
                mma_commit(smem_u32(&bars.s_full[1]));
            }
            release_parts(sk0, C::KP);
            // Q is free once the item's last Q K^T products complete: the next item's Q tiles
            // then load while this item's last softmax and PV products run.
            if (n_kv == 1) mma_commit(smem_u32(&bars.q_empty));
            for (int i = 0; i < n_kv; ++i) {
                // V_i and K_{i+1}
                const int nv = C::NPOS * (gt + i) + C::KP, nk = C::NPOS * (gt + i + 1);
                const int sv = stage_of(nv), sk = stage_of(nk);
                const uint32_t phv = parity_of(nv), phk = parity_of(nk);
                const bool more = i + 1 < n_kv;
                ok = wait_parts(sv, phv, C::VP);
                if (!ok) break;
                if (i < n0 && !(ok = pv_step(0, i, n0, sv))) break;
                if (more) {
                    ok = wait_parts(sk, phk, C::KP);
                    if (!ok) break;
                    tc_fence_after();
                    if (i + 1 < n0) {
                        issue_s(0, sk);
                        mma_commit(smem_u32(&bars.s_full[0]));
                    }
                }
                if (i < n1 && !(ok = pv_step(1, i, n1, sv))) break;
                release_parts(sv, C::VP);
                if (more) {
                    if (i + 1 < n1) {
                        issue_s(1, sk);
                        mma_commit(smem_u32(&bars.s_full[1]));
                    }
                    release_parts(sk, C::KP);
                    if (i + 2 == n_kv) mma_commit(smem_u32(&bars.q_empty));   // last Q K^T issued
                }
            }
            if (!ok) break;
            oe[0] += n0 > 0;
            oe[1] += n1 > 0;
            gt += n_kv;
        }
        if (!ok) raise_timeout(&abort_flag, p.status);
        // every MMA issued above completes before TMEM is released
        mma_commit(smem_u32(&bars.drain));
        mbar_wait(smem_u32(&bars.drain), 0, nullptr, 20000000ull);
      }
    } else {
        setmaxnreg_inc<X3 ? kSoftmaxRegsX3 : kSoftmaxRegs>();
        // ============================================================== softmax
        const int t = (warp - 4) >> 2;           // Q tile
        const int r = tid - 128 * (t + 1);       // row within the tile == TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t s_addr = lane_base + (t ? C::S_COL1 : C::S_COL0);
        const uint32_t o_addr = lane_base + (t ? C::O_COL1 : C::O_COL0);
        const uint32_t p_smem = sbase + C::P_OFF + t * C::P_TILE;   // PSMEM: this tile's P
        (void)p_smem;
        const float sl2 = p.scale_log2;
        const long long rows_total = (long long)p.B * p.Hq * p.Sq;
        bool ok = true;
        int sc = 0, oc = 0;   // S handshakes and finished O tiles so far
        Item w;
        for (int rr = 0; ok && item_at(p, n_qb, n_items, rr, w); ++rr) {
            const int nt = t ? w.n1 : w.n0;
            const int row_first = w.q0 + t * BM;   // first row of this tile
            const int row = row_first + r;
            float m_ref = -INFINITY, l = 0.f;
            for (int i = 0; i < nt; ++i) {
                ok = mbar_wait(smem_u32(&bars.s_full[t]), sc & 1, &abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                ++sc;
                tc_fence_after();
                const int key0 = (w.kt_begin + i) * BN;
                const bool need_mask = (key0 + BN > p.Sk) || (p.causal && key0 + BN - 1 > row_first + p.causal_off);
                // column j of the tile (key key0 + j) is kept iff j < lim: inside the sequence
                // and, when causal, not after the last key this row sees
                int lim = p.Sk - key0;
                if (p.causal) lim = min(lim, row + p.causal_off - key0 + 1);
                uint32_t sr[X3 ? 1 : 4][32];   // bf16 mode: the whole score row in registers
                float mx;
                if constexpr (X3) {
                    // two passes over TMEM (the row max, then P) keep one 32-column chunk in
                    // registers, which leaves room for P's two parts
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        tmem_ld32(s_addr + c * 32, sr[0]);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            const float x = (need_mask && c * 32 + k >= lim) ? -INFINITY : __uint_as_float(sr[0][k]);
                            m4[k & 3] = fmaxf(m4[k & 3], x);
                        }
                    }
                    mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + c * 32, sr[c]);
                    tmem_ld_wait();
                    if (need_mask) {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                if (c * 32 + k >= lim) sr[c][k] = __float_as_uint(-INFINITY);
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
                    mx = fmax3(fmax3(mm[0], mm[1], mm[2]), fmax3(mm[3], mm[4], mm[5]), fmaxf(mm[6], mm[7]));
                }
                const float m_tile = mx * sl2;   // -inf stays -inf (sl2 > 0)
                const float m_new = fmaxf(m_ref, m_tile);
                const bool rescale = __any_sync(0xffffffffu, m_new > m_ref + kRescaleThreshold);
                float alpha = 1.f;
                if (rescale) {
                    // the warp rescales together; a row that has seen no key yet (m_new still
                    // -inf, e.g. all keys of this split are after it) keeps l = 0, not NaN
                    alpha = ex2_approx(m_ref - (m_new == -INFINITY ? 0.f : m_new));   // m_ref == -inf -> 0
                    l *= alpha;
                    m_ref = m_new;
                }
                const float mr = (m_ref == -INFINITY) ? 0.f : m_ref;
                const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(-mr, -mr);
                float rs;
                if constexpr (X3) {
                    // chunk c (keys 32c..32c+31) puts P hi over its own first 16 columns and
                    // P lo = bf16(p - P hi) over its last 16, so no chunk overwrites unread scores
                    uint64_t acc = f2_pack(0.f, 0.f);
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        tmem_ld32(s_addr + c * 32, sr[0]);
                        tmem_ld_wait();
                        uint32_t ph[16], pl[16];
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            const float s0 = (need_mask && c * 32 + 2 * k >= lim) ? -INFINITY : __uint_as_float(sr[0][2 * k]);
                            const float s1 = (need_mask && c * 32 + 2 * k + 1 >= lim) ? -INFINITY
                                                                                     : __uint_as_float(sr[0][2 * k + 1]);
                            float p0, p1;
                            f2_unpack(f2_fma(f2_pack(s0, s1), sc2, nm2), p0, p1);
                            p0 = ex2_approx(p0);
                            p1 = ex2_approx(p1);
                            acc = f2_add(acc, f2_pack(p0, p1));
                            ph[k] = pack_bf16x2(p0, p1);
                            pl[k] = pack_bf16x2(p0 - __uint_as_float(ph[k] << 16), p1 - __uint_as_float(ph[k] & 0xffff0000u));
                        }
                        tmem_st16(s_addr + c * 32, ph[0], ph[1], ph[2], ph[3], ph[4], ph[5], ph[6], ph[7], ph[8], ph[9],
                                  ph[10], ph[11], ph[12], ph[13], ph[14], ph[15]);
                        tmem_st16(s_addr + c * 32 + 16, pl[0], pl[1], pl[2], pl[3], pl[4], pl[5], pl[6], pl[7], pl[8],
                                  pl[9], pl[10], pl[11], pl[12], pl[13], pl[14], pl[15]);
                    }
                    float lo, hi;
                    f2_unpack(acc, lo, hi);
                    rs = lo + hi;
                } else {
                    uint64_t acc[4];
                    // p = 2^(s * scale * log2e - m): pairs through one f32x2 FMA, sums in four
                    // independent f32x2 accumulators; P packed to bf16 over the first half of S.
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        acc[c] = f2_pack(0.f, 0.f);
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            float p0, p1;
                            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c][2 * k]), __uint_as_float(sr[c][2 * k + 1])),
                                             sc2, nm2),
                                      p0, p1);
                            p0 = ex2_approx(p0);
                            p1 = ex2_approx(p1);
                            acc[c] = f2_add(acc[c], f2_pack(p0, p1));
                            sr[c][k] = pack_bf16x2(p0, p1);
                        }
                        if constexpr (C::PSMEM) {
                            // keys 32c..32c+31 of row r: four 16-byte chunks of the 128-byte row in
                            // block c / 2, at chunk index (c % 2) * 4 + i, XOR-swizzled by r % 8
                            const uint32_t rowb = p_smem + (c >> 1) * C::DBLK + r * 128;
#pragma unroll
                            for (int i2 = 0; i2 < 4; ++i2) {
                                const uint32_t q = (uint32_t)((c & 1) * 4 + i2);
                                st_shared_v4(rowb + ((q ^ (uint32_t)(r & 7)) << 4), sr[c][4 * i2], sr[c][4 * i2 + 1],
                                             sr[c][4 * i2 + 2], sr[c][4 * i2 + 3]);
                            }
                        } else {
                            tmem_st16(s_addr + c * 16, sr[c][0], sr[c][1], sr[c][2], sr[c][3], sr[c][4], sr[c][5],
                                      sr[c][6], sr[c][7], sr[c][8], sr[c][9], sr[c][10], sr[c][11], sr[c][12], sr[c][13],
                                      sr[c][14], sr[c][15]);
                        }
                    }
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
                    for (int c = 0; c < C::DO / 32; ++c) {
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
                // this warp's 32 rows of P (and any rescaled O) are in TMEM (P: shared memory, made
                // visible to the tensor core's async proxy)
                tmem_st_wait();
                if constexpr (C::PSMEM) fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars.p_full[t]));
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue
            if (t < w.ntiles) {
                const bool have_o = nt > 0;
                if (have_o) {
                    ok = mbar_wait(smem_u32(&bars.o_final[t]), oc & 1, &abort_flag);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    ++oc;
                    tc_fence_after();
                }
                const long long grow = (long long)w.bh * p.Sq + row;
                const bool row_ok = row < p.Sq;
                if (X3 && p.splits == 1) {
                    // fp32 O = (O[:, :D] + O[:, D:]) / l
                    const float inv = l > 0.f ? 1.f / l : 0.f;
                    float *Og = static_cast<float *>(p.o) + o_at(p, w.b, w.hq, row);
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t oa[32], ob[32];
                        if (have_o) {
                            tmem_ld32(o_addr + c * 32, oa);
                            tmem_ld32(o_addr + D + c * 32, ob);
                            tmem_ld_wait();
                        }
                        if (row_ok) {
                            float4 *dst = reinterpret_cast<float4 *>(Og + c * 32);
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                float v[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    v[e] = have_o ? (__uint_as_float(oa[4 * k + e]) + __uint_as_float(ob[4 * k + e])) * inv
                                                  : 0.f;
                                dst[k] = make_float4(v[0], v[1], v[2], v[3]);
                            }
                        }
                    }
                    if (p.lse && row_ok) p.lse[grow] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
                } else if (p.splits == 1) {
                    const float inv = l > 0.f ? 1.f / l : 0.f;
                    __nv_bfloat16 *Og = static_cast<__nv_bfloat16 *>(p.o) + o_at(p, w.b, w.hq, row);
                    // 32-byte stores when every row starts on a 32-byte boundary
                    const bool o32 = ((reinterpret_cast<uintptr_t>(p.o) | (uintptr_t)(p.o_ss * 2) |
                                       (uintptr_t)(p.o_sh * 2) | (uintptr_t)(p.o_sb * 2)) & 31) == 0;
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
                            if (o32) {
                                st_global_v8(Og + c * 32, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
                                st_global_v8(Og + c * 32 + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
                            } else {
                                uint4 *dst = reinterpret_cast<uint4 *>(Og + c * 32);
#pragma unroll
                                for (int k = 0; k < 4; ++k)
                                    dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                            }
                        }
                    }
                    if (p.lse && row_ok) p.lse[grow] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
                } else if constexpr (MERGE) {
                    // O stays in TMEM for the merge at the end
                    fin_m = have_o ? m_ref : -INFINITY;
                    fin_l = have_o ? l : 0.f;
                    fin_have = have_o;
                } else {
                    float *A = p.part_acc + ((size_t)blockIdx.y * rows_total + grow) * D;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        if (have_o) {
                            tmem_ld32(o_addr + c * 32, o);
                            if constexpr (X3) {
                                uint32_t ob[32];
                                tmem_ld32(o_addr + D + c * 32, ob);
                                tmem_ld_wait();
#pragma unroll
                                for (int k = 0; k < 32; ++k)
                                    o[k] = __float_as_uint(__uint_as_float(o[k]) + __uint_as_float(ob[k]));
                            }
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
                if (have_o) {
                    // this warp's rows of O_t are in registers: the next item's first PV may
                    // overwrite them
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&bars.o_empty[t]));
                }
            }
        }
        if (!ok) raise_timeout(&abort_flag, p.status);
    }

    tc_fence_before();
    __syncwarp();
    __syncthreads();
    if constexpr (MERGE) {
        // ------------------------------------------------------------ split merge
        // Every MMA and copy of this CTA has completed.  Each softmax thread stages its row of O
        // (unnormalised fp32, 16-byte chunks XOR-swizzled by row) and its (m, l) at the start of
        // shared memory; after a cluster barrier, CTA k of the cluster merges rows [kR, kR + R)
        // of the item from all the cluster's stages with the log-sum-exp rule, and a second
        // barrier keeps each stage alive until every CTA has read it.  Every thread of every CTA
        // reaches both barriers.
        constexpr int CH = D / 4;   // 16-byte chunks per O row
        static_assert(2 * BM * (D * 4 + 16) + 1024 <= C::SMEM_BYTES, "merge stage does not fit");
        const uint32_t stage = sbase, ml_stage = sbase + 2 * BM * D * 4;
        if (warp >= 4) {
            const int t = (warp - 4) >> 2, rl = tid - 128;   // row of the item's 256
            const uint32_t o_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (t ? C::O_COL1 : C::O_COL0);
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(o_addr + c * 32, o);   // warp-collective: every lane loads
                tmem_ld_wait();
                if constexpr (X3) {
                    uint32_t ob[32];
                    tmem_ld32(o_addr + D + c * 32, ob);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) + __uint_as_float(ob[k]));
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int ch = c * 8 + q;
                    const uint32_t a = stage + (uint32_t)rl * (D * 4) + ((uint32_t)(ch ^ (rl & (CH - 1))) << 4);
                    if (fin_have) st_shared_v4(a, o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                    else st_shared_v4(a, 0u, 0u, 0u, 0u);
                }
            }
            st_shared_v4(ml_stage + (uint32_t)rl * 16, __float_as_uint(fin_m), __float_as_uint(fin_l), 0u, 0u);
        }
        __syncwarp();
        cluster_sync();
        const int ns = (int)gridDim.y;   // the cluster is the item's splits
        const int rank = (int)cluster_ctarank();
        const int R = (2 * BM + ns - 1) / ns;
        Item w;
        item_at(p, n_qb, n_items, 0, w);
        for (int task = tid; task < R * CH; task += NTHREADS) {
            const int rl = rank * R + task / CH, ch = task % CH;
            const int row = w.q0 + rl;
            if (rl >= 2 * BM || row >= p.Sq) break;   // tasks go by row
            float ms[8], ls[8], M = -INFINITY;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                ms[k] = -INFINITY;
                ls[k] = 0.f;
                if (k < ns) {
                    const uint32_t a = mapa_shared(ml_stage + (uint32_t)rl * 16, (uint32_t)k);
                    ms[k] = ld_shared_cluster_f32(a);
                    ls[k] = ld_shared_cluster_f32(a + 4);
                    M = fmaxf(M, ms[k]);
                }
            }
            float L = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            const uint32_t off = (uint32_t)rl * (D * 4) + ((uint32_t)(ch ^ (rl & (CH - 1))) << 4);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (k < ns && ms[k] != -INFINITY) {   // a split that saw keys of this row
                    const float wk = ex2_approx(ms[k] - M);
                    const float4 v = ld_shared_cluster_v4f(mapa_shared(stage + off, (uint32_t)k));
                    L += wk * ls[k];
                    acc.x += wk * v.x;
                    acc.y += wk * v.y;
                    acc.z += wk * v.z;
                    acc.w += wk * v.w;
                }
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            if constexpr (X3) {
                float *Og = static_cast<float *>(p.o) + o_at(p, w.b, w.hq, row) + ch * 4;
                *reinterpret_cast<float4 *>(Og) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            } else {
                __nv_bfloat16 *Og = static_cast<__nv_bfloat16 *>(p.o) + o_at(p, w.b, w.hq, row) + ch * 4;
                *reinterpret_cast<uint2 *>(Og) = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv),
                                                            pack_bf16x2(acc.z * inv, acc.w * inv));
            }
            if (ch == 0 && p.lse)
                p.lse[(long long)w.bh * p.Sq + row] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
        }
        __syncwarp();
        cluster_sync();
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------------- host side
// Q, K, V tile maps of a problem (5-D strided views); false when TMA cannot address them.
bool make_maps(const AttnProblem &p, CUtensorMap *mq, CUtensorMap *mk, CUtensorMap *mv) {
    return make_bf16_tile_map_strided(mq, p.q, p.D, p.Sq, p.Hq, p.B, p.q_ss, p.q_sh, p.q_sb, BM) &&
           make_bf16_tile_map_strided(mk, p.k, p.D, p.Sk, p.Hkv, p.B, p.k_ss, p.k_sh, p.k_sb, BN) &&
           make_bf16_tile_map_strided(mv, p.v, p.D, p.Sk, p.Hkv, p.B, p.v_ss, p.v_sh, p.v_sb, BN);
}

// x3 pre-pass: every float32 element of Q, K, V (any b/h/s strides) into its bf16 parts,
// h = bf16(x), m = bf16(x - h), l = bf16(x - h - m), written as contiguous [B, H, S, D] arrays
// Qh | Qm | Ql | Kh | Km | Kl | Vh | Vl (V keeps h and l = bf16(x - h), the "m" slot).
// blockIdx.y selects Q, K or V.
__device__ __forceinline__ uint32_t bf16_pair(float lo, float hi) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// One thread per four consecutive elements of a row (D = 64: 16 threads per row).
__global__ void __launch_bounds__(256) split_parts_kernel(const AttnProblem p, __nv_bfloat16 *ws) {
    const int which = blockIdx.y;
    const int H = which == 0 ? p.Hq : p.Hkv;
    const int S = which == 0 ? p.Sq : p.Sk;
    const long long nq = (long long)p.B * p.Hq * p.Sq * p.D, nk = (long long)p.B * p.Hkv * p.Sk * p.D;
    const long long n = which == 0 ? nq : nk;
    const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;   // group of 4 elements
    if (g * 4 >= n) return;
    const int per_row = p.D >> 2;
    const long long row = g / per_row;
    const int d = (int)(g - row * per_row) * 4;
    const long long sidx = row % S;
    const long long bh = row / S;
    const int h = (int)(bh % H), b = (int)(bh / H);
    const float *src;
    __nv_bfloat16 *out;
    if (which == 0) {
        src = static_cast<const float *>(p.q) + q_at(p, b, h, sidx) + d;
        out = ws;
    } else if (which == 1) {
        src = static_cast<const float *>(p.k) + k_at(p, b, h, sidx) + d;
        out = ws + 3 * nq;
    } else {
        src = static_cast<const float *>(p.v) + v_at(p, b, h, sidx) + d;
        out = ws + 3 * nq + 3 * nk;
    }
    float x[4];
    if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
        const float4 v = *reinterpret_cast<const float4 *>(src);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = src[e];
    }
    const long long i = row * p.D + d;   // element index in the contiguous part arrays
    // h = bf16(x), m = bf16(x - h), l = bf16(x - h - m)
    const uint32_t h01 = bf16_pair(x[0], x[1]), h23 = bf16_pair(x[2], x[3]);
    const float r[4] = {x[0] - bf16_lo(h01), x[1] - bf16_hi(h01), x[2] - bf16_lo(h23), x[3] - bf16_hi(h23)};
    const uint32_t m01 = bf16_pair(r[0], r[1]), m23 = bf16_pair(r[2], r[3]);
    *reinterpret_cast<uint2 *>(out + i) = make_uint2(h01, h23);
    *reinterpret_cast<uint2 *>(out + i + n) = make_uint2(m01, m23);
    if (which != 2) {
        const uint32_t l01 = bf16_pair(r[0] - bf16_lo(m01), r[1] - bf16_hi(m01));
        const uint32_t l23 = bf16_pair(r[2] - bf16_lo(m23), r[3] - bf16_hi(m23));
        *reinterpret_cast<uint2 *>(out + i + 2 * n) = make_uint2(l01, l23);
    }
}

template <int D, bool X3, bool MERGE>
cudaError_t set_smem_attr() {
    return set_max_dynamic_smem((const void *)attn_tc_kernel<D, X3, MERGE>, (int)TcCfg<D, X3>::SMEM_BYTES);
}

// Whether `clusters` clusters of `ns` CTAs of the merging kernel can all run at once (one wave;
// otherwise the splits are merged by the combine kernel).  Cached per device and cluster size.
template <int D, bool X3>
bool merge_fits(int clusters, int ns) {
    static std::mutex mu;
    static std::map<std::pair<int, int>, int> most;   // (device, ns) -> clusters resident at once
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lock(mu);
    auto it = most.find({dev, ns});
    if (it == most.end()) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)clusters, (unsigned)ns);
        cfg.blockDim = dim3(NTHREADS);
        cfg.dynamicSmemBytes = TcCfg<D, X3>::SMEM_BYTES;
        cudaLaunchAttribute a;
        a.id = cudaLaunchAttributeClusterDimension;
        a.val.clusterDim.x = 1;
        a.val.clusterDim.y = (unsigned)ns;
        a.val.clusterDim.z = 1;
        cfg.attrs = &a;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, attn_tc_kernel<D, X3, true>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        it = most.emplace(std::make_pair(dev, ns), n).first;
    }
    return it->second >= clusters;
}

// `merged`: the key splits were merged inside the kernel (no combine kernel needed).
template <int D, bool X3>
cudaError_t launch_t(const AttnProblem &p, const CUtensorMap (&m)[8], int sm_count, cudaStream_t s, bool &merged) {
    using C = TcCfg<D, X3>;
    merged = false;
    cudaError_t attr_err = set_smem_attr<D, X3, false>();
    if (attr_err != cudaSuccess) return attr_err;
    const int n_qb = (p.Sq + 2 * BM - 1) / (2 * BM);
    const long long items = (long long)n_qb * p.B * p.Hq;
    if (items >= (1LL << 31)) return cudaErrorInvalidValue;
    // one resident CTA per SM walks the items; fewer items than SMs: one CTA per item
    const int grid = (int)(items < sm_count ? items : (sm_count > 0 ? sm_count : 1));
    const dim3 g((unsigned)grid, (unsigned)p.splits);
    // key splits of few items: a cluster per item when its splits fit one (portable size 8)
    // and all clusters run at once
    if (p.splits > 1 && p.splits <= 8 && items < sm_count && set_smem_attr<D, X3, true>() == cudaSuccess &&
        merge_fits<D, X3>(grid, p.splits)) {
        cudaError_t e = launch_clustered(attn_tc_kernel<D, X3, true>, g, dim3(NTHREADS), C::SMEM_BYTES, s,
                                         dim3(1, (unsigned)p.splits, 1), X3, m[0], m[1], m[2], m[3], m[4], m[5], m[6],
                                         m[7], p, n_qb, (int)items);
        if (e != cudaSuccess) return e;
        merged = true;
    } else if (X3) {
        // dependent of the split pre-pass (see the producers' griddep_wait)
        cudaError_t e = launch_dependent(attn_tc_kernel<D, X3, false>, g, dim3(NTHREADS), C::SMEM_BYTES, s, m[0],
                                         m[1], m[2], m[3], m[4], m[5], m[6], m[7], p, n_qb, (int)items);
        if (e != cudaSuccess) return e;
    } else {
        attn_tc_kernel<D, X3, false><<<g, NTHREADS, C::SMEM_BYTES, s>>>(m[0], m[1], m[2], m[3], m[4], m[5], m[6], m[7],
                                                                         p, n_qb, (int)items);
    }
    count_launches(1);
    return cudaGetLastError();
}

// bf16 inputs: maps on the caller's tensors (the part maps are unused copies).
cudaError_t launch_bf16(const AttnProblem &p, int sm_count, cudaStream_t s, bool &merged) {
    CUtensorMap m[8];
    if (!make_maps(p, &m[0], &m[1], &m[2])) return cudaErrorInvalidValue;
    m[3] = m[6] = m[0];
    m[4] = m[7] = m[1];
    m[5] = m[2];
    return p.D == 64 ? launch_t<64, false>(p, m, sm_count, s, merged) : launch_t<128, false>(p, m, sm_count, s, merged);
}

// float32 inputs (D = 64): split Q, K, V into bf16 parts in the workspace, then run x3 mode on
// contiguous maps of the parts.  Map order: Qh Kh Vh Qm Km Ql Kl Vl.
cudaError_t launch_x3(const AttnProblem &p, int sm_count, cudaStream_t s, bool &merged) {
    const long long nq = (long long)p.B * p.Hq * p.Sq * p.D, nk = (long long)p.B * p.Hkv * p.Sk * p.D;
    __nv_bfloat16 *ws = static_cast<__nv_bfloat16 *>(p.x3_ws);
    if (!ws) return cudaErrorInvalidValue;
    const long long nmax = nq > nk ? nq : nk;
    const long long blocks = (nmax / 4 + 255) / 256;   // one thread per four elements (D % 4 == 0)
    if (blocks >= (1LL << 31)) return cudaErrorInvalidValue;
    split_parts_kernel<<<dim3((unsigned)blocks, 3), 256, 0, s>>>(p, ws);
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const __nv_bfloat16 *q[3] = {ws, ws + nq, ws + 2 * nq};
    const __nv_bfloat16 *k[3] = {ws + 3 * nq, ws + 3 * nq + nk, ws + 3 * nq + 2 * nk};
    const __nv_bfloat16 *v[2] = {ws + 3 * nq + 3 * nk, ws + 3 * nq + 4 * nk};
    const int D = p.D;
    const long long qs = (long long)p.Sq * D, ks = (long long)p.Sk * D;
    auto qmap = [&](CUtensorMap *m, const void *g) {
        return make_bf16_tile_map_strided(m, g, D, p.Sq, p.Hq, p.B, D, qs, qs * p.Hq, BM);
    };
    auto kmap = [&](CUtensorMap *m, const void *g) {
        return make_bf16_tile_map_strided(m, g, D, p.Sk, p.Hkv, p.B, D, ks, ks * p.Hkv, BN);
    };
    CUtensorMap m[8];
    if (!qmap(&m[0], q[0]) || !kmap(&m[1], k[0]) || !kmap(&m[2], v[0]) || !qmap(&m[3], q[1]) ||
        !kmap(&m[4], k[1]) || !qmap(&m[5], q[2]) || !kmap(&m[6], k[2]) || !kmap(&m[7], v[1]))
        return cudaErrorInvalidValue;
    return launch_t<64, true>(p, m, sm_count, s, merged);
}

// CTAs the kernel runs for a problem (before any key split).
long long tc_ctas(const AttnProblem &p) {
    return (long long)((p.Sq + 2 * BM - 1) / (2 * BM)) * p.B * p.Hq;
}



}  // namespace

bool attn_tc_supported(const AttnProblem &p, const void *Q, const void *K, const void *V, const void *O) {
    if (p.dtype == OSF_F32) {
        // x3 mode: the pre-pass reads Q, K, V with any strides; the epilogue stores 16-byte
        // pieces of each fp32 O row
        if (p.Sq < 2 || p.D != 64 || !aligned16(O) || ((p.o_ss | p.o_sh | p.o_sb) * 4) % 16 != 0) return false;
        return tc_ctas(p) < (1LL << 31) && tensor_map_encoder() != nullptr;
    }
    if (p.dtype != OSF_BF16 || p.Sq < 2 || (p.D != 64 && p.D != 128)) return false;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return false;
    // the epilogue stores 16-byte pieces of each O row
    if (((p.o_ss | p.o_sh | p.o_sb) * 2) % 16 != 0) return false;
    if (tc_ctas(p) >= (1LL << 31)) return false;
    return tensor_map_encoder() != nullptr &&
           tile_map_addressable(p.q, p.D, p.Sq, p.Hq, p.B, p.q_ss, p.q_sh, p.q_sb) &&
           tile_map_addressable(p.k, p.D, p.Sk, p.Hkv, p.B, p.k_ss, p.k_sh, p.k_sb) &&
           tile_map_addressable(p.v, p.D, p.Sk, p.Hkv, p.B, p.v_ss, p.v_sh, p.v_sb);
}

size_t attn_tc_extra_bytes(const AttnProblem &p) {
    if (p.dtype != OSF_F32) return 0;
    const size_t nq = (size_t)p.B * p.Hq * p.Sq * p.D, nk = (size_t)p.B * p.Hkv * p.Sk * p.D;
    return 2 * (3 * nq + 5 * nk);   // bf16 parts: three of Q and K, two of V
}

int attn_tc_pick_splits(const AttnProblem &p, int sm_count) {
    const long long ctas = tc_ctas(p);
    const int n_kt = (p.Sk + BN - 1) / BN;
    if (ctas >= sm_count || n_kt <= 1) return 1;
    // as many splits as keep every CTA in one wave (one CTA per SM): a second wave would cost
    // more than the extra split saves
    int want = (int)(sm_count / ctas);
    if (want > n_kt) want = n_kt;
    if (want < 2) return 1;
    const int tps = (n_kt + want - 1) / want;
    return (n_kt + tps - 1) / tps;   // no empty split
}

cudaError_t launch_attn_tc(const AttnProblem &p, int sm_count, cudaStream_t s) {
    bool merged = false;
    cudaError_t e = p.dtype == OSF_F32 ? launch_x3(p, sm_count, s, merged) : launch_bf16(p, sm_count, s, merged);
    if (e == cudaSuccess && p.splits > 1 && !merged) e = launch_attn_combine(p, s);
    return e;
}

}  // namespace osf
