// Split-K decode for bfloat16 K/V caches: one query row per head (Sq == 1), or a few (G * Sq
// <= 16: speculative decoding, where Sq draft tokens are checked against the cache at once).
//
// Decode reads the whole KV cache once per step and does only G = Hq/Hkv query rows of math
// per kv head, so it is bound by HBM bandwidth.  One CTA takes one (batch, kv head, key chunk):
// all G query heads that share the kv head ("从零开始写Qwen3（五-其一）...", "GQA") are computed
// together, so each K/V byte leaves HBM exactly once.  The key range of a kv head is cut into
// `splits` chunks so that there are several CTAs per SM; each chunk yields a partial online-softmax
// state (m, l, acc) and a second kernel merges the chunks with the log-sum-exp rule -- the
// boxed recurrence of "Softmax 算子的实现与优化", "Online Softmax", applied to whole partial
// states.  (The split is not on the pages; it is the plainest way to spread one row over the GPU.)
//
// Inside a CTA: two warps drive TMA loads of 64-key K and V tiles (one instruction per tile,
// 128-byte swizzle, so the ldmatrix reads below are bank-conflict free) into a 3-stage ring; four compute warps each
// take 16 keys of every tile and run the recurrence of "softmax_attention", "实现思路" with
// warp-level tensor-core MMAs (m16n8k16, bf16 in, fp32 accumulate): S = Q K^T with the G query
// rows padded to 16, then the S accumulator fragments are reused in registers as the P operand
// of O += P V.  At the end the four warps' states are merged through shared memory.  With
// Sq > 1 the 16 rows hold G heads x Sq query rows, each with its own causal key limit.
#include "decode.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.cuh"

namespace osf {
namespace {

using namespace ptx;

constexpr int KT = 64;                       // keys per tile
constexpr int NCW = 4;                       // compute warps, 16 keys of each tile apiece
constexpr int NTHREADS = (NCW + 2) * 32;     // + two TMA producer warps (K, V)
constexpr int STAGES = 3;
constexpr uint32_t BOXB = 64 * 128;          // one [64 keys x 64 bf16] box, 128-byte rows
constexpr int MAX_G = 16;                    // query rows per kv head: G * Sq (MMA rows)

template <int D>
struct DecCfg {
    static constexpr int BOXES = D / 64;
    static constexpr uint32_t TILE = BOXES * BOXB;          // one K or V tile
    static constexpr uint32_t K_OFF = 0, V_OFF = STAGES * TILE;
    static constexpr uint32_t SMEM = 2 * STAGES * TILE + 1024;
    static constexpr int NT = D / 8;                        // n8 tiles of an O row block
};

// Shared-memory address of the 16 bytes holding (key, d .. d+7) of a [64 x D] tile written by
// TMA with 128-byte swizzle: chunk (d % 64) / 8 of a 128-byte row sits at chunk ^ (row % 8).
__device__ __forceinline__ uint32_t swz(uint32_t tile, int key, int d) {
    return tile + (uint32_t)(d >> 6) * BOXB + (uint32_t)key * 128u + ((uint32_t)(((d & 63) >> 3) ^ (key & 7)) << 4);
}

__device__ __forceinline__ uint32_t ld_bf16x2(const __nv_bfloat16 *p) {
    return *reinterpret_cast<const uint32_t *>(p);
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 2)
decode_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
              const AttnProblem p, int tps) {
    using C = DecCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full[STAGES], empty[STAGES];
    __shared__ volatile int abort_flag;
    __shared__ float sm_m[NCW][MAX_G], sm_l[NCW][MAX_G];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int kvbh = blockIdx.x;                    // b * Hkv + kv head
    const int split = blockIdx.y;
    const int G = p.Hq / p.Hkv;
    const int b = kvbh / p.Hkv, kvh = kvbh % p.Hkv;
    const int n_kt_all = (p.Sk + KT - 1) / KT;
    const int t_begin = split * tps;
    const int t_end = min(n_kt_all, t_begin + tps);
    const int ntile = max(0, t_end - t_begin);
    const int key_end = min(p.Sk, t_end * KT);

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 2);   // the K and the V producer each arrive once
            mbar_init(smem_u32(&empty[s]), NCW);
        }
        abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();

    if (warp >= NCW) {
        // ================================================================ TMA producers
        // warp NCW streams K, warp NCW + 1 streams V; each 64-key tile is one TMA instruction.
        if (lane == 0 && ntile > 0) {
            const CUtensorMap *map = warp == NCW ? &mk : &mv;
            const uint32_t ring = sbase + (warp == NCW ? C::K_OFF : C::V_OFF);
            tma_prefetch_desc(map);
            int issued = 0;
            bool ok = true;
            for (int i = 0; i < ntile; ++i) {
                const int st = i % STAGES;
                ok = mbar_wait(smem_u32(&empty[st]), ((i / STAGES) & 1) ^ 1, &abort_flag);
                if (!ok) break;
                const uint32_t bar = smem_u32(&full[st]);
                mbar_expect_tx(bar, C::TILE);
                tma_load_5d(ring + st * C::TILE, map, bar, 0, (t_begin + i) * KT, 0, kvh, b);
                issued = i + 1;
            }
            if (!ok) {
                abort_flag = 1;
                atomicExch(p.status, kStatusTimeout);
                for (int i = max(0, issued - STAGES); i < issued; ++i)   // let issued copies land
                    mbar_wait(smem_u32(&full[i % STAGES]), (i / STAGES) & 1, nullptr, 20000000ull);
            }
        }
        // Every issued copy is consumed by the compute warps before they reuse the ring, so
        // the producer warps can leave now.
        return;
    }

    // ==================================================================== compute warps
    const int r0 = lane >> 2, r1 = r0 + 8, kc = (lane & 3) * 2;
    // row r of the 16-row tile is query row r % Sq of head kvh * G + r / Sq; rows past G * Sq
    // are zero padding
    const int R = G * p.Sq;
    const __nv_bfloat16 *Qb = static_cast<const __nv_bfloat16 *>(p.q);
    const __nv_bfloat16 *Q0 = Qb + q_at(p, b, kvh * G + r0 / p.Sq, r0 % p.Sq);
    const __nv_bfloat16 *Q1 = Qb + q_at(p, b, kvh * G + r1 / p.Sq, r1 % p.Sq);
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        qa[kk][0] = r0 < R ? ld_bf16x2(Q0 + kk * 16 + kc) : 0u;
        qa[kk][1] = r1 < R ? ld_bf16x2(Q1 + kk * 16 + kc) : 0u;
        qa[kk][2] = r0 < R ? ld_bf16x2(Q0 + kk * 16 + 8 + kc) : 0u;
        qa[kk][3] = r1 < R ? ld_bf16x2(Q1 + kk * 16 + 8 + kc) : 0u;
    }
    // last key each of this thread's two rows may see (exclusive bound)
    const int lim0 = p.causal ? min(key_end, r0 % p.Sq + p.causal_off + 1) : key_end;
    const int lim1 = p.causal ? min(key_end, r1 % p.Sq + p.causal_off + 1) : key_end;
    float o[C::NT][4];
#pragma unroll
    for (int j = 0; j < C::NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const float sl2 = p.scale_log2;
    const int mi = lane >> 3, rr = lane & 7;
    const int kb = warp * 16;                                     // this warp's keys in a tile
    const int key_k = kb + ((mi >> 1) << 3) + rr, dk = (mi & 1) << 3;   // ldmatrix rows for K
    const int key_v = kb + ((mi & 1) << 3) + rr, dv = (mi >> 1) << 3;   // ldmatrix.trans rows for V
    bool ok = true;
    for (int i = 0; i < ntile; ++i) {
        const int st = i % STAGES;
        ok = mbar_wait(smem_u32(&full[st]), (i / STAGES) & 1, &abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint32_t kt = sbase + C::K_OFF + st * C::TILE;
        const uint32_t vt = sbase + C::V_OFF + st * C::TILE;
        // S = Q K^T for this warp's 16 keys (two n8 tiles)
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(swz(kt, key_k, kk * 16 + dk), b0, b1, b2, b3);
            mma_m16n8k16_bf16(s[0], qa[kk], b0, b1);
            mma_m16n8k16_bf16(s[1], qa[kk], b2, b3);
        }
        // scale to base 2, mask keys past this chunk's end
        const int key_g = (t_begin + i) * KT + kb + kc;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool valid = key_g + n * 8 + (e & 1) < (e < 2 ? lim0 : lim1);
                s[n][e] = valid ? s[n][e] * sl2 : -INFINITY;
                if (e < 2) mx0 = fmaxf(mx0, s[n][e]); else mx1 = fmaxf(mx1, s[n][e]);
            }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        // online update: m' = max(m, m_tile), alpha = 2^(m - m'), l = l alpha + sum p
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float ref0 = mn0 == -INFINITY ? 0.f : mn0, ref1 = mn1 == -INFINITY ? 0.f : mn1;
        const float a0 = ex2_approx(m0 - ref0), a1 = ex2_approx(m1 - ref1);
        float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            s[n][0] = ex2_approx(s[n][0] - ref0);
            s[n][1] = ex2_approx(s[n][1] - ref0);
            s[n][2] = ex2_approx(s[n][2] - ref1);
            s[n][3] = ex2_approx(s[n][3] - ref1);
            rs0 += s[n][0] + s[n][1];
            rs1 += s[n][2] + s[n][3];
        }
        rs0 += __shfl_xor_sync(0xffffffffu, rs0, 1);
        rs0 += __shfl_xor_sync(0xffffffffu, rs0, 2);
        rs1 += __shfl_xor_sync(0xffffffffu, rs1, 1);
        rs1 += __shfl_xor_sync(0xffffffffu, rs1, 2);
        l0 = l0 * a0 + rs0;
        l1 = l1 * a1 + rs1;
        m0 = mn0;
        m1 = mn1;
#pragma unroll
        for (int j = 0; j < C::NT; ++j) {
            o[j][0] *= a0; o[j][1] *= a0;
            o[j][2] *= a1; o[j][3] *= a1;
        }
        // the S fragments of the two n8 tiles are exactly the A fragment of P (16 x 16)
        const uint32_t pa[4] = {pack_bf16x2(s[0][0], s[0][1]), pack_bf16x2(s[0][2], s[0][3]),
                                pack_bf16x2(s[1][0], s[1][1]), pack_bf16x2(s[1][2], s[1][3])};
#pragma unroll
        for (int j = 0; j < C::NT; j += 2) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(swz(vt, key_v, j * 8 + dv), b0, b1, b2, b3);
            mma_m16n8k16_bf16(o[j], pa, b0, b1);
            mma_m16n8k16_bf16(o[j + 1], pa, b2, b3);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
    }
    if (!ok) {
        abort_flag = 1;
        atomicExch(p.status, kStatusTimeout);
    }

    // ------------------------------------------------------- merge the four warps' states
    named_barrier(1, NCW * 32);            // every warp is done reading the K/V ring
    float *sO = reinterpret_cast<float *>(smem_raw + (sbase - smem_u32(smem_raw)));   // [NCW][16][D]
    if ((lane & 3) == 0) {
        sm_m[warp][r0] = m0; sm_l[warp][r0] = l0;
        sm_m[warp][r1] = m1; sm_l[warp][r1] = l1;
    }
    float *mine = sO + warp * MAX_G * D;
#pragma unroll
    for (int j = 0; j < C::NT; ++j) {
        *reinterpret_cast<float2 *>(mine + r0 * D + j * 8 + kc) = make_float2(o[j][0], o[j][1]);
        *reinterpret_cast<float2 *>(mine + r1 * D + j * 8 + kc) = make_float2(o[j][2], o[j][3]);
    }
    named_barrier(1, NCW * 32);
    const long long rows_total = (long long)p.B * p.Hq * p.Sq;
    for (int idx = tid; idx < R * D; idx += NCW * 32) {
        const int row = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) M = fmaxf(M, sm_m[w][row]);
        const float Mref = M == -INFINITY ? 0.f : M;
        float acc = 0.f, L = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
            const float wt = ex2_approx(sm_m[w][row] - Mref);
            acc += wt * sO[(w * MAX_G + row) * D + d];
            L += wt * sm_l[w][row];
        }
        const int hq = kvh * G + row / p.Sq, qi = row % p.Sq;
        const long long grow = ((long long)b * p.Hq + hq) * p.Sq + qi;
        if (p.splits == 1) {
            const float inv = L > 0.f ? 1.f / L : 0.f;
            static_cast<__nv_bfloat16 *>(p.o)[o_at(p, b, hq, qi) + d] = __float2bfloat16_rn(acc * inv);
            if (p.lse && d == 0) p.lse[grow] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
        } else {
            p.part_acc[((size_t)split * rows_total + grow) * D + d] = acc;
            if (d == 0) {
                p.part_m[(size_t)split * rows_total + grow] = M;
                p.part_l[(size_t)split * rows_total + grow] = L;
            }
        }
    }
}

// K and V tile maps of a problem (5-D strided views); false when TMA cannot address them.
bool make_maps(const AttnProblem &p, CUtensorMap *mk, CUtensorMap *mv) {
    return make_bf16_tile_map_strided(mk, p.k, p.D, p.Sk, p.Hkv, p.B, p.k_ss, p.k_sh, p.k_sb, KT) &&
           make_bf16_tile_map_strided(mv, p.v, p.D, p.Sk, p.Hkv, p.B, p.v_ss, p.v_sh, p.v_sb, KT);
}

template <int D>
cudaError_t launch_t(const AttnProblem &p, cudaStream_t s) {
    using C = DecCfg<D>;
    const cudaError_t attr_err = set_max_dynamic_smem((const void *)decode_kernel<D>, (int)C::SMEM);
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap mk, mv;
    if (!make_maps(p, &mk, &mv)) return cudaErrorInvalidValue;
    const int n_kt = (p.Sk + KT - 1) / KT;
    const int tps = (n_kt + p.splits - 1) / p.splits;
    dim3 grid((unsigned)(p.B * p.Hkv), (unsigned)p.splits);
    decode_kernel<D><<<grid, NTHREADS, C::SMEM, s>>>(mk, mv, p, tps);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

bool decode_supported(const AttnProblem &p, const void *Q, const void *K, const void *V, const void *O) {
    (void)O;
    if (p.dtype != OSF_BF16 || p.Sq < 1 || (p.D != 64 && p.D != 128)) return false;
    if ((long long)(p.Hq / p.Hkv) * p.Sq > MAX_G) return false;
    if (!aligned16(K) || !aligned16(V) || (reinterpret_cast<uintptr_t>(Q) & 3u) != 0) return false;
    if (((p.q_sb | p.q_sh | p.q_ss) & 1) != 0) return false;   // Q is read as bf16 pairs
    if ((long long)p.B * p.Hkv >= (1LL << 31)) return false;
    return tensor_map_encoder() != nullptr &&
           tile_map_addressable(p.k, p.D, p.Sk, p.Hkv, p.B, p.k_ss, p.k_sh, p.k_sb) &&
           tile_map_addressable(p.v, p.D, p.Sk, p.Hkv, p.B, p.v_ss, p.v_sh, p.v_sb);
}

int decode_pick_splits(const AttnProblem &p, int sm_count, int requested) {
    const int n_kt = (p.Sk + KT - 1) / KT;
    int s;
    if (requested > 0) {
        s = requested;
    } else {
        // about four waves of two CTAs per SM, so the last wave's imbalance stays small
        const long long items = (long long)p.B * p.Hkv;
        const long long slots = 2LL * sm_count;
        s = (int)((4 * slots + items / 2) / items);
        if (s < 1) s = 1;
    }
    if (s > n_kt) s = n_kt;
    if (s > 65535) s = 65535;
    const int tps = (n_kt + s - 1) / s;
    return (n_kt + tps - 1) / tps;   // no empty chunk
}

cudaError_t launch_decode(const AttnProblem &p, cudaStream_t s) {
    cudaError_t e = p.D == 64 ? launch_t<64>(p, s) : launch_t<128>(p, s);
    if (e == cudaSuccess && p.splits > 1) e = launch_attn_combine(p, s);
    return e;
}

}  // namespace osf
