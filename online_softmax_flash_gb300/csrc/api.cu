// C ABI of libosf (declared in include/osf.h): argument checks, kernel choice, workspace
// sizing and the device status word.  Every entry point validates on the host, then enqueues
// kernels on the caller's stream and returns; nothing here allocates device memory.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <map>
#include <utility>

#include "osf_internal.cuh"
#include "softmax_ex.cuh"
#include "attn_bwd.cuh"
#include "selftest.cuh"
#include "attn_tc.cuh"
#include "decode.cuh"

namespace osf {

static std::atomic<unsigned long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

cudaError_t set_max_dynamic_smem(const void *kernel, int bytes) {
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, int> done;   // (device, kernel) -> limit set
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(dev, kernel);
    auto it = done.find(key);
    if (it != done.end() && it->second >= bytes) return cudaSuccess;   // the limit is only raised
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[key] = bytes;
    return e;
}

namespace {

constexpr int kMaxDevices = 64;

// One status word per device; kernels with bounded waits write kStatusTimeout here.
__device__ int g_status_word;

struct DeviceInfo {
    int sm_count = 0;
    int *status = nullptr;   // device address of g_status_word
    std::atomic<bool> ready{false};   // set (release) after the fields above
};
DeviceInfo g_dev[kMaxDevices];

int current_device(int *dev) {
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return OSF_ERR_CUDA;
    return OSF_OK;
}

// Per-device set-up (SM count, status word address), once per device under a lock; later
// calls see the published fields through the acquire load of `ready`.
int device_info(DeviceInfo **out) {
    static std::mutex mu;
    int dev;
    if (current_device(&dev) != OSF_OK) return OSF_ERR_CUDA;
    DeviceInfo &d = g_dev[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(mu);
        if (!d.ready.load(std::memory_order_relaxed)) {
            int sms = 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return OSF_ERR_CUDA;
            void *addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return OSF_ERR_CUDA;
            d.sm_count = sms;
            d.status = static_cast<int *>(addr);
            d.ready.store(true, std::memory_order_release);
        }
    }
    *out = &d;
    return OSF_OK;
}

}  // namespace

int device_sm_count(int *sms) {
    DeviceInfo *d;
    const int st = device_info(&d);
    if (st != OSF_OK) return st;
    *sms = d->sm_count;
    return OSF_OK;
}

namespace {

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

size_t elem_size(int dtype) { return dtype == OSF_F32 ? 4 : 2; }

int launch_status(cudaError_t e) { return e == cudaSuccess ? OSF_OK : OSF_ERR_CUDA; }

// Bytes spanned by a strided [n0, n1, n2, D] tensor (strides s0..s2 in elements, d contiguous).
size_t span_bytes(long long n0, long long n1, long long n2, long long D, long long s0, long long s1,
                  long long s2, size_t es) {
    return (size_t)((n0 - 1) * s0 + (n1 - 1) * s1 + (n2 - 1) * s2 + D) * es;
}

// True when no two rows of a [n0, n1, n2, D] tensor with these strides share an element: the
// dimensions, sorted by stride, each step over the whole block of the smaller ones.
bool rows_disjoint(long long n0, long long n1, long long n2, long long D, long long s0, long long s1,
                   long long s2) {
    long long st[3] = {s0, s1, s2}, n[3] = {n0, n1, n2};
    for (int i = 0; i < 3; ++i)
        for (int j = i + 1; j < 3; ++j)
            if (st[j] < st[i]) {
                long long t = st[i]; st[i] = st[j]; st[j] = t;
                t = n[i]; n[i] = n[j]; n[j] = t;
            }
    long long block = D;
    for (int i = 0; i < 3; ++i) {
        if (n[i] <= 1) continue;
        if (st[i] < block) return false;
        block = st[i] * (n[i] - 1) + block;
    }
    return true;
}

// Shared validation of the GQA problem; fills `p` (without workspace pointers).  `strides`:
// NULL (contiguous [B, H, S, D]) or Q, K, V, O x (b, h, s) element strides.  `mask`: an
// osf_mask; the original entry point passes TOP_LEFT for causal and keeps its Sq == Sk rule.
int check_gqa_ex(const void *Q, const void *K, const void *V, void *O, int dtype, int B, int Hq,
                 int Hkv, int Sq, int Sk, int D, const long long *strides, int mask, float scale,
                 float *lse, AttnProblem &p, bool &empty) {
    empty = false;
    if (dtype != OSF_F32 && dtype != OSF_BF16) return OSF_ERR_INVALID;
    if (B < 0 || Hq < 0 || Hkv < 0 || Sq < 0 || Sk < 0 || D <= 0) return OSF_ERR_INVALID;
    if (Hq == 0 || Hkv == 0 || Hq % Hkv != 0) return OSF_ERR_INVALID;
    if (!(scale == scale)) return OSF_ERR_INVALID;  // NaN
    if (mask != OSF_MASK_NONE && mask != OSF_MASK_TOP_LEFT && mask != OSF_MASK_BOTTOM_RIGHT)
        return OSF_ERR_INVALID;
    long long st[12];
    if (strides) {
        for (int i = 0; i < 12; ++i) {
            if (strides[i] < 0) return OSF_ERR_INVALID;
            st[i] = strides[i];
        }
    } else {
        const long long q[3] = {(long long)Hq * Sq * D, (long long)Sq * D, D};
        const long long kv[3] = {(long long)Hkv * Sk * D, (long long)Sk * D, D};
        for (int i = 0; i < 3; ++i) {
            st[i] = q[i];
            st[3 + i] = kv[i];
            st[6 + i] = kv[i];
            st[9 + i] = q[i];
        }
    }
    if (D > 256) return OSF_ERR_UNSUPPORTED;
    if (B == 0 || Sq == 0 || Sk == 0) { empty = true; return OSF_OK; }
    // per-head element counts index with 32-bit row numbers inside kernels
    if ((long long)Sq * D >= (1LL << 31) || (long long)Sk * D >= (1LL << 31) ||
        (long long)B * Hq >= (1LL << 31) || (long long)B * Hq * Sq >= (1LL << 40))
        return OSF_ERR_UNSUPPORTED;
    for (int i = 0; i < 12; ++i)
        if (st[i] >= (1LL << 40)) return OSF_ERR_UNSUPPORTED;
    if (!Q || !K || !V || !O) return OSF_ERR_INVALID;
    const size_t es = elem_size(dtype);
    const size_t nq = span_bytes(B, Hq, Sq, D, st[0], st[1], st[2], es);
    const size_t nk = span_bytes(B, Hkv, Sk, D, st[3], st[4], st[5], es);
    const size_t nv = span_bytes(B, Hkv, Sk, D, st[6], st[7], st[8], es);
    const size_t no = span_bytes(B, Hq, Sq, D, st[9], st[10], st[11], es);
    if (!rows_disjoint(B, Hq, Sq, D, st[9], st[10], st[11])) return OSF_ERR_INVALID;
    if (overlaps(O, no, Q, nq) || overlaps(O, no, K, nk) || overlaps(O, no, V, nv))
        return OSF_ERR_INVALID;
    if (lse) {
        const size_t nl = (size_t)B * Hq * Sq * sizeof(float);
        if (overlaps(lse, nl, O, no) || overlaps(lse, nl, Q, nq) || overlaps(lse, nl, K, nk) ||
            overlaps(lse, nl, V, nv))
            return OSF_ERR_INVALID;
    }
    p = AttnProblem{};
    p.q = Q; p.k = K; p.v = V; p.o = O; p.lse = lse;
    p.dtype = dtype;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sq = Sq; p.Sk = Sk; p.D = D;
    p.q_sb = st[0]; p.q_sh = st[1]; p.q_ss = st[2];
    p.k_sb = st[3]; p.k_sh = st[4]; p.k_ss = st[5];
    p.v_sb = st[6]; p.v_sh = st[7]; p.v_ss = st[8];
    p.o_sb = st[9]; p.o_sh = st[10]; p.o_ss = st[11];
    // key j is visible to row i iff j <= i + off; a mask that hides nothing is dropped
    const long long off = mask == OSF_MASK_BOTTOM_RIGHT ? (long long)Sk - Sq : 0;
    const bool masks = (mask == OSF_MASK_TOP_LEFT && Sq > 1) || mask == OSF_MASK_BOTTOM_RIGHT;
    p.causal = (masks && off < (long long)Sk - 1) ? 1 : 0;
    p.causal_off = p.causal ? (int)off : 0;
    const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
    p.scale_log2 = sc * kLog2e;
    p.splits = 1;
    return OSF_OK;
}

int check_gqa(const void *Q, const void *K, const void *V, void *O, int dtype, int B, int Hq,
              int Hkv, int Sq, int Sk, int D, int causal, float scale, float *lse,
              AttnProblem &p, bool &empty) {
    // the original entry point: contiguous tensors, causal only with Sq == Sk (or Sq == 1)
    if (causal && Sq > 1 && Sq != Sk) return OSF_ERR_INVALID;
    return check_gqa_ex(Q, K, V, O, dtype, B, Hq, Hkv, Sq, Sk, D, nullptr,
                        causal ? OSF_MASK_TOP_LEFT : OSF_MASK_NONE, scale, lse, p, empty);
}

// Workspace layout for split partial states: acc | m | l (floats), 256-byte aligned pieces.
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t partial_bytes(int splits, long long rows, int D) {
    if (splits <= 1) return 0;
    return align256((size_t)splits * rows * D * 4) + 2 * align256((size_t)splits * rows * 4);
}

void carve_partials(AttnProblem &p, void *ws, long long rows) {
    char *base = static_cast<char *>(ws);
    p.part_acc = reinterpret_cast<float *>(base);
    base += align256((size_t)p.splits * rows * p.D * 4);
    p.part_m = reinterpret_cast<float *>(base);
    base += align256((size_t)p.splits * rows * 4);
    p.part_l = reinterpret_cast<float *>(base);
}

// Which kernel runs a (validated, non-empty) problem.
enum class Path { Simt, TensorCore, Decode };

Path choose_path(const AttnProblem &p, const void *Q, const void *K, const void *V, const void *O) {
    // one or a few query rows per head (G * Sq <= 16): the HBM-bound decode kernel, which reads
    // each K/V byte once for all the query heads of its kv head
    if (p.dtype == OSF_BF16 && decode_supported(p, Q, K, V, O)) return Path::Decode;
    // bf16, and fp32 with D = 64 (as bf16 high / low parts)
    if (p.Sq > 1 && attn_tc_supported(p, Q, K, V, O)) return Path::TensorCore;
    return Path::Simt;
}

int plan_splits(const AttnProblem &p, Path path, int sm_count, int requested) {
    if (path == Path::TensorCore) return attn_tc_pick_splits(p, sm_count);
    if (path == Path::Decode) return decode_pick_splits(p, sm_count, requested);
    if (requested > 0) {
        const int n_kt = (p.Sk + 63) / 64;
        return requested < n_kt ? requested : n_kt;
    }
    return attn_simt_pick_splits(p, sm_count);
}

size_t path_workspace(const AttnProblem &p, Path path, int splits) {
    // every path keeps split partial states in the same layout; the tensor-core path keeps the
    // fp32 operands' bf16 parts after them
    const size_t part = partial_bytes(splits, (long long)p.B * p.Hq * p.Sq, p.D);
    return path == Path::TensorCore ? part + align256(attn_tc_extra_bytes(p)) : part;
}

int run_gqa(AttnProblem &p, Path path, void *workspace, size_t workspace_bytes, int splits,
            DeviceInfo *dev, cudaStream_t s) {
    p.splits = splits;
    p.status = dev->status;
    const size_t need = path_workspace(p, path, splits);
    if (need > 0 && (!workspace || workspace_bytes < need)) return OSF_ERR_WORKSPACE;
    const long long rows = (long long)p.B * p.Hq * p.Sq;
    switch (path) {
        case Path::TensorCore:
            if (splits > 1) carve_partials(p, workspace, rows);
            p.x3_ws = attn_tc_extra_bytes(p) > 0
                          ? static_cast<void *>(static_cast<char *>(workspace) + partial_bytes(splits, rows, p.D))
                          : nullptr;
            return launch_status(launch_attn_tc(p, dev->sm_count, s));
        case Path::Decode:
            if (splits > 1) carve_partials(p, workspace, rows);
            return launch_status(launch_decode(p, s));
        case Path::Simt:
        default: {
            if (splits > 1) carve_partials(p, workspace, rows);
            cudaError_t e = launch_attn_simt(p, s);
            if (e == cudaSuccess && splits > 1) e = launch_attn_combine(p, s);
            return launch_status(e);
        }
    }
}

// ------------------------------------------------------------- host buffers in and out
// osf_attn_fwd_gqa_host splits the problem into chunks of whole (batch, kv head) units: unit u =
// b * Hkv + g owns the G query heads g*G .. g*G+G-1 of batch b and kv head g, so a run of
// consecutive units is one contiguous range of Q, K, V and O, and a chunk of n units is itself a
// GQA problem with B = n, Hq = G, Hkv = 1.  Each chunk's copies in, attention and copy out are
// enqueued on three streams (copy-in, the caller's, copy-out) linked by events, so the copies of
// one chunk overlap the attention of another and the two copy directions overlap each other.
constexpr int kHostChunks = 8;

struct HostUnits {
    long long units = 0;      // B * Hkv
    int chunks = 0;           // number of chunks
    long long per = 0;        // units per chunk (the last may have fewer)
    size_t q_unit = 0, kv_unit = 0;   // bytes of one unit's Q (and O) and of its K (and V)
};

HostUnits host_units(int dtype, int B, int Hq, int Hkv, int Sq, int Sk, int D) {
    HostUnits h;
    const int G = Hq / Hkv;
    h.units = (long long)B * Hkv;
    h.chunks = (int)std::min<long long>(h.units, kHostChunks);
    h.per = (h.units + h.chunks - 1) / h.chunks;
    h.chunks = (int)((h.units + h.per - 1) / h.per);
    h.q_unit = (size_t)G * Sq * D * elem_size(dtype);
    h.kv_unit = (size_t)Sk * D * elem_size(dtype);
    return h;
}

// Device-buffer layout: Q | K | V | O | chunk workspace, each piece 256-byte aligned.
struct HostLayout {
    size_t q = 0, k = 0, v = 0, o = 0, ws = 0, ws_bytes = 0, total = 0;
};

int host_layout(int dtype, int B, int Hq, int Hkv, int Sq, int Sk, int D, HostLayout &L) {
    const HostUnits h = host_units(dtype, B, Hq, Hkv, Sq, Sk, D);
    const size_t qb = h.q_unit * h.units, kvb = h.kv_unit * h.units;
    // workspace: the larger need of a full chunk and of the last (smaller) one
    size_t ws = 0;
    const long long sizes[2] = {h.per, h.units - (long long)(h.chunks - 1) * h.per};
    for (long long n : sizes) {
        size_t w = 0;
        const int st = osf_attn_workspace_bytes(dtype, (int)n, Hq / Hkv, 1, Sq, Sk, D, &w);
        if (st != OSF_OK) return st;
        ws = std::max(ws, w);
    }
    L.q = 0;
    L.k = align256(qb);
    L.v = L.k + align256(kvb);
    L.o = L.v + align256(kvb);
    L.ws = L.o + align256(qb);
    L.ws_bytes = ws;
    L.total = L.ws + align256(ws);
    return OSF_OK;
}

// Per-device copy streams and events, created on the first host-buffer call on the device.
struct HostStreams {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t landed[kHostChunks] = {}, computed[kHostChunks] = {};
    bool ready = false;
};
HostStreams g_host[kMaxDevices];
std::mutex g_host_mutex;   // held while a call enqueues its work (the events are shared)

int host_streams(HostStreams **out) {
    int dev;
    if (current_device(&dev) != OSF_OK) return OSF_ERR_CUDA;
    HostStreams &h = g_host[dev];
    if (!h.ready) {
        bool ok = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h.start, cudaEventDisableTiming) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h.done, cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; ok && i < kHostChunks; ++i)
            ok = cudaEventCreateWithFlags(&h.landed[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&h.computed[i], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            // release what was created, so a later call starts over cleanly
            if (h.in) cudaStreamDestroy(h.in);
            if (h.out) cudaStreamDestroy(h.out);
            cudaEvent_t *evs[] = {&h.start, &h.done};
            for (cudaEvent_t *e : evs)
                if (*e) cudaEventDestroy(*e);
            for (int i = 0; i < kHostChunks; ++i) {
                if (h.landed[i]) cudaEventDestroy(h.landed[i]);
                if (h.computed[i]) cudaEventDestroy(h.computed[i]);
            }
            h = HostStreams();
            return OSF_ERR_CUDA;
        }
        h.ready = true;
    }
    *out = &h;
    return OSF_OK;
}

}  // namespace
}  // namespace osf

using namespace osf;

extern "C" {

const char *osf_status_string(int status) {
    switch (status) {
        case OSF_OK: return "OSF_OK";
        case OSF_ERR_INVALID: return "OSF_ERR_INVALID: invalid argument";
        case OSF_ERR_UNSUPPORTED: return "OSF_ERR_UNSUPPORTED: unsupported size or type";
        case OSF_ERR_CUDA: return "OSF_ERR_CUDA: CUDA runtime error";
        case OSF_ERR_TIMEOUT: return "OSF_ERR_TIMEOUT: a bounded device wait expired";
        case OSF_ERR_WORKSPACE: return "OSF_ERR_WORKSPACE: workspace missing or too small";
        default: return "unknown osf status";
    }
}

int osf_version(void) { return 100; }

unsigned long long osf_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int osf_sm_count(void) {
    DeviceInfo *d;
    return device_info(&d) == OSF_OK ? d->sm_count : 0;
}

int osf_attn_fwd(const float *Q, const float *K, const float *V, float *out, int M, int N, int d,
                 osf_stream stream) {
    if (M < 0 || N < 0 || d <= 0) return OSF_ERR_INVALID;
    if (M == 0 || N == 0) return OSF_OK;
    AttnProblem p;
    bool empty;
    int st = check_gqa(Q, K, V, out, OSF_F32, 1, 1, 1, M, N, d, 0, 0.f, nullptr, p, empty);
    if (st != OSF_OK || empty) return st;
    DeviceInfo *dev;
    if (device_info(&dev) != OSF_OK) return OSF_ERR_CUDA;
    // no workspace in this signature: run unsplit
    return run_gqa(p, Path::Simt, nullptr, 0, 1, dev, (cudaStream_t)stream);
}

int osf_attn_workspace_bytes(int dtype, int B, int Hq, int Hkv, int Sq, int Sk, int D,
                             size_t *bytes) {
    if (!bytes) return OSF_ERR_INVALID;
    *bytes = 0;
    AttnProblem p;
    bool empty;
    // pointers are not known here: validate sizes with placeholder addresses
    const void *ph = reinterpret_cast<const void *>(uintptr_t(1) << 40);
    int st = check_gqa(ph, ph, ph, reinterpret_cast<void *>(uintptr_t(1) << 44), dtype, B, Hq, Hkv,
                       Sq, Sk, D, 0, 0.f, nullptr, p, empty);
    if (st != OSF_OK || empty) return st;
    DeviceInfo *dev;
    if (device_info(&dev) != OSF_OK) return OSF_ERR_CUDA;
    // the larger of the possible paths' needs (alignment decides the path at call time)
    size_t need = partial_bytes(attn_simt_pick_splits(p, dev->sm_count), (long long)B * Hq * Sq, D);
    if (Sq > 1 && ((dtype == OSF_BF16 && (D == 64 || D == 128)) || (dtype == OSF_F32 && D == 64))) {
        const size_t tc = path_workspace(p, Path::TensorCore, attn_tc_pick_splits(p, dev->sm_count));
        if (tc > need) need = tc;
    }
    if (dtype == OSF_BF16 && (long long)(Hq / Hkv) * Sq <= 16) {
        const size_t dn = partial_bytes(decode_pick_splits(p, dev->sm_count, 0), (long long)B * Hq * Sq, D);
        if (dn > need) need = dn;
    }
    *bytes = need;
    return OSF_OK;
}

int osf_attn_fwd_gqa(const void *Q, const void *K, const void *V, void *O, int dtype, int B,
                     int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale, float *lse,
                     void *workspace, size_t workspace_bytes, osf_stream stream) {
    AttnProblem p;
    bool empty;
    int st = check_gqa(Q, K, V, O, dtype, B, Hq, Hkv, Sq, Sk, D, causal, scale, lse, p, empty);
    if (st != OSF_OK || empty) return st;
    DeviceInfo *dev;
    if (device_info(&dev) != OSF_OK) return OSF_ERR_CUDA;
    const Path path = choose_path(p, Q, K, V, O);
    const int splits = plan_splits(p, path, dev->sm_count, 0);
    return run_gqa(p, path, workspace, workspace_bytes, splits, dev, (cudaStream_t)stream);
}

int osf_attn_fwd_gqa_ex(const void *Q, const void *K, const void *V, void *O, int dtype, int B,
                        int Hq, int Hkv, int Sq, int Sk, int D, const long long *strides, int mask,
                        float scale, float *lse, void *workspace, size_t workspace_bytes,
                        osf_stream stream) {
    AttnProblem p;
    bool empty;
    int st = check_gqa_ex(Q, K, V, O, dtype, B, Hq, Hkv, Sq, Sk, D, strides, mask, scale, lse, p, empty);
    if (st != OSF_OK || empty) return st;
    DeviceInfo *dev;
    if (device_info(&dev) != OSF_OK) return OSF_ERR_CUDA;
    const Path path = choose_path(p, Q, K, V, O);
    const int splits = plan_splits(p, path, dev->sm_count, 0);
    return run_gqa(p, path, workspace, workspace_bytes, splits, dev, (cudaStream_t)stream);
}

int osf_attn_host_buffer_bytes(int dtype, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal,
                               size_t *bytes) {
    if (!bytes) return OSF_ERR_INVALID;
    *bytes = 0;
    AttnProblem p;
    bool empty;
    const void *ph = reinterpret_cast<const void *>(uintptr_t(1) << 40);
    int st = check_gqa(ph, ph, ph, reinterpret_cast<void *>(uintptr_t(1) << 44), dtype, B, Hq, Hkv,
                       Sq, Sk, D, causal, 0.f, nullptr, p, empty);
    if (st != OSF_OK || empty) return st;
    HostLayout L;
    st = host_layout(dtype, B, Hq, Hkv, Sq, Sk, D, L);
    if (st != OSF_OK) return st;
    *bytes = L.total;
    return OSF_OK;
}

int osf_attn_fwd_gqa_host(const void *Q, const void *K, const void *V, void *O, int dtype, int B,
                          int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                          void *device_buffer, size_t device_buffer_bytes, osf_stream stream) {
    AttnProblem p;
    bool empty;
    // validate the sizes and the host pointers as a whole problem
    int st = check_gqa(Q, K, V, O, dtype, B, Hq, Hkv, Sq, Sk, D, causal, scale, nullptr, p, empty);
    if (st != OSF_OK || empty) return st;
    if (!device_buffer) return OSF_ERR_WORKSPACE;
    HostLayout L;
    st = host_layout(dtype, B, Hq, Hkv, Sq, Sk, D, L);
    if (st != OSF_OK) return st;
    if (device_buffer_bytes < L.total) return OSF_ERR_WORKSPACE;
    DeviceInfo *dev;
    if (device_info(&dev) != OSF_OK) return OSF_ERR_CUDA;
    HostStreams *hs;
    std::lock_guard<std::mutex> lock(g_host_mutex);
    if (host_streams(&hs) != OSF_OK) return OSF_ERR_CUDA;
    const cudaStream_t s = (cudaStream_t)stream;
    const HostUnits h = host_units(dtype, B, Hq, Hkv, Sq, Sk, D);
    char *base = static_cast<char *>(device_buffer);
    char *dq = base + L.q, *dk = base + L.k, *dv = base + L.v, *dout = base + L.o;
    void *ws = L.ws_bytes > 0 ? base + L.ws : nullptr;
    const char *hq = static_cast<const char *>(Q), *hk = static_cast<const char *>(K),
               *hv = static_cast<const char *>(V);
    char *ho = static_cast<char *>(O);
    const int G = Hq / Hkv;
    // everything earlier on the caller's stream (a previous call using this buffer) comes first
    if (cudaEventRecord(hs->start, s) != cudaSuccess || cudaStreamWaitEvent(hs->in, hs->start, 0) != cudaSuccess)
        return OSF_ERR_CUDA;
    // On an error after this point some chunks may already be queued on the copy streams: the
    // caller's stream is made to wait for both of them (best effort) so that work it enqueues
    // next still runs after them, and the error is returned.  O is then undefined.
    auto fail = [&](int code) {
        if (cudaEventRecord(hs->start, hs->in) == cudaSuccess) cudaStreamWaitEvent(s, hs->start, 0);
        if (cudaEventRecord(hs->done, hs->out) == cudaSuccess) cudaStreamWaitEvent(s, hs->done, 0);
        cudaGetLastError();
        return code;
    };
    for (int c = 0; c < h.chunks; ++c) {
        const long long u0 = (long long)c * h.per;
        const long long n = std::min<long long>(h.per, h.units - u0);
        const size_t qo = (size_t)u0 * h.q_unit, ko = (size_t)u0 * h.kv_unit;
        const size_t qn = (size_t)n * h.q_unit, kn = (size_t)n * h.kv_unit;
        if (cudaMemcpyAsync(dq + qo, hq + qo, qn, cudaMemcpyHostToDevice, hs->in) != cudaSuccess ||
            cudaMemcpyAsync(dk + ko, hk + ko, kn, cudaMemcpyHostToDevice, hs->in) != cudaSuccess ||
            cudaMemcpyAsync(dv + ko, hv + ko, kn, cudaMemcpyHostToDevice, hs->in) != cudaSuccess ||
            cudaEventRecord(hs->landed[c], hs->in) != cudaSuccess || cudaStreamWaitEvent(s, hs->landed[c], 0) != cudaSuccess)
            return fail(OSF_ERR_CUDA);
        // the chunk as its own problem: B = n units, Hq = G, Hkv = 1
        AttnProblem pc;
        bool ec;
        st = check_gqa(dq + qo, dk + ko, dv + ko, dout + qo, dtype, (int)n, G, 1, Sq, Sk, D, causal, scale, nullptr,
                       pc, ec);
        if (st != OSF_OK) return fail(st);
        const Path path = choose_path(pc, dq + qo, dk + ko, dv + ko, dout + qo);
        st = run_gqa(pc, path, ws, L.ws_bytes, plan_splits(pc, path, dev->sm_count, 0), dev, s);
        if (st != OSF_OK) return fail(st);
        if (cudaEventRecord(hs->computed[c], s) != cudaSuccess || cudaStreamWaitEvent(hs->out, hs->computed[c], 0) != cudaSuccess ||
            cudaMemcpyAsync(ho + qo, dout + qo, qn, cudaMemcpyDeviceToHost, hs->out) != cudaSuccess)
            return fail(OSF_ERR_CUDA);
    }
    // the caller's stream continues once O has reached the host
    if (cudaEventRecord(hs->done, hs->out) != cudaSuccess || cudaStreamWaitEvent(s, hs->done, 0) != cudaSuccess)
        return fail(OSF_ERR_CUDA);
    return OSF_OK;
}

int osf_attn_decode_workspace_bytes(int dtype, int B, int Hq, int Hkv, int Sk, int D,
                                    int num_splits, size_t *bytes) {
    if (!bytes) return OSF_ERR_INVALID;
    *bytes = 0;
    AttnProblem p;
    bool empty;
    const void *ph = reinterpret_cast<const void *>(uintptr_t(1) << 40);
    int st = check_gqa(ph, ph, ph, reinterpret_cast<void *>(uintptr_t(1) << 44), dtype, B, Hq, Hkv,
                       1, Sk, D, 0, 0.f, nullptr, p, empty);
    if (st != OSF_OK || empty) return st;
    DeviceInfo *dev;
    if (device_info(&dev) != OSF_OK) return OSF_ERR_CUDA;
    size_t need = partial_bytes(plan_splits(p, Path::Simt, dev->sm_count, num_splits), (long long)B * Hq, D);
    if (dtype == OSF_BF16) {
        const size_t dn = partial_bytes(decode_pick_splits(p, dev->sm_count, num_splits), (long long)B * Hq, D);
        if (dn > need) need = dn;
    }
    *bytes = need;
    return OSF_OK;
}

int osf_attn_decode_gqa(const void *Q, const void *K, const void *V, void *O, int dtype, int B,
                        int Hq, int Hkv, int Sk, int D, float scale, float *lse, int num_splits,
                        void *workspace, size_t workspace_bytes, osf_stream stream) {
    AttnProblem p;
    bool empty;
    int st = check_gqa(Q, K, V, O, dtype, B, Hq, Hkv, 1, Sk, D, 0, scale, lse, p, empty);
    if (st != OSF_OK || empty) return st;
    DeviceInfo *dev;
    if (device_info(&dev) != OSF_OK) return OSF_ERR_CUDA;
    const Path path = (dtype == OSF_BF16 && decode_supported(p, Q, K, V, O)) ? Path::Decode : Path::Simt;
    const int splits = plan_splits(p, path, dev->sm_count, num_splits);
    return run_gqa(p, path, workspace, workspace_bytes, splits, dev, (cudaStream_t)stream);
}

int osf_softmax_workspace_bytes(long long rows, long long T, size_t *bytes) {
    if (!bytes) return OSF_ERR_INVALID;
    *bytes = 0;
    if (rows < 0 || T < 0) return OSF_ERR_INVALID;
    if (rows == 0 || T == 0) return OSF_OK;
    if (rows > 65535 && T > 32768) return OSF_ERR_UNSUPPORTED;
    DeviceInfo *dev;
    if (device_info(&dev) != OSF_OK) return OSF_ERR_CUDA;
    *bytes = softmax_workspace_floats(rows, T, dev->sm_count) * sizeof(float);
    return OSF_OK;
}

int osf_softmax_rows(const float *x, float *z, long long rows, long long T, void *workspace,
                     size_t workspace_bytes, osf_stream stream) {
    if (rows < 0 || T < 0) return OSF_ERR_INVALID;
    if (rows == 0 || T == 0) return OSF_OK;
    if (!x || !z) return OSF_ERR_INVALID;
    if (rows > (1LL << 31) - 1 || (rows > 65535 && T > 32768)) return OSF_ERR_UNSUPPORTED;
    const size_t n = (size_t)rows * (size_t)T * sizeof(float);
    if ((const void *)x != (const void *)z && overlaps(x, n, z, n)) return OSF_ERR_INVALID;
    DeviceInfo *dev;
    if (device_info(&dev) != OSF_OK) return OSF_ERR_CUDA;
    const size_t need = softmax_workspace_floats(rows, T, dev->sm_count) * sizeof(float);
    if (need > 0 && (!workspace || workspace_bytes < need)) return OSF_ERR_WORKSPACE;
    return launch_status(launch_softmax_rows(x, z, rows, T, static_cast<float *>(workspace),
                                             dev->sm_count, (cudaStream_t)stream));
}

// Bytes of bf16 dS^T the tensor-core backward keeps for its separate dQ product ([128 x 128]
// tiles covering [B * Hq][Sk rounded up to 128][Sq rounded up to 128]); 0 where that path does not
// apply or the buffer would pass 16 GiB (dQ then recomputes S and dP instead).
static size_t bwd_ds_bytes(int dtype, int B, int Hq, int Sq, int Sk, int D) {
    if (dtype != OSF_BF16 || (D != 64 && D != 128) || B <= 0 || Hq <= 0 || Sq <= 0 || Sk <= 0) return 0;
    const size_t cap = (size_t)16 << 30;
    const size_t tile = ((size_t)Sk + 127) / 128 * 128 * (((size_t)Sq + 127) / 128 * 128) * 2;
    if (tile > cap / ((size_t)B * (size_t)Hq)) return 0;
    return align256(tile * (size_t)B * (size_t)Hq);
}

int osf_attn_bwd_workspace_bytes(int dtype, int B, int Hq, int Hkv, int Sq, int Sk, int D, size_t *bytes) {
    if (!bytes) return OSF_ERR_INVALID;
    *bytes = 0;
    AttnProblem p;
    bool empty;
    const void *ph = reinterpret_cast<const void *>(uintptr_t(1) << 40);
    int st = check_gqa_ex(ph, ph, ph, reinterpret_cast<void *>(uintptr_t(1) << 44), dtype, B, Hq, Hkv, Sq, Sk, D,
                          nullptr, OSF_MASK_NONE, 0.f, nullptr, p, empty);
    if (st != OSF_OK || empty) return st;
    *bytes = align256((size_t)B * Hq * Sq * sizeof(float)) + bwd_ds_bytes(dtype, B, Hq, Sq, Sk, D);
    return OSF_OK;
}

int osf_attn_bwd_gqa(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                     const float *lse, void *dQ, void *dK, void *dV, int dtype, int B, int Hq, int Hkv,
                     int Sq, int Sk, int D, int mask, float scale, void *workspace, size_t workspace_bytes,
                     osf_stream stream) {
    AttnProblem p;
    bool empty;
    // the forward problem's checks (sizes, mask, scale; dQ plays the output's part)
    int st = check_gqa_ex(Q, K, V, dQ, dtype, B, Hq, Hkv, Sq, Sk, D, nullptr, mask, scale, nullptr, p, empty);
    if (st != OSF_OK) return st;
    if (empty) {
        // no keys or no rows: gradients are zero (written when there is anything to write)
        return OSF_OK;
    }
    if (!O || !dO || !lse || !dK || !dV) return OSF_ERR_INVALID;
    const size_t es = elem_size(dtype);
    const size_t nq = (size_t)B * Hq * Sq * D * es, nkv = (size_t)B * Hkv * Sk * D * es;
    const size_t nl = (size_t)B * Hq * Sq * sizeof(float);
    const void *ins[6] = {Q, K, V, O, dO, lse};
    const size_t in_n[6] = {nq, nkv, nkv, nq, nq, nl};
    void *outs[3] = {dQ, dK, dV};
    const size_t out_n[3] = {nq, nkv, nkv};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 6; ++i)
            if (overlaps(outs[o], out_n[o], ins[i], in_n[i])) return OSF_ERR_INVALID;
        for (int o2 = o + 1; o2 < 3; ++o2)
            if (overlaps(outs[o], out_n[o], outs[o2], out_n[o2])) return OSF_ERR_INVALID;
    }
    const size_t need = align256(nl);
    if (!workspace || workspace_bytes < need) return OSF_ERR_WORKSPACE;
    DeviceInfo *dev;
    if (device_info(&dev) != OSF_OK) return OSF_ERR_CUDA;
    BwdProblem b{};
    b.q = Q; b.k = K; b.v = V; b.o = O; b.dout = dO; b.lse = lse;
    b.dq = dQ; b.dk = dK; b.dv = dV;
    b.dtype = dtype;
    b.B = B; b.Hq = Hq; b.Hkv = Hkv; b.Sq = Sq; b.Sk = Sk; b.D = D;
    b.causal = p.causal; b.causal_off = p.causal_off;
    b.scale_log2 = p.scale_log2;
    b.scale = p.scale_log2 / kLog2e;
    b.dvec = static_cast<float *>(workspace);
    // a workspace that also holds dS^T selects the tensor-core path's separate dQ product
    const size_t ds_bytes = bwd_ds_bytes(dtype, B, Hq, Sq, Sk, D);
    if (ds_bytes > 0 && workspace_bytes >= need + ds_bytes &&
        ((reinterpret_cast<uintptr_t>(workspace) + need) & 31u) == 0) {
        b.ds = static_cast<char *>(workspace) + need;
        b.ds_rows = ((long long)Sk + 127) / 128 * 128;
        b.ds_ld = ((long long)Sq + 127) / 128 * 128;
    }
    b.status = dev->status;
    return launch_status(launch_attn_bwd(b, (cudaStream_t)stream));
}

int osf_softmax_ex_workspace_bytes(long long rows, long long T, size_t *bytes) {
    if (!bytes) return OSF_ERR_INVALID;
    *bytes = 0;
    if (rows < 0 || T < 0) return OSF_ERR_INVALID;
    if (rows == 0 || T == 0) return OSF_OK;
    if (rows > 65535 && T > 32768) return OSF_ERR_UNSUPPORTED;
    DeviceInfo *dev;
    if (device_info(&dev) != OSF_OK) return OSF_ERR_CUDA;
    // the larger of the float32 path's and the general path's needs
    const size_t a = softmax_workspace_floats(rows, T, dev->sm_count);
    const size_t b = softmax_ex_workspace_floats(rows, T, dev->sm_count);
    *bytes = (a > b ? a : b) * sizeof(float);
    return OSF_OK;
}

int osf_softmax_rows_ex(const void *x, void *z, int x_dtype, int z_dtype, long long rows, long long T,
                        long long x_row_stride, long long z_row_stride, float scale, long long causal_period,
                        void *workspace, size_t workspace_bytes, osf_stream stream) {
    if ((x_dtype != OSF_F32 && x_dtype != OSF_BF16) || (z_dtype != OSF_F32 && z_dtype != OSF_BF16))
        return OSF_ERR_INVALID;
    if (rows < 0 || T < 0 || causal_period < 0 || x_row_stride < 0 || z_row_stride < 0) return OSF_ERR_INVALID;
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return OSF_ERR_INVALID;
    if (rows == 0 || T == 0) return OSF_OK;
    const long long xs = x_row_stride ? x_row_stride : T, zs = z_row_stride ? z_row_stride : T;
    if (xs < T || zs < T) return OSF_ERR_INVALID;   // rows may not overlap one another
    if (!x || !z) return OSF_ERR_INVALID;
    if (rows > (1LL << 31) - 1 || (rows > 65535 && T > 32768) || xs >= (1LL << 40) || zs >= (1LL << 40))
        return OSF_ERR_UNSUPPORTED;
    const size_t nx = (size_t)((rows - 1) * xs + T) * elem_size(x_dtype);
    const size_t nz = (size_t)((rows - 1) * zs + T) * elem_size(z_dtype);
    const bool in_place = x == (const void *)z && x_dtype == z_dtype && xs == zs;
    if (!in_place && overlaps(x, nx, z, nz)) return OSF_ERR_INVALID;
    const float sc = scale == 0.f ? 1.f : scale;
    DeviceInfo *dev;
    if (device_info(&dev) != OSF_OK) return OSF_ERR_CUDA;
    if (x_dtype == OSF_F32 && z_dtype == OSF_F32 && sc == 1.f && causal_period == 0 && xs == T && zs == T)
        return osf_softmax_rows(static_cast<const float *>(x), static_cast<float *>(z), rows, T, workspace,
                                workspace_bytes, stream);
    const size_t need = softmax_ex_workspace_floats(rows, T, dev->sm_count) * sizeof(float);
    if (need > 0 && (!workspace || workspace_bytes < need)) return OSF_ERR_WORKSPACE;
    SoftmaxExProblem q{x, z, x_dtype, z_dtype, rows, T, xs, zs, sc * kLog2e, causal_period, dev->sm_count,
                       dev->status};
    return launch_status(launch_softmax_ex(q, static_cast<float *>(workspace), (cudaStream_t)stream));
}

int osf_selftest_bounded_wait(unsigned long long limit_ns, osf_stream stream) {
    if (limit_ns == 0 || limit_ns > 2000000000ull) return OSF_ERR_INVALID;
    DeviceInfo *dev;
    if (device_info(&dev) != OSF_OK) return OSF_ERR_CUDA;
    return launch_status(launch_bounded_wait_selftest(limit_ns, dev->status, (cudaStream_t)stream));
}

int osf_device_status(osf_stream stream) {
    DeviceInfo *dev;
    if (device_info(&dev) != OSF_OK) return OSF_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return OSF_ERR_CUDA;
    int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(int)) != cudaSuccess) return OSF_ERR_CUDA;
    if (word != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return OSF_ERR_CUDA;
    }
    return word;
}

}  // extern "C"
