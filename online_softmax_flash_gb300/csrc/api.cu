// C ABI of libosf (declared in include/osf.h): argument checks, kernel choice, workspace
// sizing and the device status word.  Every entry point validates on the host, then enqueues
// kernels on the caller's stream and returns; nothing here allocates device memory.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "osf_internal.cuh"
#include "attn_tc.cuh"
#include "decode.cuh"

namespace osf {

static std::atomic<unsigned long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

namespace {

constexpr int kMaxDevices = 64;

// One status word per device; kernels with bounded waits write kStatusTimeout here.
__device__ int g_status_word;

struct DeviceInfo {
    int sm_count = 0;
    int *status = nullptr;   // device address of g_status_word
    bool ready = false;
};
DeviceInfo g_dev[kMaxDevices];

int current_device(int *dev) {
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return OSF_ERR_CUDA;
    return OSF_OK;
}

// Per-device set-up (SM count, status word address).  Idempotent; concurrent first calls
// compute the same values.
int device_info(DeviceInfo **out) {
    int dev;
    if (current_device(&dev) != OSF_OK) return OSF_ERR_CUDA;
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return OSF_ERR_CUDA;
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return OSF_ERR_CUDA;
        d.sm_count = sms;
        d.status = static_cast<int *>(addr);
        d.ready = true;
    }
    *out = &d;
    return OSF_OK;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

size_t elem_size(int dtype) { return dtype == OSF_F32 ? 4 : 2; }

int launch_status(cudaError_t e) { return e == cudaSuccess ? OSF_OK : OSF_ERR_CUDA; }

// Shared validation of the GQA problem; fills `p` (without workspace pointers).
int check_gqa(const void *Q, const void *K, const void *V, void *O, int dtype, int B, int Hq,
              int Hkv, int Sq, int Sk, int D, int causal, float scale, float *lse,
              AttnProblem &p, bool &empty) {
    empty = false;
    if (dtype != OSF_F32 && dtype != OSF_BF16) return OSF_ERR_INVALID;
    if (B < 0 || Hq < 0 || Hkv < 0 || Sq < 0 || Sk < 0 || D <= 0) return OSF_ERR_INVALID;
    if (Hq == 0 || Hkv == 0 || Hq % Hkv != 0) return OSF_ERR_INVALID;
    if (!(scale == scale)) return OSF_ERR_INVALID;  // NaN
    if (causal && Sq > 1 && Sq != Sk) return OSF_ERR_INVALID;
    if (D > 256) return OSF_ERR_UNSUPPORTED;
    if (B == 0 || Sq == 0 || Sk == 0) { empty = true; return OSF_OK; }
    // per-head element counts index with 32-bit row numbers inside kernels
    if ((long long)Sq * D >= (1LL << 31) || (long long)Sk * D >= (1LL << 31) ||
        (long long)B * Hq >= (1LL << 31) || (long long)B * Hq * Sq >= (1LL << 40))
        return OSF_ERR_UNSUPPORTED;
    if (!Q || !K || !V || !O) return OSF_ERR_INVALID;
    const size_t es = elem_size(dtype);
    const size_t nq = (size_t)B * Hq * Sq * D * es, nkv = (size_t)B * Hkv * Sk * D * es;
    if (overlaps(O, nq, Q, nq) || overlaps(O, nq, K, nkv) || overlaps(O, nq, V, nkv))
        return OSF_ERR_INVALID;
    if (lse) {
        const size_t nl = (size_t)B * Hq * Sq * sizeof(float);
        if (overlaps(lse, nl, O, nq) || overlaps(lse, nl, Q, nq) || overlaps(lse, nl, K, nkv) ||
            overlaps(lse, nl, V, nkv))
            return OSF_ERR_INVALID;
    }
    p = AttnProblem{};
    p.q = Q; p.k = K; p.v = V; p.o = O; p.lse = lse;
    p.dtype = dtype;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sq = Sq; p.Sk = Sk; p.D = D;
    p.causal = (causal && Sq > 1) ? 1 : 0;
    const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
    p.scale_log2 = sc * kLog2e;
    p.splits = 1;
    return OSF_OK;
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
    if (p.dtype == OSF_BF16 && p.Sq == 1 && decode_supported(p, Q, K, V, O)) return Path::Decode;
    if (p.dtype == OSF_BF16 && p.Sq > 1 && attn_tc_supported(p, Q, K, V, O)) return Path::TensorCore;
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
    (void)path;  // every path keeps split partial states in the same layout
    return partial_bytes(splits, (long long)p.B * p.Hq * p.Sq, p.D);
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
    if (dtype == OSF_BF16 && Sq > 1 && (D == 64 || D == 128)) {
        const size_t tc = partial_bytes(attn_tc_pick_splits(p, dev->sm_count), (long long)B * Hq * Sq, D);
        if (tc > need) need = tc;
    }
    if (dtype == OSF_BF16 && Sq == 1) {
        const size_t dn = partial_bytes(decode_pick_splits(p, dev->sm_count, 0), (long long)B * Hq, D);
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
