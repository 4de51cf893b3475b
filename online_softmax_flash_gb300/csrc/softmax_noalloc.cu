// osf_softmax_rows_noalloc: the row softmax of osf_softmax_rows for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code running while a CUDA graph is being
// captured, a host library handed only its input and output buffers by an engine that owns
// every allocation, or a process under a strict device-memory budget.  For them the chunked
// path's scratch (one (m, l) float2 per chunk of each long row) lives in a fixed file-scope
// device array instead of a caller workspace.  The array is part of the library image: every
// GPU that loads libosf holds it until the process exits.
//
// The kernels are the ones osf_softmax_rows runs; only where their scratch lives differs.
#include <mutex>

#include "osf_internal.cuh"

namespace osf {
namespace {

constexpr int kNoAllocMaxDevices = 64;

// Capacity: 16384 chunk states (128 KiB).  Rows of up to 32768 elements need none; a longer
// row needs one state per chunk (the 1-D vector of 2^26 elements uses about 4 per SM).
constexpr long long kNoAllocMaxStates = 16384;

static __device__ __align__(256) float2 g_noalloc_scratch[kNoAllocMaxStates];

float *g_na_scratch[kNoAllocMaxDevices];   // device address of g_noalloc_scratch, per device
std::mutex g_na_mutex;

// One-time set-up per device, with that device current: the array's device address (in host
// code its name is only a host-side stand-in, never a usable pointer).
int noalloc_scratch(float **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return OSF_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_na_mutex);
    if (!g_na_scratch[dev]) {
        float *ptr = nullptr;
        if (cudaGetSymbolAddress((void **)&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return OSF_ERR_CUDA;
        g_na_scratch[dev] = ptr;
    }
    *out = g_na_scratch[dev];
    return OSF_OK;
}

}  // namespace
}  // namespace osf

extern "C" int osf_softmax_rows_noalloc(const float *x, float *z, long long rows, long long T,
                                        osf_stream stream) {
    using namespace osf;
    if (rows < 0 || T < 0) return OSF_ERR_INVALID;
    if (rows == 0 || T == 0) return OSF_OK;
    if (!x || !z) return OSF_ERR_INVALID;
    if (rows > (1LL << 31) - 1 || (rows > 65535 && T > 32768)) return OSF_ERR_UNSUPPORTED;
    const size_t n = (size_t)rows * (size_t)T * sizeof(float);
    const uintptr_t a = reinterpret_cast<uintptr_t>(x), b = reinterpret_cast<uintptr_t>(z);
    if (a != b && a < b + n && b < a + n) return OSF_ERR_INVALID;  // partial overlap
    // the SM count every entry point uses: the capacity check and the launch geometry agree
    // with osf_softmax_rows
    int sms = 0;
    int st = device_sm_count(&sms);
    if (st != OSF_OK) return st;
    float *scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != OSF_OK) return st;
    const size_t states = softmax_workspace_floats(rows, T, sms) / 2;
    if ((long long)states > kNoAllocMaxStates) return OSF_ERR_WORKSPACE;
    return launch_softmax_rows(x, z, rows, T, scratch, sms, (cudaStream_t)stream) == cudaSuccess ? OSF_OK
                                                                                                  : OSF_ERR_CUDA;
}
