/*
 * osf.h -- C ABI of libosf: single-pass (online-softmax) attention and streaming softmax
 * for one NVIDIA GB300 GPU (sm_103a).
 *
 * Sources (cited by page title and section):
 *   [SA] "softmax_attention" (blog.euler0525.cn/posts/3fb3592b), "实现思路" and "附录":
 *        solve(Q, K, V, output, M, N, d) on row-major [M,d] / [N,d] tensors already on the GPU,
 *        scale d^-0.5, keys streamed in blocks with a running max / rescale / denominator /
 *        numerator, -inf for keys past N.
 *   [Q3] "从零开始写Qwen3（五-其一）使用Triton实现自注意力" (gitcode.csdn.net), "自注意力原理",
 *        "多头自注意力", "stride的作用", "GQA": O = softmax(mask(QK^T/sqrt(D)))V on [B,H,S,D]
 *        tensors, Hq divisible by Hkv, kv head = q head // (Hq/Hkv), causal tril mask applied
 *        only when the query length is > 1.
 *   [TP] Triton-Puzzles write-up (fadingcoder.top/post/105980), "Puzzle 8: Long Softmax":
 *        softmax of each row of a [rows, T] matrix; two-loop online form.
 *   [SO] "Softmax 算子的实现与优化" (blog.euler0525.cn/posts/5db73590), "Online Softmax" and
 *        "CUDA 版本": the boxed (m, l) recurrence; extern "C" solve(const float* input,
 *        float* output, int N) on device pointers, returning without work when N <= 0.
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE pointers (cudaMalloc / torch CUDA memory) on the current device,
 *     except where a parameter says otherwise.  The caller owns every buffer; the library
 *     never allocates or frees device memory in these calls.
 *   - Work is enqueued on `stream` (NULL = legacy default stream) and the call returns without
 *     waiting (unlike [SO]'s solve, which synchronises the device).  A returned OSF_OK means
 *     the arguments were valid and the launches were accepted.
 *   - Layouts are contiguous row-major: [M,d], [N,d], [B,H,S,D] (D fastest), [rows,T].
 *   - Return value: an osf_status code.  No entry point traps or asserts on the device.
 *     Device-side failures (a bounded wait that ran out) are recorded in a device status word
 *     read by osf_device_status().
 *   - Thread safety: entry points may be called concurrently from several host threads on
 *     different streams; calls sharing a workspace buffer must be ordered by the caller.
 */
#ifndef OSF_H
#define OSF_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *osf_stream;

typedef enum osf_status {
    OSF_OK = 0,
    OSF_ERR_INVALID = 1,     /* invalid argument: NULL with non-zero size, negative size,
                                Hq % Hkv != 0, causal with 1 < Sq != Sk, forbidden aliasing */
    OSF_ERR_UNSUPPORTED = 2, /* valid but outside what the library implements (e.g. D > 256,
                                or a size whose element count exceeds 2^31 per head) */
    OSF_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    OSF_ERR_TIMEOUT = 4,     /* a bounded device-side wait expired (osf_device_status) */
    OSF_ERR_WORKSPACE = 5    /* workspace NULL or smaller than the *_workspace_bytes query */
} osf_status;

typedef enum osf_dtype {
    OSF_F32 = 0,   /* IEEE float32 inputs and outputs */
    OSF_BF16 = 1   /* bfloat16 Q/K/V/O; accumulation and softmax state in float32 */
} osf_dtype;

/* Human-readable name of a status code (static string; never NULL). */
const char *osf_status_string(int status);

/* Library ABI version, major * 10000 + minor * 100 + patch. */
int osf_version(void);

/*
 * osf_attn_fwd -- single-head attention, [SA] "实现思路" / "附录" solve(Q, K, V, output, M, N, d):
 *     out[i, :] = sum_j softmax_j(Q[i,:] . K[j,:] * d^-0.5) V[j, :]
 * Q: [M, d] float32, K: [N, d], V: [N, d], out: [M, d]; all row-major contiguous, device.
 * M == 0 or N == 0: returns OSF_OK and touches nothing (the pages return early on empty input).
 * d must be 1..256 (OSF_ERR_UNSUPPORTED above).  out must not overlap Q, K or V.
 */
int osf_attn_fwd(const float *Q, const float *K, const float *V, float *out,
                 int M, int N, int d, osf_stream stream);

/*
 * osf_attn_fwd_gqa -- batched grouped-query attention with optional causal mask,
 * [Q3] "自注意力原理" + "GQA":
 *     O[b,h,i,:] = sum_j softmax_j(mask(Q[b,h,i,:] . K[b,h/G,j,:] * scale)) V[b,h/G,j,:]
 *     G = Hq / Hkv.  mask: when causal && Sq > 1, key j is excluded for j > i (top-left
 *     aligned tril(ones(Sq, Sk))); when Sq == 1 every key is used, as on the page.
 * Q: [B, Hq, Sq, D], K and V: [B, Hkv, Sk, D], O: [B, Hq, Sq, D], all of `dtype`.
 * scale <= 0 selects D^-0.5.
 * lse: optional (NULL) float32 [B, Hq, Sq] receiving the natural-log log-sum-exp of each row's
 *      scaled, masked scores (m + ln l).
 * workspace: device scratch for split-K partial states; query the size with
 *      osf_attn_workspace_bytes (may be 0, then workspace may be NULL).
 * Sq == 0 or Sk == 0 or B == 0: OSF_OK, nothing written.  Hq % Hkv != 0, causal with
 * Sq > 1 && Sq != Sk, or O overlapping Q/K/V: OSF_ERR_INVALID.  D must be 1..256.
 * Kernel choice (internal), bf16 with D in {64, 128}: when (Hq / Hkv) * Sq <= 16 (decode,
 * or a few speculative rows) the split-K decode kernel and a log-sum-exp combine; otherwise
 * the tensor-core (tcgen05/TMEM/TMA) prefill kernel.  Everything else runs the general
 * CUDA-core kernel.
 */
int osf_attn_fwd_gqa(const void *Q, const void *K, const void *V, void *O, int dtype,
                     int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                     float *lse, void *workspace, size_t workspace_bytes, osf_stream stream);

/*
 * osf_attn_bwd_gqa -- gradients of batched GQA attention (the backward pass of
 * osf_attn_fwd_gqa_ex on contiguous tensors).  The pages describe only the forward pass,
 * [Q3] "自注意力原理" + "GQA"; this is the chain rule through that definition for a loss whose
 * gradient with respect to O is dO:
 *     P = softmax(mask(Q K^T * scale)),  D_i = sum_d dO[i,d] O[i,d],
 *     dV = P^T dO,  dS = P * (dO V^T - D),  dQ = scale * dS K,  dK = scale * dS^T Q,
 * with P rebuilt from lse; a kv head's dK, dV sum over its Hq / Hkv query heads.
 * Q, O, dO, dQ: [B, Hq, Sq, D]; K, V, dK, dV: [B, Hkv, Sk, D]; all of `dtype`, contiguous,
 * device.  lse: float32 [B, Hq, Sq], the natural-log log-sum-exp the forward call returned.
 * mask, scale: as given to the forward call (an osf_mask; scale <= 0 selects D^-0.5).
 * workspace: osf_attn_bwd_workspace_bytes bytes: one float per query row (the row sums D), then,
 * for bf16 with D in {64, 128} while it stays within 16 GiB, room for dS^T in bf16
 * (B * Hq * ceil(Sk/128)*128 * ceil(Sq/128)*128 elements).  A workspace of at least the first
 * part (256-byte rounded) but short of the whole selects the path that keeps no dS.
 * dQ, dK, dV must not overlap one another or any input -> else OSF_ERR_INVALID.
 * B, Sq or Sk == 0: OSF_OK, nothing written.  Other errors as in osf_attn_fwd_gqa.
 * Kernel choice: bf16 with D in {64, 128} whose tensors TMA can address (16-byte aligned
 * pointers) runs a row-sum pre-pass and then tcgen05 tensor-core kernels (accumulators in TMEM,
 * tiles streamed by TMA): with the full workspace, dK/dV CTAs per key tile that also store dS^T,
 * then dQ = scale * dS K as one product over the stored dS (three launches); with the shorter
 * workspace, one grid of dK/dV CTAs and dQ CTAs that recompute S and dP (two launches).  Other
 * bf16 D in {64, 128} cases run the warp-level mma.sync kernels; everything else a CUDA-core
 * kernel with one warp per row.
 */
int osf_attn_bwd_gqa(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                     const float *lse, void *dQ, void *dK, void *dV, int dtype, int B, int Hq, int Hkv,
                     int Sq, int Sk, int D, int mask, float scale, void *workspace, size_t workspace_bytes,
                     osf_stream stream);

/* Bytes of workspace osf_attn_bwd_gqa needs for these sizes (written to *bytes). */
int osf_attn_bwd_workspace_bytes(int dtype, int B, int Hq, int Hkv, int Sq, int Sk, int D, size_t *bytes);

/* Mask modes of osf_attn_fwd_gqa_ex. */
typedef enum {
    OSF_MASK_NONE = 0,          /* every key */
    OSF_MASK_TOP_LEFT = 1,      /* Sq > 1: row i sees keys 0..i (tril(ones(Sq, Sk)), [Q3] "自注意力原理");
                                   Sq == 1: every key, as on the page */
    OSF_MASK_BOTTOM_RIGHT = 2   /* row i sees keys 0..i + Sk - Sq: the Sq new rows follow a cache of
                                   Sk - Sq keys (not on the pages; equals TOP_LEFT when Sq == Sk) */
} osf_mask;

/*
 * osf_attn_fwd_gqa_ex -- osf_attn_fwd_gqa on strided tensors, with a mask mode.
 * The operation is the one of osf_attn_fwd_gqa, [Q3] "自注意力原理" + "GQA".  [Q3] "stride的作用":
 * a head split or a transpose of any but the last dimension only changes strides, and an
 * expanded (broadcast) dimension has stride 0; so every tensor is addressed through its own
 * element strides instead of being copied to [B, H, S, D] first.
 *
 * strides: NULL (all four tensors contiguous [B, H, S, D]) or 12 element strides, in order
 *     Q: b, h, s   K: b, h, s   V: b, h, s   O: b, h, s.
 *     The d stride is 1.  E.g. a [B, S, H, D] tensor has b = S*H*D, h = D, s = H*D.
 *     Strides must be >= 0 (0 broadcasts an input); O's rows must not overlap one another,
 *     and O must not overlap Q, K, V or lse (checked on address ranges) -> else OSF_ERR_INVALID.
 * mask: an osf_mask; any Sq, Sk.  A row that sees no key (BOTTOM_RIGHT with i < Sq - Sk)
 *     gets O = 0 and lse = -inf.
 * lse: optional contiguous float32 [B, Hq, Sq], natural-log log-sum-exp of each row.
 * Workspace: osf_attn_workspace_bytes with the same dtype and sizes gives enough.
 * Kernel choice as in osf_attn_fwd_gqa.  The TMA kernels need 16-byte aligned bases and
 * strides (multiples of 8 bf16 elements); other layouts run on the CUDA-core kernel.
 * Errors, emptiness and ownership as in osf_attn_fwd_gqa.
 */
int osf_attn_fwd_gqa_ex(const void *Q, const void *K, const void *V, void *O, int dtype,
                        int B, int Hq, int Hkv, int Sq, int Sk, int D, const long long *strides,
                        int mask, float scale, float *lse, void *workspace, size_t workspace_bytes,
                        osf_stream stream);

/* Bytes of workspace osf_attn_fwd_gqa needs for these arguments (written to *bytes). */
int osf_attn_workspace_bytes(int dtype, int B, int Hq, int Hkv, int Sq, int Sk, int D,
                             size_t *bytes);

/*
 * osf_attn_fwd_gqa_host -- osf_attn_fwd_gqa on HOST buffers: the attention of [Q3]
 * "自注意力原理" + "GQA" (the same operation, mask rule and scale as osf_attn_fwd_gqa; the pages
 * pass tensors that are already on the GPU, so this copying variant has no counterpart there).
 * Q, K, V: host pointers to contiguous [B, Hq, Sq, D] / [B, Hkv, Sk, D] arrays of `dtype`;
 * O: host pointer to [B, Hq, Sq, D], written.  Page-locked (pinned) host memory lets the copies
 * run asynchronously and overlap; pageable memory works but the copies then block the host.
 * device_buffer: caller-owned device memory of at least osf_attn_host_buffer_bytes bytes; it
 *     receives device copies of Q, K, V, O and the kernels' scratch (too small or NULL ->
 *     OSF_ERR_WORKSPACE).
 * The problem is cut into up to 8 chunks of whole (batch, kv head) units, each a contiguous
 * range of every tensor; chunk c's host-to-device copies, its attention and its device-to-host
 * copy are enqueued on an internal copy-in stream, `stream` and an internal copy-out stream,
 * linked by events, so copies overlap computation and each other.  All of it is ordered after
 * the work already on `stream`, and work enqueued on `stream` afterwards runs after O has
 * reached the host: synchronise `stream` before reading O.  The first call on a device creates
 * the two copy streams and their events (kept until exit); calls are serialised while they
 * enqueue.  lse is not produced.  Sizes, errors and emptiness as in osf_attn_fwd_gqa.
 * After a non-OK return the contents of O are undefined (some chunks may have been copied back,
 * others not); `stream` is still ordered after every copy and kernel the call had queued, so
 * work enqueued on it afterwards, or a synchronisation of it, waits for them.
 */
int osf_attn_fwd_gqa_host(const void *Q, const void *K, const void *V, void *O, int dtype,
                          int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                          void *device_buffer, size_t device_buffer_bytes, osf_stream stream);

/* Device bytes osf_attn_fwd_gqa_host needs in device_buffer for these arguments. */
int osf_attn_host_buffer_bytes(int dtype, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal,
                               size_t *bytes);

/*
 * osf_attn_decode_gqa -- the Sq == 1 path of osf_attn_fwd_gqa with an explicit split count.
 * The Sk keys of each (b, kv head) are cut into `num_splits` contiguous chunks; each chunk
 * yields a partial state (m_s, l_s, acc_s) and a combine step merges them with the
 * log-sum-exp rule (the [SO] "Online Softmax" recurrence applied to whole partial states;
 * the pages do not describe the split itself).  num_splits <= 0 picks a count from the SM
 * count.  Q: [B, Hq, 1, D], K/V: [B, Hkv, Sk, D], O: [B, Hq, 1, D].  Workspace size:
 * osf_attn_decode_workspace_bytes with the same num_splits.
 */
int osf_attn_decode_gqa(const void *Q, const void *K, const void *V, void *O, int dtype,
                        int B, int Hq, int Hkv, int Sk, int D, float scale, float *lse,
                        int num_splits, void *workspace, size_t workspace_bytes,
                        osf_stream stream);
int osf_attn_decode_workspace_bytes(int dtype, int B, int Hq, int Hkv, int Sk, int D,
                                    int num_splits, size_t *bytes);

/*
 * osf_softmax_rows -- row softmax, [TP] "Puzzle 8: Long Softmax" / [SO] "Online Softmax":
 *     z[r, j] = exp(x[r, j] - m_r) / l_r,  m_r = max_j x[r, j],  l_r = sum_j exp(x[r, j] - m_r)
 * x, z: [rows, T] float32 row-major, device.  z == x (in place) is allowed; any other overlap
 * is OSF_ERR_INVALID.  rows == 0 or T == 0: OSF_OK, nothing written.
 * Rows of up to 32768 elements are held on chip (one read, one write); longer rows -- e.g.
 * one 1-D vector, rows == 1 -- are cut into chunks processed by many CTAs, whose partial
 * (m, l) states are merged and followed by a normalising pass (two reads, one write).  That
 * path needs workspace: osf_softmax_workspace_bytes (0 when not needed).
 */
int osf_softmax_rows(const float *x, float *z, long long rows, long long T,
                     void *workspace, size_t workspace_bytes, osf_stream stream);
int osf_softmax_workspace_bytes(long long rows, long long T, size_t *bytes);

/*
 * osf_softmax_rows_noalloc -- osf_softmax_rows for callers that cannot allocate device memory.
 * The pages have no counterpart: this entry point exists for callers such as code running
 * while a CUDA graph is captured, a library that is handed only its input and output buffers
 * by an engine owning every allocation, or a process under a fixed device-memory budget.
 * Same arguments, result and in-place rule as osf_softmax_rows, minus the workspace: the
 * chunked path keeps its per-chunk (m, l) states in a fixed device array inside the library
 * (16384 states, 128 KiB, held on every GPU that loads the library until the process exits).
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - The first call on a device, with that device current, looks up the array's device
 *     address; make that first call before any stream capture.
 *   - Every call shares the one array per device: calls that may run at the same time on the
 *     GPU (different streams, or different host threads) race and must be serialised by the
 *     caller.  Nothing in the array needs to start at zero; each call overwrites what it reads.
 *   - A problem needing more states than the array holds (only rows longer than 32768
 *     elements use any: rows x chunks per row > 16384) returns OSF_ERR_WORKSPACE and launches
 *     nothing; use osf_softmax_rows with a caller workspace instead.
 */
int osf_softmax_rows_noalloc(const float *x, float *z, long long rows, long long T,
                             osf_stream stream);

/*
 * osf_softmax_rows_ex -- row softmax of scale * x with an optional in-row causal mask, on
 * float32 or bfloat16 rows with row strides: the softmax of [Q3] "softmax的triton实现", a kernel
 * over attention-weight rows taking a row stride and a scale, whose causal variant keeps column
 * <= row (-inf elsewhere, 0 after the exponential); values are widened to float32 on load as
 * in [SO] "Online Softmax".
 *     kept(r, j) = (causal_period == 0) || (j <= r % causal_period)
 *     z[r, j] = kept ? exp(scale*x[r, j] - m_r) / l_r : 0, over the kept columns of row r
 * x: rows of T elements of x_dtype (OSF_F32 or OSF_BF16), row r at x + r * x_row_stride
 *    elements; z likewise with z_dtype and z_row_stride.  A stride of 0 means T; strides < T
 *    -> OSF_ERR_INVALID.  z == x with the same dtype and stride is in place; any other overlap
 *    -> OSF_ERR_INVALID.
 * scale: 0 -> 1; NaN or infinite -> OSF_ERR_INVALID.
 * causal_period: 0 -> no mask; P > 0 -> row r keeps columns 0 .. r % P (stacked [Sq, Sk]
 *    score matrices use P = Sq; a single matrix P = rows).
 * workspace: osf_softmax_ex_workspace_bytes(rows, T) bytes (0 for T <= 32768).
 * Kernel choice: contiguous float32 with scale 1 and no mask runs osf_softmax_rows; rows of up
 * to 32768 elements with 16-byte aligned starts are held on chip (columns past the causal limit
 * are not read); others stream through one CTA per row or, beyond 32768, chunks over the GPU.
 */
int osf_softmax_rows_ex(const void *x, void *z, int x_dtype, int z_dtype, long long rows, long long T,
                        long long x_row_stride, long long z_row_stride, float scale, long long causal_period,
                        void *workspace, size_t workspace_bytes, osf_stream stream);

/* Bytes of workspace osf_softmax_rows_ex needs for [rows, T] (written to *bytes). */
int osf_softmax_ex_workspace_bytes(long long rows, long long T, size_t *bytes);

/*
 * osf_selftest_bounded_wait -- diagnostic of the failure-detection mechanism (the pages have no
 * counterpart).  Launches one CTA that waits, with the bounded-wait helper every TMA /
 * tensor-core kernel uses, on an mbarrier nothing arrives on; after limit_ns (1 .. 2e9) the wait
 * gives up and records OSF_ERR_TIMEOUT in the device status word, which osf_device_status then
 * returns.  The kernel exits normally: the context stays usable.  limit_ns out of range ->
 * OSF_ERR_INVALID.
 */
int osf_selftest_bounded_wait(unsigned long long limit_ns, osf_stream stream);

/*
 * osf_device_status -- synchronise `stream`, then return (and reset to OSF_OK) the device
 * status word of the current device: OSF_ERR_TIMEOUT if any kernel gave up a bounded wait
 * since the last call, OSF_ERR_CUDA if the synchronisation itself failed, else OSF_OK.
 */
int osf_device_status(osf_stream stream);

/* Number of streaming multiprocessors of the current device (0 on error). */
int osf_sm_count(void);

/* Total number of kernels this library has launched in this process (all devices, all
 * threads); a diagnostic for counting launches in a timed region. */
unsigned long long osf_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* OSF_H */
