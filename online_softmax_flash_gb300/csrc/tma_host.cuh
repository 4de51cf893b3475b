// Host-side construction of TMA tensor maps (driver entry point looked up through the runtime,
// so the library does not link libcuda directly).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace osf {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 3-D map over a contiguous bf16 tensor [Z][Y][D]: box [1][box_rows][64] (128-byte rows),
// 128-byte swizzle, out-of-range elements read as zero.
inline bool make_bf16_map_3d(CUtensorMap *m, const void *g, int D, long long Y, long long Z, uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Y, (cuuint64_t)Z};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * 2 * (cuuint64_t)Y};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(g), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over a contiguous bf16 tensor [Z][Y][X] for stores of [32 x 32] boxes (64-byte rows,
// 64-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ ((r / 2) % 4) in shared memory).
inline bool make_bf16_store_map_32x32(CUtensorMap *m, const void *g, long long X, long long Y, long long Z) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)X, (cuuint64_t)Y, (cuuint64_t)Z};
    cuuint64_t strides[2] = {(cuuint64_t)X * 2, (cuuint64_t)X * 2 * (cuuint64_t)Y};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(g), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D view (d % 64, y, d / 64, z) of a contiguous bf16 tensor [Z][Y][D], D a multiple of 64:
// one box {64, box_rows, D/64, 1} brings a whole [box_rows x D] tile in a single TMA
// instruction, laid out in shared memory as D/64 consecutive [box_rows][64] blocks (128-byte
// rows, 128-byte swizzle) -- the K-major layout the tcgen05 descriptors expect.  A TMA
// instruction has a fixed cost of several hundred cycles on this part whatever its size, so
// fewer, larger boxes keep the copy engine ahead of the tensor core.
// `box_dblocks` (default all D/64) 64-column blocks per box: a box of one block loads a
// [box_rows x 64] column slice.
inline bool make_bf16_tile_map(CUtensorMap *m, const void *g, int D, long long Y, long long Z, uint32_t box_rows,
                               uint32_t box_dblocks = 0) {
    auto enc = tensor_map_encoder();
    if (!enc || D % 64 != 0) return false;
    if (box_dblocks == 0) box_dblocks = (uint32_t)(D / 64);
    cuuint64_t dims[4] = {64, (cuuint64_t)Y, (cuuint64_t)(D / 64), (cuuint64_t)Z};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, 128, (cuuint64_t)D * 2 * (cuuint64_t)Y};
    cuuint32_t box[4] = {64, box_rows, box_dblocks, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(g), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 5-D view (d % 64, s, d / 64, h, b) of a bf16 tensor [B][H][S][D] with element strides sb, sh,
// ss (d contiguous, D a multiple of 64): one box {64, box_rows, D/64, 1, 1} brings a whole
// [box_rows x D] tile of one (b, h) in a single TMA instruction, laid out as in
// make_bf16_tile_map.  TMA needs 16-byte aligned strides (multiples of 8 elements); a
// dimension of extent 1 takes a placeholder stride.  False when the map cannot be encoded.
inline bool make_bf16_tile_map_strided(CUtensorMap *m, const void *g, int D, long long S, long long H,
                                       long long B, long long ss, long long sh, long long sb,
                                       uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc || D % 64 != 0) return false;
    auto fix = [](long long extent, long long stride_elems) -> cuuint64_t {
        return extent > 1 ? (cuuint64_t)stride_elems * 2 : (cuuint64_t)128;
    };
    cuuint64_t dims[5] = {64, (cuuint64_t)S, (cuuint64_t)(D / 64), (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[4] = {fix(S, ss), 128, fix(H, sh), fix(B, sb)};
    for (int i = 0; i < 4; ++i)
        if (strides[i] == 0 || strides[i] % 16 != 0) return false;
    cuuint32_t box[5] = {64, box_rows, (cuuint32_t)(D / 64), 1, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(g), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// True when make_bf16_tile_map_strided can describe the tensor (no encoding call): 16-byte
// aligned base, D a multiple of 64, and every stride of a dimension longer than one a non-zero
// multiple of 16 bytes below 2^40.
inline bool tile_map_addressable(const void *g, int D, long long S, long long H, long long B, long long ss,
                                 long long sh, long long sb) {
    if ((reinterpret_cast<uintptr_t>(g) & 15u) != 0 || D % 64 != 0) return false;
    const long long ext[3] = {S, H, B}, st[3] = {ss, sh, sb};
    for (int i = 0; i < 3; ++i)
        if (ext[i] > 1 && (st[i] <= 0 || (st[i] * 2) % 16 != 0 || st[i] * 2 >= (1LL << 40))) return false;
    return true;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace osf
