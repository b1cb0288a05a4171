// fa_tma_host.h -- host helpers shared by the tcgen05 kernels' launchers:
// the driver's tensor-map encoder (looked up once through the runtime), the
// tiled maps of [B, H, T, d] tensors with the 128-byte swizzle, and the SM
// count of the current device.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace fa {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (fn == nullptr) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// A tensor map of bf16 (elem = 2) or e4m3 (elem = 1, as bytes) over `rank`
// dimensions, dims[0] = d contiguous, the others with element strides; boxes
// of 128 bytes of columns by box[1..] elements with the 128-byte swizzle.
// Coordinates outside the tensor read as zero (loads) or are dropped
// (stores).  A dimension of extent 1 is never stepped, so it gets a packed
// stride whatever the caller's.
inline bool encode_map(EncodeTiledFn enc, CUtensorMap *map, const void *base, int rank, const int64_t *dims,
                const int64_t *strides, const uint32_t *box, int elem) {
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    uint64_t packed = (uint64_t)dims[0] * elem;
    for (int i = 0; i < rank; ++i) {
        gd[i] = (cuuint64_t)dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i > 0) {
            gs[i - 1] = dims[i] > 1 ? (cuuint64_t)strides[i] * elem : (cuuint64_t)packed;
            packed = (uint64_t)gs[i - 1] * (uint64_t)dims[i];
        }
    }
    return enc(map, elem == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank,
               const_cast<void *>(base), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [B, H, T, d] with element strides (sb, sh, st) as the 4-D map (d, T, H, B);
// boxes of 128 bytes of columns x box_rows rows of one (batch, head).
inline bool make_map(EncodeTiledFn enc, CUtensorMap *map, const void *base, int d, int T, int H, int B, int64_t st,
              int64_t sh, int64_t sb, int box_rows, int elem = 2) {
    const int64_t dims[4] = {d, T, H, B}, strides[4] = {1, st, sh, sb};
    const uint32_t box[4] = {(uint32_t)(128 / elem), (uint32_t)box_rows, 1, 1};
    return encode_map(enc, map, base, 4, dims, strides, box, elem);
}

// Streaming multiprocessors of the current device (cached per device).
inline int sm_count() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;
    }
    return cached[dev];
}

}  // namespace fa
