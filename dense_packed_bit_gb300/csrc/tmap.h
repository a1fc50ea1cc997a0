// tmap.h -- host-side creation of 2-D TMA tensor maps.
//
// cuTensorMapEncodeTiled is a driver API entry point; it is looked up at run
// time through the CUDA runtime, so libmm does not link libcuda and still
// loads on a machine without a GPU driver.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

namespace mm {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder(cudaError_t *err) {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static cudaError_t e = cudaSuccess;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (e == cudaSuccess && q != cudaDriverEntryPointSuccess) e = cudaErrorSymbolNotFound;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    *err = e;
    return fn;
}

// Row-major 2-D tensor: `inner` contiguous elements per row, `outer` rows,
// rows `row_stride_bytes` apart.  Box of box_inner x box_outer elements.
// Out-of-range elements of a box read as zero.
inline cudaError_t make_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t elem_bytes, const void *base,
                                uint64_t inner, uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                                uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    cudaError_t err;
    auto enc = tmap_encoder(&err);
    if (err != cudaSuccess) return err;
    (void)elem_bytes;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// A batch of row-major 2-D tensors: `inner` x `outer` each, rows `row_stride_bytes`
// apart, `batch` matrices `mat_stride_bytes` apart (both multiples of 16).  Box of
// box_inner x box_outer x 1.  Out-of-range elements of a box read as zero.
inline cudaError_t make_tmap_3d(CUtensorMapDataType dtype, CUtensorMap *map, const void *base, uint64_t inner,
                                uint64_t outer, uint64_t batch, uint64_t row_stride_bytes, uint64_t mat_stride_bytes,
                                uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    cudaError_t err;
    auto enc = tmap_encoder(&err);
    if (err != cudaSuccess) return err;
    cuuint64_t dims[3] = {inner, outer, batch};
    cuuint64_t strides[2] = {row_stride_bytes, mat_stride_bytes};
    cuuint32_t box[3] = {box_inner, box_outer, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, dtype, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace mm
