// tmap.h -- host-side construction of TMA tensor maps (CUtensorMap) through
// the driver entry point, so that the library needs no link against libcuda.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Tiled tensor map of `rank` dims.  dims[0] is the contiguous dim; strides_b
// holds the byte strides of dims 1..rank-1 (multiples of 16); box[i] elements
// per copy along dim i.  Out-of-range elements read as zero.
inline bool make_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank,
                            const void* base, const uint64_t* dims, const uint64_t* strides_b,
                            const uint32_t* box, CUtensorMapSwizzle swizzle) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    uint32_t estride[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, dtype, rank, const_cast<void*>(base), dims, strides_b, box, estride,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace kda
