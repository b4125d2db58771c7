// Host-side TMA tensor-map encoding shared by the kernels that use tensor
// copies.  cuTensorMapEncodeTiled comes from the driver through the runtime's
// entry-point query, so the library links only the CUDA runtime.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "xs_paged.h"

namespace xs {

using TensorMapEncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                       const cuuint64_t *, const cuuint64_t *,
                                       const cuuint32_t *, const cuuint32_t *,
                                       CUtensorMapInterleave, CUtensorMapSwizzle,
                                       CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline TensorMapEncodeFn tensor_map_encoder() {
    static std::once_flag once;
    static TensorMapEncodeFn fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<TensorMapEncodeFn>(ptr);
        cudaGetLastError();
    });
    return fn;
}

// A bf16 tensor map of rank R with 128-byte swizzle (zero fill outside the
// tensor).  strides: bytes, for dims 1 .. R-1.
template <int R>
int encode_bf16_map(CUtensorMap *tm, const void *base, const cuuint64_t (&dims)[R],
                    const cuuint64_t (&strides)[R - 1], const cuuint32_t (&box)[R]) {
    TensorMapEncodeFn fn = tensor_map_encoder();
    if (!fn) return XS_EDEVICE;
    cuuint32_t estr[R];
    for (int i = 0; i < R; ++i) estr[i] = 1;
    const CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, R, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? XS_OK : XS_EUNSUPPORTED;
}

}  // namespace xs
