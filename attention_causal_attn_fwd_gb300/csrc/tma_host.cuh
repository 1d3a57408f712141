// Host-side TMA tensor-map encoding (driver entry point fetched through the
// runtime, so the library does not link libcuda directly).
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace pathattn {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 3-D map over [bh][rows][cols] with 128-byte-wide boxes (64 bf16 or 32 fp32
// columns) of 128 rows and 128-byte swizzle.
inline bool make_map_t(CUtensorMap* m, const void* base, int cols, int rows, int bh, bool f32) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t elt = f32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)bh};
    cuuint64_t strides[2] = {(cuuint64_t)cols * elt, (cuuint64_t)rows * cols * elt};
    cuuint32_t box[3] = {f32 ? 32u : 64u, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
inline bool make_map(CUtensorMap* m, const void* base, int cols, int rows, int bh) {
    return make_map_t(m, base, cols, rows, bh, false);
}

}  // namespace pathattn
