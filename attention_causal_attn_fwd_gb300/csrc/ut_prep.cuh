// Shared-memory row loader and the UT-prep launcher shared by both forward paths.
#pragma once
#include "common.cuh"

namespace pathattn {

// Load rows [r0, r0+R) x [0, D) of a row-major [*, D] array into shared memory
// (leading dimension LDS), converting to S; rows >= nrows read as zero.
template <int R, int D, int LDS, int NT, typename S, typename G>
__device__ __forceinline__ void load_rows(S* dst, const G* src, int r0, int nrows) {
    for (int idx = threadIdx.x; idx < R * D; idx += NT) {
        const int r = idx / D, c = idx % D;
        const int row = r0 + r;
        float x = row < nrows ? to_f<G>(src[(size_t)row * D + c]) : 0.f;
        dst[r * LDS + c] = from_f<S>(x);
    }
}

// Inclusive cumulative sum of log f per head into cum [BH, Lp] (ut_prep.cu).
__global__ void __launch_bounds__(1024) fox_cumsum(const float* __restrict__ log_f, int L, int Lp,
                                                   float* __restrict__ cum);

// Launch the per-chunk UT-prep kernel (and, when log_f is given, the FoX
// cumulative sum) for chunk size C, filling the workspace regions of `lay`.
cudaError_t launch_ut_prep(int dtype, int C, int d, const void* q, const void* k, const void* w, const float* beta,
                           const float* log_f, int BH, int L, unsigned char* ws, const FwdLayout& lay,
                           cudaStream_t st);

}  // namespace pathattn
