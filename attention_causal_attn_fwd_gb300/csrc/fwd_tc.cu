// bf16 forward entry (staging: routes to the CUDA-core kernel at chunk 64).
#include "common.cuh"

namespace pathattn {
cudaError_t fwd_simt_bf16(const void* q, const void* k, const void* v, const void* w, const float* beta,
                          const float* log_f, void* o, float* lse, int BH, int L, int d, float scale,
                          unsigned char* ws, const FwdLayout& lay, cudaStream_t st);
int tc_chunk(int d) { (void)d; return 64; }
bool tc_supported(int d) { return d == 64 || d == 128; }
cudaError_t fwd_tc_bf16(const void* q, const void* k, const void* v, const void* w, const float* beta,
                        const float* log_f, void* o, float* lse, int BH, int L, int d, float scale,
                        unsigned char* ws, const FwdLayout& lay, int fault_mask, cudaStream_t st) {
    (void)fault_mask;
    return fwd_simt_bf16(q, k, v, w, beta, log_f, o, lse, BH, L, d, scale, ws, lay, st);
}
}  // namespace pathattn
