// Prefill -> decode hand-off: the transported key cache of a whole prompt.
//
// "Resumo Técnico: Atenção PaTH" (gist.science/pt/paper/2505.16381), §3
// "Inferência": during decoding the cache holds keys updated in place by
// every later transition.  After a prompt of L tokens the cache must hold
//     k~_j = H_{L-1} H_{L-2} ... H_{j+1} k_j          (j < L),
// exactly what token-by-token decoding from an empty cache would leave.
//
// With chunks of C positions and the UT representation of each chunk's
// product P_c = H_start ... H_end = I - W_c^T A_c W_c (§3 "Representação de
// Transformação UT"), a key of chunk m is first transported to its chunk end,
// khat_j = H_end ... H_{j+1} k_j (from the UT prep), then through every later
// chunk in order:  k~_j = P_last^T ... P_{m+1}^T khat_j.  Row-wise,
//     r <- r P_c = r - (r W_c^T)(A_c W_c) = r - (r W_c^T) V_c,
// a left-to-right scan over later chunks with the factor V_c = A_c W_c, which
// the UT prep writes when asked to.  This kernel runs that scan on CUDA cores
// in fp32 (one CTA per key chunk and head); it serves fp32 and bf16 at d = 64.
// bf16 at d = 128 uses the tensor-core suffix-product form (prefill_tc.cu).
#include "common.cuh"
#include "simt_gemm.cuh"
#include "ut_prep.cuh"

namespace pathattn {

template <typename T, int C, int D, int NT>
struct PrefillSmem {
    static constexpr int LDT = D + 1, LDS = C + 1;
    static constexpr size_t bytes = (size_t)C * LDT * sizeof(float) + 2 * (size_t)C * LDT * sizeof(T) +
                                    (size_t)C * LDS * sizeof(float);
};

template <typename T, int C, int D, int NT>
__global__ void __launch_bounds__(NT) prefill_key_transport(const T* __restrict__ w, const T* __restrict__ khat,
                                                            const T* __restrict__ vfac, T* __restrict__ kcache,
                                                            int L, int Lp, int n_max) {
    using SM = PrefillSmem<T, C, D, NT>;
    constexpr int LDT = SM::LDT, LDS = SM::LDS;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* sR = reinterpret_cast<float*>(smem_raw);
    T* sW = reinterpret_cast<T*>(sR + C * LDT);
    T* sV = sW + C * LDT;
    float* sS = reinterpret_cast<float*>(sV + C * LDT);

    const int m = blockIdx.x, bh = blockIdx.y;  // m = 0 has the most later chunks: launched first
    const int nch = gridDim.x;
    const size_t woff = (size_t)bh * Lp;
    load_rows<C, D, LDT, NT>(sR, khat + woff * D, m * C, Lp);
    for (int c = m + 1; c < nch; ++c) {
        load_rows<C, D, LDT, NT>(sW, w + (size_t)bh * L * D, c * C, L);
        load_rows<C, D, LDT, NT>(sV, vfac + woff * D, c * C, Lp);
        __syncthreads();
        // S = R W_c^T
        block_gemm<C, C, D, NT>([&](int i, int kk) { return sR[i * LDT + kk]; },
                                [&](int kk, int n) { return to_f<T>(sW[n * LDT + kk]); },
                                [&](int i, int n, float acc) { sS[i * LDS + n] = acc; });
        // R <- R - S V_c
        block_gemm<C, D, C, NT>([&](int i, int kk) { return sS[i * LDS + kk]; },
                                [&](int kk, int n) { return to_f<T>(sV[kk * LDT + n]); },
                                [&](int i, int n, float acc) { sR[i * LDT + n] -= acc; });
    }
    T* dst = kcache + (size_t)bh * n_max * D;
    for (int idx = threadIdx.x; idx < C * D; idx += NT) {
        const int r = idx / D, c = idx % D;
        const int j = m * C + r;
        if (j < L) dst[(size_t)j * D + c] = from_f<T>(sR[r * LDT + c]);
    }
}

template <typename T, int C, int D>
static cudaError_t launch_prefill_t(const void* w, void* kcache, int BH, int L, int n_max, unsigned char* ws,
                                    const FwdLayout& lay, cudaStream_t st) {
    constexpr int NT = 256;
    auto kern = prefill_key_transport<T, C, D, NT>;
    const size_t smem = PrefillSmem<T, C, D, NT>::bytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    mark_start(st);
    kern<<<dim3(cdiv(L, C), BH), NT, smem, st>>>(static_cast<const T*>(w), reinterpret_cast<const T*>(ws + lay.khat),
                                               reinterpret_cast<const T*>(ws + lay.vfac), static_cast<T*>(kcache), L,
                                               lay.Lp, n_max);
    mark_end(st);
    return cudaGetLastError();
}

// Tensor-core suffix-product transport for bf16, d = 128 (prefill_tc.cu).
cudaError_t launch_prefill_tc(const void* w, void* kcache, int BH, int L, int n_max, unsigned char* ws,
                              const FwdLayout& lay, cudaStream_t st);

// UT prep (with the V factor) followed by the key transport.  C is the
// dtype's forward chunk size; the prompt's q is not needed, k stands in for it.
cudaError_t prefill_kcache(int dtype, int C, int d, const void* k, const void* w, const float* beta, void* kcache,
                           int BH, int L, int n_max, unsigned char* ws, const FwdLayout& lay, cudaStream_t st) {
    cudaError_t e = launch_ut_prep(dtype, C, d, k, k, w, beta, nullptr, BH, L, ws, lay, st);
    if (e != cudaSuccess) return e;
    using bf = __nv_bfloat16;
    if (dtype == PATH_F32) {
        if (C == 16 && d == 16) return launch_prefill_t<float, 16, 16>(w, kcache, BH, L, n_max, ws, lay, st);
        if (C == 32 && d == 32) return launch_prefill_t<float, 32, 32>(w, kcache, BH, L, n_max, ws, lay, st);
        if (C == 32 && d == 64) return launch_prefill_t<float, 32, 64>(w, kcache, BH, L, n_max, ws, lay, st);
        if (C == 32 && d == 128) return launch_prefill_t<float, 32, 128>(w, kcache, BH, L, n_max, ws, lay, st);
    } else {
        if (C == 128 && d == 64) return launch_prefill_t<bf, 128, 64>(w, kcache, BH, L, n_max, ws, lay, st);
        if (C == 128 && d == 128) return launch_prefill_tc(w, kcache, BH, L, n_max, ws, lay, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pathattn
