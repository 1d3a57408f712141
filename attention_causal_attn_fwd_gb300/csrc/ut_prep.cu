// UT-transform preparation per chunk of C positions (fp32 arithmetic on CUDA cores).
//
// "Resumo Técnico: Atenção PaTH" (gist.science/pt/paper/2505.16381), §3
// "Representação de Transformação UT": the product of a chunk's transitions,
// P = H_0 ... H_{C-1}, is written compactly as I - W^T A W with
//     A = (I + D triu_1(W W^T))^{-1} D,   D = diag(beta),
// the division-free form of I - W^T T^{-1} W (T = D^{-1} + triu_1(W W^T),
// triangular and built from beta).  §3 "Algoritmo Estilo FlashAttention",
// first sub-bullet: from A the kernel derives the chunk's boundary-adjusted
// queries and keys,
//     qhat_i = H_start ... H_i q_i   = q_i - (Y W)_i,    Y = tril(Q W^T) A^T
//     khat_j = H_end ... H_{j+1} k_j = k_j - (Z A W)_j,  Z = triu_1(K W^T)
// and the scan factor -U = -A^T W, so that the query transport through the
// whole chunk is  q~ <- P q~ = q~ + (q~ W^T)(-U)  row-wise.  The diagonal
// block's logits are q_i.k_j - Y_i.Z_j (j <= i).
#include "common.cuh"
#include "ut_prep.cuh"
#include "simt_gemm.cuh"

namespace pathattn {

cudaError_t launch_ut_prep_tc(int d, const void* q, const void* k, const void* w, const float* beta, int BH, int L,
                              unsigned char* ws, const FwdLayout& lay, bool want_kmax, cudaStream_t st,
                              bool reset_header = true);

template <typename T, int C, int D, int NT>
struct UtSmem {
    static constexpr int LDT = D + 1;  // T arrays [C][D]
    static constexpr int LDF = C + 1;  // float arrays [C][C]
    static constexpr size_t bytes = 2 * (size_t)C * LDT * sizeof(T) + 2 * (size_t)C * LDF * sizeof(float) +
                                    C * sizeof(float);
};

template <typename T, int C, int D, int NT>
__global__ void __launch_bounds__(NT) ut_prep_simt(const T* __restrict__ q, const T* __restrict__ k,
                                                   const T* __restrict__ w, const float* __restrict__ beta,
                                                   int L, int Lp, float* __restrict__ qhat,
                                                   T* __restrict__ khat, T* __restrict__ un,
                                                   T* __restrict__ y, T* __restrict__ zn, T* __restrict__ vfac,
                                                   WsHeader* hdr) {
    using SM = UtSmem<T, C, D, NT>;
    constexpr int LDT = SM::LDT, LDF = SM::LDF;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* sW = reinterpret_cast<T*>(smem_raw);
    T* sX = sW + C * LDT;
    float* sA = reinterpret_cast<float*>(sX + C * LDT);
    float* sY = sA + C * LDF;
    float* sBeta = sY + C * LDF;

    const int chunk = blockIdx.x, bh = blockIdx.y;
    const int r0 = chunk * C;
    if (chunk == 0 && bh == 0 && threadIdx.x == 0) hdr->status = 0;
    const T* qh = q + (size_t)bh * L * D;
    const T* kh = k + (size_t)bh * L * D;
    const T* wh = w + (size_t)bh * L * D;
    const size_t wrow = (size_t)bh * Lp + r0;  // first workspace row of this chunk

    load_rows<C, D, LDT, NT>(sW, wh, r0, L);
    for (int i = threadIdx.x; i < C; i += NT) sBeta[i] = (r0 + i < L) ? beta[(size_t)bh * L + r0 + i] : 0.f;
    __syncthreads();

    // G = W W^T, strictly upper part kept (N = triu_1(G)).
    block_gemm<C, C, D, NT>([&](int m, int kk) { return to_f<T>(sW[m * LDT + kk]); },
                            [&](int kk, int n) { return to_f<T>(sW[n * LDT + kk]); },
                            [&](int m, int n, float acc) { sA[m * LDF + n] = n > m ? acc : 0.f; });

    // A = (I + D N)^{-1} D, rows from the bottom:  A_ii = beta_i,
    // A_ij = -beta_i sum_{k=i+1}^{j} G_ik A_kj  (j > i), in place over G's rows.
    {
        constexpr int P = NT / C >= 1 ? NT / C : 1;  // threads per column
        const int j = threadIdx.x / P, p = threadIdx.x % P;
        for (int i = C - 1; i >= 0; --i) {
            float acc = 0.f;
            if (j < C && j > i)
                for (int kk = i + 1 + p; kk <= j; kk += P) acc = fmaf(sA[i * LDF + kk], sA[kk * LDF + j], acc);
#pragma unroll
            for (int off = P / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            __syncthreads();
            if (j < C && p == 0) sA[i * LDF + j] = j > i ? -sBeta[i] * acc : (j == i ? sBeta[i] : 0.f);
            __syncthreads();
        }
    }

    // -U = -A^T W
    block_gemm<C, D, C, NT>([&](int m, int kk) { return sA[kk * LDF + m]; },
                            [&](int kk, int n) { return to_f<T>(sW[kk * LDT + n]); },
                            [&](int m, int n, float acc) { un[(wrow + m) * D + n] = from_f<T>(-acc); });
    // V = A W (key-side transport factor, prefill cache only)
    if (vfac)
        block_gemm<C, D, C, NT>([&](int m, int kk) { return sA[m * LDF + kk]; },
                                [&](int kk, int n) { return to_f<T>(sW[kk * LDT + n]); },
                                [&](int m, int n, float acc) { vfac[(wrow + m) * D + n] = from_f<T>(acc); });

    // Queries: Y' = tril(Q W^T), Y = Y' A^T, qhat = Q - Y W.
    load_rows<C, D, LDT, NT>(sX, qh, r0, L);
    __syncthreads();
    block_gemm<C, C, D, NT>([&](int m, int kk) { return to_f<T>(sX[m * LDT + kk]); },
                            [&](int kk, int n) { return to_f<T>(sW[n * LDT + kk]); },
                            [&](int m, int n, float acc) { sY[m * LDF + n] = n <= m ? acc : 0.f; });
    block_gemm<C, C, C, NT>([&](int m, int kk) { return sY[m * LDF + kk]; },
                            [&](int kk, int n) { return sA[n * LDF + kk]; },
                            [&](int m, int n, float acc) {
                                sY[m * LDF + n] = acc;
                                y[(wrow + m) * C + n] = from_f<T>(acc);
                            });
    block_gemm<C, D, C, NT>([&](int m, int kk) { return sY[m * LDF + kk]; },
                            [&](int kk, int n) { return to_f<T>(sW[kk * LDT + n]); },
                            [&](int m, int n, float acc) {
                                qhat[(wrow + m) * D + n] = to_f<T>(sX[m * LDT + n]) - acc;
                            });

    // Keys: Z = triu_1(K W^T), khat = K - (Z A) W.
    load_rows<C, D, LDT, NT>(sX, kh, r0, L);
    __syncthreads();
    block_gemm<C, C, D, NT>([&](int m, int kk) { return to_f<T>(sX[m * LDT + kk]); },
                            [&](int kk, int n) { return to_f<T>(sW[n * LDT + kk]); },
                            [&](int m, int n, float acc) {
                                const float z = n > m ? acc : 0.f;
                                sY[m * LDF + n] = z;
                                zn[(wrow + m) * C + n] = from_f<T>(-z);
                            });
    block_gemm<C, C, C, NT>([&](int m, int kk) { return sY[m * LDF + kk]; },
                            [&](int kk, int n) { return sA[kk * LDF + n]; },
                            [&](int m, int n, float acc) { sY[m * LDF + n] = acc; });
    block_gemm<C, D, C, NT>([&](int m, int kk) { return sY[m * LDF + kk]; },
                            [&](int kk, int n) { return to_f<T>(sW[kk * LDT + n]); },
                            [&](int m, int n, float acc) {
                                khat[(wrow + m) * D + n] = from_f<T>(to_f<T>(sX[m * LDT + n]) - acc);
                            });
}

// Inclusive cumulative sum of log f per head (PaTH-FoX bias c_i - c_j =
// sum_{s=j+1..i} log f_s), accumulated in fp64 and stored as fp32 for every
// position below Lp (positions >= L add zero).  One CTA per head walks the head
// in segments of 1024 x kCumRun positions: each thread sums its run of kCumRun
// consecutive positions serially, the run totals are scanned across the CTA
// (warp shuffles, then the 32 warp totals), and each thread writes its run with
// the prefix and the carry of the earlier segments.
constexpr int kCumRun = 16;
__global__ void __launch_bounds__(1024) fox_cumsum(const float* __restrict__ log_f, int L, int Lp,
                                                   float* __restrict__ cum) {
    __shared__ double warp_tot[32];
    __shared__ double carry_s;
    const int bh = blockIdx.x;
    const float* src = log_f + (size_t)bh * L;
    float* dst = cum + (size_t)bh * Lp;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry_s = 0.0;
    __syncthreads();
    for (int base = 0; base < Lp; base += 1024 * kCumRun) {
        const int i0 = base + (int)threadIdx.x * kCumRun;
        double run[kCumRun];
        double acc = 0.0;
#pragma unroll
        for (int e = 0; e < kCumRun; ++e) {
            acc += i0 + e < L ? (double)src[i0 + e] : 0.0;
            run[e] = acc;
        }
        double x = acc;  // inclusive scan of the run totals over the CTA
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) warp_tot[wid] = x;
        __syncthreads();
        if (wid == 0) {
            double t = warp_tot[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const double y = __shfl_up_sync(0xffffffffu, t, off);
                if (lane >= off) t += y;
            }
            warp_tot[lane] = t;
        }
        __syncthreads();
        const double prefix = carry_s + (wid > 0 ? warp_tot[wid - 1] : 0.0) + (x - acc);
#pragma unroll
        for (int e = 0; e < kCumRun; ++e)
            if (i0 + e < Lp) dst[i0 + e] = (float)(prefix + run[e]);
        __syncthreads();
        if (threadIdx.x == 1023) carry_s = prefix + acc;
        __syncthreads();
    }
}


template <typename T, int C, int D>
static cudaError_t launch_ut_t(const void* q, const void* k, const void* w, const float* beta, const float* log_f,
                               int BH, int L, unsigned char* ws, const FwdLayout& lay, cudaStream_t st) {
    constexpr int NT = 256;
    auto ut = ut_prep_simt<T, C, D, NT>;
    const size_t smem = UtSmem<T, C, D, NT>::bytes;
    cudaError_t e = cudaFuncSetAttribute(ut, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ut<<<dim3(cdiv(L, C), BH), NT, smem, st>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(w), beta, L, lay.Lp,
        reinterpret_cast<float*>(ws + lay.qhat), reinterpret_cast<T*>(ws + lay.khat), reinterpret_cast<T*>(ws + lay.un),
        reinterpret_cast<T*>(ws + lay.y), reinterpret_cast<T*>(ws + lay.zn),
        lay.vfac ? reinterpret_cast<T*>(ws + lay.vfac) : nullptr, reinterpret_cast<WsHeader*>(ws));
    if (log_f) fox_cumsum<<<BH, 1024, 0, st>>>(log_f, L, lay.Lp, reinterpret_cast<float*>(ws + lay.cum));
    return cudaGetLastError();
}

cudaError_t launch_ut_prep(int dtype, int C, int d, const void* q, const void* k, const void* w, const float* beta,
                           const float* log_f, int BH, int L, unsigned char* ws, const FwdLayout& lay,
                           cudaStream_t st) {
    if (dtype == PATH_F32) {
        if (C == 16 && d == 16) return launch_ut_t<float, 16, 16>(q, k, w, beta, log_f, BH, L, ws, lay, st);
        if (C == 32 && d == 32) return launch_ut_t<float, 32, 32>(q, k, w, beta, log_f, BH, L, ws, lay, st);
        if (C == 32 && d == 64) return launch_ut_t<float, 32, 64>(q, k, w, beta, log_f, BH, L, ws, lay, st);
        if (C == 32 && d == 128) return launch_ut_t<float, 32, 128>(q, k, w, beta, log_f, BH, L, ws, lay, st);
    } else if (C == 128) {  // bf16: tensor-core UT prep (ut_prep_tc.cu)
        cudaError_t e = launch_ut_prep_tc(d, q, k, w, beta, BH, L, ws, lay, log_f != nullptr, st);
        if (e == cudaSuccess && log_f)
            fox_cumsum<<<BH, 1024, 0, st>>>(log_f, L, lay.Lp, reinterpret_cast<float*>(ws + lay.cum));
        return e == cudaSuccess ? cudaGetLastError() : e;
    }
    return cudaErrorInvalidValue;
}

}  // namespace pathattn
