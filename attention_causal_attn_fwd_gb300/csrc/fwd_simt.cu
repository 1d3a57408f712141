// PaTH causal attention forward on CUDA cores (fp32 arithmetic).
//
// Two kernels, following the blockwise algorithm of "Resumo Técnico: Atenção
// PaTH" (gist.science/pt/paper/2505.16381), §3 "Treinamento e Inferência
// Eficientes":
//
//  ut_prep_simt   — per chunk of C positions, the UT representation of the
//                   chunk's transition product (§3 "Representação de
//                   Transformação UT"), P = H_0 ... H_{C-1} = I - W^T A W with
//                   A = (I + D triu_1(W W^T))^{-1} D, D = diag(beta) (the
//                   division-free form of I - W^T T^{-1} W); and from it the
//                   "boundary-adjusted" queries and keys (§3 "Algoritmo Estilo
//                   FlashAttention", first sub-bullet):
//                     qhat_i = H_start ... H_i q_i       = q_i - (Y W)_i
//                     khat_j = H_end ... H_{j+1} k_j     = k_j - (Z A W)_j
//                   with Y = tril(Q W^T) A^T and Z = triu_1(K W^T), plus the
//                   scan factor -U = -A^T W (so that P q = q - W^T (A W q),
//                   i.e. row-wise  q~ <- q~ + (q~ W^T)(-U)).
//  path_fwd_simt  — per query chunk n: the diagonal block from
//                   s_ij = q_i.k_j - Y_i.Z_j, then the right-to-left scan over
//                   key/value chunks m = n-1 ... 0 (second sub-bullet):
//                   S = q~ khat_m^T, online softmax, O += P V_m, and the query
//                   transport q~ <- P_m q~ = q~ + (q~ W_m^T)(-U_m).
//
// This is the fp32 path (no TF32) and the reference-quality path for small
// head dimensions.  The bf16 tensor-core path lives in fwd_tc.cu.
#include "common.cuh"
#include "simt_gemm.cuh"

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
                                                   T* __restrict__ y, T* __restrict__ zn, WsHeader* hdr) {
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
// sum_{s=j+1..i} log f_s), accumulated in fp64 and stored as fp32.
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
    for (int base = 0; base < Lp; base += 1024) {
        const int i = base + threadIdx.x;
        double x = i < L ? (double)src[i] : 0.0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            double y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) warp_tot[wid] = x;
        __syncthreads();
        if (wid == 0) {
            double t = warp_tot[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                double y = __shfl_up_sync(0xffffffffu, t, off);
                if (lane >= off) t += y;
            }
            warp_tot[lane] = t;
        }
        __syncthreads();
        const double carry = carry_s;
        x += carry + (wid > 0 ? warp_tot[wid - 1] : 0.0);
        if (i < Lp) dst[i] = (float)x;
        __syncthreads();
        if (threadIdx.x == 1023) carry_s = x;
        __syncthreads();
    }
}

template <typename T, int C, int D, int NT>
struct FwdSmem {
    static constexpr int LDT = D + 1;
    static constexpr int LDS = 2 * C + 1;
    static constexpr size_t bytes = 2 * (size_t)C * LDT * sizeof(float)   // sQt, sO
                                    + 4 * (size_t)C * LDT * sizeof(T)     // sK, sW, sV, sU
                                    + (size_t)C * LDS * sizeof(float)     // sS
                                    + 5 * C * sizeof(float);              // m, l, alpha, ci, cj
};

// One CTA per (query chunk, head).  Query chunks are visited longest-first.
template <typename T, int C, int D, int NT, bool FOX>
__global__ void __launch_bounds__(NT) path_fwd_simt(const T* __restrict__ q, const T* __restrict__ k,
                                                    const T* __restrict__ v, const T* __restrict__ w,
                                                    const float* __restrict__ qhat,
                                                    const T* __restrict__ khat, const T* __restrict__ un,
                                                    const T* __restrict__ y, const T* __restrict__ zn,
                                                    const float* __restrict__ cum, T* __restrict__ o,
                                                    float* __restrict__ lse, int L, int Lp, float scale) {
    using SM = FwdSmem<T, C, D, NT>;
    constexpr int LDT = SM::LDT, LDS = SM::LDS;
    constexpr int RG = NT / C;  // threads per row in the softmax
    static_assert(NT % C == 0 && RG <= 32 && (RG & (RG - 1)) == 0, "row groups");
    static_assert(C <= D, "Y/Z chunk blocks are staged in [C][D] buffers");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* sQt = reinterpret_cast<float*>(smem_raw);
    float* sO = sQt + C * LDT;
    T* sK = reinterpret_cast<T*>(sO + C * LDT);
    T* sW = sK + C * LDT;
    T* sV = sW + C * LDT;
    T* sU = sV + C * LDT;
    float* sS = reinterpret_cast<float*>(sU + C * LDT);
    float* sM = sS + C * LDS;
    float* sL = sM + C;
    float* sAl = sL + C;
    float* sCi = sAl + C;
    float* sCj = sCi + C;

    const int nchunks = gridDim.x;
    const int n = nchunks - 1 - blockIdx.x;  // longest first
    const int bh = blockIdx.y;
    const int r0 = n * C;
    const size_t hoff = (size_t)bh * L * D;
    const size_t woff = (size_t)bh * Lp;
    const float sl2 = scale * 1.4426950408889634f;  // logits in log2 units
    constexpr float kLog2e = 1.4426950408889634f;

    if (FOX)
        for (int i = threadIdx.x; i < C; i += NT) sCi[i] = cum[woff + r0 + i];

    // ---- diagonal block: s_ij = q_i.k_j - Y_i.Z_j  (j <= i within the chunk)
    load_rows<C, D, LDT, NT>(sQt, q + hoff, r0, L);
    load_rows<C, D, LDT, NT>(sK, k + hoff, r0, L);
    load_rows<C, D, LDT, NT>(sV, v + hoff, r0, L);
    load_rows<C, C, LDT, NT>(sU, y + woff * C, r0, Lp);   // Y
    load_rows<C, C, LDT, NT>(sW, zn + woff * C, r0, Lp);  // -Z
    __syncthreads();
    block_gemm<C, C, D, NT>([&](int m, int kk) { return sQt[m * LDT + kk]; },
                            [&](int kk, int nn) { return to_f<T>(sK[nn * LDT + kk]); },
                            [&](int m, int nn, float acc) { sS[m * LDS + nn] = acc; });
    block_gemm<C, C, C, NT>([&](int m, int kk) { return to_f<T>(sU[m * LDT + kk]); },
                            [&](int kk, int nn) { return to_f<T>(sW[nn * LDT + kk]); },
                            [&](int m, int nn, float acc) { sS[m * LDS + nn] += acc; });
    {
        const int r = threadIdx.x / RG, g = threadIdx.x % RG;
        float mx = -INFINITY;
        for (int j = g; j < C; j += RG) {
            float s = sS[r * LDS + j] * sl2;
            if (FOX) s += (sCi[r] - sCi[j]) * kLog2e;
            if (j > r) s = -INFINITY;
            sS[r * LDS + j] = s;
            mx = fmaxf(mx, s);
        }
#pragma unroll
        for (int off = RG / 2; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        float sum = 0.f;
        for (int j = g; j < C; j += RG) {
            float p = exp2f(sS[r * LDS + j] - mx);
            sS[r * LDS + j] = p;
            sum += p;
        }
#pragma unroll
        for (int off = RG / 2; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (g == 0) {
            sM[r] = mx;
            sL[r] = sum;
        }
    }
    __syncthreads();
    block_gemm<C, D, C, NT>([&](int m, int kk) { return sS[m * LDS + kk]; },
                            [&](int kk, int nn) { return to_f<T>(sV[kk * LDT + nn]); },
                            [&](int m, int nn, float acc) { sO[m * LDT + nn] = acc; });

    // ---- right-to-left scan over key/value chunks m = n-1 ... 0
    load_rows<C, D, LDT, NT>(sQt, qhat + woff * D, r0, Lp);
    __syncthreads();
    for (int mb = n - 1; mb >= 0; --mb) {
        const int c0 = mb * C;
        load_rows<C, D, LDT, NT>(sK, khat + woff * D, c0, Lp);
        load_rows<C, D, LDT, NT>(sW, w + hoff, c0, L);
        load_rows<C, D, LDT, NT>(sV, v + hoff, c0, L);
        load_rows<C, D, LDT, NT>(sU, un + woff * D, c0, Lp);
        if (FOX)
            for (int i = threadIdx.x; i < C; i += NT) sCj[i] = cum[woff + c0 + i];
        __syncthreads();
        // [S_k | S_w] = q~ [khat_m ; W_m]^T
        block_gemm<C, 2 * C, D, NT>(
            [&](int m, int kk) { return sQt[m * LDT + kk]; },
            [&](int kk, int nn) { return nn < C ? to_f<T>(sK[nn * LDT + kk]) : to_f<T>(sW[(nn - C) * LDT + kk]); },
            [&](int m, int nn, float acc) { sS[m * LDS + nn] = acc; });
        {
            const int r = threadIdx.x / RG, g = threadIdx.x % RG;
            float mx = -INFINITY;
            for (int j = g; j < C; j += RG) {
                float s = sS[r * LDS + j] * sl2;
                if (FOX) s += (sCi[r] - sCj[j]) * kLog2e;
                sS[r * LDS + j] = s;
                mx = fmaxf(mx, s);
            }
#pragma unroll
            for (int off = RG / 2; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_old = sM[r];
            const float m_new = fmaxf(m_old, mx);
            float sum = 0.f;
            for (int j = g; j < C; j += RG) {
                float p = exp2f(sS[r * LDS + j] - m_new);
                sS[r * LDS + j] = p;
                sum += p;
            }
#pragma unroll
            for (int off = RG / 2; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            __syncwarp();
            if (g == 0) {
                const float alpha = exp2f(m_old - m_new);
                sAl[r] = alpha;
                sL[r] = sL[r] * alpha + sum;
                sM[r] = m_new;
            }
        }
        __syncthreads();
        // O = alpha O + P V_m
        block_gemm<C, D, C, NT>([&](int m, int kk) { return sS[m * LDS + kk]; },
                                [&](int kk, int nn) { return to_f<T>(sV[kk * LDT + nn]); },
                                [&](int m, int nn, float acc) { sO[m * LDT + nn] = sAl[m] * sO[m * LDT + nn] + acc; });
        // q~ <- P_m q~ = q~ + S_w (-U_m)   (not needed after the last chunk)
        if (mb > 0)
            block_gemm<C, D, C, NT>([&](int m, int kk) { return sS[m * LDS + C + kk]; },
                                    [&](int kk, int nn) { return to_f<T>(sU[kk * LDT + nn]); },
                                    [&](int m, int nn, float acc) { sQt[m * LDT + nn] += acc; });
    }

    // ---- epilogue: o = O / l, lse = (m + log2 l) ln 2
    for (int idx = threadIdx.x; idx < C * D; idx += NT) {
        const int r = idx / D, c = idx % D;
        if (r0 + r < L) o[hoff + (size_t)(r0 + r) * D + c] = from_f<T>(sO[r * LDT + c] / sL[r]);
    }
    if (lse)
        for (int r = threadIdx.x; r < C; r += NT)
            if (r0 + r < L) lse[(size_t)bh * L + r0 + r] = (sM[r] + log2f(sL[r])) * 0.6931471805599453f;
}

// ----------------------------------------------------------------------------- host launchers
template <typename T, int C, int D>
static cudaError_t launch_simt(const void* q, const void* k, const void* v, const void* w, const float* beta,
                               const float* log_f, void* o, float* lse, int BH, int L, float scale,
                               unsigned char* ws, const FwdLayout& lay, cudaStream_t st) {
    constexpr int NT = 256;
    const int nch = cdiv(L, C);
    const T* tq = static_cast<const T*>(q);
    const T* tk = static_cast<const T*>(k);
    const T* tv = static_cast<const T*>(v);
    const T* tw = static_cast<const T*>(w);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    float* qhat = reinterpret_cast<float*>(ws + lay.qhat);
    T* khat = reinterpret_cast<T*>(ws + lay.khat);
    T* un = reinterpret_cast<T*>(ws + lay.un);
    T* y = reinterpret_cast<T*>(ws + lay.y);
    T* zn = reinterpret_cast<T*>(ws + lay.zn);
    float* cum = reinterpret_cast<float*>(ws + lay.cum);

    auto ut = ut_prep_simt<T, C, D, NT>;
    const size_t ut_smem = UtSmem<T, C, D, NT>::bytes;
    cudaError_t e = cudaFuncSetAttribute(ut, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ut_smem);
    if (e != cudaSuccess) return e;
    ut<<<dim3(nch, BH), NT, ut_smem, st>>>(tq, tk, tw, beta, L, lay.Lp, qhat, khat, un, y, zn, hdr);
    if (log_f) fox_cumsum<<<BH, 1024, 0, st>>>(log_f, L, lay.Lp, cum);

    const size_t fsm = FwdSmem<T, C, D, NT>::bytes;
    if (log_f) {
        auto kf = path_fwd_simt<T, C, D, NT, true>;
        e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fsm);
        if (e != cudaSuccess) return e;
        mark_start(st);
        kf<<<dim3(nch, BH), NT, fsm, st>>>(tq, tk, tv, tw, qhat, khat, un, y, zn, cum, static_cast<T*>(o), lse, L,
                                           lay.Lp, scale);
        mark_end(st);
    } else {
        auto kf = path_fwd_simt<T, C, D, NT, false>;
        e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fsm);
        if (e != cudaSuccess) return e;
        mark_start(st);
        kf<<<dim3(nch, BH), NT, fsm, st>>>(tq, tk, tv, tw, qhat, khat, un, y, zn, cum, static_cast<T*>(o), lse, L,
                                           lay.Lp, scale);
        mark_end(st);
    }
    return cudaGetLastError();
}

// Chunk size of the CUDA-core path for head dimension d.
int simt_chunk(int d) { return d <= 16 ? 16 : 32; }

cudaError_t fwd_simt_f32(const void* q, const void* k, const void* v, const void* w, const float* beta,
                         const float* log_f, void* o, float* lse, int BH, int L, int d, float scale,
                         unsigned char* ws, const FwdLayout& lay, cudaStream_t st) {
    switch (d) {
        case 16: return launch_simt<float, 16, 16>(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, lay, st);
        case 32: return launch_simt<float, 32, 32>(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, lay, st);
        case 64: return launch_simt<float, 32, 64>(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, lay, st);
        case 128: return launch_simt<float, 32, 128>(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, lay, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pathattn

namespace pathattn {
// bf16 inputs on the CUDA-core path (chunk 64); staging path until the
// tensor-core kernel covers bf16.
cudaError_t fwd_simt_bf16(const void* q, const void* k, const void* v, const void* w, const float* beta,
                          const float* log_f, void* o, float* lse, int BH, int L, int d, float scale,
                          unsigned char* ws, const FwdLayout& lay, cudaStream_t st) {
    switch (d) {
        case 64: return launch_simt<__nv_bfloat16, 64, 64>(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, lay, st);
        case 128: return launch_simt<__nv_bfloat16, 64, 128>(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, lay, st);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace pathattn
