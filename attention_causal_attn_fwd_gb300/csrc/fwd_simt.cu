// PaTH causal attention forward on CUDA cores (fp32 arithmetic).
//
// Two kernels, following the blockwise algorithm of "Resumo Técnico: Atenção
// PaTH" (gist.science/pt/paper/2505.16381), §3 "Treinamento e Inferência
// Eficientes":
//
//  ut_prep_simt   — (ut_prep.cu) per chunk of C positions, the UT representation of the
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
#include "ut_prep.cuh"

namespace pathattn {

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
// MODE 0: PaTH; 1: PaTH-FoX (bias c_i - c_j from the log-gate cumsum);
// 2: relative-position bias rel[h][i - j] ([H, L] table).
template <typename T, int C, int D, int NT, int MODE>
__global__ void __launch_bounds__(NT) path_fwd_simt(const T* __restrict__ q, const T* __restrict__ k,
                                                    const T* __restrict__ v, const T* __restrict__ w,
                                                    const float* __restrict__ qhat,
                                                    const T* __restrict__ khat, const T* __restrict__ un,
                                                    const T* __restrict__ y, const T* __restrict__ zn,
                                                    const float* __restrict__ cum, const float* __restrict__ rel,
                                                    int H, T* __restrict__ o, float* __restrict__ lse, int L, int Lp,
                                                    float scale) {
    constexpr bool FOX = MODE == 1, REL = MODE == 2;
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
    const float* relh = REL ? rel + (size_t)(bh % H) * L : nullptr;  // this head's bias by distance

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
            if (REL) s += __ldg(relh + min(max(r - j, 0), L - 1)) * kLog2e;
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
                if (REL) s += __ldg(relh + min(r0 + r - c0 - j, L - 1)) * kLog2e;  // padding rows clamp
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
                               const float* log_f, const float* rel_bias, int H, void* o, float* lse, int BH, int L,
                               float scale, unsigned char* ws, const FwdLayout& lay, cudaStream_t st) {
    constexpr int NT = 256;
    const int nch = cdiv(L, C);
    cudaError_t e = launch_ut_prep(PATH_F32, C, D, q, k, w, beta, log_f, BH, L, ws, lay, st);
    if (e != cudaSuccess) return e;
    const T* tq = static_cast<const T*>(q);
    const T* tk = static_cast<const T*>(k);
    const T* tv = static_cast<const T*>(v);
    const T* tw = static_cast<const T*>(w);
    const float* qhat = reinterpret_cast<const float*>(ws + lay.qhat);
    const T* khat = reinterpret_cast<const T*>(ws + lay.khat);
    const T* un = reinterpret_cast<const T*>(ws + lay.un);
    const T* y = reinterpret_cast<const T*>(ws + lay.y);
    const T* zn = reinterpret_cast<const T*>(ws + lay.zn);
    const float* cum = reinterpret_cast<const float*>(ws + lay.cum);
    const size_t fsm = FwdSmem<T, C, D, NT>::bytes;
    auto kf = log_f ? path_fwd_simt<T, C, D, NT, 1> : rel_bias ? path_fwd_simt<T, C, D, NT, 2>
                                                               : path_fwd_simt<T, C, D, NT, 0>;
    e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fsm);
    if (e != cudaSuccess) return e;
    mark_start(st);
    kf<<<dim3(nch, BH), NT, fsm, st>>>(tq, tk, tv, tw, qhat, khat, un, y, zn, cum, rel_bias, H,
                                       static_cast<T*>(o), lse, L, lay.Lp, scale);
    mark_end(st);
    return cudaGetLastError();
}

// Chunk size of the CUDA-core path for head dimension d.
int simt_chunk(int d) { return d <= 16 ? 16 : 32; }

cudaError_t fwd_simt_f32(const void* q, const void* k, const void* v, const void* w, const float* beta,
                         const float* log_f, const float* rel_bias, int H, void* o, float* lse, int BH, int L, int d,
                         float scale, unsigned char* ws, const FwdLayout& lay, cudaStream_t st) {
#define PATH_SIMT_ARGS q, k, v, w, beta, log_f, rel_bias, H, o, lse, BH, L, scale, ws, lay, st
    switch (d) {
        case 16: return launch_simt<float, 16, 16>(PATH_SIMT_ARGS);
        case 32: return launch_simt<float, 32, 32>(PATH_SIMT_ARGS);
        case 64: return launch_simt<float, 32, 64>(PATH_SIMT_ARGS);
        case 128: return launch_simt<float, 32, 128>(PATH_SIMT_ARGS);
#undef PATH_SIMT_ARGS
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pathattn
