// PaTH forward with value-side transport, on CUDA cores (fp32 arithmetic).
//
// "Resumo Técnico: Por que Transformações Acumuladas Extrapolam?"
// (gist.science/pt/paper/2606.24975), §"Metodologia" 1: the route transport
// P_{j->i} is the product of the per-token steps from source j to query i;
// §"Principais Contribuições" 3 "Proteção do Lado de Valor": the same
// accumulated transport is applied to the values.  With the PaTH steps
// H_s = I - beta_s w_s w_s^T ("Resumo Técnico: Atenção PaTH", §2 "Mecanismo
// Central") the route operator of the logit is H_i ... H_{j+1}, so
//     o_i = sum_j softmax_j(s_i.) H_i ... H_{j+1} v_j,
// with the PaTH(-FoX) logits s_ij = scale k_j^T H_{j+1} ... H_i q_i (+ bias).
//
// One warp per query row, two walks over the row's keys:
//   1. right to left, the query carried backwards (u <- H_j u): the logits,
//      kept in shared memory (so L is bounded by the shared memory);
//   2. left to right, the output accumulated along the route
//      (acc <- H_j acc + alpha_ij v_j), which leaves o_i = acc.
// Each step is a d-vector update with a warp reduction, so the kernel is
// bound by the reduction latency: it is the direct, unblocked form of the
// operator (a blockwise tensor-core version would carry per-chunk d x d route
// products, which this library does not implement).  No waits, no barriers
// between warps.
#include "common.cuh"

namespace pathattn {

constexpr int kVtWarps = 4;
constexpr int kVtMaxL = 8192;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}
__device__ __forceinline__ float2 warp_sum2(float2 x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        x.x += __shfl_xor_sync(0xffffffffu, x.x, off);
        x.y += __shfl_xor_sync(0xffffffffu, x.y, off);
    }
    return x;
}

// grid (ceil(L / kVtWarps), B*H), kVtWarps warps; warp = one query row.
// Element c = 32 e + lane of a row (e < E = ceil(D / 32); lanes beyond D idle).
template <typename T, int D>
__global__ void __launch_bounds__(32 * kVtWarps) path_fwd_vt_rows(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, const T* __restrict__ w,
    const float* __restrict__ beta, const float* __restrict__ log_f, T* __restrict__ o, float* __restrict__ lse,
    int L, float scale, WsHeader* hdr) {
    constexpr int E = (D + 31) / 32;
    extern __shared__ float s_all[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y;
    const int i = blockIdx.x * kVtWarps + warp;
    if (blockIdx.x == 0 && bh == 0 && threadIdx.x == 0) hdr->status = 0;
    if (i >= L) return;
    float* s = s_all + (size_t)warp * L;
    const size_t hoff = (size_t)bh * L;
    const T* kh = k + hoff * D;
    const T* vh = v + hoff * D;
    const T* wh = w + hoff * D;
    const float* bh_beta = beta + hoff;
    const float* lf = log_f ? log_f + hoff : nullptr;
    auto ld = [&](const T* row, int e) -> float {
        const int c = 32 * e + lane;
        return c < D ? to_f<T>(row[c]) : 0.f;
    };
    // rows of this head read or written below lie inside the [B*H, L, D] tensors (checked in
    // the bounds-checked build only)
    const long long n_rows = (long long)gridDim.y * L;
    auto row_ok = [&](int j, int site) { return in_bounds((long long)(hoff + j) * D, D, n_rows * D, hdr, site); };
    if (!row_ok(i, 224) || !in_bounds((long long)hoff, i + 1, n_rows, hdr, 225)) return;

    // walk 1: logits, the query carried backwards through H_i, H_{i-1}, ...
    float u[E];
#pragma unroll
    for (int e = 0; e < E; ++e) u[e] = ld(q + (hoff + i) * D, e);
    float bias = 0.f;  // sum_{s=j+1..i} log f_s
    for (int j = i; j >= 0; --j) {
        if (!row_ok(j, 226)) break;
        float2 part = make_float2(0.f, 0.f);
        float wj[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            wj[e] = ld(wh + (size_t)j * D, e);
            part.x = fmaf(ld(kh + (size_t)j * D, e), u[e], part.x);
            part.y = fmaf(wj[e], u[e], part.y);
        }
        part = warp_sum2(part);
        if (lane == 0) s[j] = scale * part.x + bias;
        const float t = bh_beta[j] * part.y;
#pragma unroll
        for (int e = 0; e < E; ++e) u[e] = fmaf(-t, wj[e], u[e]);
        if (lf) bias += lf[j];
    }
    __syncwarp();
    float m = -INFINITY;
    for (int j = lane; j <= i; j += 32) m = fmaxf(m, s[j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float l = 0.f;
    for (int j = lane; j <= i; j += 32) l += expf(s[j] - m);
    l = warp_sum(l);
    const float inv_l = 1.f / l;

    // walk 2: the output carried forward along the route
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    for (int j = 0; j <= i; ++j) {
        if (!row_ok(j, 227)) break;
        float wj[E];
        if (j > 0) {
            float part = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                wj[e] = ld(wh + (size_t)j * D, e);
                part = fmaf(wj[e], acc[e], part);
            }
            const float t = bh_beta[j] * warp_sum(part);
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = fmaf(-t, wj[e], acc[e]);
        }
        const float a = expf(s[j] - m) * inv_l;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(a, ld(vh + (size_t)j * D, e), acc[e]);
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int c = 32 * e + lane;
        if (c < D) o[(hoff + i) * D + c] = from_f<T>(acc[e]);
    }
    if (lse && lane == 0) lse[hoff + i] = m + logf(l);
}

bool fwd_vt_supported(int d, int L) { return (d == 16 || d == 32 || d == 64 || d == 128) && L <= kVtMaxL; }

template <typename T, int D>
static cudaError_t launch_vt(const void* q, const void* k, const void* v, const void* w, const float* beta,
                             const float* log_f, void* o, float* lse, int BH, int L, float scale, unsigned char* ws,
                             cudaStream_t st) {
    auto kern = path_fwd_vt_rows<T, D>;
    const size_t smem = (size_t)kVtWarps * L * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    mark_start(st);
    kern<<<dim3(cdiv(L, kVtWarps), BH), 32 * kVtWarps, smem, st>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), static_cast<const T*>(w),
        beta, log_f, static_cast<T*>(o), lse, L, scale, reinterpret_cast<WsHeader*>(ws));
    mark_end(st);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_vt_d(int d, const void* q, const void* k, const void* v, const void* w, const float* beta,
                               const float* log_f, void* o, float* lse, int BH, int L, float scale,
                               unsigned char* ws, cudaStream_t st) {
    switch (d) {
        case 16: return launch_vt<T, 16>(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, st);
        case 32: return launch_vt<T, 32>(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, st);
        case 64: return launch_vt<T, 64>(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, st);
        case 128: return launch_vt<T, 128>(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t fwd_vt(int dtype, int d, const void* q, const void* k, const void* v, const void* w, const float* beta,
                   const float* log_f, void* o, float* lse, int BH, int L, float scale, unsigned char* ws,
                   cudaStream_t st) {
    if (dtype == PATH_F32) return launch_vt_d<float>(d, q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, st);
    return launch_vt_d<__nv_bfloat16>(d, q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, st);
}

}  // namespace pathattn
