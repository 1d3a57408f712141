// The two CUDA-core stages of the blockwise value-transport forward (bf16,
// d = 128, chunks of 128); the tensor-core stages are the UT prep and the scan
// (csrc/ut_prep_tc.cu, csrc/fwd_tc.cu, fwd_tc_vt_bf16).
//
// "Resumo Técnico: Por que Transformações Acumuladas Extrapolam?", §"Principais
// Contribuições" 3: o_i = sum_j alpha_ij H_i ... H_{j+1} v_j with the PaTH steps
// H_s = I - beta_s w_s w_s^T ("Resumo Técnico: Atenção PaTH", §2 "Mecanismo
// Central"), blocked as in that page's §3 "Algoritmo Estilo FlashAttention".
// With P_c = H_{e_c} ... H_{b_c} the transition of chunk c and vhat_j the value
// moved to the end of its chunk:
//   vt_value_chain  Vtil_{n,m} = Vhat_m (P_{n-1} ... P_{m+1})^T for every pair m < n:
//                   row j of it is v_j carried to the position just before chunk n;
//   vt_diag_walks   o_i = H_i ... H_b X_i + sum_{b <= j <= i} alpha_ij H_i ... H_{j+1} v_j,
//                   X_i = sum_{j < b} alpha_ij (row j of Vtil_{n,m(j)}) from the scan,
//                   alpha_ij = exp(s_ij - lse_i) with the scan's LSE.
#include "common.cuh"

namespace pathattn {

namespace {

constexpr int kVcC = 128;  // chunk (= d)
constexpr int kVcLd = kVcC + 4;
constexpr int kVcThreads = 256;
constexpr size_t kVcSmem = 2 * kVcC * kVcLd * sizeof(float);

__device__ __forceinline__ long long pair_index(int n, int m) { return (long long)n * (n - 1) / 2 + m; }

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&p);
}
__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// grid (B*H, N - 1), 256 threads; CTA (bh, m) runs the chain of key chunk m (N - 2 - m
// products), so the longest chains, of every head, are launched first.
// Vtil is kept transposed in shared memory (VT[k][i] = Vtil[i][k], fp32) so that
// each thread's 8 x 8 output tile reads 8 consecutive floats of each operand row.
// P_c^T = I + (P - I) as the UT prep stores it (its row k, column c is entry
// (k, c) of P_c^T - I), so one step is Vtil += Vtil (P - I).
__global__ void __launch_bounds__(kVcThreads, 1)
    vt_value_chain(const __nv_bfloat16* __restrict__ vhat, const __nv_bfloat16* __restrict__ pmi,
                   __nv_bfloat16* __restrict__ pairs, int Lp, int N, long long pair_rows) {
    extern __shared__ float vc_smem[];
    float* VT = vc_smem;                // [k][i]
    float* PM = vc_smem + kVcC * kVcLd;  // [k][c]
    const int bh = blockIdx.x, m = blockIdx.y;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    if (m >= N - 1) return;
    const __nv_bfloat16* vh = vhat + ((size_t)bh * Lp + (size_t)m * kVcC) * kVcC;
    __nv_bfloat16* ph = pairs + (size_t)bh * (size_t)pair_rows * kVcC;
    {  // Vtil_{m+1,m} = Vhat_m: to the pair store as it is, and transposed to fp32
        __nv_bfloat16* dst = ph + (size_t)pair_index(m + 1, m) * kVcC * kVcC;
        for (int idx = tid; idx < kVcC * 16; idx += kVcThreads) {
            const int i = idx >> 4, g = idx & 15;
            const uint4 raw = *reinterpret_cast<const uint4*>(vh + (size_t)i * kVcC + 8 * g);
            *reinterpret_cast<uint4*>(dst + (size_t)i * kVcC + 8 * g) = raw;
            const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                VT[(8 * g + 2 * e) * kVcLd + i] = bf_lo(w4[e]);
                VT[(8 * g + 2 * e + 1) * kVcLd + i] = bf_hi(w4[e]);
            }
        }
    }
    for (int n = m + 1; n <= N - 2; ++n) {  // Vtil_{n+1,m} = Vtil_{n,m} P_n^T
        const __nv_bfloat16* pm = pmi + ((size_t)bh * Lp + (size_t)n * kVcC) * kVcC;
        for (int idx = tid; idx < kVcC * 16; idx += kVcThreads) {
            const int k = idx >> 4, g = idx & 15;
            const uint4 raw = *reinterpret_cast<const uint4*>(pm + (size_t)k * kVcC + 8 * g);
            float4* d4 = reinterpret_cast<float4*>(PM + k * kVcLd + 8 * g);
            d4[0] = make_float4(bf_lo(raw.x), bf_hi(raw.x), bf_lo(raw.y), bf_hi(raw.y));
            d4[1] = make_float4(bf_lo(raw.z), bf_hi(raw.z), bf_lo(raw.w), bf_hi(raw.w));
        }
        __syncthreads();
        float acc[8][8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[r][q] = 0.f;
#pragma unroll 4
        for (int k = 0; k < kVcC; ++k) {
            const float4 a0 = *reinterpret_cast<const float4*>(VT + k * kVcLd + 8 * ty);
            const float4 a1 = *reinterpret_cast<const float4*>(VT + k * kVcLd + 8 * ty + 4);
            const float4 b0 = *reinterpret_cast<const float4*>(PM + k * kVcLd + 8 * tx);
            const float4 b1 = *reinterpret_cast<const float4*>(PM + k * kVcLd + 8 * tx + 4);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[r][q] = fmaf(a[r], b[q], acc[r][q]);
        }
        __syncthreads();  // every read of Vtil_{n,m} is done
        __nv_bfloat16* dst = ph + (size_t)pair_index(n + 1, m) * kVcC * kVcC;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int i = 8 * ty + r;
            float v8[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int c = 8 * tx + q;
                v8[q] = VT[c * kVcLd + i] + acc[r][q];
                VT[c * kVcLd + i] = v8[q];
            }
            uint4 o;
            o.x = pack_bf16x2_rn(v8[0], v8[1]);
            o.y = pack_bf16x2_rn(v8[2], v8[3]);
            o.z = pack_bf16x2_rn(v8[4], v8[5]);
            o.w = pack_bf16x2_rn(v8[6], v8[7]);
            *reinterpret_cast<uint4*>(dst + (size_t)i * kVcC + 8 * tx) = o;
        }
        __syncthreads();
    }
}

// ----------------------------------------------------------------------------- diagonal walks
constexpr int kDwRows = 4;   // query rows per warp, in lockstep
constexpr int kDwWarps = 8;

// Sums 8 values over the warp; every lane returns the total of value (lane >> 2) & 7.
__device__ __forceinline__ float dw_sum_8(const float (&x)[8], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float y[4], z[2];
#pragma unroll
    for (int v = 0; v < 4; ++v)
        y[v] = (b4 ? x[v + 4] : x[v]) + __shfl_xor_sync(0xffffffffu, b4 ? x[v] : x[v + 4], 16);
#pragma unroll
    for (int v = 0; v < 2; ++v)
        z[v] = (b3 ? y[v + 2] : y[v]) + __shfl_xor_sync(0xffffffffu, b3 ? y[v] : y[v + 2], 8);
    float a = (b2 ? z[1] : z[0]) + __shfl_xor_sync(0xffffffffu, b2 ? z[0] : z[1], 4);
    a += __shfl_xor_sync(0xffffffffu, a, 2);
    a += __shfl_xor_sync(0xffffffffu, a, 1);
    return a;
}
// Sums 4 values over the warp; every lane returns the total of value (lane >> 3) & 3.
__device__ __forceinline__ float dw_sum_4(const float (&x)[4], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8;
    float y[2];
#pragma unroll
    for (int v = 0; v < 2; ++v)
        y[v] = (b4 ? x[v + 2] : x[v]) + __shfl_xor_sync(0xffffffffu, b4 ? x[v] : x[v + 2], 16);
    float a = (b3 ? y[1] : y[0]) + __shfl_xor_sync(0xffffffffu, b3 ? y[0] : y[1], 8);
    a += __shfl_xor_sync(0xffffffffu, a, 4);
    a += __shfl_xor_sync(0xffffffffu, a, 2);
    a += __shfl_xor_sync(0xffffffffu, a, 1);
    return a;
}

// grid (ceil(B*H*L / 4 / kDwWarps)), kDwWarps warps; warp = 4 consecutive query rows of one
// head (one chunk, since 128 is a multiple of 4).  A lane holds 4 consecutive elements of
// every d = 128 vector.  Walk 1 (right to left, j = i .. b): the logits s_ij of the diagonal
// chunk, staged in shared memory; walk 2 (left to right, j = b .. i): acc <- H_j acc +
// alpha_ij v_j from acc = X_i.
template <bool FOX>
__global__ void __launch_bounds__(32 * kDwWarps) vt_diag_walks(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
    const __nv_bfloat16* __restrict__ w, const float* __restrict__ beta, const float* __restrict__ log_f,
    const __nv_bfloat16* __restrict__ x, const float* __restrict__ lse_in, __nv_bfloat16* __restrict__ o,
    float* __restrict__ lse_out, int BH, int L, float scale, WsHeader* hdr) {
    constexpr int D = 128, E = 4, R = kDwRows;
    __shared__ float4 stage_all[kDwWarps][kVcC];  // [j - b][row]: logits, then weights
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ngr = cdiv(L, R);
    const long long g = (long long)blockIdx.x * kDwWarps + warp;
    if (g >= (long long)BH * ngr) return;
    const int bh = (int)(g / ngr);
    const int i0 = (int)(g % ngr) * R;
    const int imax = min(i0 + R, L) - 1;
    const int jlo = (i0 / kVcC) * kVcC;
    const int hr = bh * L;           // the head's first row (B*H*L*D < 2^31)
    const int ho = hr * D + lane * E;
    if (!in_bounds((long long)hr * D, (long long)L * D, (long long)BH * L * D, hdr, 230)) return;
    float4* st = stage_all[warp];
    const int r_l = lane >> 3;
    int ir[R];
#pragma unroll
    for (int r = 0; r < R; ++r) ir[r] = i0 + r <= imax ? i0 + r : -1;
    const int il = i0 + r_l <= imax ? i0 + r_l : -1;
    auto ld4 = [&](const __nv_bfloat16* p, float (&f)[E]) {
        const uint2 raw = *reinterpret_cast<const uint2*>(p);
        f[0] = bf_lo(raw.x); f[1] = bf_hi(raw.x); f[2] = bf_lo(raw.y); f[3] = bf_hi(raw.y);
    };

    // walk 1: the diagonal chunk's logits, each query carried backwards through H_i, H_{i-1}, ...
    float u[R][E];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (ir[r] >= 0) ld4(q + ho + (i0 + r) * D, u[r]);
        else
#pragma unroll
            for (int e = 0; e < E; ++e) u[r][e] = 0.f;
    }
    float bias = 0.f;  // of row r_l: sum_{s=j+1..i} log f_s
    for (int j = imax; j >= jlo; --j) {
        float kj[E], wj[E];
        ld4(k + ho + j * D, kj);
        ld4(w + ho + j * D, wj);
        const float bj = beta[hr + j];
        float xs[2 * R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float a = 0.f, b = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                a = fmaf(kj[e], u[r][e], a);
                b = fmaf(wj[e], u[r][e], b);
            }
            xs[2 * r] = a;
            xs[2 * r + 1] = b;
        }
        const float sum = dw_sum_8(xs, lane);  // lanes 8r..8r+3: k_j . u_r; 8r+4..8r+7: w_j . u_r
        const float s = fmaf(scale, sum, bias);
        if (FOX && j <= il) bias += log_f[hr + j];
        if ((lane & 7) == 0) reinterpret_cast<float*>(&st[j - jlo])[r_l] = s;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float t = j <= ir[r] ? bj * __shfl_sync(0xffffffffu, sum, 8 * r + 4) : 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) u[r][e] = fmaf(-t, wj[e], u[r][e]);
        }
    }
    __syncwarp();
    // weights alpha_ij = exp(s_ij - lse_i), 32 keys at a time (lane = key)
    float lse_r[R];
#pragma unroll
    for (int r = 0; r < R; ++r) lse_r[r] = ir[r] >= 0 ? lse_in[hr + i0 + r] : 0.f;
    for (int jb = jlo; jb <= imax; jb += 32) {
        const int j = jb + lane;
        float4 sv = j <= imax ? st[j - jlo] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float sr[R] = {sv.x, sv.y, sv.z, sv.w};
        float ew[R];
#pragma unroll
        for (int r = 0; r < R; ++r) ew[r] = j <= ir[r] ? expf(sr[r] - lse_r[r]) : 0.f;
        __syncwarp();
        if (j <= imax) st[j - jlo] = make_float4(ew[0], ew[1], ew[2], ew[3]);
    }
    __syncwarp();

    // walk 2: from acc = X_i, the diagonal chunk's steps and terms
    float acc[R][E];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (ir[r] >= 0) ld4(x + ho + (i0 + r) * D, acc[r]);
        else
#pragma unroll
            for (int e = 0; e < E; ++e) acc[r][e] = 0.f;
    }
    for (int j = jlo; j <= imax; ++j) {
        float wj[E], vj[E];
        ld4(w + ho + j * D, wj);
        ld4(v + ho + j * D, vj);
        const float bj = beta[hr + j];
        const float4 a4 = st[j - jlo];
        const float a[R] = {a4.x, a4.y, a4.z, a4.w};
        float xs[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float p = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) p = fmaf(wj[e], acc[r][e], p);
            xs[r] = p;
        }
        const float sum = dw_sum_4(xs, lane);  // lanes 8r..8r+7: w_j . acc_r
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float t = j <= ir[r] ? bj * __shfl_sync(0xffffffffu, sum, 8 * r) : 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[r][e] = fmaf(a[r], vj[e], fmaf(-t, wj[e], acc[r][e]));
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (ir[r] < 0) continue;
        uint2 out;
        out.x = pack_bf16x2_rn(acc[r][0], acc[r][1]);
        out.y = pack_bf16x2_rn(acc[r][2], acc[r][3]);
        *reinterpret_cast<uint2*>(o + ho + (i0 + r) * D) = out;
        if (lse_out && lane == 0) lse_out[hr + i0 + r] = lse_r[r];
    }
}

}  // namespace

cudaError_t launch_vt_chain(const void* vhat, const void* pmi, void* pairs, int BH, int Lp, int N,
                            long long pair_rows, cudaStream_t st) {
    if (N < 2) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(vt_value_chain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kVcSmem);
    if (e != cudaSuccess) return e;
    vt_value_chain<<<dim3(BH, N - 1), kVcThreads, kVcSmem, st>>>(
        static_cast<const __nv_bfloat16*>(vhat), static_cast<const __nv_bfloat16*>(pmi),
        static_cast<__nv_bfloat16*>(pairs), Lp, N, pair_rows);
    return cudaGetLastError();
}

cudaError_t launch_vt_diag(const void* q, const void* k, const void* v, const void* w, const float* beta,
                           const float* log_f, const void* x, const float* lse_in, void* o, float* lse_out, int BH,
                           int L, float scale, WsHeader* hdr, cudaStream_t st) {
    const long long groups = (long long)BH * cdiv(L, kDwRows);
    const int ctas = (int)((groups + kDwWarps - 1) / kDwWarps);
    auto kern = log_f ? vt_diag_walks<true> : vt_diag_walks<false>;
    mark_start(st);
    kern<<<ctas, 32 * kDwWarps, 0, st>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
        static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(w), beta, log_f,
        static_cast<const __nv_bfloat16*>(x), lse_in, static_cast<__nv_bfloat16*>(o), lse_out, BH, L, scale, hdr);
    mark_end(st);
    return cudaGetLastError();
}

}  // namespace pathattn
