// Two stages of the blockwise value-transport forward (bf16, d = 128, chunks of
// 128): the value chains (tensor cores) and the diagonal walks (CUDA cores); the
// other stages are the UT prep and the scan (csrc/ut_prep_tc.cu, csrc/fwd_tc.cu,
// fwd_tc_vt_bf16).
//
// "Resumo Técnico: Por que Transformações Acumuladas Extrapolam?", §"Principais
// Contribuições" 3: o_i = sum_j alpha_ij H_i ... H_{j+1} v_j with the PaTH steps
// H_s = I - beta_s w_s w_s^T ("Resumo Técnico: Atenção PaTH", §2 "Mecanismo
// Central"), blocked as in that page's §3 "Algoritmo Estilo FlashAttention".
// With P_c = H_{e_c} ... H_{b_c} the transition of chunk c and vhat_j the value
// moved to the end of its chunk:
//   vt_value_chain  Vtil_{n,m} = Vhat_m (P_{n-1} ... P_{m+1})^T for every pair m < n
//                   (tensor cores): row j of it is v_j carried to the position just
//                   before chunk n;
//   vt_diag_walks   o_i = H_i ... H_b X_i + sum_{b <= j <= i} alpha_ij H_i ... H_{j+1} v_j,
//                   X_i = sum_{j < b} alpha_ij (row j of Vtil_{n,m(j)}) from the scan,
//                   alpha_ij = exp(s_ij - lse_i) from the scan's diagonal P and LSE.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.cuh"

namespace pathattn {

namespace {

constexpr int kVcC = 128;  // chunk (= d)
constexpr int kVcThreads = 128;
constexpr uint32_t VC_SLOT = 32768;                 // one P - I tile (two 64-column boxes of 16 KB)
constexpr uint32_t VC_BAR = 2 * VC_SLOT;            // full0, full1, mma, drain; then TMEM address, abort
constexpr size_t kVcSmem = VC_BAR + 64 + 1024;      // + alignment slack
constexpr uint32_t VC_TM_M = 0, VC_TM_A = 128;      // TMEM: fp32 master [0,128), bf16 copy [128,192)
enum VcBar { VB_FULL0 = 0, VB_FULL1, VB_MMA, VB_DRAIN };

__device__ __forceinline__ long long pair_index(int n, int m) { return (long long)n * (n - 1) / 2 + m; }

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&p);
}
__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// grid (B*H, N - 1), 128 threads (thread = row of the block = TMEM lane); CTA (bh, m)
// runs the chain of key chunk m, N - 2 - m products, the longest chains of every head
// launched first.  The fp32 master of Vtil stays in TMEM and each step accumulates
// bf16(Vtil) (P_n - I)^T-as-the-UT-prep-stores-it into it (one M128 N128 K128 product,
// A from TMEM, P - I from shared memory as an MN-major B operand, as V is in the
// scan), so the identity part is exact and only the correction is rounded, as for
// the scan's query transport.  The bf16 copy of each step's result is both the
// next product's A operand and the pair store's block.  Thread 0 issues the TMA
// copies (two P - I tiles in flight) and the MMAs; every wait is bounded.
__global__ void __launch_bounds__(kVcThreads, 2)
    vt_value_chain(const __grid_constant__ CUtensorMap tm_pm, const __nv_bfloat16* __restrict__ vhat,
                   __nv_bfloat16* __restrict__ pairs, int Lp, int N, long long pair_rows, WsHeader* hdr,
                   unsigned long long limit_ns) {
    using namespace sm100;
    extern __shared__ uint8_t vc_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(vc_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    auto bar = [&](int k) { return sb + VC_BAR + 8u * (uint32_t)k; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + VC_BAR + 32);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + VC_BAR + 36);
    const int bh = blockIdx.x, m = blockIdx.y;
    const int i = threadIdx.x, warp = i >> 5;
    if (m >= N - 1) return;
    const int steps = N - 2 - m;
    constexpr uint32_t IDESC = idesc_bf16(kVcC, true);
    if (i == 0) {
        for (int k = 0; k < 4; ++k) mbar_init(bar(k), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
    const WaitCtl wc{abort_flag, hdr, limit_ns};
    int issued[2] = {0, 0};  // thread 0: copies issued per slot
    bool mma_issued = false; // thread 0
    if (i == 0) {
        prefetch_tmap(&tm_pm);
        for (int t = 0; t < 2 && t < steps; ++t) {
            mbar_expect_tx(bar(VB_FULL0 + t), VC_SLOT);
            for (int c = 0; c < 2; ++c)
                tma_load_3d(sb + (uint32_t)t * VC_SLOT + c * 16384, &tm_pm, bar(VB_FULL0 + t), c * 64,
                            (m + 1 + t) * kVcC, bh);
            ++issued[t];
        }
    }
    __nv_bfloat16* ph = pairs + (size_t)bh * (size_t)pair_rows * kVcC;
    {  // Vtil_{m+1,m} = Vhat_m: to the pair store as it is, to the master and its bf16 copy
        const uint4* src = reinterpret_cast<const uint4*>(vhat + ((size_t)bh * Lp + (size_t)m * kVcC + i) * kVcC);
        uint4* dst = reinterpret_cast<uint4*>(ph + ((size_t)pair_index(m + 1, m) * kVcC + i) * kVcC);
        uint32_t raw[64];
#pragma unroll
        for (int g = 0; g < 16; ++g) {
            const uint4 x = src[g];
            dst[g] = x;
            raw[4 * g] = x.x; raw[4 * g + 1] = x.y; raw[4 * g + 2] = x.z; raw[4 * g + 3] = x.w;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t f[32];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                f[2 * j] = raw[16 * c + j] << 16;
                f[2 * j + 1] = raw[16 * c + j] & 0xffff0000u;
            }
            tmem_st32(tl + VC_TM_M + 32 * c, f);
            tmem_st16(tl + VC_TM_A + 16 * c, &raw[16 * c]);
        }
        tmem_wait_st();
    }
    bool ok = true;
    for (int t = 0; t < steps; ++t) {  // Vtil_{n+1,m} = Vtil_{n,m} P_n^T, n = m + 1 + t
        const int n = m + 1 + t, s = t & 1;
        tc_fence_before();
        __syncthreads();  // the bf16 copy of Vtil_{n,m} is in TMEM
        if (i == 0) {
            if (mbar_wait(bar(VB_FULL0 + s), (uint32_t)((t >> 1) & 1), wc, 70)) {
                tc_fence_after();
                for (int kk = 0; kk < kVcC / 16; ++kk)
                    mma_ts(tmem + VC_TM_M, tmem + VC_TM_A + kk * 8, mnmajor_desc(sb + (uint32_t)s * VC_SLOT, kk),
                           IDESC, 1);
                mma_commit(bar(VB_MMA));
                mma_issued = true;
            }
        }
        ok = __syncthreads_and(mbar_wait(bar(VB_MMA), (uint32_t)(t & 1), wc, 71)) != 0;
        if (!ok) break;
        tc_fence_after();
        if (i == 0 && t + 2 < steps) {  // the slot is free again: P - I of step t + 2
            mbar_expect_tx(bar(VB_FULL0 + s), VC_SLOT);
            for (int c = 0; c < 2; ++c)
                tma_load_3d(sb + (uint32_t)s * VC_SLOT + c * 16384, &tm_pm, bar(VB_FULL0 + s), c * 64,
                            (n + 2) * kVcC, bh);
            ++issued[s];
        }
        uint4* dst = reinterpret_cast<uint4*>(ph + ((size_t)pair_index(n + 1, m) * kVcC + i) * kVcC);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t f[32], pk[16];
            tmem_ld32(tl + VC_TM_M + 32 * c, f);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2_rn(__uint_as_float(f[2 * j]), __uint_as_float(f[2 * j + 1]));
            tmem_st16(tl + VC_TM_A + 16 * c, pk);
#pragma unroll
            for (int g = 0; g < 4; ++g) dst[4 * c + g] = make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
        }
        tmem_wait_st();
    }
    // copies and MMAs in flight land before TMEM is released
    if (i == 0) {
        if (mma_issued) {
            mma_commit(bar(VB_DRAIN));
            drain_wait(bar(VB_DRAIN), 0, limit_ns, hdr, 95);
        }
        for (int k = 0; k < 2; ++k)
            if (issued[k] > 0) drain_wait(bar(VB_FULL0 + k), (uint32_t)((issued[k] - 1) & 1), limit_ns, hdr, 96);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ----------------------------------------------------------------------------- diagonal walks
constexpr int kDwRows = 4;   // query rows per warp, in lockstep
constexpr int kDwWarps = 8;

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
// head (one chunk, since 128 is a multiple of 4), walked in lockstep.  A lane holds 4
// consecutive elements of every d = 128 vector.  The weights of the diagonal chunk come
// from the scan: alpha_ij = P_ij 2^(m0_i - lse_i log2 e), with P the diagonal block's
// bf16 probabilities formed against the max m0_i; 32 keys at a time, one per lane.  The
// walk (left to right, j = b .. i) is acc <- H_j acc + alpha_ij v_j from acc = X_i.  The
// walk is latency-bound: four CTAs per SM (64 registers) beat three (A/B 0.574 against 0.611 ms
// for the whole B1 H12 L4096 call), eight rows per warp or two were slower.
__global__ void __launch_bounds__(32 * kDwWarps, 4) vt_diag_walks(
    const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ w, const float* __restrict__ beta,
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ pdiag, const float* __restrict__ m0,
    const float* __restrict__ lse_in, __nv_bfloat16* __restrict__ o, float* __restrict__ lse_out, int BH, int L,
    WsHeader* hdr) {
    constexpr int D = 128, E = 4, R = kDwRows;
    constexpr float kL2e = 1.4426950408889634f;
    __shared__ float4 stage_all[kDwWarps][kVcC];  // [j - b][row]: weights
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
    int ir[R];
#pragma unroll
    for (int r = 0; r < R; ++r) ir[r] = i0 + r <= imax ? i0 + r : -1;
    auto ld4 = [&](const __nv_bfloat16* p, float (&f)[E]) {
        const uint2 raw = *reinterpret_cast<const uint2*>(p);
        f[0] = bf_lo(raw.x); f[1] = bf_hi(raw.x); f[2] = bf_lo(raw.y); f[3] = bf_hi(raw.y);
    };
    float lse_r[R], fac[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        lse_r[r] = ir[r] >= 0 ? lse_in[hr + i0 + r] : 0.f;
        fac[r] = ir[r] >= 0 ? exp2f(m0[hr + i0 + r] - lse_r[r] * kL2e) : 0.f;
    }
    for (int jb = jlo; jb <= imax; jb += 32) {
        const int j = jb + lane;
        float ew[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            ew[r] = 0.f;
            if (j <= ir[r]) {
                const unsigned short raw =
                    *reinterpret_cast<const unsigned short*>(pdiag + ((size_t)hr + i0 + r) * kVcC + (j - jlo));
                ew[r] = __uint_as_float((uint32_t)raw << 16) * fac[r];
            }
        }
        if (j <= imax) st[j - jlo] = make_float4(ew[0], ew[1], ew[2], ew[3]);
    }
    __syncwarp();

    float acc[R][E];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (ir[r] >= 0) ld4(x + ho + (i0 + r) * D, acc[r]);
        else
#pragma unroll
            for (int e = 0; e < E; ++e) acc[r][e] = 0.f;
    }
    float wn[E], vn[E];
    ld4(w + ho + jlo * D, wn);
    ld4(v + ho + jlo * D, vn);
    float bn = beta[hr + jlo];
    for (int j = jlo; j <= imax; ++j) {
        float wj[E], vj[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            wj[e] = wn[e];
            vj[e] = vn[e];
        }
        const float bj = bn;
        const int jn = min(j + 1, imax);
        ld4(w + ho + jn * D, wn);
        ld4(v + ho + jn * D, vn);
        bn = beta[hr + jn];
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
                            long long pair_rows, WsHeader* hdr, cudaStream_t st) {
    if (N < 2) return cudaSuccess;
    CUtensorMap mpm;
    if (!make_map(&mpm, pmi, kVcC, Lp, BH)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(vt_value_chain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kVcSmem);
    if (e != cudaSuccess) return e;
    vt_value_chain<<<dim3(BH, N - 1), kVcThreads, kVcSmem, st>>>(
        mpm, static_cast<const __nv_bfloat16*>(vhat), static_cast<__nv_bfloat16*>(pairs), Lp, N, pair_rows, hdr,
        2000000000ull);
    return cudaGetLastError();
}

cudaError_t launch_vt_diag(const void* v, const void* w, const float* beta, const void* x, const void* pdiag,
                           const float* m0, const float* lse_in, void* o, float* lse_out, int BH, int L,
                           WsHeader* hdr, cudaStream_t st) {
    const long long groups = (long long)BH * cdiv(L, kDwRows);
    const int ctas = (int)((groups + kDwWarps - 1) / kDwWarps);
    mark_start(st);
    vt_diag_walks<<<ctas, 32 * kDwWarps, 0, st>>>(
        static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(w), beta,
        static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(pdiag), m0, lse_in,
        static_cast<__nv_bfloat16*>(o), lse_out, BH, L, hdr);
    mark_end(st);
    return cudaGetLastError();
}

}  // namespace pathattn
