// Prefill -> decode hand-off on GB300 tensor cores (bf16, d = 128).
//
// "Resumo Técnico: Atenção PaTH" (gist.science/pt/paper/2505.16381), §3
// "Inferência": after a prompt of L tokens the decode cache must hold
//     k~_j = H_{L-1} ... H_{j+1} k_j          (j < L).
// With the chunk products of §3 "Representação de Transformação UT",
// P_c = I - W_c^T A_c W_c = I - W_c^T V_c (V_c = A_c W_c), a key row of chunk
// m transported to its chunk end (khat, from the UT prep) continues as
//     k~ = khat P_{m+1} P_{m+2} ... P_last.
// Instead of carrying every chunk through every later chunk (a quadratic
// number of chunk pairs), this kernel walks the chunks of one head right to
// left and keeps the suffix product
//     N_c = P_c P_{c+1} ... P_last = N_{c+1} - W_c^T (V_c N_{c+1}),  N_{last+1} = I,
// a d x d matrix, so that each chunk's keys need one product:
//     k~ (chunk c-1) = khat_{c-1} N_c.
// Per chunk that is three 128 x 128 x 128 products on the tensor cores:
//     T   = V_c N              (A = V_c, K-major;   B = N, MN-major)
//     N  += W_c^T (-T)         (A = W_c^T, MN-major view of the W tile; B = -T, MN-major)
//     K~  = khat_{c-1} N_c     (A = khat, K-major;  B = N, MN-major)
// N (fp32 master in TMEM) and T change every step and are not exact in bf16:
// they are split into hi + lo bf16 operands and multiplied term by term,
// which keeps the products near fp32 accuracy; W, V and khat are bf16 values
// already (the UT prep stores them that way).
//
// One CTA per head, 320 threads: warp 0 TMA, warp 1 MMA issue, warps 2-9
// conversions (one TMEM lane = one matrix row; the two warps of a lane quarter
// split the columns).  Every wait is bounded; on expiry the kernel records
// PATH_ERR_TIMEOUT, every role stops, copies and MMAs drain and TMEM is freed.
#include "common.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.cuh"
#include "ut_prep.cuh"

namespace pathattn {
using namespace sm100;

namespace pfk {
constexpr int C = 128, D = 128;
constexpr int kThreads = 320;
constexpr int kConv = 256;  // warps 2-9
constexpr uint32_t TILE = 32768;  // 128 x 128 bf16
constexpr uint32_t RV = 0, RW = 32768, RK = 65536, RNH = 98304, RNL = 131072, RTH = 163840, RTL = 196608;
constexpr uint32_t RB = 229376;
constexpr size_t kSmem = RB + 256 + 1024;  // + alignment slack
constexpr uint32_t TM_N = 0, TM_T = 128, TM_K = 256;
enum {
    B_VFULL = 0, B_WFULL, B_KFULL, B_VEMPTY, B_WEMPTY, B_KEMPTY,
    B_T, B_N, B_KOUT, B_TREADY, B_NREADY, B_KREAD, B_DRAIN, B_COUNT
};
static_assert(B_COUNT * 8 <= 128, "barriers overlap the TMEM slot and abort flag at +128");
}  // namespace pfk

struct PfParams {
    int L, Lp, nch;
    const __nv_bfloat16* khat;  // [BH, Lp, D] (workspace)
    __nv_bfloat16* kcache;      // [BH, n_max, D]
    int n_max;
    WsHeader* hdr;
    unsigned long long limit_ns;
};

__global__ void __launch_bounds__(pfk::kThreads, 1)
    prefill_suffix_tc(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ CUtensorMap tm_khat, const PfParams p) {
    using namespace pfk;
    constexpr uint32_t ID_KMN = idesc_bf16_ab(D, false, true);   // A K-major, B MN-major
    constexpr uint32_t ID_MNMN = idesc_bf16_ab(D, true, true);   // A MN-major, B MN-major

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    auto bar = [&](int i) { return sb + RB + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + RB + 128);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + RB + 132);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int S = p.nch - 1;  // steps: chunks c = nch-1 .. 1

    if (threadIdx.x == 0) {
        for (int i = 0; i < B_COUNT; ++i)
            mbar_init(bar(i), (i == B_TREADY || i == B_NREADY || i == B_KREAD) ? kConv : 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl wc{abort_flag, p.hdr, p.limit_ns};

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_v); prefetch_tmap(&tm_w); prefetch_tmap(&tm_khat);
            int issued[3] = {0, 0, 0};  // V, W, khat loads issued
            bool ok = true;
            for (int s = 0; s < S && ok; ++s) {
                const int c = p.nch - 1 - s;
                // each slot is refilled once its consumer (GEMM 1, 2, 3 of step s-1) has completed
                if (s > 0) ok = mbar_wait(bar(B_VEMPTY), (s - 1) & 1, wc, 60);
                if (!ok) break;
                mbar_expect_tx(bar(B_VFULL), TILE);
                for (int h = 0; h < 2; ++h) tma_load_3d(sb + RV + h * 16384, &tm_v, bar(B_VFULL), h * 64, c * C, bh);
                ++issued[0];
                if (s > 0) ok = mbar_wait(bar(B_WEMPTY), (s - 1) & 1, wc, 61);
                if (!ok) break;
                mbar_expect_tx(bar(B_WFULL), TILE);
                for (int h = 0; h < 2; ++h) tma_load_3d(sb + RW + h * 16384, &tm_w, bar(B_WFULL), h * 64, c * C, bh);
                ++issued[1];
                if (s > 0) ok = mbar_wait(bar(B_KEMPTY), (s - 1) & 1, wc, 62);
                if (!ok) break;
                mbar_expect_tx(bar(B_KFULL), TILE);
                for (int h = 0; h < 2; ++h)
                    tma_load_3d(sb + RK + h * 16384, &tm_khat, bar(B_KFULL), h * 64, (c - 1) * C, bh);
                ++issued[2];
            }
            // copies still in flight must land before the CTA exits
            const int ful[3] = {B_VFULL, B_WFULL, B_KFULL};
            for (int i = 0; i < 3; ++i)
                if (issued[i] > 0) drain_wait(bar(ful[i]), (uint32_t)((issued[i] - 1) & 1), p.limit_ns, p.hdr, 95);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0 && S > 0) {
            bool ok = mbar_wait(bar(B_NREADY), 0, wc, 63);  // N = I written
            for (int s = 0; s < S && ok; ++s) {
                if (!(ok = mbar_wait(bar(B_VFULL), s & 1, wc, 64))) break;
                tc_fence_after();
                // T = V_c (N_hi + N_lo)
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + TM_T, kmajor_desc(sb + RV, kk, 16384), mnmajor_desc(sb + RNH, kk), ID_KMN, kk > 0);
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + TM_T, kmajor_desc(sb + RV, kk, 16384), mnmajor_desc(sb + RNL, kk), ID_KMN, 1);
                mma_commit(bar(B_VEMPTY));
                mma_commit(bar(B_T));
                if (!(ok = mbar_wait(bar(B_TREADY), s & 1, wc, 65) && mbar_wait(bar(B_WFULL), s & 1, wc, 66))) break;
                tc_fence_after();
                // N += W_c^T ((-T)_hi + (-T)_lo)
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tmem + TM_N, mnmajor_desc(sb + RW, kk), mnmajor_desc(sb + RTH, kk), ID_MNMN, 1);
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tmem + TM_N, mnmajor_desc(sb + RW, kk), mnmajor_desc(sb + RTL, kk), ID_MNMN, 1);
                mma_commit(bar(B_WEMPTY));
                mma_commit(bar(B_N));
                if (!(ok = mbar_wait(bar(B_NREADY), (s + 1) & 1, wc, 67) && mbar_wait(bar(B_KFULL), s & 1, wc, 68) &&
                           (s == 0 || mbar_wait(bar(B_KREAD), (s - 1) & 1, wc, 69))))
                    break;
                tc_fence_after();
                // K~ = khat_{c-1} (N_hi + N_lo)
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + TM_K, kmajor_desc(sb + RK, kk, 16384), mnmajor_desc(sb + RNH, kk), ID_KMN, kk > 0);
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + TM_K, kmajor_desc(sb + RK, kk, 16384), mnmajor_desc(sb + RNL, kk), ID_KMN, 1);
                mma_commit(bar(B_KEMPTY));
                mma_commit(bar(B_KOUT));
            }
            // every issued MMA completes before TMEM is released
            mma_commit(bar(B_DRAIN));
            drain_wait(bar(B_DRAIN), 0, p.limit_ns, p.hdr, 96);
        }
    } else {
        // ------------------------------------------------------------------ conversion warps
        const int r = 32 * (warp & 3) + lane;  // matrix row = TMEM lane
        const int h = (warp - 2) >> 2;         // column half
        const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        __nv_bfloat16* cache = p.kcache + (size_t)bh * p.n_max * D;
        uint8_t* nhi = sm + RNH;
        uint8_t* nlo = sm + RNL;
        {  // the last chunk is already at its end: khat is its transported key
            const int j = (p.nch - 1) * C + r;
            if (j < p.L) {
                uint4* dst = reinterpret_cast<uint4*>(cache + (size_t)j * D + 64 * h);
#pragma unroll
                for (int g = 0; g < 8; ++g) dst[g] = ld_global_nc_v4(p.khat + ((size_t)bh * p.Lp + j) * D + 64 * h + 8 * g);
            }
        }
        // N_{last+1} = I: the fp32 master in TMEM and its hi / lo operands
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            uint32_t v[32];
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                x[j] = (64 * h + 32 * c + j == r) ? 1.0f : 0.0f;
                v[j] = __float_as_uint(x[j]);
            }
            tmem_st32(tl + TM_N + 64 * h + 32 * c, v);
#pragma unroll
            for (int g = 0; g < 4; ++g) put_hilo(nhi, nlo, r, 8 * h + 4 * c + g, x + 8 * g);
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(B_NREADY));

        bool ok = true;
        for (int s = 0; s < S && ok; ++s) {
            const int c = p.nch - 1 - s;
            // -T row -> hi / lo operand
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(B_T), s & 1, wc, 70)))) break;
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t v[32];
                tmem_ld32(tl + TM_T + 64 * h + 32 * cc, v);
                tmem_wait_ld();
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    float t8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) t8[e] = -__uint_as_float(v[8 * g + e]);
                    put_hilo(sm + RTH, sm + RTL, r, 8 * h + 4 * cc + g, t8);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B_TREADY));
            // N_c row -> hi / lo operand
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(B_N), s & 1, wc, 71)))) break;
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t v[32];
                tmem_ld32(tl + TM_N + 64 * h + 32 * cc, v);
                tmem_wait_ld();
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    float n8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) n8[e] = __uint_as_float(v[8 * g + e]);
                    put_hilo(nhi, nlo, r, 8 * h + 4 * cc + g, n8);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B_NREADY));
            // K~ rows of chunk c-1 -> the cache
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(B_KOUT), s & 1, wc, 72)))) break;
            tc_fence_after();
            const int j = (c - 1) * C + r;  // < L: only the last chunk can be partial
            uint4* dst = reinterpret_cast<uint4*>(cache + (size_t)j * D + 64 * h);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t v[32];
                tmem_ld32(tl + TM_K + 64 * h + 32 * cc, v);
                tmem_wait_ld();
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    dst[4 * cc + g] = make_uint4(
                        pack_bf16x2(__uint_as_float(v[8 * g + 0]), __uint_as_float(v[8 * g + 1])),
                        pack_bf16x2(__uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3])),
                        pack_bf16x2(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5])),
                        pack_bf16x2(__uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7])));
            }
            tc_fence_before();
            mbar_arrive(bar(B_KREAD));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// The V factor and khat come from the UT prep (run before this launch on the
// same stream); w is the caller's [BH, L, D] tensor.
cudaError_t launch_prefill_tc(const void* w, void* kcache, int BH, int L, int n_max, unsigned char* ws,
                              const FwdLayout& lay, cudaStream_t st) {
    using namespace pfk;
    CUtensorMap mv, mw, mkh;
    if (!make_map(&mv, ws + lay.vfac, D, lay.Lp, BH) || !make_map(&mw, w, D, L, BH) ||
        !make_map(&mkh, ws + lay.khat, D, lay.Lp, BH))
        return cudaErrorInvalidValue;
    PfParams p;
    p.L = L;
    p.Lp = lay.Lp;
    p.nch = lay.Lp / C;
    p.khat = reinterpret_cast<const __nv_bfloat16*>(ws + lay.khat);
    p.kcache = static_cast<__nv_bfloat16*>(kcache);
    p.n_max = n_max;
    p.hdr = reinterpret_cast<WsHeader*>(ws);
    p.limit_ns = 2000000000ull;
    cudaError_t e = cudaFuncSetAttribute(prefill_suffix_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    mark_start(st);
    prefill_suffix_tc<<<BH, kThreads, kSmem, st>>>(mv, mw, mkh, p);
    mark_end(st);
    return cudaGetLastError();
}

}  // namespace pathattn
