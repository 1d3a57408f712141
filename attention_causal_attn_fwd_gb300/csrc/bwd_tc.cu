// Backward chunk-pair reduction on GB300 tensor cores (bf16, d = 128).
//
// The backward of "Resumo Técnico: Atenção PaTH" (gist.science/pt/paper/2505.16381)
// is organised in chunks of C = 64 positions (csrc/bwd.cu).  For one key chunk m
// this kernel sums, over every later query chunk n, the per-pair products
//     dV_m^T    += dO_n^T P_nm          (d x C)
//     dKhat_m^T += U_{n,m}^T dS_nm      (d x C; scaled on output)
//     dP_m      += G_{n,m-1}^T U_{n,m}  (d x d; m >= 1)
// from the bf16 pair store that bwd_chain writes and the caller's dO.  Every
// operand is read MN-major: the tiles are [64 rows = K][64- or 128-column = M/N]
// as TMA writes them (128-byte swizzle, two 64-column halves 8 KB apart), so one
// tile layout serves as the transposed A operand and as the B operand.
//
// One CTA per (key chunk, head), 192 threads: warp 0 TMA, warp 1 MMA issue,
// warps 2-5 the epilogue (one TMEM lane = one output row).  Three stages of
// operands (64 KB each) keep the loads ahead of the MMAs; the accumulators stay
// in TMEM (dV^T and dKhat^T 64 columns each, dP 128) for the whole key chunk.
// Every wait is bounded; on expiry the kernel records PATH_ERR_TIMEOUT, every
// role stops, copies and MMAs drain and TMEM is freed.
#include "common.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.cuh"

namespace pathattn {
using namespace sm100;

namespace rtk {
constexpr int C = 64, D = 128;
constexpr int kThreads = 192;
constexpr int kStages = 3;
constexpr uint32_t S_O = 0, S_U = 16384, S_G = 32768, S_S = 49152, S_P = 57344, STAGE = 65536;
constexpr uint32_t RB = kStages * STAGE;  // barriers
enum { B_FULL = 0, B_EMPTY = kStages, B_DONE = 2 * kStages, B_COUNT };
constexpr uint32_t R_SLOT = RB + 64;  // TMEM address, then the abort flag
static_assert(B_COUNT * 8 <= 64, "barriers overlap the TMEM slot");
constexpr size_t kSmem = RB + 128 + 1024;  // + alignment slack
constexpr uint32_t TM_V = 0, TM_K = 64, TM_P = 128;
}  // namespace rtk

struct RtParams {
    int N;
    size_t head_pairs;
    int Lp;
    float scale;
    float *dvoff, *dkhat, *dpm;
    WsHeader* hdr;
    unsigned long long limit_ns;
};

// MN-major operand of 64 K-rows: 64-column halves 8 KB apart, 8-row groups 1 KB apart;
// k-step kk = 16 rows.
__device__ __forceinline__ uint64_t mn64_desc(uint32_t base, int kk) {
    return sdesc_sw128(base + (uint32_t)kk * 2048u, 8192, 1024);
}

__global__ void __launch_bounds__(rtk::kThreads, 1)
    bwd_reduce_tc(const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_u,
                  const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_s,
                  const __grid_constant__ CUtensorMap tm_p, const RtParams p) {
    using namespace rtk;
    constexpr uint32_t ID64 = idesc_bf16_ab(64, true, true);    // N = 64, A and B MN-major
    constexpr uint32_t ID128 = idesc_bf16_ab(128, true, true);  // N = 128

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    auto bar = [&](int i) { return sb + RB + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + R_SLOT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + R_SLOT + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m = blockIdx.x, bh = blockIdx.y;  // m = 0 has the most query chunks: launched first
    const int np = p.N - 1 - m;                 // query chunks n = m + 1 .. N - 1

    if (threadIdx.x == 0) {
        for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), 1);
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
    const WaitCtl wc{abort_flag, p.hdr, p.limit_ns};

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_do); prefetch_tmap(&tm_u); prefetch_tmap(&tm_g);
            prefetch_tmap(&tm_s); prefetch_tmap(&tm_p);
            const uint32_t bytes = m >= 1 ? STAGE : STAGE - 16384;  // G only past the first key chunk
            int issued = 0;
            bool ok = true;
            for (int i = 0; i < np && ok; ++i) {
                const int n = m + 1 + i, st = i % kStages;
                // a stage is refilled once the MMAs that read it (pair i - kStages) have completed
                if (i >= kStages && !(ok = mbar_wait(bar(B_EMPTY + st), (uint32_t)((i / kStages - 1) & 1), wc, 110)))
                    break;
                const uint32_t base = sb + (uint32_t)st * STAGE;
                const int pz = (int)((size_t)bh * p.head_pairs + (size_t)n * (n - 1) / 2 + m);
                mbar_expect_tx(bar(B_FULL + st), bytes);
                for (int h = 0; h < 2; ++h) {
                    tma_load_3d(base + S_O + h * 8192, &tm_do, bar(B_FULL + st), h * 64, n * C, bh);
                    tma_load_3d(base + S_U + h * 8192, &tm_u, bar(B_FULL + st), h * 64, 0, pz);
                    if (m >= 1) tma_load_3d(base + S_G + h * 8192, &tm_g, bar(B_FULL + st), h * 64, 0, pz);
                }
                tma_load_3d(base + S_S, &tm_s, bar(B_FULL + st), 0, 0, pz);
                tma_load_3d(base + S_P, &tm_p, bar(B_FULL + st), 0, 0, pz);
                ++issued;
            }
            // copies still in flight must land before the CTA exits: the last fill of each stage
            for (int st = 0; st < kStages && st < issued; ++st) {
                const int fills = (issued - st + kStages - 1) / kStages;
                drain_wait(bar(B_FULL + st), (uint32_t)((fills - 1) & 1), p.limit_ns, p.hdr, 111);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = true;
            for (int i = 0; i < np && ok; ++i) {
                const int st = i % kStages;
                if (!(ok = mbar_wait(bar(B_FULL + st), (uint32_t)((i / kStages) & 1), wc, 112))) break;
                tc_fence_after();
                const uint32_t base = sb + (uint32_t)st * STAGE;
                for (int kk = 0; kk < C / 16; ++kk) {
                    const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                    mma_ss(tmem + TM_V, mn64_desc(base + S_O, kk), mn64_desc(base + S_P, kk), ID64, acc);
                    mma_ss(tmem + TM_K, mn64_desc(base + S_U, kk), mn64_desc(base + S_S, kk), ID64, acc);
                    if (m >= 1)
                        mma_ss(tmem + TM_P, mn64_desc(base + S_G, kk), mn64_desc(base + S_U, kk), ID128, acc);
                }
                mma_commit(bar(B_EMPTY + st));
            }
            // every issued MMA completes before the epilogue reads TMEM and TMEM is released
            mma_commit(bar(B_DONE));
            drain_wait(bar(B_DONE), 0, p.limit_ns, p.hdr, 113);
        }
    } else {
        // ------------------------------------------------------------------ epilogue (warps 2-5)
        const int r = 32 * (warp & 3) + lane;  // TMEM lane = output row (a column of d)
        const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const bool ok = __all_sync(0xffffffffu, mbar_wait_sleep(bar(B_DONE), 0, wc, 114));
        tc_fence_after();
        if (ok) {
            const size_t row0 = (size_t)bh * p.Lp + (size_t)m * C;  // first key row of the chunk
            // dV^T row r -> column r of dV (consecutive threads write consecutive columns)
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t v[32], k[32];
                tmem_ld32(tl + TM_V + 32 * cc, v);
                tmem_ld32(tl + TM_K + 32 * cc, k);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const size_t o = (row0 + 32 * cc + j) * D + r;
                    p.dvoff[o] = __uint_as_float(v[j]);
                    p.dkhat[o] = p.scale * __uint_as_float(k[j]);
                }
            }
            if (m >= 1) {
                float* dst = p.dpm + (((size_t)bh * p.N + m) * D + r) * D;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t v[32];
                    tmem_ld32(tl + TM_P + 32 * cc, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(dst + 32 * cc + j) =
                            make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                                        __uint_as_float(v[j + 3]));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

namespace {
// 3-D bf16 map [depth][rows][cols] with explicit strides and a {64, 64} box (128-byte swizzle).
bool make_map_rows64(CUtensorMap* mp, const void* base, uint64_t cols, uint64_t rows, uint64_t depth,
                     uint64_t row_bytes, uint64_t depth_bytes) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {cols, rows, depth};
    cuuint64_t strides[2] = {row_bytes, depth_bytes};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(mp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

// dO: the caller's [BH, L, 128] bf16; pairs: the bf16 pair store of bwd_chain
// (per pair U [64][128], G [64][128], dS [64][64], P [64][64]).
cudaError_t launch_bwd_reduce_tc(const void* dO, const void* pairs, float* dvoff, float* dkhat, float* dpm, int BH,
                                 int L, int Lp, int N, size_t head_pairs, float scale, WsHeader* hdr,
                                 cudaStream_t st) {
    using namespace rtk;
    if (N < 2) return cudaSuccess;
    const uint64_t pair_elems = 2ull * C * D + 2ull * C * C, pair_bytes = pair_elems * 2;
    const uint64_t npairs = (uint64_t)BH * head_pairs;
    const uint8_t* pb = static_cast<const uint8_t*>(pairs);
    CUtensorMap mo, mu, mg, ms, mp;
    if (!make_map_rows64(&mo, dO, D, (uint64_t)L, (uint64_t)BH, D * 2, (uint64_t)L * D * 2) ||
        !make_map_rows64(&mu, pb, D, C, npairs, D * 2, pair_bytes) ||
        !make_map_rows64(&mg, pb + (size_t)C * D * 2, D, C, npairs, D * 2, pair_bytes) ||
        !make_map_rows64(&ms, pb + (size_t)2 * C * D * 2, C, C, npairs, C * 2, pair_bytes) ||
        !make_map_rows64(&mp, pb + ((size_t)2 * C * D + C * C) * 2, C, C, npairs, C * 2, pair_bytes))
        return cudaErrorInvalidValue;
    RtParams p;
    p.N = N;
    p.head_pairs = head_pairs;
    p.Lp = Lp;
    p.scale = scale;
    p.dvoff = dvoff;
    p.dkhat = dkhat;
    p.dpm = dpm;
    p.hdr = hdr;
    p.limit_ns = 2000000000ull;
    cudaError_t e = cudaFuncSetAttribute(bwd_reduce_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    bwd_reduce_tc<<<dim3(N - 1, BH), kThreads, kSmem, st>>>(mo, mu, mg, ms, mp, p);
    return cudaGetLastError();
}

}  // namespace pathattn
