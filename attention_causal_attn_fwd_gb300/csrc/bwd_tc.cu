// Backward kernels on GB300 tensor cores (bf16, d = 128): the per-key-chunk
// reduction bwd_reduce_tc, and further down the query-side chunk chains
// bwd_chain_tc that write its input.
//
// The backward of "Resumo Técnico: Atenção PaTH" (gist.science/pt/paper/2505.16381)
// is organised in chunks of C = 64 positions (csrc/bwd.cu).  For one key chunk m
// this kernel sums, over every later query chunk n, the per-pair products
//     dV_m^T    += dO_n^T P_nm          (d x C)
//     dKhat_m^T += U_{n,m}^T dS_nm      (d x C; scaled on output)
//     dP_m      += G_{n,m-1}^T U_{n,m}  (d x d; m >= 1)
// from the bf16 pair store that bwd_chain_tc writes and the caller's dO.  Every
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

// ============================================================================ chunk chains
// The query-side chains of the backward for bf16 at d = 128 (the CUDA-core
// version is bwd_chain in csrc/bwd.cu).  A CTA runs two query chunks, nA and
// nB = nA - 1, as the 128 rows of one MMA tile (rows 0-63 chunk nA, rows
// 64-127 chunk nB), walking the key chunks m = nA - 1 .. 0 and back:
//   down:  S = U khat_m^T,  dP = dO v_m^T   (N = 64)
//          P = exp(scale S + c_i - c_j - lse_i),  dS = P o (dP - Delta)
//          U <- U P_m^T                      (N = 128; fp32 master in TMEM)
//   up:    G <- scale dS khat_m + G P_m      (N = 128; fp32 master in TMEM)
// Chunk nB's rows join the down chain after key chunk nB (its U is set to
// qbar there) and leave the up chain after it; meanwhile they are masked.
// U and G are carried as fp32 in TMEM and fed back as hi + lo bf16 operands
// (three MMAs per product: hi*hi + hi*lo + lo*hi), P_m likewise; S uses U's hi
// part and bf16 khat, like the forward's scan.  Per pair the epilogue writes
// U, G, dS and P (bf16) for bwd_reduce_tc and the FoX row / column sums.
//
// Roles (320 threads): warp 0 TMA, warp 1 MMA issue, warps 2-9 the epilogue,
// two warps per TMEM lane quarter (one TMEM lane = one query row) that split
// every row's columns.  FoX is a template parameter, so the non-FoX dS loop
// carries no per-element test.  Every wait is bounded; on expiry the kernel
// records PATH_ERR_TIMEOUT, every role stops, copies and MMAs drain and TMEM is
// freed.
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

namespace ctk {
constexpr int C = 64, D = 128;
constexpr int kThreads = 320;
constexpr int kEpi = 256;          // warps 2-9: two per TMEM lane quarter, each owning half the columns
constexpr uint32_t R_O = 0;        // dO [128][128] (down); dS [128][64] (up)
constexpr uint32_t R_UH = 32768;   // U (then G) hi  [128][128]
constexpr uint32_t R_UL = 65536;   // U (then G) lo  [128][128]
constexpr uint32_t R_K = 98304;    // khat_m [64][128]
constexpr uint32_t R_V = 114688;   // v_m [64][128]
constexpr uint32_t R_PH = 131072;  // P_m hi [128][128]
constexpr uint32_t R_PL = 163840;  // P_m lo [128][128]
constexpr uint32_t R_ST = 196608;  // per epilogue warp: its 32 rows x 32 columns of dS, then of P, 64-byte rows
constexpr uint32_t RB = 229376;    // barriers
enum { B_DO = 0, B_KV, B_KVE, B_P, B_PE, B_S, B_U, B_UP, B_READY, B_DRAIN, B_COUNT };
constexpr uint32_t R_SLOT = RB + 96;  // TMEM address, abort flag
static_assert(B_COUNT * 8 <= 96, "barriers overlap the TMEM slot");
constexpr size_t kSmem = RB + 128 + 1024;
static_assert(R_ST + 8 * 4096 <= RB && kSmem <= 227 * 1024, "shared memory per CTA");
constexpr uint32_t TM_S = 0, TM_DP = 64, TM_U = 128, TM_T = 256;  // TM_U holds U, then G P
}  // namespace ctk

struct CtParams {
    int N, L, Lp;
    size_t head_pairs;
    float scale;
    int fox;
    const float *qbar, *lse, *delta, *cum;
    float *dqbar, *dcrow, *dccol;
    __nv_bfloat16* pairs;  // [pairs][U | G | dS | P]
    WsHeader* hdr;
    unsigned long long limit_ns;
};

// 8 bf16 of row r, granule g (columns 8g..8g+7) of a 128-byte-swizzled K-major
// tile whose 64-column halves are `half` bytes apart.
__device__ __forceinline__ uint32_t sw_off(int r, int g, uint32_t half) {
    return (uint32_t)(g >> 3) * half + (uint32_t)r * 128u + ((uint32_t)((g & 7) ^ (r & 7)) << 4);
}

template <bool FOX>
__global__ void __launch_bounds__(ctk::kThreads, 1)
    bwd_chain_tc(const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_ph,
                 const __grid_constant__ CUtensorMap tm_pl, const __grid_constant__ CUtensorMap tm_ds,
                 const CtParams p) {
    using namespace ctk;
    constexpr uint32_t ID_S = idesc_bf16_ab(64, false, false);    // U khat^T, dO v^T: K-major A and B
    constexpr uint32_t ID_U = idesc_bf16_ab(128, false, false);   // U P^T: K-major B (rows of P)
    constexpr uint32_t ID_G = idesc_bf16_ab(128, false, true);    // dS khat, G P: MN-major B

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    auto bar = [&](int i) { return sb + RB + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + R_SLOT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + R_SLOT + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y;
    const int nA = p.N - 1 - 2 * (int)blockIdx.x, nB = nA - 1;  // longest chains first
    const int steps = 2 * nA;                                      // nA down, nA up

    if (threadIdx.x == 0) {
        for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), i == B_READY ? kEpi : 1);
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
    const size_t pair0 = (size_t)bh * p.head_pairs;
    auto pair_index = [&](int n, int m) { return pair0 + (size_t)n * (n - 1) / 2 + m; };
    // key chunk of step s: down steps s < nA walk m = nA-1 .. 0, up steps walk m = 0 .. nA-1
    auto key_of = [&](int s) { return s < nA ? nA - 1 - s : s - nA; };

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_do); prefetch_tmap(&tm_k); prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_ph); prefetch_tmap(&tm_pl); prefetch_tmap(&tm_ds);
            mbar_expect_tx(bar(B_DO), 32768);
            for (int h = 0; h < 2; ++h) {
                tma_load_3d(sb + R_O + h * 16384, &tm_do, bar(B_DO), h * 64, nA * C, bh);
                tma_load_3d(sb + R_O + h * 16384 + 8192, &tm_do, bar(B_DO), h * 64, nB * C, bh);
            }
            int kv = 0, pp = 0;  // fills issued
            bool ok = true;
            for (int s = 0; s < steps && ok; ++s) {
                const int m = key_of(s);
                const bool up = s >= nA;
                if (kv > 0 && !(ok = mbar_wait(bar(B_KVE), (uint32_t)((kv - 1) & 1), wc, 120))) break;
                // the upward walk reads dS back from the pair store: wait until the epilogue has
                // written (and fenced) every down step's dS (READY completion nA)
                if (s == nA && !(ok = mbar_wait(bar(B_READY), (uint32_t)(nA & 1), wc, 119))) break;
                uint32_t bytes = 16384 + (up ? 8192u + (m < nB ? 8192u : 0u) : 16384u);
                mbar_expect_tx(bar(B_KV), bytes);
                for (int h = 0; h < 2; ++h)
                    tma_load_3d(sb + R_K + h * 8192, &tm_k, bar(B_KV), h * 64, m * C, bh);
                if (!up) {
                    for (int h = 0; h < 2; ++h) tma_load_3d(sb + R_V + h * 8192, &tm_v, bar(B_KV), h * 64, m * C, bh);
                } else {  // dS of both chunks into the rows of the (free) dO tile
                    tma_load_3d(sb + R_O, &tm_ds, bar(B_KV), 0, 0, (int)pair_index(nA, m));
                    if (m < nB) tma_load_3d(sb + R_O + 8192, &tm_ds, bar(B_KV), 0, 0, (int)pair_index(nB, m));
                }
                ++kv;
                if (m >= 1) {
                    if (pp > 0 && !(ok = mbar_wait(bar(B_PE), (uint32_t)((pp - 1) & 1), wc, 121))) break;
                    mbar_expect_tx(bar(B_P), 65536);
                    const int z = bh * p.N + m;
                    for (int h = 0; h < 2; ++h) {
                        tma_load_3d(sb + R_PH + h * 16384, &tm_ph, bar(B_P), h * 64, 0, z);
                        tma_load_3d(sb + R_PL + h * 16384, &tm_pl, bar(B_P), h * 64, 0, z);
                    }
                    ++pp;
                }
            }
            // copies in flight land before the CTA exits
            drain_wait(bar(B_DO), 0, p.limit_ns, p.hdr, 122);
            if (kv > 0) drain_wait(bar(B_KV), (uint32_t)((kv - 1) & 1), p.limit_ns, p.hdr, 123);
            if (pp > 0) drain_wait(bar(B_P), (uint32_t)((pp - 1) & 1), p.limit_ns, p.hdr, 124);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int pp = 0;
            bool ok = mbar_wait(bar(B_DO), 0, wc, 125);
            for (int s = 0; s < steps && ok; ++s) {
                const int m = key_of(s);
                const bool up = s >= nA;
                // operands of step s loaded; the epilogue has consumed step s-1 and written U or G
                if (!(ok = mbar_wait(bar(B_KV), (uint32_t)(s & 1), wc, 126) &&
                           mbar_wait(bar(B_READY), (uint32_t)(s & 1), wc, 127)))
                    break;
                tc_fence_after();
                if (!up) {
                    for (int kk = 0; kk < D / 16; ++kk) {
                        mma_ss(tmem + TM_S, kmajor_desc(sb + R_UH, kk, 16384), kmajor_desc(sb + R_K, kk, 8192), ID_S,
                               kk > 0);
                        mma_ss(tmem + TM_DP, kmajor_desc(sb + R_O, kk, 16384), kmajor_desc(sb + R_V, kk, 8192), ID_S,
                               kk > 0);
                    }
                    mma_commit(bar(B_S));
                } else {
                    for (int kk = 0; kk < C / 16; ++kk)  // T = dS khat (K = 64)
                        mma_ss(tmem + TM_T, kmajor_desc(sb + R_O, kk, 16384),
                               sdesc_sw128(sb + R_K + (uint32_t)kk * 2048u, 8192, 1024), ID_G, kk > 0);
                }
                if (m >= 1) {
                    if (!(ok = mbar_wait(bar(B_P), (uint32_t)(pp & 1), wc, 128))) break;
                    tc_fence_after();
                    // down: U P^T (B = rows of P, K-major); up: G P (B = P, MN-major)
                    for (int t = 0; t < 3; ++t) {
                        const uint32_t a = t == 2 ? R_UL : R_UH, b = t == 1 ? R_PL : R_PH;
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint64_t bd = up ? mnmajor_desc(sb + b, kk) : kmajor_desc(sb + b, kk, 16384);
                            mma_ss(tmem + TM_U, kmajor_desc(sb + a, kk, 16384), bd, up ? ID_G : ID_U,
                                   (t > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    mma_commit(bar(B_PE));
                    ++pp;
                }
                mma_commit(bar(B_KVE));
                mma_commit(up ? bar(B_UP) : bar(B_U));
            }
            mma_commit(bar(B_DRAIN));
            drain_wait(bar(B_DRAIN), 0, p.limit_ns, p.hdr, 129);
        }
    } else {
        // ------------------------------------------------------------------ epilogue (warps 2-9)
        // Warp w reads TMEM lanes 32 (w % 4) .. + 31 (the quarter its SM sub-partition may access);
        // warps w and w + 4 share those rows, `half` 0 taking the first half of every row's columns
        // (S / dP columns 0-31, U / G / T columns 0-63) and `half` 1 the second.  Each warp writes
        // and copies out only its own columns, so the two need no synchronisation beyond READY.
        const int qw = warp & 3, half = (warp - 2) >> 2;
        const int i = 32 * qw + lane;  // tile row = TMEM lane
        const uint32_t tl = tmem + ((uint32_t)(32 * qw) << 16);
        const int chunk = i < 64 ? nA : nB, r = i & 63;
        const int g = chunk * C + r;  // query position
        const bool valid = g < p.L;
        const size_t hrow = (size_t)bh * p.L + g, prow = (size_t)bh * p.Lp + g;
        const float lse = valid ? p.lse[hrow] : 0.f, del = valid ? p.delta[prow] : 0.f;
        const float ci = (FOX && valid) ? p.cum[prow] : 0.f;
        // p_ij = 2^(scale log2e S_ij + off - log2e c_j); off = -inf for rows the chain does not cover
        // at this key chunk gives p_ij = 0 without a select per element
        constexpr float kLog2e = 1.4426950408889634f;
        const float l2s = p.scale * kLog2e, off_in = (ci - lse) * kLog2e;
        uint8_t* uh = sm + R_UH;
        uint8_t* ul = sm + R_UL;
        uint8_t* stg = sm + R_ST + (uint32_t)(warp - 2) * 4096u;
        const int r0 = r & ~31;  // the warp's first row within its chunk
        float rowsum = 0.f;
        // the hi parts of the warp's columns (64 of 128) of its 32 rows of U (or G) to the rows at dst
        // (row stride 128 elements): one 128-byte segment per row, four rows per instruction
        auto copy_rows = [&](__nv_bfloat16* dst) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int row = 4 * k + (lane >> 3), gg = lane & 7;
                *reinterpret_cast<uint4*>(dst + row * D + 64 * half + 8 * gg) =
                    *reinterpret_cast<const uint4*>(uh + sw_off(32 * qw + row, 8 * half + gg, 16384));
            }
        };
        // initial U: qbar of chunk nA (chunk nB's rows start at zero and take qbar after key chunk nB)
        auto put_row = [&](const float* src) {  // src: the row's 128 fp32 values (global) or nullptr for zeros
#pragma unroll 4
            for (int gr = 8 * half; gr < 8 * half + 8; ++gr) {
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = src ? src[8 * gr + e] : 0.f;
                put_hilo(uh, ul, i, gr, v);
            }
        };
        put_row(i < 64 && valid ? p.qbar + prow * D : nullptr);
        fence_proxy_async_smem();
        mbar_arrive(bar(B_READY));
        int su = 0, sd = 0, upw = 0;  // completed waits on B_S, B_U, B_UP
        bool ok = true;
        for (int s = 0; s < steps && ok; ++s) {
            const int m = key_of(s);
            const bool up = s >= nA;
            const bool act = valid && m < chunk;  // this row's chain covers key chunk m
            // every row of a covered pair is written (padded rows of a ragged chunk carry zeros), so
            // the reduction never reads uninitialised rows
            __nv_bfloat16* rec =
                m < chunk ? p.pairs + pair_index(chunk, m) * (size_t)(2 * C * D + 2 * C * C) : nullptr;
            if (!up) {
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(B_S), (uint32_t)(sd & 1), wc, 130)))) break;
                ++sd;
                tc_fence_after();
                const float off = act ? off_in : -INFINITY;
                float csum[32];
                {
                    const int h = half;
                    uint32_t sv[32], dv[32];
                    tmem_ld32(tl + TM_S + 32 * h, sv);
                    tmem_ld32(tl + TM_DP + 32 * h, dv);
                    tmem_wait_ld();
                    uint32_t pw[16], dw[16];
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        float pr[2], ds[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int jj = 32 * h + j + e;  // key column
                            float x = fmaf(l2s, __uint_as_float(sv[j + e]), off);
                            if constexpr (FOX) x -= kLog2e * p.cum[(size_t)bh * p.Lp + m * C + jj];
                            pr[e] = ex2_approx(x);
                            ds[e] = pr[e] * (__uint_as_float(dv[j + e]) - del);
                            if constexpr (FOX) {
                                csum[j + e] = ds[e];
                                rowsum += ds[e];
                            }
                        }
                        pw[j / 2] = pack_bf16x2(pr[0], pr[1]);
                        dw[j / 2] = pack_bf16x2(ds[0], ds[1]);
                    }
                    if (rec) {  // row `lane` of the warp's staging tiles, 16-byte granules XOR-swizzled by row pair
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint32_t o = (uint32_t)lane * 64u + (uint32_t)((q ^ ((lane >> 1) & 3)) << 4);
                            *reinterpret_cast<uint4*>(stg + o) = make_uint4(dw[4 * q], dw[4 * q + 1], dw[4 * q + 2], dw[4 * q + 3]);
                            *reinterpret_cast<uint4*>(stg + 2048 + o) =
                                make_uint4(pw[4 * q], pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]);
                        }
                    }
                }
                if constexpr (FOX) {  // column sums of dS over the 32 rows of the warp, then across warps
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        float t = csum[jj];
#pragma unroll
                        for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                        if (lane == jj) atomicAdd(p.dccol + (size_t)bh * p.Lp + m * C + 32 * half + jj, t);
                    }
                }
                if (rec) {  // the warp's columns of its 32 rows of dS, P and U_{chunk,m} (the hi part the logits
                            // used) to the pair store, whole 32-byte sectors, eight or four rows per instruction
                    __syncwarp();
                    __nv_bfloat16* dsd = rec + 2 * C * D + r0 * C + 32 * half;
                    __nv_bfloat16* pd = dsd + C * C;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int row = 8 * k + (lane >> 2), gg = lane & 3;
                        const uint32_t o = (uint32_t)row * 64u + (uint32_t)((gg ^ ((row >> 1) & 3)) << 4);
                        *reinterpret_cast<uint4*>(dsd + row * C + 8 * gg) = *reinterpret_cast<const uint4*>(stg + o);
                        *reinterpret_cast<uint4*>(pd + row * C + 8 * gg) = *reinterpret_cast<const uint4*>(stg + 2048 + o);
                    }
                    copy_rows(rec + r0 * D);
                    __syncwarp();
                }
                if (m >= 1) {  // U <- U P_m^T, or qbar for chunk nB's rows once key chunk nB is passed
                    if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(B_U), (uint32_t)(su & 1), wc, 131)))) break;
                    ++su;
                    tc_fence_after();
                    if (i >= 64 && m == nB) {
                        put_row(valid ? p.qbar + prow * D : nullptr);
                    } else {
#pragma unroll
                        for (int h = 2 * half; h < 2 * half + 2; ++h) {
                            uint32_t v[32];
                            tmem_ld32(tl + TM_U + 32 * h, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int gr = 0; gr < 4; ++gr) {
                                float x[8];
#pragma unroll
                                for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(v[8 * gr + e]);
                                put_hilo(uh, ul, i, 4 * h + gr, x);
                            }
                        }
                    }
                }
            } else {
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(B_UP), (uint32_t)(upw & 1), wc, 132)))) break;
                ++upw;
                tc_fence_after();
                if (rec && m >= 1) {  // G_{chunk,m-1} (hi part) of the warp's rows to the pair store
                    __syncwarp();  // rows written by other lanes in the previous step
                    copy_rows(rec + C * D + r0 * D);
                    __syncwarp();
                }
                const bool last = valid && m == chunk - 1;  // the row's chain ends here: G is dqbar
#pragma unroll
                for (int h = 2 * half; h < 2 * half + 2; ++h) {
                    uint32_t tv[32], gv[32];
                    tmem_ld32(tl + TM_T + 32 * h, tv);
                    if (m >= 1) tmem_ld32(tl + TM_U + 32 * h, gv);
                    tmem_wait_ld();
                    float x[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        x[e] = p.scale * __uint_as_float(tv[e]) + (m >= 1 ? __uint_as_float(gv[e]) : 0.f);
#pragma unroll
                    for (int gr = 0; gr < 4; ++gr) put_hilo(uh, ul, i, 4 * h + gr, x + 8 * gr);
                    if (last) {
                        float4* dq = reinterpret_cast<float4*>(p.dqbar + prow * D + 32 * h);
#pragma unroll
                        for (int q = 0; q < 8; ++q) dq[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
                    }
                }
            }
            fence_proxy_async_smem();
            if (!up) fence_proxy_async_global();  // dS / P / U rows are read back by TMA
            tc_fence_before();
            mbar_arrive(bar(B_READY));
        }
        // the two warps of a row each hold the sum over their columns; dcrow was zeroed by the launcher,
        // and a sum of two terms does not depend on their order
        if (FOX && valid && chunk >= 1) atomicAdd(p.dcrow + prow, rowsum);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}


// The chains for bf16, d = 128: dO and v the caller's [BH, L, 128] bf16; khat16, phi,
// plo the bf16 copies bwd_prep writes; pairs the bf16 pair store (written here).
cudaError_t launch_bwd_chain_tc(const void* dO, const void* v, const void* khat16, const void* phi, const void* plo,
                                void* pairs, const float* qbar, const float* lse, const float* delta,
                                const float* cum, float* dqbar, float* dcrow, float* dccol, int fox, int BH, int L,
                                int Lp, int N, size_t head_pairs, float scale, WsHeader* hdr, cudaStream_t st) {
    using namespace ctk;
    if (N < 2) return cudaSuccess;
    const uint64_t pair_bytes = (2ull * C * D + 2ull * C * C) * 2;
    const uint64_t npairs = (uint64_t)BH * head_pairs;
    CUtensorMap mdo, mk, mv, mph, mpl, mds;
    if (!make_map_rows64(&mdo, dO, D, (uint64_t)L, (uint64_t)BH, D * 2, (uint64_t)L * D * 2) ||
        !make_map_rows64(&mk, khat16, D, (uint64_t)Lp, (uint64_t)BH, D * 2, (uint64_t)Lp * D * 2) ||
        !make_map_rows64(&mv, v, D, (uint64_t)L, (uint64_t)BH, D * 2, (uint64_t)L * D * 2) ||
        !make_map_t(&mph, phi, D, D, BH * N, false) || !make_map_t(&mpl, plo, D, D, BH * N, false) ||
        !make_map_rows64(&mds, static_cast<const uint8_t*>(pairs) + (size_t)2 * C * D * 2, C, C, npairs, C * 2,
                         pair_bytes))
        return cudaErrorInvalidValue;
    CtParams p;
    p.N = N;
    p.L = L;
    p.Lp = Lp;
    p.head_pairs = head_pairs;
    p.scale = scale;
    p.fox = fox;
    p.qbar = qbar;
    p.lse = lse;
    p.delta = delta;
    p.cum = cum;
    p.dqbar = dqbar;
    p.dcrow = dcrow;
    p.dccol = dccol;
    p.pairs = static_cast<__nv_bfloat16*>(pairs);
    p.hdr = hdr;
    p.limit_ns = 2000000000ull;
    auto kern = fox ? bwd_chain_tc<true> : bwd_chain_tc<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    mark_start(st);
    kern<<<dim3(N / 2, BH), kThreads, kSmem, st>>>(mdo, mk, mv, mph, mpl, mds, p);
    mark_end(st);
    return cudaGetLastError();
}

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
