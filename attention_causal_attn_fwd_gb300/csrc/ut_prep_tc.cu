// UT-transform preparation on GB300 tensor cores (bf16 inputs, chunk C = 128).
//
// "Resumo Técnico: Atenção PaTH" (gist.science/pt/paper/2505.16381), §3
// "Representação de Transformação UT": the product of a chunk's transitions
// is P = I - W^T A W with A = (I + D triu_1(W W^T))^{-1} D, D = diag(beta); §3
// "Algoritmo Estilo FlashAttention", first sub-bullet: the chunk's
// boundary-adjusted queries and keys.  Per chunk this kernel writes
//     P - I = W^T (-V),  V = A W          (scan transition, bf16, d x d)
//      Y   = tril(Q W^T) A^T              (diagonal block, bf16)
//     qhat = Q - Y W                      (fp32)
//     -Z   = -triu_1(K W^T)               (diagonal block, bf16)
//     khat = K - (Z A) W = K - Z V        (bf16)
// and, for the prefill hand-off, V itself.  (The fp32 CUDA-core version in
// ut_prep.cu writes -U = -A^T W in place of P - I: its scan applies the
// transition as two products.)
//
// Products run as tcgen05 MMAs (M = 128) with fp32 accumulation in TMEM.
// Operands that are not exact in bf16 (A, tril(QW^T), Y, Z, V) are split
// into hi + lo bf16 parts and multiplied term by term (hi*hi + hi*lo + lo*hi),
// which keeps those products close to fp32 accuracy; -V enters P - I as one
// bf16 operand (P - I is itself stored in bf16).  A = X D with the unit upper-
// triangular X = (I + D triu_1(G))^{-1} is solved in fp32 on CUDA cores,
// blocked: the 16 x 16 diagonal blocks of X by back substitution, scaled by D
// into those of A, then three doubling merges A_PQ = -A_PP G_PQ A_QQ (which
// is X_PQ D_Q for X_PQ = -X_PP D_P G_PQ X_QQ) on a dense copy of A kept in the
// shared memory that held Q and K.
//
// One shared-memory layout — rows of 64-element, 128-byte-swizzled chunks,
// exactly what a TMA box {64, 128} writes — serves as a K-major operand, an
// MN-major B operand and an MN-major ("transposed") A operand, so W and A are
// staged once each.
//
// Roles (320 threads): warp 0 TMA loads, TMEM allocation and the workspace
// stores (bulk tensor stores of staged tiles), warp 1 MMA issue,
// warps 2-9 solve, conversions and stores (one TMEM lane = one chunk row; the
// two warps sharing a lane quarter split the columns).  Waits are bounded;
// a timeout sets PATH_ERR_TIMEOUT and every role stops, drains and frees TMEM.
#include <cstdio>

#include "common.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.cuh"
#include "ut_prep.cuh"

namespace pathattn {
using namespace sm100;

namespace utk {
constexpr int C = 128;
constexpr int kThreads = 320;
constexpr int kCompute = 256;   // warps 2-9: two warps per TMEM lane quarter
constexpr uint32_t R0 = 0;        // W            (K-major / MN-major source), then qhat staging
constexpr uint32_t R1 = 32768;    // Q, then solve temp, then A_hi, then V_hi
constexpr uint32_t R2 = 65536;    // K, then A_lo, then V_lo, then khat staging
constexpr uint32_t R3 = 98304;    // G fp32 [128][132] for the solve, then hi/lo operand (hi, hi + 32 KB = lo)
constexpr int LDG = 132;          // rows start on 16-byte boundaries
constexpr uint32_t RB = R3 + 128 * LDG * 4;  // barriers, beta
constexpr uint32_t RT = RB + 1024;            // solve temp T [64][68] fp32
constexpr int LDT = 68;
constexpr uint32_t RS = RT + 64 * LDT * 4;    // output staging tile for TMA stores (32 KB)
static_assert(RS % 1024 == 0, "128-byte-swizzled tiles start on 1024-byte boundaries");
constexpr uint32_t TOTAL = RS + 32768;
// Operand tiles of the level-64 merge on the tensor cores (hi part, lo part
// 16 KB / 8 KB after it): G_PQ, then A_PP (rows 0-63 of an M = 128 K-major
// tile) in the staging tile; A_QQ, then T, as a 64-row MN-major B in the
// solve temp.
constexpr uint32_t RM_A = RS, RM_B = RT;
static_assert(64 * LDT * 4 >= 16384, "the solve temp holds the hi and lo 8 KB B tiles");
constexpr size_t kSmem = TOTAL + 1024;
constexpr uint32_t T0 = 0, T128 = 128, T256 = 256, T384 = 384;
// B_STG*: a workspace-store group is staged (compute warps); B_FREE*: its
// tiles have been read by the bulk stores (store thread).  Groups: 0 Y (R3);
// 1 P - I (staging tile, which held -V as the operand of P - I); 2 -Z (R3),
// qhat columns 0-31 of each half (staging tile); 3 qhat columns 32-63
// (d = 128; R0, free once Y W and P - I have completed); last khat (R2, free
// once Z V has completed).
// B_M64*: the merge at level 64 on the tensor cores (operands staged, T done,
// T staged, A_PQ done).
enum { B_LOAD = 0, B_G, B_QK, B_M64A, B_M64T, B_M64B, B_M64R, B_OPS1, B_UY, B_OPS2, B_Q, B_OPS3, B_K, B_DRAIN,
       B_STG0, B_STG1, B_STG2, B_STG3, B_STG4, B_FREE0, B_FREE1, B_FREE2, B_FREE3, B_FREE4, B_COUNT };
constexpr uint32_t RB_SLOT = 200;  // TMEM address and abort flag after the barriers
static_assert(B_COUNT * 8 <= RB_SLOT && RB_SLOT + 8 <= 256, "barriers overlap the TMEM slot, abort flag or beta");
}  // namespace utk

// Phase timestamps of one CTA in the middle of the grid (SM cycle counter),
// compiled in only for instrumented builds (-DPATH_TRACE).
#ifdef PATH_TRACE
#define UT_TRACE(slot) \
    do { if (p.trace && blockIdx.x == 10 && blockIdx.y == 40) p.trace[(slot)] = clock64(); } while (0)
// Per-CTA global-timer stamps (every CTA): 0 entry, 1 compute warps' start, 2 exit, 3 SM id.
constexpr int kUtTraceCtaBase = 64, kUtTraceMaxCtas = 65536;
#define UT_CTA(slot, val)                                                                           \
    do {                                                                                            \
        const unsigned cta_ = blockIdx.y * gridDim.x + blockIdx.x;                                  \
        if (p.trace && cta_ < kUtTraceMaxCtas) p.trace[kUtTraceCtaBase + cta_ * 4 + (slot)] = (val); \
    } while (0)
#else
#define UT_TRACE(slot) do { } while (0)
#define UT_CTA(slot, val) do { } while (0)
#endif

struct UtParams {
    int L, Lp, BH;
    const float* beta;           // [BH, L]
    const __nv_bfloat16* q;      // [BH, L, d] (row reads for the "Q -" epilogue)
    const __nv_bfloat16* k;
    float* qhat;                 // [BH, Lp, d]
    __nv_bfloat16* khat;         // [BH, Lp, d]
    __nv_bfloat16* un;           // [BH, Lp, d]
    __nv_bfloat16* y;            // [BH, Lp, C]
    __nv_bfloat16* zn;           // [BH, Lp, C]
    __nv_bfloat16* vfac;         // [BH, Lp, d] V = A W (prefill cache only) or null
    float* kmax2;                // [BH, nch] max |khat|^2 per chunk (PaTH-FoX) or null
    int nch;
    int ahead;                   // L2 prefetch of the inputs of the CTA launched `ahead` later (0: none)
    int reset;                   // the first CTA clears the workspace header's status and visited count
    WsHeader* hdr;
    unsigned long long limit_ns;
#ifdef PATH_TRACE
    unsigned long long* trace;
#endif
};

__device__ __forceinline__ uint4 pack8(const float* v) {
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
}
// 16 bytes of row r into a staging tile laid out as a TMA store box sequence:
// 128-byte rows, 128 rows per 16 KB box, 128-byte swizzle; `box` selects the
// box and `g` the 16-byte granule of the row.
__device__ __forceinline__ void stage16(uint8_t* base, int r, int box, int g, uint4 v) {
    *reinterpret_cast<uint4*>(base + (uint32_t)box * 16384u + (uint32_t)r * 128u +
                              ((uint32_t)((g & 7) ^ (r & 7)) << 4)) = v;
}

// One doubling merge of the blocked factor A = X D, for 256 threads t: for each
// pair of S-blocks (P, Q = P + S) on the diagonal,
//     T    = G_PQ A_QQ
//     A_PQ = -A_PP T
// with A dense (zeros below the diagonal), so the products are plain
// register-tiled loops.  The k loop takes 4 steps at a time so that
// every operand is read as 16- or 8-byte row segments (rows of G, X and T
// start on 16-byte boundaries): 2 x (TM + 4) vector loads per 4 x TM x TN FMAs.
template <int TN>
__device__ __forceinline__ void ld_row(float (&dst)[TN], const float* src) {
    static_assert(TN == 2 || TN == 4, "row segment");
    if constexpr (TN == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
    } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        dst[0] = v.x; dst[1] = v.y;
    }
}
template <int S, int TM, int TN>
__device__ __forceinline__ void merge_level(const float* sG, float* sX, float* sT, int t) {
    using namespace utk;
    constexpr int NP = C / (2 * S);
    constexpr int TR = S / TM, TC = S / TN;
    static_assert(NP * TR * TC == kCompute, "one tile per thread");
    static_assert(S % 4 == 0 && LDG % 4 == 0 && LDT % 4 == 0 && C % 4 == 0, "16-byte row segments");
    const int p = t / (TR * TC), rem = t % (TR * TC);
    const int i0 = (rem / TC) * TM, j0 = (rem % TC) * TN;
    const int P = 2 * p * S, Q = P + S;
    float acc[TM][TN];
#pragma unroll
    for (int u = 0; u < TM; ++u)
#pragma unroll
        for (int v = 0; v < TN; ++v) acc[u][v] = 0.f;
#pragma unroll 2
    for (int k4 = 0; k4 < S; k4 += 4) {
        float g[TM][4], x[4][TN];
#pragma unroll
        for (int u = 0; u < TM; ++u) ld_row<4>(g[u], sG + (P + i0 + u) * LDG + Q + k4);
#pragma unroll
        for (int e = 0; e < 4; ++e) ld_row<TN>(x[e], sX + (Q + k4 + e) * C + Q + j0);
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int u = 0; u < TM; ++u)
#pragma unroll
                for (int v = 0; v < TN; ++v) acc[u][v] = fmaf(g[u][e], x[e][v], acc[u][v]);
    }
#pragma unroll
    for (int u = 0; u < TM; ++u)
#pragma unroll
        for (int v = 0; v < TN; ++v) sT[(p * S + i0 + u) * LDT + j0 + v] = acc[u][v];
    named_bar_sync(1, kCompute);
#pragma unroll
    for (int u = 0; u < TM; ++u)
#pragma unroll
        for (int v = 0; v < TN; ++v) acc[u][v] = 0.f;
#pragma unroll 2
    for (int k4 = 0; k4 < S; k4 += 4) {
        float xp[TM][4], tv[4][TN];
#pragma unroll
        for (int u = 0; u < TM; ++u) ld_row<4>(xp[u], sX + (P + i0 + u) * C + P + k4);
#pragma unroll
        for (int e = 0; e < 4; ++e) ld_row<TN>(tv[e], sT + (p * S + k4 + e) * LDT + j0);
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int u = 0; u < TM; ++u)
#pragma unroll
                for (int v = 0; v < TN; ++v) acc[u][v] = fmaf(xp[u][e], tv[e][v], acc[u][v]);
    }
#pragma unroll
    for (int u = 0; u < TM; ++u)
#pragma unroll
        for (int v = 0; v < TN; ++v) sX[(P + i0 + u) * C + Q + j0 + v] = -acc[u][v];
    named_bar_sync(1, kCompute);
}

// The same merge without the zero halves of the triangular factors:
// T = G_PQ A_QQ needs only k <= j and A_PQ = -A_PP T only k >= i (both A
// blocks are upper triangular).  Pass 1 gives each warp WC adjacent column
// tiles and pass 2 WR adjacent row tiles, so a warp's k range is uniform; the
// two warps that share a scheduler (compute warps cw and cw + 4) get
// complementary ranges.  G is symmetric, so the G column needed for row
// segment i0.. is read as 16- or 8-byte segments of row Q + k.
template <int S, int TM, int TN>
__device__ __forceinline__ void merge_level_tri(const float* sG, float* sX, float* sT, int t) {
    using namespace utk;
    constexpr int NP = C / (2 * S);
    constexpr int TR = S / TM, TC = S / TN;
    constexpr int WPP = TR * TC / 32;  // warps per diagonal pair
    constexpr int WC = 32 / TR, WR = 32 / TC;
    static_assert(NP * WPP == kCompute / 32 && 32 % TR == 0 && 32 % TC == 0, "warp tiling");
    static_assert((WC * TN) % 4 == 0 && (WR * TM) % 4 == 0, "k ranges in steps of 4");
    const int cw = t >> 5, lane = t & 31;
    const int pr = cw / WPP;
    const int wp = cw < 4 ? cw % WPP : WPP - 1 - (cw - 4) % WPP;
    const int P = 2 * pr * S, Q = P + S;
    float acc[TM][TN];
    {  // pass 1: T = G_PQ A_QQ over k < kend
        const int i0 = (lane % TR) * TM, j0 = (wp * WC + lane / TR) * TN;
        const int kend = (wp + 1) * WC * TN;
#pragma unroll
        for (int u = 0; u < TM; ++u)
#pragma unroll
            for (int v = 0; v < TN; ++v) acc[u][v] = 0.f;
#pragma unroll 2
        for (int k4 = 0; k4 < kend; k4 += 4) {
            float g[4][TM], x[4][TN];
#pragma unroll
            for (int e = 0; e < 4; ++e) ld_row<TM>(g[e], sG + (Q + k4 + e) * LDG + P + i0);
#pragma unroll
            for (int e = 0; e < 4; ++e) ld_row<TN>(x[e], sX + (Q + k4 + e) * C + Q + j0);
#pragma unroll
            for (int e = 0; e < 4; ++e)
#pragma unroll
                for (int u = 0; u < TM; ++u)
#pragma unroll
                    for (int v = 0; v < TN; ++v) acc[u][v] = fmaf(g[e][u], x[e][v], acc[u][v]);
        }
#pragma unroll
        for (int u = 0; u < TM; ++u)
#pragma unroll
            for (int v = 0; v < TN; ++v) sT[(pr * S + i0 + u) * LDT + j0 + v] = acc[u][v];
    }
    named_bar_sync(1, kCompute);
    {  // pass 2: A_PQ = -A_PP T over k >= kbeg
        const int i0 = (wp * WR + lane / TC) * TM, j0 = (lane % TC) * TN;
        const int kbeg = wp * WR * TM;
#pragma unroll
        for (int u = 0; u < TM; ++u)
#pragma unroll
            for (int v = 0; v < TN; ++v) acc[u][v] = 0.f;
#pragma unroll 2
        for (int k4 = kbeg; k4 < S; k4 += 4) {
            float xp[TM][4], tv[4][TN];
#pragma unroll
            for (int u = 0; u < TM; ++u) ld_row<4>(xp[u], sX + (P + i0 + u) * C + P + k4);
#pragma unroll
            for (int e = 0; e < 4; ++e) ld_row<TN>(tv[e], sT + (pr * S + k4 + e) * LDT + j0);
#pragma unroll
            for (int e = 0; e < 4; ++e)
#pragma unroll
                for (int u = 0; u < TM; ++u)
#pragma unroll
                    for (int v = 0; v < TN; ++v) acc[u][v] = fmaf(xp[u][e], tv[e][v], acc[u][v]);
        }
#pragma unroll
        for (int u = 0; u < TM; ++u)
#pragma unroll
            for (int v = 0; v < TN; ++v) sX[(P + i0 + u) * C + Q + j0 + v] = -acc[u][v];
    }
    named_bar_sync(1, kCompute);
}

// The 16 x 16 diagonal blocks of X = (I + D triu_1(G))^{-1} (unit upper
// triangular) by back substitution, written as those of A = X D (column j
// scaled by beta_j) into the dense, zeroed sX [128][128], for 256 threads t
// (the merges above then fill the rest); sG holds G (upper part read).
__device__ __forceinline__ void solve_diag_blocks(const float* sG, const float* sB, float* sX, int t) {
    using namespace utk;
    if (t < 128) {  // 16 x 16 diagonal blocks: thread (block I, column j) back-substitutes its column
        const int I = t >> 4, j = t & 15, b0 = I * 16;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
        for (int i = 14; i >= 0; --i) {
            float acc = 0.f;
#pragma unroll
            for (int kk = i + 1; kk < 16; ++kk) acc = fmaf(sG[(b0 + i) * LDG + b0 + kk], x[kk], acc);
            const float val = -sB[b0 + i] * acc;
            if (i < j) x[i] = val;
        }
        const float bj = sB[b0 + j];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (i <= j) sX[(b0 + i) * C + b0 + j] = x[i] * bj;
    }
    named_bar_sync(1, kCompute);
}

template <int D>
__global__ void __launch_bounds__(utk::kThreads, 1)
    ut_prep_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_un,
               const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ CUtensorMap tm_zn,
               const __grid_constant__ CUtensorMap tm_khat, const __grid_constant__ CUtensorMap tm_qhat,
               const UtParams p) {
    using namespace utk;
    static_assert(D == 64 || D == 128, "head dim");
    constexpr int KCH = D / 64;
    constexpr uint32_t TILE = 128u * D * 2u;
    constexpr uint32_t ID_KK128 = idesc_bf16_ab(128, false, false);
    constexpr uint32_t ID_KMN_D = idesc_bf16_ab(D, false, true);
    constexpr uint32_t ID_MNMN_D = idesc_bf16_ab(D, true, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    auto bar = [&](int i) { return sb + RB + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + RB + RB_SLOT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + RB + RB_SLOT + 4);
    float* sBeta = reinterpret_cast<float*>(sm + RB + 256);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Heads run last to first: the scan starts with the first head group, whose
    // outputs are then the most recently written (still in L2).
    const int chunk = blockIdx.x, bh = (int)gridDim.y - 1 - (int)blockIdx.y;
    const int row0 = chunk * C;
    if (p.reset && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {  // the first CTA launched
        p.hdr->status = 0;
        p.hdr->visited = 0;
    }
    if (threadIdx.x == 0) {
        UT_CTA(0, globaltimer());
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        UT_CTA(3, smid);
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < B_COUNT; ++i)
            mbar_init(bar(i), (i == B_OPS1 || i == B_OPS2 || i == B_OPS3 || i == B_M64A || i == B_M64B ||
                               (i >= B_STG0 && i <= B_STG4))
                                  ? kCompute : 1);
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
        if (lane == 0) {
            prefetch_tmap(&tm_q); prefetch_tmap(&tm_k); prefetch_tmap(&tm_w);
            mbar_expect_tx(bar(B_LOAD), 3 * TILE);
            for (int c = 0; c < KCH; ++c) {
                tma_load_3d(sb + R0 + c * 16384, &tm_w, bar(B_LOAD), c * 64, row0, bh);
                tma_load_3d(sb + R1 + c * 16384, &tm_q, bar(B_LOAD), c * 64, row0, bh);
                tma_load_3d(sb + R2 + c * 16384, &tm_k, bar(B_LOAD), c * 64, row0, bh);
            }
            // warm L2 for the inputs of the CTA launched `ahead` after this one
            if (p.ahead > 0) {
                const int lin = (int)(blockIdx.y * gridDim.x + blockIdx.x) + p.ahead;
                if (lin < (int)(gridDim.x * gridDim.y)) {
                    const int c2 = lin % (int)gridDim.x, bh2 = (int)gridDim.y - 1 - lin / (int)gridDim.x;
                    for (int c = 0; c < KCH; ++c) {
                        tma_prefetch_3d(&tm_w, c * 64, c2 * C, bh2);
                        tma_prefetch_3d(&tm_q, c * 64, c2 * C, bh2);
                        tma_prefetch_3d(&tm_k, c * 64, c2 * C, bh2);
                    }
                }
            }
            drain_wait(bar(B_LOAD), 0, p.limit_ns, p.hdr, 98);
            // Workspace stores: this thread issues each group once the compute
            // warps have staged it and frees its tiles once the stores have read
            // them, so no compute thread waits on a bulk store.
            constexpr int kGroups = D == 128 ? 5 : 4;
            bool ok = true;
            for (int g = 0; g < kGroups && ok; ++g) {
                if (!(ok = mbar_wait_sleep(bar(B_STG0 + g), 0, wc, 45 + g))) break;
                if (g == 0) {
                    for (int b = 0; b < 2; ++b) tma_store_3d(&tm_y, sb + R3 + b * 16384, 64 * b, row0, bh);
                } else if (g == 1) {
                    for (int b = 0; b < D / 64; ++b) tma_store_3d(&tm_un, sb + RS + b * 16384, 64 * b, row0, bh);
                } else if (g == 2 || (D == 128 && g == 3)) {
                    const int c = g - 2;  // qhat columns 32c .. 32c+31 of each half
                    const uint32_t src = sb + (c == 0 ? RS : R0);
                    for (int b = 0; b < 2; ++b)
                        tma_store_3d(&tm_qhat, src + b * 16384, (D / 2) * b + 32 * c, row0, bh);
                    if (g == 2)
                        for (int b = 0; b < 2; ++b) tma_store_3d(&tm_zn, sb + R3 + b * 16384, 64 * b, row0, bh);
                } else {
                    for (int b = 0; b < D / 64; ++b) tma_store_3d(&tm_khat, sb + R2 + b * 16384, 64 * b, row0, bh);
                }
                bulk_commit();
                bulk_wait_read0();
                mbar_arrive(bar(B_FREE0 + g));
            }
            bulk_wait0();  // the workspace stores have landed before the CTA exits
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = mbar_wait(bar(B_LOAD), 0, wc, 40);
            UT_TRACE(13);
            if (ok) {
                tc_fence_after();
                // G = W W^T first, on its own barrier (the solve needs only G), then Q W^T, K W^T
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + T0, kmajor_desc(sb + R0, kk, 16384), kmajor_desc(sb + R0, kk, 16384), ID_KK128, kk > 0);
                mma_commit(bar(B_G));
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t bw = kmajor_desc(sb + R0, kk, 16384);
                    mma_ss(tmem + T128, kmajor_desc(sb + R1, kk, 16384), bw, ID_KK128, kk > 0);
                    mma_ss(tmem + T256, kmajor_desc(sb + R2, kk, 16384), bw, ID_KK128, kk > 0);
                }
                mma_commit(bar(B_QK));
                UT_TRACE(14);
                // the merge at level 64: T = G_PQ A_QQ, then A_PQ = -(A_PP T), both as
                // hi*hi + hi*lo + lo*hi with M = 128 (rows 64-127 unused), N = 64, K = 64
                constexpr uint32_t ID_M64 = idesc_bf16_ab(64, false, true);
                ok = mbar_wait(bar(B_M64A), 0, wc, 46);
                if (ok) {
                    tc_fence_after();
                    for (int part = 0; part < 3; ++part) {
                        const uint32_t a = sb + RM_A + (part == 2 ? 16384u : 0u);
                        const uint32_t b = sb + RM_B + (part == 1 ? 8192u : 0u);
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ss(tmem + T384, kmajor_desc(a, kk, 16384), mnmajor_desc(b, kk), ID_M64,
                                   (part > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(bar(B_M64T));
                    ok = mbar_wait(bar(B_M64B), 0, wc, 47);
                }
                if (ok) {
                    tc_fence_after();
                    for (int part = 0; part < 3; ++part) {
                        const uint32_t a = sb + RM_A + (part == 2 ? 16384u : 0u);
                        const uint32_t b = sb + RM_B + (part == 1 ? 8192u : 0u);
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ss(tmem + T384 + 64, kmajor_desc(a, kk, 16384), mnmajor_desc(b, kk), ID_M64,
                                   (part > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(bar(B_M64R));
                    ok = mbar_wait(bar(B_OPS1), 0, wc, 41);
                }
                UT_TRACE(15);
            }
            if (ok) {
                tc_fence_after();
                // Y = Y' A^T = Y'hi Ahi + Y'hi Alo + Y'lo Ahi  (A rows as K-major B)
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tmem + T0, kmajor_desc(sb + R3, kk, 16384), kmajor_desc(sb + R1, kk, 16384), ID_KK128, kk > 0);
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tmem + T0, kmajor_desc(sb + R3, kk, 16384), kmajor_desc(sb + R2, kk, 16384), ID_KK128, 1);
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tmem + T0, kmajor_desc(sb + R3 + 32768, kk, 16384), kmajor_desc(sb + R1, kk, 16384),
                           ID_KK128, 1);
                // V = A W = Ahi W + Alo W (A rows as K-major A operand)
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tmem + T128, kmajor_desc(sb + R1, kk, 16384), mnmajor_desc(sb + R0, kk), ID_KMN_D, kk > 0);
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tmem + T128, kmajor_desc(sb + R2, kk, 16384), mnmajor_desc(sb + R0, kk), ID_KMN_D, 1);
                mma_commit(bar(B_UY));
                UT_TRACE(16);
                ok = mbar_wait(bar(B_OPS2), 0, wc, 42);
                UT_TRACE(17);
            }
            if (ok) {
                tc_fence_after();
                // Y W  (W as MN-major B)
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tmem + T384, kmajor_desc(sb + R3, kk, 16384), mnmajor_desc(sb + R0, kk), ID_KMN_D, kk > 0);
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tmem + T384, kmajor_desc(sb + R3 + 32768, kk, 16384), mnmajor_desc(sb + R0, kk), ID_KMN_D, 1);
                // P - I = W^T (-V): W^T is the MN-major view of the W tile (rows n >= d of
                // that view are the zeroed second box when d = 64), -V the MN-major B
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tmem + T128, mnmajor_desc(sb + R0, kk), mnmajor_desc(sb + RS, kk), ID_MNMN_D, kk > 0);
                mma_commit(bar(B_Q));
                UT_TRACE(18);
                ok = mbar_wait(bar(B_OPS3), 0, wc, 43);
                UT_TRACE(19);
            }
            if (ok) {
                tc_fence_after();
                // (Z A) W = Z V: -(Z V) = (-Z)hi Vhi + (-Z)hi Vlo + (-Z)lo Vhi  (V as MN-major B)
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tmem + T0, kmajor_desc(sb + R3, kk, 16384), mnmajor_desc(sb + R1, kk), ID_KMN_D, kk > 0);
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tmem + T0, kmajor_desc(sb + R3, kk, 16384), mnmajor_desc(sb + R2, kk), ID_KMN_D, 1);
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tmem + T0, kmajor_desc(sb + R3 + 32768, kk, 16384), mnmajor_desc(sb + R1, kk), ID_KMN_D,
                           1);
                mma_commit(bar(B_K));
                UT_TRACE(20);
            }
            mma_commit(bar(B_DRAIN));
            drain_wait(bar(B_DRAIN), 0, p.limit_ns, p.hdr, 99);
        }
    } else {
        // ---------------------------------------------------------------- compute warps (rows)
        const int t = threadIdx.x - 64;         // 0..255
        const int r = 32 * (warp & 3) + lane;    // chunk row = TMEM lane
        const int h = (warp - 2) >> 2;           // column half handled by this warp
        const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const int grow = row0 + r;               // sequence position of this row
        const size_t ws_row = (size_t)bh * p.Lp + grow;
        float* sG = reinterpret_cast<float*>(sm + R3);
        float* sX = reinterpret_cast<float*>(sm + R1);  // dense X [128][128], over Q and K
        float* sT = reinterpret_cast<float*>(sm + RT);
        uint8_t* opHi = sm + R3;
        uint8_t* opLo = sm + R3 + 32768;
        const long long n_bhl = (long long)p.BH * p.L;
        if (h == 0)
            sBeta[r] = grow < p.L && in_bounds((long long)bh * p.L + grow, 1, n_bhl, p.hdr, 210)
                           ? p.beta[(size_t)bh * p.L + grow] : 0.f;
        if (D == 64) {  // rows 64-127 of the W^T view (the unused second box of the W tile) read as zero
            uint4* z = reinterpret_cast<uint4*>(sm + R0 + 16384);
            for (int i = t; i < 16384 / 16; i += kCompute) z[i] = make_uint4(0, 0, 0, 0);
        }
        // All compute warps wait on the same barriers, so they agree on `ok`
        // and reach the named barriers below together.
        if (t == 0) UT_TRACE(0);
        if (t == 0) UT_CTA(1, globaltimer());
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar(B_G), 0, wc, 50));
        if (t == 0) UT_TRACE(1);
        if (ok) {
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 2; ++c) {  // G row -> shared fp32 (this warp's half)
                uint32_t v[32];
                tmem_ld32(tl + T0 + 64 * h + 32 * c, v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4*>(sG + r * LDG + 64 * h + 32 * c + j) =
                        make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                                    __uint_as_float(v[j + 3]));
            }
            // Q and K (under the dense A) must be consumed by Q W^T and K W^T first
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B_QK), 0, wc, 58));
        }
        if (ok) {
            {  // zero the dense A
                float4* x4 = reinterpret_cast<float4*>(sX);
                for (int i = t; i < C * C / 4; i += kCompute) x4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            named_bar_sync(1, kCompute);
            if (t == 0) UT_TRACE(2);
            solve_diag_blocks(sG, sBeta, sX, t);
            if (t == 0) UT_TRACE(23);
            merge_level<16, 2, 2>(sG, sX, sT, t);
            if (t == 0) UT_TRACE(24);
            merge_level_tri<32, 2, 4>(sG, sX, sT, t);
            if (t == 0) UT_TRACE(25);
            // The merge at level 64 (P = rows 0-63, Q = rows 64-127) on the tensor
            // cores: G_PQ and A_QQ to hi/lo bf16 tiles, T = G_PQ A_QQ; T and A_PP to
            // hi/lo, A_PQ = -(A_PP T) back into the dense A.  Y' = tril(Q W^T) goes to
            // its hi/lo operand tiles (over G, no longer read) while A_PP T runs.
            {
                const int row = t >> 2, c0 = 16 * (t & 3);  // 64 rows x 4 segments of 16 columns
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    const int col = c0 + 8 * g;
                    const float4 g0 = *reinterpret_cast<const float4*>(sG + row * LDG + 64 + col);
                    const float4 g1 = *reinterpret_cast<const float4*>(sG + row * LDG + 64 + col + 4);
                    const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                    put_hilo(sm + RM_A, sm + RM_A + 16384, row, col >> 3, gv);
                    const float4 a0 = *reinterpret_cast<const float4*>(sX + (64 + row) * C + 64 + col);
                    const float4 a1 = *reinterpret_cast<const float4*>(sX + (64 + row) * C + 64 + col + 4);
                    const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                    put_hilo(sm + RM_B, sm + RM_B + 8192, row, col >> 3, av);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B_M64A));
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B_M64T), 0, wc, 59));
            if (ok) {
                tc_fence_after();
                if (r < 64) {  // T row r (this warp's 32 columns) -> MN-major B rows
                    uint32_t v[32];
                    tmem_ld32(tl + T384 + 32 * h, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        float v8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) v8[e] = __uint_as_float(v[8 * g + e]);
                        put_hilo(sm + RM_B, sm + RM_B + 8192, r, 4 * h + g, v8);
                    }
                } else {  // A_PP row r - 64 (32 columns) -> K-major A rows, over G_PQ
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const int col = 32 * h + 8 * g;
                        const float4 a0 = *reinterpret_cast<const float4*>(sX + (r - 64) * C + col);
                        const float4 a1 = *reinterpret_cast<const float4*>(sX + (r - 64) * C + col + 4);
                        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                        put_hilo(sm + RM_A, sm + RM_A + 16384, r - 64, col >> 3, av);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar(B_M64B));
                // Y' = tril(Q W^T) -> hi/lo operand (every thread's G reads came before B_M64T)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tl + T128 + 64 * h + 32 * c, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        float y8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int b = 64 * h + 32 * c + 8 * g + e;
                            y8[e] = b <= r ? __uint_as_float(v[8 * g + e]) : 0.f;
                        }
                        put_hilo(opHi, opLo, r, 8 * h + 4 * c + g, y8);
                    }
                }
                ok = __all_sync(0xffffffffu, mbar_wait(bar(B_M64R), 0, wc, 60));
            }
            if (ok) {
                tc_fence_after();
                if (r < 64) {  // A_PQ row r = -(A_PP T) row r
                    uint32_t v[32];
                    tmem_ld32(tl + T384 + 64 + 32 * h, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(sX + r * C + 64 + 32 * h + j) =
                            make_float4(-__uint_as_float(v[j]), -__uint_as_float(v[j + 1]), -__uint_as_float(v[j + 2]),
                                        -__uint_as_float(v[j + 3]));
                }
            }
            named_bar_sync(1, kCompute);
            if (t == 0) UT_TRACE(3);
            // A as hi/lo bf16 tiles.  The tiles overwrite the dense A, so
            // each thread first reads its 8 granules (8 consecutive columns of
            // one row; consecutive threads walk along a row, free of bank
            // conflicts) into registers, then writes them after a barrier.
            {
                float a[8][8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int q = t + kCompute * i, row = q >> 4, G = q & 15;
                    const float4 x0 = *reinterpret_cast<const float4*>(sX + row * C + 8 * G);
                    const float4 x1 = *reinterpret_cast<const float4*>(sX + row * C + 8 * G + 4);
                    const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) a[i][e] = xv[e];
                }
                named_bar_sync(1, kCompute);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int q = t + kCompute * i;
                    put_hilo(sm + R1, sm + R2, q >> 4, q & 15, a[i]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B_OPS1));
            if (t == 0) UT_TRACE(4);
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B_UY), 0, wc, 51));
            if (t == 0) UT_TRACE(5);
        }
        if (ok) {
            tc_fence_after();
            // V = A W row -> -V (bf16 MN-major B operand of P - I) and V as a hi/lo
            // MN-major B operand of Z V over A (A is no longer read once Y and V
            // have completed)
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t v[32];
                const int col = (D / 2) * h + 32 * c;
                tmem_ld32(tl + T128 + col, v);
                tmem_wait_ld();
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    float v8[8], nv8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        v8[e] = __uint_as_float(v[8 * g + e]);
                        nv8[e] = -v8[e];
                    }
                    stage16(sm + RS, r, (col + 8 * g) >> 6, ((col + 8 * g) & 63) >> 3, pack8(nv8));
                    put_hilo(sm + R1, sm + R2, r, (col + 8 * g) >> 3, v8);
                    if (p.vfac && in_bounds((long long)ws_row * D + col + 8 * g, 8, (long long)p.BH * p.Lp * D, p.hdr,
                                            213))  // the prefill hand-off's key-side factor V
                        st_global_v4(p.vfac + ws_row * D + col + 8 * g, pack8(v8));
                }
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {  // Y row -> hi/lo operand; its hi part is the bf16 Y output
                uint32_t v[32];
                const int col = 64 * h + 32 * c;
                tmem_ld32(tl + T0 + col, v);
                tmem_wait_ld();
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    float y8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) y8[e] = __uint_as_float(v[8 * g + e]);
                    put_hilo(opHi, opLo, r, 8 * h + 4 * c + g, y8);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B_OPS2));
            mbar_arrive(bar(B_STG0));  // Y tile -> workspace
            if (t == 0) UT_TRACE(6);
        }
        // This thread's half of the Q row, loaded while Y W runs on the tensor cores.
        uint4 qpre[D / 16];
        {
            const __nv_bfloat16* qrow = p.q + ((size_t)bh * p.L + grow) * D;
#pragma unroll
            for (int i = 0; i < D / 16; ++i)
                qpre[i] = (ok && grow < p.L &&
                           in_bounds(((long long)bh * p.L + grow) * D + (D / 2) * h + 8 * i, 8, n_bhl * D, p.hdr, 211))
                              ? ld_global_nc_v4(qrow + (D / 2) * h + 8 * i) : make_uint4(0, 0, 0, 0);
        }
        // qhat = Q - Y W (fp32, Y W in TMEM at T384), columns 32c .. 32c+31 of this
        // thread's half, into a staging tile laid out as two 32-column boxes
        auto stage_qhat = [&](int c, uint8_t* dst) {
            uint32_t v[32];
            const int col = (D / 2) * h + 32 * c;
            tmem_ld32(tl + T384 + col, v);
            tmem_wait_ld();
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                Vec16<__nv_bfloat16> qv;
                qv.raw = qpre[4 * c + g];
                float q8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) q8[e] = qv.get(e) - __uint_as_float(v[8 * g + e]);
                stage16(dst, r, h, 2 * g, make_uint4(__float_as_uint(q8[0]), __float_as_uint(q8[1]),
                                                     __float_as_uint(q8[2]), __float_as_uint(q8[3])));
                stage16(dst, r, h, 2 * g + 1, make_uint4(__float_as_uint(q8[4]), __float_as_uint(q8[5]),
                                                         __float_as_uint(q8[6]), __float_as_uint(q8[7])));
            }
        };
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(B_Q), 0, wc, 52));
        if (t == 0) UT_TRACE(7);
        if (ok) {
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {  // P - I row (n) -> staging tile (bf16); -V there is consumed
                uint32_t v[32];
                const int col = (D / 2) * h + 32 * c;
                tmem_ld32(tl + T128 + col, v);
                tmem_wait_ld();
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    float m8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) m8[e] = __uint_as_float(v[8 * g + e]);
                    stage16(sm + RS, r, (col + 8 * g) >> 6, ((col + 8 * g) & 63) >> 3, pack8(m8));
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(B_STG1));  // P - I -> workspace
            // the Y store has read R3 before it is rewritten
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B_FREE0), 0, wc, 55));
        }
        if (ok) {
            // Z = triu_1(K W^T) -> hi/lo operand, negated: its hi part is the bf16 -Z
            // output, and Z V comes out as -(Z V)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t v[32];
                const int col = 64 * h + 32 * c;
                tmem_ld32(tl + T256 + col, v);
                tmem_wait_ld();
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    float nz8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int b = col + 8 * g + e;
                        nz8[e] = b > r ? -__uint_as_float(v[8 * g + e]) : 0.f;
                    }
                    put_hilo(opHi, opLo, r, 8 * h + 4 * c + g, nz8);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B_OPS3));
            if (t == 0) UT_TRACE(8);
            // qhat = Q - Y W (fp32) while Z V runs: columns 0-31 of each half into the
            // staging tile (once the P - I store has read it), columns 32-63 into R0
            // (W is no longer read once Y W and P - I have completed)
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B_FREE1), 0, wc, 56));
            if (ok) {
                stage_qhat(0, sm + RS);
                fence_proxy_async_smem();
                mbar_arrive(bar(B_STG2));  // with the -Z tile
                if (D == 128) {
                    stage_qhat(1, sm + R0);
                    fence_proxy_async_smem();
                    mbar_arrive(bar(B_STG3));
                }
            }
        }
        // This thread's half of the K row, loaded while Z V runs.
        uint4 kpre[D / 16];
        {
            const __nv_bfloat16* krow = p.k + ((size_t)bh * p.L + grow) * D;
#pragma unroll
            for (int i = 0; i < D / 16; ++i)
                kpre[i] = (ok && grow < p.L &&
                           in_bounds(((long long)bh * p.L + grow) * D + (D / 2) * h + 8 * i, 8, n_bhl * D, p.hdr, 212))
                              ? ld_global_nc_v4(krow + (D / 2) * h + 8 * i) : make_uint4(0, 0, 0, 0);
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(B_K), 0, wc, 54));
        if (t == 0) UT_TRACE(11);

        if (ok) {
            tc_fence_after();
            float n2 = 0.f;  // this thread's part of |khat_row|^2
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {  // khat = K - Z V; TMEM holds -(Z V)
                uint32_t v[32];
                const int col = (D / 2) * h + 32 * c;
                tmem_ld32(tl + T0 + col, v);
                tmem_wait_ld();
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    Vec16<__nv_bfloat16> kv;
                    kv.raw = kpre[4 * c + g];
                    float k8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        k8[e] = kv.get(e) + __uint_as_float(v[8 * g + e]);
                        n2 = fmaf(k8[e], k8[e], n2);
                    }
                    stage16(sm + R2, r, (col + 8 * g) >> 6, ((col + 8 * g) & 63) >> 3, pack8(k8));
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(B_STG2 + D / 64));  // khat tile (R2, free since Z V) -> workspace
            if (p.kmax2) {  // chunk max of |khat|^2 over rows < L (the solve temp is free)
                float* red = reinterpret_cast<float*>(sm + RT);
                red[r + 128 * h] = grow < p.L ? n2 : 0.f;
                named_bar_sync(1, kCompute);
                if (h == 0) {
                    float x = red[r] + red[r + 128];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
                    if (lane == 0) red[256 + (warp & 3)] = x;
                }
                named_bar_sync(1, kCompute);
                if (t == 0 && in_bounds((long long)bh * p.nch + chunk, 1, (long long)p.BH * p.nch, p.hdr, 214))
                    p.kmax2[(size_t)bh * p.nch + chunk] = fmaxf(fmaxf(red[256], red[257]), fmaxf(red[258], red[259]));
            }
        }
    }

    if (threadIdx.x == 64) UT_TRACE(12);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0) UT_CTA(2, globaltimer());
}

#ifdef PATH_TRACE
static unsigned long long* ut_trace_buffer() {
    static unsigned long long* buf = nullptr;
    const size_t n = kUtTraceCtaBase + (size_t)kUtTraceMaxCtas * 4;
    if (!buf && cudaMalloc(&buf, n * sizeof(unsigned long long)) == cudaSuccess)
        cudaMemset(buf, 0, n * sizeof(unsigned long long));
    return buf;
}
}  // namespace pathattn
extern "C" void path_ut_trace_dump(unsigned long long* host) {
    cudaDeviceSynchronize();
    cudaMemcpy(host, pathattn::ut_trace_buffer(), 64 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
}
// Per-CTA stamps of the last launch: ncta x {entry, compute start, exit, SM id}.
extern "C" void path_ut_trace_cta_dump(unsigned long long* host, int ncta) {
    cudaDeviceSynchronize();
    cudaMemcpy(host, pathattn::ut_trace_buffer() + pathattn::kUtTraceCtaBase,
               (size_t)ncta * 4 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
}
namespace pathattn {
#endif

template <int D>
static cudaError_t launch_ut_tc_d(const void* q, const void* k, const void* w, const float* beta, int BH, int L,
                                  unsigned char* ws, const FwdLayout& lay, bool want_kmax, cudaStream_t st,
                                  bool reset_header) {
    CUtensorMap mq, mk, mw, mun, my, mzn, mkh, mqh;
    if (!make_map(&mq, q, D, L, BH) || !make_map(&mk, k, D, L, BH) || !make_map(&mw, w, D, L, BH) ||
        !make_map(&mun, ws + lay.un, D, lay.Lp, BH) || !make_map(&my, ws + lay.y, utk::C, lay.Lp, BH) ||
        !make_map(&mzn, ws + lay.zn, utk::C, lay.Lp, BH) || !make_map(&mkh, ws + lay.khat, D, lay.Lp, BH) ||
        !make_map_t(&mqh, ws + lay.qhat, D, lay.Lp, BH, true))
        return cudaErrorInvalidValue;
    UtParams p;
    p.L = L;
    p.Lp = lay.Lp;
    p.BH = BH;
    p.beta = beta;
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.qhat = reinterpret_cast<float*>(ws + lay.qhat);
    p.khat = reinterpret_cast<__nv_bfloat16*>(ws + lay.khat);
    p.un = reinterpret_cast<__nv_bfloat16*>(ws + lay.un);
    p.y = reinterpret_cast<__nv_bfloat16*>(ws + lay.y);
    p.zn = reinterpret_cast<__nv_bfloat16*>(ws + lay.zn);
    p.vfac = lay.vfac ? reinterpret_cast<__nv_bfloat16*>(ws + lay.vfac) : nullptr;
    p.kmax2 = want_kmax ? reinterpret_cast<float*>(ws + lay.kmax) : nullptr;
    p.nch = lay.Lp / utk::C;
    {  // one CTA per SM is resident: prefetch for the CTA half a wave ahead (A/B: anything from an
       // eighth to three quarters of a wave does equally well, a whole wave or more is slower)
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) ==
                                                      cudaSuccess)
            p.ahead = sms / 2;
        else
            p.ahead = 0;
    }
    p.reset = reset_header ? 1 : 0;
    p.hdr = reinterpret_cast<WsHeader*>(ws);
    p.limit_ns = 2000000000ull;
#ifdef PATH_TRACE
    p.trace = ut_trace_buffer();
#endif
    auto kern = ut_prep_tc<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)utk::kSmem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(cdiv(L, utk::C), BH), utk::kThreads, utk::kSmem, st>>>(mq, mk, mw, mun, my, mzn, mkh, mqh, p);
    return cudaGetLastError();
}

cudaError_t launch_ut_prep_tc(int d, const void* q, const void* k, const void* w, const float* beta, int BH, int L,
                              unsigned char* ws, const FwdLayout& lay, bool want_kmax, cudaStream_t st,
                              bool reset_header) {
    if (d == 64) return launch_ut_tc_d<64>(q, k, w, beta, BH, L, ws, lay, want_kmax, st, reset_header);
    if (d == 128) return launch_ut_tc_d<128>(q, k, w, beta, BH, L, ws, lay, want_kmax, st, reset_header);
    return cudaErrorInvalidValue;
}

}  // namespace pathattn
