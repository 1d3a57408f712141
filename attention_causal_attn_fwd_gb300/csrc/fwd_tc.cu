// PaTH causal attention forward on GB300 tensor cores (bf16 in, fp32 accumulate).
//
// Blockwise algorithm of "Resumo Técnico: Atenção PaTH"
// (gist.science/pt/paper/2505.16381), §3 "Algoritmo Estilo FlashAttention":
// boundary-adjusted queries/keys per chunk (from the UT-prep kernel,
// ut_prep_tc.cu), then a right-to-left scan over key/value blocks that carries
// the Householder product on the query side, never forming the L x L matrix.
//
// One CTA owns a tile of 128 queries (= one chunk n of one head) and walks the
// key/value blocks m = n (diagonal), n-1, ..., 0.  Per block m < n, with the
// transported query q~ (fp32 master and its bf16 copy, both in TMEM), one
// accumulating product gives the block's logits and the query's step through
// the block:
//   [S | q~] += bf16(q~) [khat_m ; P_m - I]^T             (M=128, N=128+d, K=d)
//   O += P V_m,  P = exp2(S * scale*log2e - m)            (M=128, N=d,     K=128)
// (the softmax warps zero S after reading it, so S starts from zero).
// where P_m = I - W_m^T A_m W_m is the chunk's transition in the UT form of §3
// "Representação de Transformação UT" (the UT prep writes P_m - I in bf16), so
// the query moves through a whole chunk in one d x d product, and S and dq
// share the A operand, which makes the instruction N = 256 wide (d = 128): a
// single thread cannot issue the 128-wide ones fast enough to keep the pipe
// busy.  The diagonal block uses S = Q K^T + Y (-Z)^T with the causal mask.
// The logits may carry an additive bias (MODE 1 PaTH-FoX, MODE 2 relative
// position).
// Online softmax keeps one query row per thread (TMEM lane = row), so row
// max and sum need no cross-thread reduction.  The running max is only
// raised (and O rescaled) when it grows by more than 2^8, which keeps every
// exponent <= 2^8 and makes rescales rare.
//
// Warp roles (320 threads):
//   warp 0      TMA producer (one lane) + TMEM allocation
//   warp 1      tcgen05.mma issuer (one lane), per block in the order
//               [S | q~](it), P V(it-1): the transport of the next query
//               overlaps P V, and the softmax of block it overlaps P V
//   warps 2-5   softmax: S -> P (bf16, into TMEM), row statistics, epilogue
//   warps 6-9   query transport: fp32 q~ master -> bf16 q~ (TMEM), the first half of
//               its columns released before the second is converted
// Every MMA reads its A operand from TMEM except the diagonal block's, so
// shared memory carries only the B tiles (khat, P - I, V) and their TMA writes.
//
// TMEM (512 columns x 128 lanes, 32-bit): [0,128) S (fp32), [128,128+d) q~
// master (fp32), [256,320) P (bf16 pairs), [320,320+d/2) bf16 q~ (pairs),
// [384,384+d) O.
// Shared memory (1024-aligned, 128-byte swizzled tiles as TMA writes them,
// 64-column boxes of 16 KB), double-buffered by block parity:
//   KM0/KM1  per 64-column box c (32 KB): rows 0-127 khat_m, rows 128-255
//            P_m - I (one K-major B operand of N = 128 + d rows); KM0 holds K
//            and Y of the diagonal in the same places
//   V0/V1    V_m, MN-major B            (V0: V of the diagonal, V1: -Z)
//   Q        Q of the diagonal; once the diagonal's product has completed, the
//            softmax warps stage each block's bias values there (FoX: c_j;
//            relative bias: the table window of the block)
// Every mbarrier wait is bounded (globaltimer); on expiry the kernel records
// PATH_ERR_TIMEOUT in the workspace status word, every role stops, pending
// copies and MMAs are drained (bounded) and TMEM is freed before exit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.cuh"
#include "ut_prep.cuh"

namespace pathattn {
using namespace sm100;

constexpr int kTcC = 128;
constexpr int kTcThreads = 320;
constexpr uint32_t SM_KM0 = 0, SM_V0 = 131072, SM_V1 = 163840, SM_Q = 196608, SM_BAR = 229376;
constexpr uint32_t KM_SLOT = 65536;  // SM_KM1 = SM_KM0 + KM_SLOT
constexpr uint32_t SM_TOTAL = SM_BAR + 256;
constexpr size_t kTcSmem = SM_TOTAL + 1024;  // + alignment slack
constexpr uint32_t TM_S = 0, TM_QM = 128, TM_P = 256, TM_QB = 320, TM_O = 384;

// Every barrier below is waited on in a way that it can never run two phases
// ahead of its waiter (a parity wait cannot tell those apart): each one's next
// completion needs an action its waiter takes after the current wait.
enum Bar { B_QFULL = 0, B_KMFULL0, B_KMFULL1, B_KMEMPTY0, B_KMEMPTY1, B_VFULL0, B_VFULL1, B_VEMPTY0, B_VEMPTY1,
           B_SDONE, B_ODONE, B_DRAIN, B_COUNT };
// Named (hardware) barriers between the warps and the MMA warp; id 2 is the
// softmax warps' own vote barrier.  Counts are threads: the MMA warp syncs,
// the others arrive.
constexpr int NB_SK = 3, NB_SK_COUNT = 32 + 128 + 128;  // MMA warp + softmax warps + transport warps
constexpr int NB_PV = 4, NB_PV_COUNT = 32 + 128;        // MMA warp + softmax warps
constexpr int NB_SKB = 5, NB_SKB_COUNT = 32 + 128;      // MMA warp + transport warps
// Barriers at SM_BAR, then the control words (TMEM address, abort flag, FoX
// stop index and votes, max |khat|^2) at SM_CTL, all inside SM_BAR + 256.
constexpr uint32_t SM_CTL = SM_BAR + 192;
static_assert(B_COUNT * 8 <= 192, "barriers overlap the control words");
static_assert(SM_CTL + 52 <= SM_TOTAL, "control words exceed the barrier region");

constexpr int kHeadGroup = 4;

// Use index of the V slot (it & 1) for block iteration it: slot 1 holds -Z of
// the diagonal first, so its V_m uses are shifted by one.
__host__ __device__ constexpr int v_use(int it) { return (it >> 1) + (it & 1); }

// Phase timestamps of one CTA (SM cycle counter), compiled in only for
// instrumented builds (-DPATH_TRACE): slot s of block iteration it.  CTA 773
// is a 32-block tile of the fourth head group at L = 4096 (a later wave, so
// its code is warm in the instruction cache).
#ifndef PATH_TRACE_CTA
#define PATH_TRACE_CTA 773
#endif
constexpr int kTraceCta = PATH_TRACE_CTA;
#ifdef PATH_TRACE
#define TC_TRACE(slot, it) \
    do { if (p.trace && blockIdx.x == kTraceCta && (it) < 64) p.trace[(it) * 32 + (slot)] = clock64(); } while (0)
// Per-CTA global-timer stamps (every CTA): 0 entry, 1 diagonal issued, 2 exit, 3 SM id.
constexpr int kTraceCtaBase = 64 * 32, kTraceMaxCtas = 65536;
#define TC_CTA(slot, val) \
    do { if (p.trace && blockIdx.x < kTraceMaxCtas) p.trace[kTraceCtaBase + blockIdx.x * 4 + (slot)] = (val); } while (0)
#else
#define TC_TRACE(slot, it) do { } while (0)
#define TC_CTA(slot, val) do { } while (0)
#endif

struct TcParams {
    int L, Lp, ntiles, BH;
    float sl2;                 // scale * log2(e)
    const float* qhat;         // [BH, Lp, d] fp32
    const float* cum;          // [BH, Lp] fp32 (FoX)
    __nv_bfloat16* o;          // [BH, L, d]
    float* lse;                // [BH, L] or null
    WsHeader* hdr;
    unsigned long long limit_ns;
    const __nv_bfloat16* q;    // [BH, L, d] (FoX: query norms for far-block skipping)
    const float* kmax2;        // [BH, nch] max |khat|^2 per chunk (FoX)
    const float* rbias;        // [H, L] bias by distance i - j (relative-bias mode)
    int H;
    int nch;
    int fault;                 // test hook: skip one producer signal
    int no_skip;               // FoX: visit every block (the far-block stop disabled)
    unsigned* visited;         // (query tile, key block) pairs visited, summed over tiles
    __nv_bfloat16* pdiag;      // VT: the diagonal block's P, [BH, L, 128] bf16
    float* m0;                 // VT: the max the diagonal's P was formed with (log2 units), [BH, L]
#ifdef PATH_TRACE
    unsigned long long* trace;
#endif
};

// MODE 0: PaTH; 1: PaTH-FoX (forget-gate bias, far blocks skipped); 2: PaTH
// with a relative-position bias table rel[h][i - j].
// VT (value-side transport, the blockwise form): key block m of query tile n
// takes its values from the pair store (tm_vp: the block's values carried to
// the start of chunk n, rows (n (n - 1) / 2 + m) * 128 of the head), and the
// diagonal block's values are zero (the TMA fill of rows below 0), so O holds
// only the earlier blocks' terms; the diagonal's are added by the walks that
// follow (csrc/fwd_vt.cu).
template <int D, int MODE, bool VT = false>
__global__ void __launch_bounds__(kTcThreads, 1)
    path_fwd_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_khat,
                const __grid_constant__ CUtensorMap tm_pm, const __grid_constant__ CUtensorMap tm_y,
                const __grid_constant__ CUtensorMap tm_zn, const __grid_constant__ CUtensorMap tm_vp,
                const TcParams p) {
    static_assert(D == 64 || D == 128, "head dim");
    constexpr bool FOX = MODE == 1, REL = MODE == 2;
    constexpr bool BIASED = MODE != 0;   // logits carry an additive bias (log2 units in the softmax)
    constexpr int KCH = D / 64;          // 64-column boxes of the head dim
    constexpr uint32_t ROWB = 128u * D * 2u;  // bytes of one [128 x D] bf16 tile
    constexpr uint32_t IDESC_S = idesc_bf16(128, false);      // N = 128 keys, B K-major (diagonal)
    constexpr uint32_t IDESC_SQ = idesc_bf16(128 + D, false); // N = 128 keys + d, B K-major [khat; P - I]
    static_assert(TM_QM == TM_S + 128, "S and the q~ master form one N = 128 + d accumulator");
    constexpr uint32_t IDESC_PV = idesc_bf16(D, true);        // N = d, B MN-major (V)

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    const uint32_t bar0 = sb + SM_BAR;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + SM_CTL);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + SM_CTL + 4);
    // PaTH-FoX far-block skipping: the scan stops before block iteration
    // *stop_it (n + 1 = never); set by the softmax warps before they release S.
    volatile int* stop_it = reinterpret_cast<volatile int*>(sm + SM_CTL + 8);
    int* votes = reinterpret_cast<int*>(sm + SM_CTL + 16);     // [2][4]
    float* s_kmax2 = reinterpret_cast<float*>(sm + SM_CTL + 48);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        TC_CTA(0, globaltimer());
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        TC_CTA(3, smid);
    }
    // Launch order: heads in groups of kHeadGroup; inside a group, tiles
    // longest first with the heads interleaved.  The ~150 resident CTAs then
    // cover a few heads each, so their key/value blocks are re-read from L2,
    // and the short tiles of the last group fill the tail.
    int bh, n;
    {
        const int idx = (int)blockIdx.x;
        const int per_group = kHeadGroup * p.ntiles;
        const int g = idx / per_group, rem = idx - g * per_group;
        const int gsize = min(kHeadGroup, p.BH - g * kHeadGroup);
        n = p.ntiles - 1 - rem / gsize;
        bh = g * kHeadGroup + rem % gsize;
    }
    const int row0 = n * kTcC;

    if (threadIdx.x == 0) {
        uint32_t counts[B_COUNT];
        for (int i = 0; i < B_COUNT; ++i) counts[i] = 1;
        for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), counts[i]);
        *abort_flag = 0;
        *stop_it = n + 1;
        for (int i = 0; i < 8; ++i) votes[i] = 0;
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
            prefetch_tmap(&tm_q); prefetch_tmap(&tm_k); prefetch_tmap(&tm_v); prefetch_tmap(&tm_khat);
            prefetch_tmap(&tm_pm); prefetch_tmap(&tm_y); prefetch_tmap(&tm_zn);
            if (VT) prefetch_tmap(&tm_vp);
            // diagonal block: Q, K and Y (KM slot 0), -Z (V slot 1), V (V slot 0)
            mbar_expect_tx(bar(B_QFULL), ROWB);
            for (int c = 0; c < KCH; ++c) tma_load_3d(sb + SM_Q + c * 16384, &tm_q, bar(B_QFULL), c * 64, row0, bh);
            mbar_expect_tx(bar(B_KMFULL0), ROWB + 32768);
            for (int c = 0; c < KCH; ++c) tma_load_3d(sb + SM_KM0 + c * 32768, &tm_k, bar(B_KMFULL0), c * 64, row0, bh);
            for (int c = 0; c < 2; ++c)
                tma_load_3d(sb + SM_KM0 + c * 32768 + 16384, &tm_y, bar(B_KMFULL0), c * 64, row0, bh);
            mbar_expect_tx(bar(B_VFULL1), 32768);
            for (int c = 0; c < 2; ++c) tma_load_3d(sb + SM_V1 + c * 16384, &tm_zn, bar(B_VFULL1), c * 64, row0, bh);
            mbar_expect_tx(bar(B_VFULL0), ROWB);
            for (int c = 0; c < KCH; ++c)
                tma_load_3d(sb + SM_V0 + c * 16384, &tm_v, bar(B_VFULL0), c * 64, VT ? -kTcC : row0, bh);
            // Scan blocks, two streams: khat with P - I (one KM slot; the last block,
            // m = 0, needs no P - I) and V, each block iteration it into slot it & 1
            // once that slot's previous contents were consumed (their empty
            // barrier's matching completion).
            int nxt[2] = {1, 1};
            int issued[5] = {1, 1, 0, 1, 1};  // Q, KM0, KM1, V0, V1 (loads per full barrier)
            const uint64_t t0 = globaltimer();
            bool ok = true;
            for (uint32_t spin = 0; ok; ++spin) {
                const int lim = FOX ? min(n, *stop_it - 1) : n;
                if (nxt[0] > lim && nxt[1] > lim) break;
                for (int sl = 0; sl < 2; ++sl) {
                    const int it = nxt[sl];
                    if (it > lim) continue;
                    const int s = it & 1;
                    const int u = sl == 1 ? v_use(it) : (it >> 1);
                    const int eb = (sl == 0 ? B_KMEMPTY0 : B_VEMPTY0) + s;
                    if (u >= 1 && !mbar_test_wait(bar(eb), (uint32_t)((u - 1) & 1))) continue;
                    nxt[sl] = it + 1;
                    if (sl == 1 && p.fault && it == 1) continue;  // test hook: the consumer's wait must expire
                    const int r = (n - it) * kTcC;
                    if (sl == 0) {
                        const uint32_t dst = sb + SM_KM0 + (uint32_t)s * KM_SLOT;
                        const bool pm = n - it > 0;
                        mbar_expect_tx(bar(B_KMFULL0 + s), pm ? 2 * ROWB : ROWB);
                        for (int c = 0; c < KCH; ++c) {
                            tma_load_3d(dst + c * 32768, &tm_khat, bar(B_KMFULL0 + s), c * 64, r, bh);
                            if (pm) tma_load_3d(dst + c * 32768 + 16384, &tm_pm, bar(B_KMFULL0 + s), c * 64, r, bh);
                        }
                    } else {
                        mbar_expect_tx(bar(B_VFULL0 + s), ROWB);
                        const int vr = VT ? (n * (n - 1) / 2 + (n - it)) * kTcC : r;
                        for (int c = 0; c < KCH; ++c)
                            tma_load_3d(sb + SM_V0 + (uint32_t)s * 32768u + c * 16384, VT ? &tm_vp : &tm_v,
                                        bar(B_VFULL0 + s), c * 64, vr, bh);
                    }
                    ++issued[1 + 2 * sl + s];
                    TC_TRACE(12 + sl, it);
                }
                if ((spin & 255u) == 255u) {
                    if (*abort_flag) { ok = false; break; }
                    if (globaltimer() - t0 > p.limit_ns * (uint64_t)(n + 1)) {
                        report_status(p.hdr, PATH_ERR_TIMEOUT, 1);
                        *abort_flag = 1;
                        ok = false;
                    }
                }
            }
            // copies still in flight must land before the CTA exits
            const int ful[5] = {B_QFULL, B_KMFULL0, B_KMFULL1, B_VFULL0, B_VFULL1};
            for (int i = 0; i < 5; ++i)
                if (issued[i] > 0) drain_wait(bar(ful[i]), (uint32_t)((issued[i] - 1) & 1), p.limit_ns, p.hdr, 91);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        // Issue blocks for about as long as a group executes and the tensor pipe
        // queues little, so every pause between groups is a bubble.  This warp
        // therefore waits on nothing but two named barriers per block (no
        // shared-memory round trip): the warps that signal it have already
        // waited for the copies the next MMAs read.
        //   NB_SK(it)   the first half (in K) of [S | q~](it) may go: the first half
        //               of bf16 q~(it) is in TMEM and khat_m, P_m - I have landed
        //               (transport warps); S(it-1) has been read and zeroed and, with
        //               FoX, block it is known to be visited (softmax warps)
        //   NB_SKB(it)  its second half may go: the rest of bf16 q~(it) (transport)
        //   NB_PV(it)   P V(it) may go: P(it) is in TMEM and V_m has landed (softmax)
        // Lane 0 issues; the whole warp takes the barriers.
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar(B_QFULL), 0, wc, 10) && mbar_wait(bar(B_KMFULL0), 0, wc, 11) &&
                                              mbar_wait(bar(B_VFULL1), 0, wc, 12));
        if (ok && lane == 0) {
            tc_fence_after();
            // diagonal: S = Q K^T + Y (-Z)^T
            for (int kk = 0; kk < D / 16; ++kk)
                mma_ss(tmem + TM_S, kmajor_desc(sb + SM_Q, kk, 16384), kmajor_desc(sb + SM_KM0, kk, 32768), IDESC_S,
                       kk > 0);
            for (int kk = 0; kk < kTcC / 16; ++kk)
                mma_ss(tmem + TM_S, kmajor_desc(sb + SM_KM0 + 16384, kk, 32768), kmajor_desc(sb + SM_V1, kk, 16384),
                       IDESC_S, 1);
            mma_commit(bar(B_SDONE));
            mma_commit(bar(B_KMEMPTY0));
            mma_commit(bar(B_VEMPTY1));
            TC_TRACE(0, 0);
            TC_CTA(1, globaltimer());
        }
        __syncwarp();
        auto issue_pv = [&](int blk) {  // O (+)= P V for block iteration blk (P in TMEM)
            named_bar_sync(NB_PV, NB_PV_COUNT);
            if (lane == 0) {
                TC_TRACE(18, blk);
                tc_fence_after();
                const int s = blk & 1;
                const uint32_t vbuf = sb + SM_V0 + (uint32_t)s * 32768u;
                for (int kk = 0; kk < kTcC / 16; ++kk)
                    mma_ts(tmem + TM_O, tmem + TM_P + kk * 8, mnmajor_desc(vbuf, kk), IDESC_PV,
                           (blk > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bar(B_ODONE));
                mma_commit(bar(B_VEMPTY0 + s));
                TC_TRACE(2, blk);
            }
            __syncwarp();
        };
        int last = n;  // last block iteration whose P V is issued
        // The rounds of both named barriers run whatever happens: a warp that
        // gives up (a bounded wait expired) still arrives on every remaining
        // round, so this warp never blocks for good; MMAs issued after such a
        // failure read stale but valid addresses and their results are unused.
        if (ok) {
            for (int it = 1; it <= n; ++it) {
                const int s = it & 1;
                named_bar_sync(NB_SK, NB_SK_COUNT);
                if (FOX && *stop_it <= it) {  // every block from here on contributes exactly zero
                    last = it - 1;
                    break;
                }
                // [S | q~] += bf16(q~) [khat ; P_m - I]^T  (for m = 0 the q~ half reads
                // stale slot contents; the master is not used again), in two halves of K:
                // the first half of bf16 q~ is released (NB_SK) before the transport warps
                // convert the second (NB_SKB)
                if (lane == 0) {
                    TC_TRACE(15, it);
                    tc_fence_after();
                    for (int kk = 0; kk < D / 32; ++kk)
                        mma_ts(tmem + TM_S, tmem + TM_QB + kk * 8, kmajor_desc(sb + SM_KM0 + s * KM_SLOT, kk, 32768),
                               IDESC_SQ, 1);
                }
                __syncwarp();
                named_bar_sync(NB_SKB, NB_SKB_COUNT);
                if (lane == 0) {
                    tc_fence_after();
                    for (int kk = D / 32; kk < D / 16; ++kk)
                        mma_ts(tmem + TM_S, tmem + TM_QB + kk * 8, kmajor_desc(sb + SM_KM0 + s * KM_SLOT, kk, 32768),
                               IDESC_SQ, 1);
                    mma_commit(bar(B_SDONE));
                    mma_commit(bar(B_KMEMPTY0 + s));
                    TC_TRACE(1, it);
                }
                __syncwarp();
                issue_pv(it - 1);
            }
            issue_pv(last);  // the last block's P V
        }
        // every MMA this warp issued completes before TMEM is released
        if (lane == 0) {
            mma_commit(bar(B_DRAIN));
            drain_wait(bar(B_DRAIN), 0, p.limit_ns, p.hdr, 92);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------------------------ softmax warps
        const int r = 32 * (warp & 3) + lane;  // query row within the tile (= TMEM lane)
        const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const float* cumh = FOX ? p.cum + (size_t)bh * p.Lp : nullptr;
        const float* relh = REL ? p.rbias + (size_t)(bh % p.H) * p.L : nullptr;
        const long long n_bhlp = (long long)p.BH * p.Lp, n_bhl = (long long)p.BH * p.L;
        const float ci = FOX && in_bounds((long long)bh * p.Lp + row0 + r, 1, n_bhlp, p.hdr, 200) ? cumh[row0 + r] : 0.f;
        constexpr float kL2e = 1.4426950408889634f;
        float m_run = -INFINITY, l_run = 0.f;
        float m_true = -INFINITY;  // largest logit seen (log2 units)
        float qk_bound = 0.f;      // FoX: scale log2e |q_i| max_j |khat_j|, with a 2x margin
        int sk_sent = 0, pv_sent = 0;  // named-barrier rounds this warp has arrived on (NB_SK from 1, NB_PV from 0)
        if (FOX && n > 0) {
            if (warp == 2) {  // max |khat|^2 over the chunks left of this tile
                float x = 0.f;
                for (int c = lane; c < n; c += 32)
                    if (in_bounds((long long)bh * p.nch + c, 1, (long long)p.BH * p.nch, p.hdr, 201))
                        x = fmaxf(x, p.kmax2[(size_t)bh * p.nch + c]);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
                if (lane == 0) *s_kmax2 = x;
            }
            float qn2 = 0.f;
            if (row0 + r < p.L && in_bounds(((long long)bh * p.L + row0 + r) * D, D, n_bhl * D, p.hdr, 202)) {
                const uint4* qv = reinterpret_cast<const uint4*>(p.q + ((size_t)bh * p.L + row0 + r) * D);
                Vec16<__nv_bfloat16> v[D / 8];  // every load in flight before the first use
#pragma unroll
                for (int g = 0; g < D / 8; ++g) v[g].raw = __ldg(qv + g);
#pragma unroll
                for (int g = 0; g < D / 8; ++g)
#pragma unroll
                    for (int e = 0; e < 8; ++e) qn2 = fmaf(v[g].get(e), v[g].get(e), qn2);
            }
            named_bar_sync(2, 128);
            // |q~_i . khat_j| <= |q_i| |khat_j|: the transitions are non-expansive for
            // beta in [0, 2] and unit w; the factor 2 covers bf16 rounding of w.
            qk_bound = 2.0f * p.sl2 * sqrtf(qn2 * *s_kmax2);
        }
        int last = n;
        bool ok = true;
        // FoX: c_j of the block's 128 keys, one float4 per lane, loaded a block ahead and
        // staged per warp in the Q tile (free once the diagonal's product has completed)
        float4 c_next = make_float4(0.f, 0.f, 0.f, 0.f);
        if (FOX && in_bounds((long long)bh * p.Lp + n * kTcC, kTcC, n_bhlp, p.hdr, 203))
            c_next = __ldg(reinterpret_cast<const float4*>(cumh + n * kTcC) + lane);
        // relative bias: the 159 table entries (distances) this warp's rows meet in key
        // block mb, five per lane, loaded a block ahead and staged like c_j
        const bool rel_ok = REL && in_bounds((long long)(bh % p.H) * p.L, p.L, (long long)p.H * p.L, p.hdr, 204);
        float r_next[5];
        auto load_rel = [&](int mb) {
            const int dmin = row0 - mb * kTcC + 32 * (warp & 3) - 127;
#pragma unroll
            for (int k = 0; k < 5; ++k) r_next[k] = __ldg(relh + min(max(dmin + lane + 32 * k, 0), p.L - 1));
        };
        if (rel_ok) load_rel(n);
        for (int it = 0; it <= n; ++it) {
            const int m = n - it;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B_SDONE), it & 1, wc, 20));
            if (!ok) break;
            if (r == 0) TC_TRACE(4, it);
            tc_fence_after();
            float s[128];
            {
                uint32_t raw[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(tl + TM_S + 32 * c, raw[c]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int j = 0; j < 32; ++j) s[32 * c + j] = __uint_as_float(raw[c][j]);
            }
            if (it < n) {  // the next block's product accumulates into S
                uint32_t z[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) z[j] = 0u;
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_st32(tl + TM_S + 32 * c, z);
                tmem_wait_st();
            }
            // Without a bias the scores stay raw (the scale is applied inside the
            // exponent, one FFMA each); with one (FoX, relative) they become
            // log2-unit logits.
            const float sl2 = p.sl2;
            // S is in registers: the next block's S_k may overwrite it (FoX first
            // decides whether there is a next block)
            if (!FOX && it < n) {
                tc_fence_before();
                named_bar_arrive(NB_SK, NB_SK_COUNT);
                sk_sent = it + 1;
            }
            if (r == 0) TC_TRACE(5, it);
            if (FOX) {
                float4* cs = reinterpret_cast<float4*>(sm + SM_Q) + (warp & 3) * 64 + (it & 1) * 32;
                cs[lane] = c_next;
                __syncwarp();
                if (m > 0 && in_bounds((long long)bh * p.Lp + (m - 1) * kTcC, kTcC, n_bhlp, p.hdr, 203))
                    c_next = __ldg(reinterpret_cast<const float4*>(cumh + (m - 1) * kTcC) + lane);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float4* cj = cs + 8 * c;
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 cv = cj[j4];
                        s[32 * c + 4 * j4 + 0] = fmaf(s[32 * c + 4 * j4 + 0], sl2, (ci - cv.x) * kL2e);
                        s[32 * c + 4 * j4 + 1] = fmaf(s[32 * c + 4 * j4 + 1], sl2, (ci - cv.y) * kL2e);
                        s[32 * c + 4 * j4 + 2] = fmaf(s[32 * c + 4 * j4 + 2], sl2, (ci - cv.z) * kL2e);
                        s[32 * c + 4 * j4 + 3] = fmaf(s[32 * c + 4 * j4 + 3], sl2, (ci - cv.w) * kL2e);
                    }
                }
            }
            if (rel_ok) {
                // bias at distance i - j, clamped into the table (masked or padding entries):
                // entry lane - j + 127 of the warp's window.  The window is stored four
                // times (168 floats apart, which spreads a phase of eight lanes over all banks),
                // copy c shifted down by c entries, so that the four entries a lane
                // needs for keys 4t .. 4t + 3 (lane + 124 - 4t .. lane + 127 - 4t) form one
                // aligned float4 of copy lane & 3.  Entries are stored in log2 units.
                float* rs = reinterpret_cast<float*>(sm + SM_Q) + (warp & 3) * 1344 + (it & 1) * 672;
#pragma unroll
                for (int k = 0; k < 5; ++k)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int y = lane + 32 * k - c;
                        if (y >= 0) rs[c * 168 + y] = r_next[k] * kL2e;
                    }
                __syncwarp();
                if (m > 0) load_rel(m - 1);
                const float4* rq = reinterpret_cast<const float4*>(rs + (lane & 3) * 168 + (lane & ~3) + 124);
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const float4 b = rq[-t];
                    s[4 * t + 3] = fmaf(s[4 * t + 3], sl2, b.x);
                    s[4 * t + 2] = fmaf(s[4 * t + 2], sl2, b.y);
                    s[4 * t + 1] = fmaf(s[4 * t + 1], sl2, b.z);
                    s[4 * t + 0] = fmaf(s[4 * t + 0], sl2, b.w);
                }
            }
            if (it == 0) {
#pragma unroll
                for (int j = 0; j < 128; ++j)
                    if (j > r) s[j] = -INFINITY;
            }
            float mx;  // row max in log2 units (8 independent chains of three-input maxima)
            {
                float pm[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) pm[u] = fmaxf(s[u], s[u + 8]);
#pragma unroll
                for (int j = 16; j < 128; j += 16)
#pragma unroll
                    for (int u = 0; u < 8; ++u) pm[u] = fmax3(pm[u], s[j + u], s[j + 8 + u]);
                mx = fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
                if (!BIASED) mx *= sl2;  // sl2 > 0: the max of raw scores scales
            }
            bool stop = false;
            if (FOX) {
                m_true = fmaxf(m_true, mx);
                // The warps vote on every fourth block only: a vote holds them together
                // for a shared-memory round trip, and a stop found up to three blocks late
                // only adds blocks whose P is exactly zero (A/B at L = 16384: 6 % more
                // blocks, 4 % less time than a vote per block).
                if (m > 0 && !p.no_skip && (it & 3) == 0) {
                    // Every key left of this block has bias <= c_i - c_(128 m - 1) and
                    // |logit| <= qk_bound: below m_true - 160 (log2) its exp2 is 0 in fp32.
                    const float cprev = in_bounds((long long)bh * p.Lp + m * kTcC - 1, 1, n_bhlp, p.hdr, 205)
                                            ? cumh[m * kTcC - 1] : ci;
                    const float bound = qk_bound + (ci - cprev) * kL2e - m_true;
                    const bool sat = (row0 + r >= p.L) || bound < -160.0f;
                    const int vote = __all_sync(0xffffffffu, sat);
                    // Votes carry the iteration (2 (it + 1) + vote), double-buffered by
                    // it & 1: no warp can post iteration it + 2 before every warp has
                    // read iteration it.  The poll is bounded (a warp that gave up on a
                    // wait raises the abort flag instead of voting).
                    volatile int* vv = votes + (it & 1) * 4;
                    if (lane == 0) vv[warp & 3] = 2 * (it + 1) + vote;
                    __syncwarp();
                    int all = 1;
                    const uint64_t tv = globaltimer();
                    for (int w4 = 0; w4 < 4 && ok; ++w4) {
                        int x;
                        for (uint32_t spin = 0; ((x = vv[w4]) >> 1) != it + 1; ++spin)
                            if ((spin & 255u) == 255u && (*abort_flag || globaltimer() - tv > p.limit_ns)) {
                                if (!*abort_flag) { report_status(p.hdr, PATH_ERR_TIMEOUT, 23); *abort_flag = 1; }
                                ok = false;
                                break;
                            }
                        all &= x & 1;
                    }
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    stop = all != 0;
                    if (stop && warp == 2 && lane == 0) *stop_it = it + 1;
                }
                if (it < n) {
                    tc_fence_before();
                    named_bar_arrive(NB_SK, NB_SK_COUNT);  // with the decision on block it + 1
                    sk_sent = it + 1;
                }
            }
            const float m_new = fmaxf(m_run, mx);
            const bool rescale = m_new > m_run + 8.0f;
            const float m_use = rescale ? m_new : m_run;
            const float alpha = rescale ? ex2_approx(m_run - m_use) : 1.0f;
            // P and O are single-buffered: the previous block's P V must have completed
            // before P is rewritten and O rescaled; waiting here, before the
            // exponentials, lets P go to TMEM 32 columns at a time as it is formed
            // (fewer live registers than holding the whole row).
            if (it > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(B_ODONE), (uint32_t)((it - 1) & 1), wc, 21));
                if (!ok) break;
                if (r == 0) TC_TRACE(11, it);
                tc_fence_after();
            }
            // V_m of this block is probed mid-loop so its shared-memory round trip
            // overlaps the exponentials; a blocking wait follows only if not ready.
            bool v_ready = false;
            uint64_t psum[4];  // packed partial row sums (8 chains)
#pragma unroll
            for (int u = 0; u < 4; ++u) psum[u] = 0ull;
            const float neg_m = -m_use;
            const uint64_t nm2 = f32x2(neg_m, neg_m), sl2x2 = f32x2(sl2, sl2);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (c == 2) v_ready = mbar_test_wait(bar(B_VFULL0 + (it & 1)), (uint32_t)(v_use(it) & 1));
                uint32_t pk[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int j = 16 * c + jj;
                    const uint64_t sv = f32x2(s[2 * j], s[2 * j + 1]);
                    const uint64_t xv = BIASED ? add_f32x2(sv, nm2) : fma_f32x2(sv, sl2x2, nm2);
                    float x0, x1;
                    f32x2_split(xv, x0, x1);
                    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                    psum[jj & 3] = add_f32x2(psum[jj & 3], f32x2(p0, p1));
                    pk[jj] = pack_bf16x2(p0, p1);
                }
                tmem_st16(tl + TM_P + 16 * c, pk);
                if (VT && it == 0 && row0 + r < p.L) {  // the diagonal's P for the walks that follow
                    uint4* pd = reinterpret_cast<uint4*>(p.pdiag + ((size_t)bh * p.L + row0 + r) * kTcC + 32 * c);
#pragma unroll
                    for (int g = 0; g < 4; ++g) pd[g] = make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
                }
            }
            float sum;
            {
                const uint64_t t = add_f32x2(add_f32x2(psum[0], psum[1]), add_f32x2(psum[2], psum[3]));
                float a, b;
                f32x2_split(t, a, b);
                sum = a + b;
            }
            l_run = l_run * alpha + sum;
            if (r == 0) TC_TRACE(6, it);
            // The O rescale (rare: the running max grew by more than 2^8) uses
            // warp-collective TMEM loads/stores, so the whole warp takes it when any
            // of its rows needs it (alpha = 1 elsewhere).
            if (it > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t ov[32];
                    tmem_ld32(tl + TM_O + 32 * c, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
                    tmem_st32(tl + TM_O + 32 * c, ov);
                }
            }
            if (VT && it == 0 && row0 + r < p.L) p.m0[(size_t)bh * p.L + row0 + r] = m_use;
            m_run = m_use;
            tmem_wait_st();
            // V_m of this block has landed before P V may go
            ok = __all_sync(0xffffffffu,
                            v_ready || mbar_wait(bar(B_VFULL0 + (it & 1)), (uint32_t)(v_use(it) & 1), wc, 24));
            if (!ok) break;
            tc_fence_before();
            named_bar_arrive(NB_PV, NB_PV_COUNT);
            pv_sent = it + 1;
            if (r == 0) TC_TRACE(7, it);
            if (lane == 0) TC_TRACE(20 + (warp & 3), it);  // 20..23: P-ready arrival per softmax warp
            if (stop) {
                last = it;
                break;
            }
        }
        if (!ok) {  // give the MMA warp every round it may still wait for
            for (int rr = sk_sent + 1; rr <= n; ++rr) named_bar_arrive(NB_SK, NB_SK_COUNT);
            for (int rr = pv_sent; rr <= n; ++rr) named_bar_arrive(NB_PV, NB_PV_COUNT);
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(B_ODONE), (uint32_t)(last & 1), wc, 22));
        if (ok) {
            tc_fence_after();
            const int row = row0 + r;
            const float inv = 1.0f / l_run;
            __nv_bfloat16* orow = p.o + ((size_t)bh * p.L + row) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                tmem_ld32(tl + TM_O + 32 * c, ov);
                tmem_wait_ld();
                if (row < p.L && in_bounds(((long long)bh * p.L + row) * D + 32 * c, 32, n_bhl * D, p.hdr, 206)) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(ov[8 * g + 0]) * inv, __uint_as_float(ov[8 * g + 1]) * inv);
                        v.y = pack_bf16x2(__uint_as_float(ov[8 * g + 2]) * inv, __uint_as_float(ov[8 * g + 3]) * inv);
                        v.z = pack_bf16x2(__uint_as_float(ov[8 * g + 4]) * inv, __uint_as_float(ov[8 * g + 5]) * inv);
                        v.w = pack_bf16x2(__uint_as_float(ov[8 * g + 6]) * inv, __uint_as_float(ov[8 * g + 7]) * inv);
                        st_global_v4(orow + 32 * c + 8 * g, v);
                    }
                }
            }
            if (p.lse && row < p.L && in_bounds((long long)bh * p.L + row, 1, n_bhl, p.hdr, 207))
                p.lse[(size_t)bh * p.L + row] = (m_run + log2f(l_run)) * 0.6931471805599453f;
            if (r == 0) atomicAdd(p.visited, (unsigned)(last + 1));
        }
    } else {
        // ------------------------------------------------------------------ query-transport warps
        const int r = 32 * (warp & 3) + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        int sk_sent = 0;   // NB_SK rounds this warp has arrived on
        int skb_sent = 0;  // NB_SKB rounds (the second half of bf16 q~)
        auto release_second = [&](int it) {
            tc_fence_before();
            named_bar_arrive(NB_SKB, NB_SKB_COUNT);
            skb_sent = it;
        };
        // bf16 copy of 32 fp32 columns (raw bits) -> 16 packed columns of TMEM
        auto put_bf16 = [&](int c, const uint32_t (&v)[32]) {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            tmem_st16(tl + TM_QB + 16 * c, pk);
        };
        // Wait for barrier `b` (parity `par`) unless the FoX scan has stopped before
        // block iteration `it`: 1 ready, 2 stopped, 3 failed.
        auto wait_or_stop = [&](int b, uint32_t par, int it, int site) -> int {
            if (!FOX) return __all_sync(0xffffffffu, mbar_wait(bar(b), par, wc, site)) ? 1 : 3;
            int st = 0;
            const uint64_t t0 = globaltimer();
            for (uint32_t spin = 0; st == 0; ++spin) {
                if (mbar_test_wait(bar(b), par)) st = 1;
                else if (*stop_it <= it) st = 2;
                else if ((spin & 255u) == 255u && (*abort_flag || globaltimer() - t0 > p.limit_ns)) {
                    if (!*abort_flag) { report_status(p.hdr, PATH_ERR_TIMEOUT, site); *abort_flag = 1; }
                    st = 3;
                }
            }
            return (int)__reduce_max_sync(0xffffffffu, (unsigned)st);
        };
        // The copies block iteration it reads (khat, and P - I unless m = 0) have
        // landed, then NB_SK(it) may complete.  A FoX scan that stops before block
        // it still syncs NB_SK(it) (that is where the MMA warp learns of the stop),
        // so the round is arrived on then too, without waiting for copies the
        // producer may never issue.
        auto release_block = [&](int it) -> int {
            const int st = wait_or_stop(B_KMFULL0 + (it & 1), (uint32_t)((it >> 1) & 1), it, 34);
            if (st == 1 || st == 2) {
                tc_fence_before();
                named_bar_arrive(NB_SK, NB_SK_COUNT);
                sk_sent = it;
            }
            return st;
        };
        bool ok = n > 0;
        int st = 1;
        if (ok) {
            // qhat (fp32) of this row becomes the q~ master and its bf16 copy
            const bool src_ok =
                in_bounds(((long long)bh * p.Lp + row0 + r) * D, D, (long long)p.BH * p.Lp * D, p.hdr, 208);
            const float4* src = reinterpret_cast<const float4*>(p.qhat + (src_ok ? ((size_t)bh * p.Lp + row0 + r) * D : 0));
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 x = __ldg(src + 8 * c + j4);
                    v[4 * j4 + 0] = __float_as_uint(x.x);
                    v[4 * j4 + 1] = __float_as_uint(x.y);
                    v[4 * j4 + 2] = __float_as_uint(x.z);
                    v[4 * j4 + 3] = __float_as_uint(x.w);
                }
                tmem_st32(tl + TM_QM + 32 * c, v);
                put_bf16(c, v);
            }
            tmem_wait_st();
            // A parity wait names a phase correctly only once the phase before it is
            // known to be complete: a barrier still in phase k - 1 satisfies a wait
            // for phase k at once.  The first phases of SDONE and of KM slot 0 belong
            // to the diagonal block, so this warp observes the diagonal's product
            // (SDONE phase 0, which follows its copies) before it waits for SDONE
            // phase 1 and KM slot 0 phase 1 below.  SDONE cannot move past phase 1
            // before this warp arrives on NB_SK(1).
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B_SDONE), 0, wc, 30));
            if (ok) {
                st = release_block(1);
                ok = st == 1;
                if (ok) release_second(1);
            }
        }
        for (int it = 1; it < n && ok; ++it) {  // q~ for block iteration it + 1 (m = n - it > 0)
            // [S | q~](it) has completed: the master moved through chunk m and bf16
            // q~(it) is no longer read
            st = wait_or_stop(B_SDONE, (uint32_t)(it & 1), it, 31);
            if (st != 1) break;
            if (r == 0) TC_TRACE(8, it);
            tc_fence_after();
            uint32_t v[D / 32][32];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tmem_ld32(tl + TM_QM + 32 * c, v[c]);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < D / 64; ++c) put_bf16(c, v[c]);
            tmem_wait_st();
            st = release_block(it + 1);
            if (st != 1) break;
#pragma unroll
            for (int c = D / 64; c < D / 32; ++c) put_bf16(c, v[c]);
            tmem_wait_st();
            release_second(it + 1);
            if (r == 0) TC_TRACE(9, it);
        }
        if (st == 3) ok = false;
        if (!ok && n > 0) {  // give the MMA warp every round it may still wait for
            for (int rr = sk_sent + 1; rr <= n; ++rr) named_bar_arrive(NB_SK, NB_SK_COUNT);
            for (int rr = skb_sent + 1; rr <= n; ++rr) named_bar_arrive(NB_SKB, NB_SKB_COUNT);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0) TC_CTA(2, globaltimer());
}

// ----------------------------------------------------------------------------- host side
int tc_chunk(int d) { (void)d; return kTcC; }
bool tc_supported(int d) { return d == 64 || d == 128; }

#ifdef PATH_TRACE
static unsigned long long* trace_buffer() {
    static unsigned long long* buf = nullptr;
    const size_t n = kTraceCtaBase + (size_t)kTraceMaxCtas * 4;
    if (!buf && cudaMalloc(&buf, n * sizeof(unsigned long long)) == cudaSuccess)
        cudaMemset(buf, 0, n * sizeof(unsigned long long));
    return buf;
}
}  // namespace pathattn
extern "C" void path_trace_dump(unsigned long long* host) {
    cudaDeviceSynchronize();
    cudaMemcpy(host, pathattn::trace_buffer(), 64 * 32 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
}
// Per-CTA stamps of the last launch: ncta x {entry, diagonal issued, exit, SM id}.
extern "C" void path_trace_cta_dump(unsigned long long* host, int ncta) {
    cudaDeviceSynchronize();
    cudaMemcpy(host, pathattn::trace_buffer() + pathattn::kTraceCtaBase,
               (size_t)ncta * 4 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
}
namespace pathattn {
#endif

template <int D>
static cudaError_t launch_tc(const void* q, const void* k, const void* v, const float* log_f, const float* rel_bias,
                             int H, void* o, float* lse, int BH, int L, float scale, unsigned char* ws,
                             const FwdLayout& lay, int fault, const FwdOptions& opt, cudaStream_t st,
                             const void* vpairs = nullptr, void* pdiag = nullptr, float* m0 = nullptr) {
    CUtensorMap mq, mk, mv, mkh, mpm, my, mzn, mvp;
    const int ntiles = cdiv(L, kTcC);
    const int pair_rows = max(1, ntiles * (ntiles - 1) / 2) * kTcC;
    if (!make_map(&mq, q, D, L, BH) || !make_map(&mk, k, D, L, BH) || !make_map(&mv, v, D, L, BH) ||
        !make_map(&mkh, ws + lay.khat, D, lay.Lp, BH) || !make_map(&mpm, ws + lay.un, D, lay.Lp, BH) ||
        !make_map(&my, ws + lay.y, kTcC, lay.Lp, BH) || !make_map(&mzn, ws + lay.zn, kTcC, lay.Lp, BH) ||
        !make_map(&mvp, vpairs ? vpairs : v, D, vpairs ? pair_rows : L, BH))
        return cudaErrorInvalidValue;
    TcParams p;
    p.L = L;
    p.Lp = lay.Lp;
    p.ntiles = cdiv(L, kTcC);
    p.BH = BH;
    p.sl2 = scale * 1.4426950408889634f;
    p.qhat = reinterpret_cast<const float*>(ws + lay.qhat);
    p.cum = reinterpret_cast<const float*>(ws + lay.cum);
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.hdr = reinterpret_cast<WsHeader*>(ws);
    p.limit_ns = fault ? 20000000ull : 2000000000ull;  // 20 ms under the test hook, else 2 s
    p.fault = fault;
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.kmax2 = reinterpret_cast<const float*>(ws + lay.kmax);
    p.nch = lay.Lp / kTcC;
    p.rbias = rel_bias;
    p.H = H;
    p.no_skip = opt.no_skip;
    p.visited = &p.hdr->visited;
    p.pdiag = static_cast<__nv_bfloat16*>(pdiag);
    p.m0 = m0;
#ifdef PATH_TRACE
    p.trace = trace_buffer();
#endif
    auto kern = vpairs ? (log_f ? path_fwd_tc<D, 1, true> : path_fwd_tc<D, 0, true>)
                       : log_f ? path_fwd_tc<D, 1> : rel_bias ? path_fwd_tc<D, 2> : path_fwd_tc<D, 0>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
    if (e != cudaSuccess) return e;
    mark_start(st);
    kern<<<dim3(BH * p.ntiles), kTcThreads, kTcSmem, st>>>(mq, mk, mv, mkh, mpm, my, mzn, mvp, p);
    mark_end(st);
    return cudaGetLastError();
}

cudaError_t launch_ut_prep_tc(int d, const void* q, const void* k, const void* w, const float* beta, int BH, int L,
                              unsigned char* ws, const FwdLayout& lay, bool want_kmax, cudaStream_t st,
                              bool reset_header);
cudaError_t launch_vt_chain(const void* vhat, const void* pmi, void* pairs, int BH, int Lp, int N,
                            long long pair_rows, WsHeader* hdr, cudaStream_t st);
cudaError_t launch_vt_diag(const void* v, const void* w, const float* beta, const void* x, const void* pdiag,
                           const float* m0, const float* lse_in, void* o, float* lse_out, int BH, int L,
                           WsHeader* hdr, cudaStream_t st);

// PaTH(-FoX) forward with value-side transport in the blockwise form (bf16, d = 128):
//   1. the UT prep and FoX sums of the key side, as for path_attn_fwd;
//   2. the UT prep run with v in the key slot, whose khat is each value moved to
//      the end of its chunk (vhat_j = H_e ... H_{j+1} v_j);
//   3. the value chains: per key chunk m, Vtil_{m+1,m} = Vhat_m and
//      Vtil_{n+1,m} = Vtil_{n,m} P_n^T (tensor cores, fp32 master in TMEM, stored
//      bf16 per pair);
//   4. the scan with the pair store as the value operand and a zero diagonal:
//      X_i = sum over earlier chunks of alpha_ij (H_{b-1} ... H_{j+1} v_j), LSE, and
//      the diagonal block's P (bf16) with the max it was formed with;
//   5. per row, the walk of the diagonal chunk: acc <- H_j acc + alpha_ij v_j from
//      acc = X_i over j = b .. i (alpha from that P, the max and the LSE), which
//      applies H_i ... H_b to X_i and adds the diagonal's terms.
cudaError_t fwd_tc_vt_bf16(const void* q, const void* k, const void* v, const void* w, const float* beta,
                           const float* log_f, void* o, float* lse, int BH, int L, float scale, unsigned char* ws,
                           const VtBlockLayout& vl, cudaStream_t st) {
    cudaError_t e = launch_ut_prep(PATH_BF16, kTcC, 128, q, k, w, beta, log_f, BH, L, ws, vl.lay, st);
    if (e != cudaSuccess) return e;
    e = launch_ut_prep_tc(128, q, v, w, beta, BH, L, ws, vl.lay2, false, st, false);
    if (e != cudaSuccess) return e;
    e = launch_vt_chain(ws + vl.lay2.khat, ws + vl.lay.un, ws + vl.pairs, BH, vl.lay.Lp, vl.N, vl.pair_rows,
                        reinterpret_cast<WsHeader*>(ws), st);
    if (e != cudaSuccess) return e;
    FwdOptions opt;
    opt.no_skip = 0;
    e = launch_tc<128>(q, k, v, log_f, nullptr, 1, ws + vl.x, reinterpret_cast<float*>(ws + vl.lse), BH, L, scale,
                       ws, vl.lay, 0, opt, st, ws + vl.pairs, ws + vl.pdiag, reinterpret_cast<float*>(ws + vl.m0));
    if (e != cudaSuccess) return e;
    return launch_vt_diag(v, w, beta, ws + vl.x, ws + vl.pdiag, reinterpret_cast<const float*>(ws + vl.m0),
                          reinterpret_cast<const float*>(ws + vl.lse), o, lse, BH, L, reinterpret_cast<WsHeader*>(ws),
                          st);
}

cudaError_t fwd_tc_bf16(const void* q, const void* k, const void* v, const void* w, const float* beta,
                        const float* log_f, const float* rel_bias, int H, void* o, float* lse, int BH, int L, int d,
                        float scale, unsigned char* ws, const FwdLayout& lay, int fault_mask, const FwdOptions& opt,
                        cudaStream_t st) {
    cudaError_t e = launch_ut_prep(PATH_BF16, kTcC, d, q, k, w, beta, log_f, BH, L, ws, lay, st);
    if (e != cudaSuccess) return e;
    if (d == 64) return launch_tc<64>(q, k, v, log_f, rel_bias, H, o, lse, BH, L, scale, ws, lay, fault_mask, opt, st);
    if (d == 128) return launch_tc<128>(q, k, v, log_f, rel_bias, H, o, lse, BH, L, scale, ws, lay, fault_mask, opt, st);
    return cudaErrorInvalidValue;
}

}  // namespace pathattn
