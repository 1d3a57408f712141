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
// transported query q~ (fp32 master in TMEM, bf16 copy in shared memory):
//   S_w   S_w = q~ W_m^T                               (M=128, N=128, K=d)
//   S_k   S_k = q~ khat_m^T                            (M=128, N=128, K=d)
//   MMA3  q~ += bf16(S_w) (-U_m)                       (M=128, N=d, K=128)
//   P V   O  += P V_m,  P = exp2(S_k * scale*log2e - m)  (M=128, N=d, K=128)
// and the diagonal block uses S = Q K^T + Y (-Z)^T with the causal mask.  The
// logits may carry an additive bias (MODE 1 PaTH-FoX, MODE 2 relative position).
// Online softmax keeps one query row per thread (TMEM lane = row), so row
// max and sum need no cross-thread reduction.  The running max is only
// raised (and O rescaled) when it grows by more than 2^8, which keeps every
// exponent <= 2^8 and makes rescales rare.
//
// Warp roles (352 threads):
//   warp 0      TMA producer (one lane) + TMEM allocation
//   warp 1      tcgen05.mma issuer (one lane): S_w and MMA3 (with FoX: all MMAs)
//   warps 2-5   softmax: S_k -> P (bf16, into TMEM), row statistics, epilogue
//   warps 6-9   query transport: S_w -> bf16 (TMEM), fp32 q~ -> bf16 q~ (smem)
//   warp 10     tcgen05.mma issuer (one lane): diagonal, S_k and P V (idle with FoX)
//
// TMEM (512 columns x 128 lanes, fp32): [0,128) S_k / P (bf16), [128,256) S_w /
// bf16(S_w), [256,256+d) O, [384,384+d) q~ master.
// Shared memory (1024-aligned, 128-byte swizzled tiles as TMA writes them):
//   SM_Q  32 KB  Q (diagonal) then bf16 q~, K-major, 64-column chunks of 16 KB
//   SM_KW 64 KB  per 64-column chunk c (32 KB): rows 0-127 khat_m (or K),
//                rows 128-255 W_m of even block iterations (or -Z)
//   SM_V  64 KB  V_m, MN-major B operand (64-column boxes of 16 KB), two
//                slots by block parity
//   SM_U  32 KB  -U_m (MN-major) or, on the diagonal, Y (K-major)
//   SM_P  32 KB  W slot 1 (W of odd block iterations; slot 0 is interleaved
//                with khat in SM_KW)
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
constexpr int kTcThreads = 352;
constexpr uint32_t SM_Q = 0, SM_KW = 32768, SM_V = 98304, SM_U = 163840, SM_P = 196608, SM_BAR = 229376;
constexpr uint32_t SM_TOTAL = SM_BAR + 256;
constexpr size_t kTcSmem = SM_TOTAL + 1024;  // + alignment slack
constexpr uint32_t TM_S = 0, TM_SW = 128, TM_O = 256, TM_Q = 384;

// Every barrier below is waited on in a way that it can never run two phases
// ahead of its waiter (a parity wait cannot tell those apart).
// Each operand slot (khat, W, -U, V) has its own full/empty pair, released
// by the MMA that consumes it, so every refill starts as early as possible.
// W and V are double-buffered by block parity (slot it & 1).
enum Bar { B_QFULL = 0, B_KFULL, B_WFULL0, B_UFULL, B_VFULL0, B_KEMPTY, B_WEMPTY0, B_UEMPTY, B_VEMPTY0, B_SFULL,
           B_SWREADY, B_PREADY, B_QUPD, B_QTREADY, B_ODONE, B_DRAIN, B_SREAD, B_VFULL1, B_VEMPTY1, B_WFULL1,
           B_WEMPTY1, B_SWFULL, B_DRAIN2, B_COUNT };
// Barriers at SM_BAR, then the control words (TMEM address, abort flag, FoX
// stop index and votes, max |khat|^2) at SM_CTL, all inside SM_BAR + 256.
constexpr uint32_t SM_CTL = SM_BAR + 192;
static_assert(B_COUNT * 8 <= 192, "barriers overlap the control words");
static_assert(SM_CTL + 52 <= SM_TOTAL, "control words exceed the barrier region");

constexpr int kHeadGroup = 8;

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
#else
#define TC_TRACE(slot, it) do { } while (0)
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
#ifdef PATH_TRACE
    unsigned long long* trace;
#endif
};

// MODE 0: PaTH; 1: PaTH-FoX (forget-gate bias, far blocks skipped); 2: PaTH
// with a relative-position bias table rel[h][i - j].
template <int D, int MODE>
__global__ void __launch_bounds__(kTcThreads, 1)
    path_fwd_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_w,
                const __grid_constant__ CUtensorMap tm_khat, const __grid_constant__ CUtensorMap tm_un,
                const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ CUtensorMap tm_zn,
                const TcParams p) {
    static_assert(D == 64 || D == 128, "head dim");
    constexpr bool FOX = MODE == 1, REL = MODE == 2;
    constexpr bool BIASED = MODE != 0;   // logits carry an additive bias (log2 units in the softmax)
    constexpr int KCH = D / 64;          // 64-column chunks of the head dim
    constexpr uint32_t ROWB = 128u * D * 2u;  // bytes of one [128 x D] bf16 tile
    constexpr uint32_t IDESC_S128 = idesc_bf16(128, false);
    constexpr uint32_t IDESC_PV = idesc_bf16(D, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    const uint32_t bar0 = sb + SM_BAR;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    // control words after the barriers (B_COUNT * 8 bytes)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + SM_CTL);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + SM_CTL + 4);
    // PaTH-FoX far-block skipping: the scan stops before block iteration
    // *stop_it (n + 1 = never); set by the softmax warps before they release S_k.
    volatile int* stop_it = reinterpret_cast<volatile int*>(sm + SM_CTL + 8);
    int* votes = reinterpret_cast<int*>(sm + SM_CTL + 16);     // [2][4]
    float* s_kmax2 = reinterpret_cast<float*>(sm + SM_CTL + 48);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
        counts[B_SWREADY] = counts[B_PREADY] = counts[B_QTREADY] = counts[B_SREAD] = 128;
        for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), counts[i]);
        *abort_flag = 0;
        *stop_it = n + 1;
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
            prefetch_tmap(&tm_q); prefetch_tmap(&tm_k); prefetch_tmap(&tm_v); prefetch_tmap(&tm_w);
            prefetch_tmap(&tm_khat); prefetch_tmap(&tm_un); prefetch_tmap(&tm_y); prefetch_tmap(&tm_zn);
            bool ok = true;
            // diagonal block: Q, K (khat slot), -Z (W slot), Y (-U slot), V
            mbar_expect_tx(bar(B_QFULL), ROWB);
            for (int c = 0; c < KCH; ++c) tma_load_3d(sb + SM_Q + c * 16384, &tm_q, bar(B_QFULL), c * 64, row0, bh);
            mbar_expect_tx(bar(B_KFULL), ROWB);
            for (int c = 0; c < KCH; ++c) tma_load_3d(sb + SM_KW + c * 32768, &tm_k, bar(B_KFULL), c * 64, row0, bh);
            mbar_expect_tx(bar(B_WFULL0), 32768);
            for (int c = 0; c < 2; ++c)
                tma_load_3d(sb + SM_KW + c * 32768 + 16384, &tm_zn, bar(B_WFULL0), c * 64, row0, bh);
            mbar_expect_tx(bar(B_UFULL), 32768);
            for (int c = 0; c < 2; ++c) tma_load_3d(sb + SM_U + c * 16384, &tm_y, bar(B_UFULL), c * 64, row0, bh);
            mbar_expect_tx(bar(B_VFULL0), ROWB);
            for (int c = 0; c < KCH; ++c) tma_load_3d(sb + SM_V + c * 16384, &tm_v, bar(B_VFULL0), c * 64, row0, bh);
            // scan blocks: refill each slot as soon as its consumer has finished.
            // khat / -U for block iteration it need the (it)-th completion of
            // their empty barrier; W and V use slot it & 1 and, from it = 2 on,
            // the (it >> 1)-th completion of that slot's empty barrier.  W and
            // -U are not used by the last block (m = 0).
            enum { SW = 0, SK, SU, SV };
            // issued: W slot 0, khat, -U, V slot 0, V slot 1, W slot 1
            int nxt[4] = {1, 1, 1, 1}, issued[6] = {1, 1, 1, 1, 0, 0};
            const int emp[3] = {B_WEMPTY0, B_KEMPTY, B_UEMPTY};
            const uint64_t t0 = globaltimer();
            for (uint32_t spin = 0; ok && (nxt[0] <= n || nxt[1] <= n || nxt[2] <= n || nxt[3] <= n); ++spin) {
                const int stop = FOX ? *stop_it : n + 1;
                for (int sl = 0; sl < 4; ++sl) {
                    const int it = nxt[sl];
                    if (it > n) continue;
                    if (it >= stop) { nxt[sl] = n + 1; continue; }  // beyond the last block the scan visits
                    if ((sl == SW || sl == SU) && it == n) { nxt[sl] = n + 1; continue; }
                    if (sl == SV || sl == SW) {
                        const int eb = sl == SV ? ((it & 1) ? B_VEMPTY1 : B_VEMPTY0) : ((it & 1) ? B_WEMPTY1 : B_WEMPTY0);
                        if (it >= 2 && !mbar_test_wait(bar(eb), (uint32_t)(((it >> 1) - 1) & 1))) continue;
                    } else if (!mbar_test_wait(bar(emp[sl]), (it - 1) & 1)) {
                        continue;
                    }
                    const int r = (n - it) * kTcC;
                    nxt[sl] = it + 1;
                    if (sl == SV && p.fault && it == 1) continue;  // test hook: the consumer's wait must expire
                    const int fb = sl == SW ? ((it & 1) ? B_WFULL1 : B_WFULL0)
                                   : sl == SK ? B_KFULL : sl == SU ? B_UFULL : ((it & 1) ? B_VFULL1 : B_VFULL0);
                    mbar_expect_tx(bar(fb), ROWB);
                    for (int c = 0; c < KCH; ++c) {
                        if (sl == SK) tma_load_3d(sb + SM_KW + c * 32768, &tm_khat, bar(fb), c * 64, r, bh);
                        if (sl == SW) {
                            const uint32_t dst = (it & 1) ? sb + SM_P + c * 16384 : sb + SM_KW + c * 32768 + 16384;
                            tma_load_3d(dst, &tm_w, bar(fb), c * 64, r, bh);
                        }
                        if (sl == SU) tma_load_3d(sb + SM_U + c * 16384, &tm_un, bar(fb), c * 64, r, bh);
                        if (sl == SV) tma_load_3d(sb + SM_V + (it & 1) * 32768 + c * 16384, &tm_v, bar(fb), c * 64, r, bh);
                    }
                    ++issued[sl == SV ? 3 + (it & 1) : (sl == SW && (it & 1)) ? 5 : sl];
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
            drain_wait(bar(B_QFULL), 0, p.limit_ns, p.hdr, 90);
            const int ful[6] = {B_WFULL0, B_KFULL, B_UFULL, B_VFULL0, B_VFULL1, B_WFULL1};
            for (int sl = 0; sl < 6; ++sl)
                if (issued[sl] > 0) drain_wait(bar(ful[sl]), (uint32_t)((issued[sl] - 1) & 1), p.limit_ns, p.hdr, 91);
        }
    } else if (warp == 1 || warp == 10) {
        // ------------------------------------------------------------------ MMA issuers
        // Issue is blocking (an MMA group's issue returns about when it has
        // executed), and every barrier poll costs a few hundred cycles while SS
        // MMAs hold the shared-memory port.  Without FoX two threads issue:
        //   warp 1  (transport chain)  S_w(it), MMA3(it)             it = 1 .. n-1
        //   warp 10 (softmax chain)    diagonal, P V(it-1), S_k(it)   it = 1 .. n
        // so that one thread's waits overlap the other's MMAs.  Their TMEM
        // columns are disjoint (S_w / q~ against S_k, P / O); the transport
        // warps wait for S_k(it) as well as MMA3(it) before they overwrite the
        // shared q~ tile.  With FoX (far-block stopping) warp 1 issues all of
        // it in the order S_w(it), P V(it-1), S_k(it), MMA3(it).
        const bool issuer_b = FOX ? warp == 1 : warp == 10;  // diagonal, P V, S_k
        const bool issuer_a = warp == 1;                      // S_w, MMA3
        if (lane == 0 && (issuer_a || issuer_b)) {
            auto issue_pv = [&](int blk) {  // O (+)= P V for block iteration blk (P in TMEM)
                tc_fence_after();
                const uint32_t vbuf = sb + SM_V + (uint32_t)(blk & 1) * 32768u;
                for (int kk = 0; kk < kTcC / 16; ++kk)
                    mma_ts(tmem + TM_O, tmem + TM_S + kk * 8, mnmajor_desc(vbuf, kk), IDESC_PV,
                           (blk > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bar(B_ODONE));
                mma_commit(bar((blk & 1) ? B_VEMPTY1 : B_VEMPTY0));
            };
            // P V of block blk needs its P (p_ready, (blk+1)-th completion) and
            // its V slot (blk & 1, (blk >> 1)+1-th completion).  Without FoX the
            // warps that arrive on P-ready, q~-ready and S_w-ready first wait for
            // the V, khat / W and -U copies of that block, so the issuers only
            // wait for the handoffs.
            auto wait_pv = [&](int blk) {
                return mbar_wait(bar(B_PREADY), (uint32_t)(blk & 1), wc, 18) &&
                       (!FOX || mbar_wait(bar((blk & 1) ? B_VFULL1 : B_VFULL0), (uint32_t)((blk >> 1) & 1), wc, 19));
            };
            auto issue_sw = [&](int it) {  // S_w = q~ W^T (W slot it & 1)
                tc_fence_after();
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t bdesc = (it & 1) ? kmajor_desc(sb + SM_P, kk, 16384)
                                                    : kmajor_desc(sb + SM_KW + 16384, kk, 32768);
                    mma_ss(tmem + TM_SW, kmajor_desc(sb + SM_Q, kk, 16384), bdesc, IDESC_S128, kk > 0);
                }
                mma_commit(bar(B_SWFULL));
                mma_commit(bar((it & 1) ? B_WEMPTY1 : B_WEMPTY0));
                TC_TRACE(0, it);
            };
            auto issue_sk = [&](int it) {  // S_k = q~ khat^T
                tc_fence_after();
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + TM_S, kmajor_desc(sb + SM_Q, kk, 16384), kmajor_desc(sb + SM_KW, kk, 32768),
                           IDESC_S128, kk > 0);
                mma_commit(bar(B_SFULL));
                mma_commit(bar(B_KEMPTY));
                TC_TRACE(1, it);
            };
            auto issue_m3 = [&](int it) {  // q~ += bf16(S_w) (-U)
                tc_fence_after();
                for (int kk = 0; kk < kTcC / 16; ++kk)
                    mma_ts(tmem + TM_Q, tmem + TM_SW + kk * 8, mnmajor_desc(sb + SM_U, kk), IDESC_PV, 1);
                mma_commit(bar(B_QUPD));
                mma_commit(bar(B_UEMPTY));
                TC_TRACE(3, it);
            };
            bool ok = true;
            if (issuer_b) {
                ok = mbar_wait(bar(B_QFULL), 0, wc, 10) && mbar_wait(bar(B_KFULL), 0, wc, 11) &&
                     mbar_wait(bar(B_WFULL0), 0, wc, 12) && mbar_wait(bar(B_UFULL), 0, wc, 12);
                if (ok) {
                    tc_fence_after();
                    // diagonal: S = Q K^T + Y (-Z)^T
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tmem + TM_S, kmajor_desc(sb + SM_Q, kk, 16384), kmajor_desc(sb + SM_KW, kk, 32768),
                               IDESC_S128, kk > 0);
                    for (int kk = 0; kk < kTcC / 16; ++kk)
                        mma_ss(tmem + TM_S, kmajor_desc(sb + SM_U, kk, 16384),
                               kmajor_desc(sb + SM_KW + 16384, kk, 32768), IDESC_S128, 1);
                    mma_commit(bar(B_SFULL));
                    mma_commit(bar(B_KEMPTY));
                    mma_commit(bar(B_WEMPTY0));
                    mma_commit(bar(B_UEMPTY));
                }
            }
            if (FOX) {
                // single issuer: S_w(it) -> P V(it-1) -> S_k(it) -> MMA3(it); P V and S_k
                // cover the conversion of S_w, and S_k follows P V because it
                // overwrites the TMEM columns that hold P.
                int last = n;  // last block iteration whose P V is issued
                for (int it = 1; it <= n && ok; ++it) {
                    const int m = n - it;
                    // the softmax warps decide first whether block it is visited
                    if (!(ok = mbar_wait(bar(B_SREAD), (it - 1) & 1, wc, 15))) break;
                    if (*stop_it <= it) {  // every block from here on contributes exactly zero
                        last = it - 1;
                        break;
                    }
                    if (!(ok = mbar_wait(bar(B_QTREADY), (it - 1) & 1, wc, 14))) break;
                    if (m > 0) {
                        if (!(ok = mbar_wait(bar((it & 1) ? B_WFULL1 : B_WFULL0), (uint32_t)((it >> 1) & 1), wc, 15)))
                            break;
                        issue_sw(it);
                    }
                    if (!(ok = wait_pv(it - 1))) break;
                    issue_pv(it - 1);
                    TC_TRACE(2, it);
                    if (!(ok = mbar_wait(bar(B_KFULL), it & 1, wc, 15))) break;
                    issue_sk(it);
                    if (m > 0) {
                        if (!(ok = mbar_wait(bar(B_UFULL), it & 1, wc, 16))) break;
                        if (!(ok = mbar_wait(bar(B_SWREADY), (it - 1) & 1, wc, 17))) break;
                        issue_m3(it);
                    }
                }
                if (ok && wait_pv(last)) issue_pv(last);  // the last block's P V
            } else if (issuer_b) {
                for (int it = 1; it <= n && ok; ++it) {
                    if (!(ok = wait_pv(it - 1))) break;
                    TC_TRACE(20, it);
                    issue_pv(it - 1);
                    TC_TRACE(2, it);
                    issue_sk(it);  // its khat and q~ were awaited before P-ready (softmax warps 3, 4)
                }
                if (ok && wait_pv(n)) issue_pv(n);  // the last block's P V
            } else {
                for (int it = 1; it < n && ok; ++it) {
                    if (!(ok = mbar_wait(bar(B_QTREADY), (it - 1) & 1, wc, 14))) break;
                    issue_sw(it);
                    if (!(ok = mbar_wait(bar(B_SWREADY), (it - 1) & 1, wc, 17))) break;
                    TC_TRACE(23, it);
                    issue_m3(it);
                }
            }
            // every MMA this thread issued completes before TMEM is released
            const int drain = (FOX || issuer_a) ? B_DRAIN : B_DRAIN2;
            mma_commit(bar(drain));
            drain_wait(bar(drain), 0, p.limit_ns, p.hdr, 92);
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------------ softmax warps
        const int r = 32 * (warp & 3) + lane;  // query row within the tile (= TMEM lane)
        const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const float* cumh = FOX ? p.cum + (size_t)bh * p.Lp : nullptr;
        const float* relh = REL ? p.rbias + (size_t)(bh % p.H) * p.L : nullptr;
        const float ci = FOX ? cumh[row0 + r] : 0.f;
        constexpr float kL2e = 1.4426950408889634f;
        float m_run = -INFINITY, l_run = 0.f;
        float m_true = -INFINITY;  // largest logit seen (log2 units)
        float qk_bound = 0.f;      // FoX: scale log2e |q_i| max_j |khat_j|, with a 2x margin
        if (FOX && n > 0) {
            if (warp == 2) {  // max |khat|^2 over the chunks left of this tile
                float x = 0.f;
                for (int c = lane; c < n; c += 32) x = fmaxf(x, p.kmax2[(size_t)bh * p.nch + c]);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
                if (lane == 0) *s_kmax2 = x;
            }
            float qn2 = 0.f;
            if (row0 + r < p.L) {
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
        for (int it = 0; it <= n; ++it) {
            const int m = n - it;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B_SFULL), it & 1, wc, 20));
            if (!ok) break;
            if (r == 0) TC_TRACE(4, it);
            tc_fence_after();
            float s[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t raw[32];
                tmem_ld32(tl + TM_S + 32 * c, raw);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) s[32 * c + j] = __uint_as_float(raw[j]);
            }
            // Without a bias the scores stay raw (the scale is applied inside the
            // exponent, one FFMA each); with one (FoX, relative) they become
            // log2-unit logits.
            const float sl2 = p.sl2;
            // S_k is in registers: the next block's S_k may overwrite it (FoX
            // first decides whether there is a next block)
            if (!FOX) {
                tc_fence_before();
                mbar_arrive(bar(B_SREAD));
            }
            if (r == 0) TC_TRACE(5, it);
            if (FOX) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float4* cj = reinterpret_cast<const float4*>(cumh + m * kTcC + 32 * c);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 cv = __ldg(cj + j4);
                        s[32 * c + 4 * j4 + 0] = fmaf(s[32 * c + 4 * j4 + 0], sl2, (ci - cv.x) * kL2e);
                        s[32 * c + 4 * j4 + 1] = fmaf(s[32 * c + 4 * j4 + 1], sl2, (ci - cv.y) * kL2e);
                        s[32 * c + 4 * j4 + 2] = fmaf(s[32 * c + 4 * j4 + 2], sl2, (ci - cv.z) * kL2e);
                        s[32 * c + 4 * j4 + 3] = fmaf(s[32 * c + 4 * j4 + 3], sl2, (ci - cv.w) * kL2e);
                    }
                }
            }
            if (REL) {  // bias at distance i - j, clamped into the table (masked or padding entries)
                const int base = row0 + r - m * kTcC;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float bv[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) bv[j] = __ldg(relh + min(max(base - 32 * c - j, 0), p.L - 1));
#pragma unroll
                    for (int j = 0; j < 32; ++j) s[32 * c + j] = fmaf(s[32 * c + j], sl2, bv[j] * kL2e);
                }
            }
            if (it == 0) {
#pragma unroll
                for (int j = 0; j < 128; ++j)
                    if (j > r) s[j] = -INFINITY;
            }
            float mx;  // row max in log2 units (8 independent partial maxima)
            {
                float pm[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) pm[u] = s[u];
#pragma unroll
                for (int j = 8; j < 128; ++j) pm[j & 7] = fmaxf(pm[j & 7], s[j]);
                mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])), fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
                if (!BIASED) mx *= sl2;  // sl2 > 0: the max of raw scores scales
            }
            bool stop = false;
            if (FOX) {
                m_true = fmaxf(m_true, mx);
                if (m > 0) {
                    // Every key left of this block has bias <= c_i - c_(128 m - 1) and
                    // |logit| <= qk_bound: below m_true - 160 (log2) its exp2 is 0 in fp32.
                    const float bound = qk_bound + (ci - cumh[m * kTcC - 1]) * kL2e - m_true;
                    const bool sat = (row0 + r >= p.L) || bound < -160.0f;
                    const int vote = __all_sync(0xffffffffu, sat);
                    if (lane == 0) votes[(it & 1) * 4 + (warp & 3)] = vote;
                    named_bar_sync(2, 128);
                    const int* vv = votes + (it & 1) * 4;
                    stop = vv[0] && vv[1] && vv[2] && vv[3];
                    if (stop && warp == 2 && lane == 0) *stop_it = it + 1;
                }
                tc_fence_before();
                mbar_arrive(bar(B_SREAD));
            }
            const float m_new = fmaxf(m_run, mx);
            const bool rescale = m_new > m_run + 8.0f;
            const float m_use = rescale ? m_new : m_run;
            const float alpha = rescale ? ex2_approx(m_run - m_use) : 1.0f;
            float psum[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) psum[u] = 0.f;
            uint32_t pk[64];
            const float neg_m = -m_use;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const float p0 = ex2_approx(BIASED ? s[2 * j] + neg_m : fmaf(s[2 * j], sl2, neg_m));
                const float p1 = ex2_approx(BIASED ? s[2 * j + 1] + neg_m : fmaf(s[2 * j + 1], sl2, neg_m));
                psum[j & 7] += p0 + p1;
                pk[j] = pack_bf16x2(p0, p1);
            }
            const float sum = ((psum[0] + psum[1]) + (psum[2] + psum[3])) + ((psum[4] + psum[5]) + (psum[6] + psum[7]));
            l_run = l_run * alpha + sum;
            if (r == 0) TC_TRACE(6, it);
            // The O rescale uses warp-collective TMEM loads/stores, so the whole
            // warp takes it when any of its rows needs it (alpha = 1 elsewhere).
            if (__any_sync(0xffffffffu, rescale && it > 0)) {
                // O is stable once the previous block's P V has completed
                const bool ok2 = __all_sync(0xffffffffu, mbar_wait(bar(B_ODONE), (it - 1) & 1, wc, 21));
                if (!ok2) { ok = false; break; }
                tc_fence_after();
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
            m_run = m_use;
            // P (bf16 pairs) over S_k's first 64 columns: the A operand of P V.  The
            // next S_k is issued after this P V, so it cannot overwrite P early.
            tmem_st32(tl + TM_S, *reinterpret_cast<const uint32_t(*)[32]>(pk));
            tmem_st32(tl + TM_S + 32, *reinterpret_cast<const uint32_t(*)[32]>(pk + 32));
            tmem_wait_st();
            // Without FoX, P-ready also stands for the inputs of the issuer's next two
            // MMAs: warp 2 waits for this block's V (P V), warp 3 for the next
            // block's khat and warp 4 for the next q~ (S_k of block it + 1), each in
            // parallel, so the issuer polls P-ready alone.
            if (!FOX && warp == 2) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar((it & 1) ? B_VFULL1 : B_VFULL0), (uint32_t)((it >> 1) & 1), wc, 24));
                if (!ok) break;
            }
            if (!FOX && warp == 3 && it < n) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(B_KFULL), (it + 1) & 1, wc, 25));
                if (!ok) break;
            }
            if (!FOX && warp == 4 && it < n) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(B_QTREADY), it & 1, wc, 26));
                if (!ok) break;
            }
            tc_fence_before();
            mbar_arrive(bar(B_PREADY));
            if (r == 0) TC_TRACE(7, it);
            if (lane == 0) TC_TRACE(14 + warp, it);  // 16..19: P-ready arrival of warps 2..5
            if (stop) {
                last = it;
                break;
            }
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
                if (row < p.L) {
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
            if (p.lse && row < p.L) p.lse[(size_t)bh * p.L + row] = (m_run + log2f(l_run)) * 0.6931471805599453f;
        }
    } else {
        // ------------------------------------------------------------------ query-transport warps
        const int r = 32 * (warp & 3) + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        uint8_t* qrow_s = sm + SM_Q + r * 128;  // this row's 128-byte line in chunk 0
        const int sw = r & 7;
        // bf16 q~ row -> swizzled K-major tile (16-byte granule g of chunk c at (g ^ (r & 7)))
        auto put_granule = [&](int G, uint4 v) {
            *reinterpret_cast<uint4*>(qrow_s + (G >> 3) * 16384 + (((G & 7) ^ sw) << 4)) = v;
        };
        // Without FoX, warp 6 waits for the W copy of block blk before q~-ready
        // (S_w is the first MMA that reads q~), and for -U before S_w-ready.
        auto loads_for_q = [&](int blk) -> bool {
            if (FOX || warp != 6 || n - blk == 0) return true;
            return __all_sync(0xffffffffu, mbar_wait(bar((blk & 1) ? B_WFULL1 : B_WFULL0),
                                                     (uint32_t)((blk >> 1) & 1), wc, 35));
        };
        // This row of qhat (fp32), the initial q~: every load is issued before
        // the wait for the diagonal, so their latency hides behind it (issued
        // chunk by chunk between the TMEM stores, the loads were serialised).
        float4 qh[D / 4];
        if (n > 0) {
            const float4* src = reinterpret_cast<const float4*>(p.qhat + ((size_t)bh * p.Lp + row0 + r) * D);
#pragma unroll
            for (int i = 0; i < D / 4; ++i) qh[i] = __ldg(src + i);
        }
        bool ok = n > 0 && __all_sync(0xffffffffu, mbar_wait(bar(B_SFULL), 0, wc, 30));
        if (ok) {
            // the diagonal MMA has consumed Q: qhat becomes the fp32 master and its bf16 copy
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 x = qh[8 * c + j4];
                    v[4 * j4 + 0] = __float_as_uint(x.x);
                    v[4 * j4 + 1] = __float_as_uint(x.y);
                    v[4 * j4 + 2] = __float_as_uint(x.z);
                    v[4 * j4 + 3] = __float_as_uint(x.w);
                }
                tmem_st32(tl + TM_Q + 32 * c, v);
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    uint4 q;
                    q.x = pack_bf16x2(__uint_as_float(v[8 * g + 0]), __uint_as_float(v[8 * g + 1]));
                    q.y = pack_bf16x2(__uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3]));
                    q.z = pack_bf16x2(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5]));
                    q.w = pack_bf16x2(__uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7]));
                    put_granule(4 * c + g, q);
                }
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            ok = loads_for_q(1);
            tc_fence_before();
            if (ok) mbar_arrive(bar(B_QTREADY));
        }
        for (int it = 1; it < n && ok; ++it) {  // block m = n - it > 0 needs the transport
            if (FOX) {  // S_w of block iteration it, unless the scan stopped before it
                int st = 0;  // 0 waiting, 1 ready, 2 stopped, 3 failed
                const uint64_t t0 = globaltimer();
                for (uint32_t spin = 0; st == 0; ++spin) {
                    if (mbar_test_wait(bar(B_SWFULL), (it - 1) & 1)) st = 1;
                    else if (*stop_it <= it) st = 2;
                    else if ((spin & 255u) == 255u && (*abort_flag || globaltimer() - t0 > p.limit_ns)) {
                        if (!*abort_flag) { report_status(p.hdr, PATH_ERR_TIMEOUT, 33); *abort_flag = 1; }
                        st = 3;
                    }
                }
                st = __reduce_max_sync(0xffffffffu, (unsigned)st);
                if (st == 2) break;
                ok = st == 1;
            } else {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(B_SWFULL), (it - 1) & 1, wc, 31));
            }
            if (!ok) break;
            if (r == 0) TC_TRACE(8, it);
            tc_fence_after();
            // S_w (fp32, columns [128,256)) -> bf16 pairs in columns [128,192)
            {
                uint32_t v[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(tl + TM_SW + 32 * c, v[c]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        pk[j] = pack_bf16x2(__uint_as_float(v[c][2 * j]), __uint_as_float(v[c][2 * j + 1]));
                    tmem_st16(tl + TM_SW + 16 * c, pk);
                }
            }
            tmem_wait_st();
            if (!FOX && warp == 6 && !(ok = __all_sync(0xffffffffu, mbar_wait(bar(B_UFULL), it & 1, wc, 36)))) break;
            tc_fence_before();
            mbar_arrive(bar(B_SWREADY));
            if (lane == 0) TC_TRACE(22 + warp, it);  // 28..31: S_w-ready arrival of warps 6..9
            if (r == 0) TC_TRACE(9, it);
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B_QUPD), (it - 1) & 1, wc, 32));
            // with two issuers S_k(it), which also reads the q~ tile, completes on its own
            if (!FOX && ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(B_SFULL), it & 1, wc, 37));
            if (!ok) break;
            if (r == 0) TC_TRACE(10, it);
            tc_fence_after();
            {
                uint32_t v[D / 32][32];
#pragma unroll
                for (int c = 0; c < D / 32; ++c) tmem_ld32(tl + TM_Q + 32 * c, v[c]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < D / 32; ++c)
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        uint4 q;
                        q.x = pack_bf16x2(__uint_as_float(v[c][8 * g + 0]), __uint_as_float(v[c][8 * g + 1]));
                        q.y = pack_bf16x2(__uint_as_float(v[c][8 * g + 2]), __uint_as_float(v[c][8 * g + 3]));
                        q.z = pack_bf16x2(__uint_as_float(v[c][8 * g + 4]), __uint_as_float(v[c][8 * g + 5]));
                        q.w = pack_bf16x2(__uint_as_float(v[c][8 * g + 6]), __uint_as_float(v[c][8 * g + 7]));
                        put_granule(4 * c + g, q);
                    }
            }
            fence_proxy_async_smem();
            if (!(ok = loads_for_q(it + 1))) break;
            tc_fence_before();
            mbar_arrive(bar(B_QTREADY));
            if (r == 64) TC_TRACE(11, it);
            if (lane == 0) TC_TRACE(18 + warp, it);  // 24..27: q~-ready arrival of warps 6..9
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ----------------------------------------------------------------------------- host side
int tc_chunk(int d) { (void)d; return kTcC; }
bool tc_supported(int d) { return d == 64 || d == 128; }

#ifdef PATH_TRACE
static unsigned long long* trace_buffer() {
    static unsigned long long* buf = nullptr;
    if (!buf && cudaMalloc(&buf, 64 * 32 * sizeof(unsigned long long)) == cudaSuccess)
        cudaMemset(buf, 0, 64 * 32 * sizeof(unsigned long long));
    return buf;
}
}  // namespace pathattn
extern "C" void path_trace_dump(unsigned long long* host) {
    cudaDeviceSynchronize();
    cudaMemcpy(host, pathattn::trace_buffer(), 64 * 32 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
}
namespace pathattn {
#endif

template <int D>
static cudaError_t launch_tc(const void* q, const void* k, const void* v, const void* w, const float* log_f,
                            const float* rel_bias, int H, void* o, float* lse, int BH, int L, float scale,
                            unsigned char* ws, const FwdLayout& lay, int fault, cudaStream_t st) {
    CUtensorMap mq, mk, mv, mw, mkh, mun, my, mzn;
    if (!make_map(&mq, q, D, L, BH) || !make_map(&mk, k, D, L, BH) || !make_map(&mv, v, D, L, BH) ||
        !make_map(&mw, w, D, L, BH) || !make_map(&mkh, ws + lay.khat, D, lay.Lp, BH) ||
        !make_map(&mun, ws + lay.un, D, lay.Lp, BH) || !make_map(&my, ws + lay.y, kTcC, lay.Lp, BH) ||
        !make_map(&mzn, ws + lay.zn, kTcC, lay.Lp, BH))
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
#ifdef PATH_TRACE
    p.trace = trace_buffer();
#endif
    auto kern = log_f ? path_fwd_tc<D, 1> : rel_bias ? path_fwd_tc<D, 2> : path_fwd_tc<D, 0>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
    if (e != cudaSuccess) return e;
    mark_start(st);
    kern<<<dim3(BH * p.ntiles), kTcThreads, kTcSmem, st>>>(mq, mk, mv, mw, mkh, mun, my, mzn, p);
    mark_end(st);
    return cudaGetLastError();
}

cudaError_t fwd_tc_bf16(const void* q, const void* k, const void* v, const void* w, const float* beta,
                        const float* log_f, const float* rel_bias, int H, void* o, float* lse, int BH, int L, int d,
                        float scale, unsigned char* ws, const FwdLayout& lay, int fault_mask, cudaStream_t st) {
    cudaError_t e = launch_ut_prep(PATH_BF16, kTcC, d, q, k, w, beta, log_f, BH, L, ws, lay, st);
    if (e != cudaSuccess) return e;
    if (d == 64) return launch_tc<64>(q, k, v, w, log_f, rel_bias, H, o, lse, BH, L, scale, ws, lay, fault_mask, st);
    if (d == 128) return launch_tc<128>(q, k, v, w, log_f, rel_bias, H, o, lse, BH, L, scale, ws, lay, fault_mask, st);
    return cudaErrorInvalidValue;
}

}  // namespace pathattn
