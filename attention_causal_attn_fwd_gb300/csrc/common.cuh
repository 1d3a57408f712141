// Shared device/host helpers for libpathattn (PaTH causal attention on sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "path_attn.h"

namespace pathattn {

// ----------------------------------------------------------------------------- element conversion
template <typename T> struct Elt;
template <> struct Elt<float> {
    static __device__ __forceinline__ float to_f(float x) { return x; }
    static __device__ __forceinline__ float from_f(float x) { return x; }
};
template <> struct Elt<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};
template <typename T> __device__ __forceinline__ float to_f(T x) { return Elt<T>::to_f(x); }
template <typename T> __device__ __forceinline__ T from_f(float x) { return Elt<T>::from_f(x); }

// 16-byte vector of T: 4 floats or 8 bf16.
template <typename T> struct Vec16 {
    static constexpr int N = 16 / sizeof(T);
    uint4 raw;
    __device__ __forceinline__ float get(int i) const {
        const T* p = reinterpret_cast<const T*>(&raw);
        return to_f<T>(p[i]);
    }
    __device__ __forceinline__ void set(int i, float x) {
        T* p = reinterpret_cast<T*>(&raw);
        p[i] = from_f<T>(x);
    }
};

__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ uint4 ld_global_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
// Streaming load (no L1 allocation): data touched once per step.
__device__ __forceinline__ uint4 ld_global_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ void st_global_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// ----------------------------------------------------------------------------- status word
// The first 256 bytes of every workspace form a header; word 0 is the status.
struct WsHeader {
    int status;
    int fault_site;     // which wait expired (debugging aid)
    unsigned work_next; // tile counter for persistent schedulers
    unsigned visited;   // tensor-core forward: (query tile, key block) pairs visited, diagonal included
    int pad[60];
};
static_assert(sizeof(WsHeader) == 256, "header size");

__device__ __forceinline__ void report_status(WsHeader* h, int code, int site) {
    if (atomicCAS(&h->status, 0, code) == 0) h->fault_site = site;
}

// Index checks of the plain (non-TMA) global loads and stores, compiled in only
// for the bounds-checked build (-DPATH_DEBUG_BOUNDS): an element range
// [first, first + count) outside [0, size) records PATH_ERR_BOUNDS and the site
// in the status word, and the caller skips the access.  The normal build
// checks nothing.
#ifdef PATH_DEBUG_BOUNDS
__device__ __forceinline__ bool in_bounds(long long first, long long count, long long size, WsHeader* h,
                                          int site) {
    if (first >= 0 && count >= 0 && first + count <= size) return true;
    report_status(h, PATH_ERR_BOUNDS, site);
    return false;
}
#else
__device__ __forceinline__ bool in_bounds(long long, long long, long long, WsHeader*, int) { return true; }
#endif

// Optional events recorded around the dominant kernel of each call (set by
// path_debug_set_timing_events; both null when unused).
void timing_events(cudaEvent_t* start, cudaEvent_t* end);
inline void mark_start(cudaStream_t st) {
    cudaEvent_t a, b;
    timing_events(&a, &b);
    if (a && b) cudaEventRecord(a, st);
}
inline void mark_end(cudaStream_t st) {
    cudaEvent_t a, b;
    timing_events(&a, &b);
    if (a && b) cudaEventRecord(b, st);
}

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
__host__ __device__ constexpr int cdiv(int a, int b) { return (a + b - 1) / b; }

// ----------------------------------------------------------------------------- forward workspace
// Per-chunk UT-transform products for a forward call with chunk size C.
// Every per-head array is padded to Lp = ceil(L / C) * C rows so that chunk
// reads never cross into the next head; padded rows hold zeros.
//   qhat : float [BH, Lp, d]  queries transported to their chunk start
//   khat : T     [BH, Lp, d]  keys transported to their chunk end
//   un   : T     [BH, Lp, d]  query-side scan factor per chunk: -U = -A^T W
//                             (fp32 CUDA-core path), or the transition
//                             P - I = -W^T A W, d x d in the chunk's first d
//                             rows (bf16 tensor-core path)
//   y    : T     [BH, Lp, C]  Y = tril(Q W^T) A^T per chunk (diagonal blocks)
//   zn   : T     [BH, Lp, C]  -Z = -triu_1(K W^T) per chunk (diagonal blocks)
//   cum  : float [BH, Lp]     inclusive cumulative sum of log f (PaTH-FoX)
//   vfac : T     [BH, Lp, d]  V = A W per chunk (key-side transport; prefill
//                             cache only, absent from forward workspaces)
//   kmax : float [BH, Lp / C] max over the chunk of |khat_j|^2 (PaTH-FoX
//                             far-block skipping)
struct FwdLayout {
    size_t qhat, khat, un, y, zn, cum, vfac, kmax, total;
    int Lp;
};
inline FwdLayout fwd_layout(int B, int H, int L, int d, int C, size_t elt, bool with_vfac = false) {
    FwdLayout s;
    s.Lp = cdiv(L, C) * C;
    const size_t rows = (size_t)B * H * s.Lp;
    size_t off = sizeof(WsHeader);
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 1024); return o; };
    s.qhat = take(rows * d * sizeof(float));
    s.khat = take(rows * d * elt);
    s.un = take(rows * d * elt);
    s.y = take(rows * C * elt);
    s.zn = take(rows * C * elt);
    s.cum = take(rows * sizeof(float));
    s.vfac = with_vfac ? take(rows * d * elt) : 0;
    s.kmax = take((size_t)B * H * (s.Lp / C) * sizeof(float));
    s.total = off;
    return s;
}

// Workspace of the blockwise value-transport forward (bf16, d = 128, chunks of 128):
// the forward's layout for the key side (lay), a second copy of it for the UT prep
// run with v in the key slot (lay2, same offsets shifted past lay; only its khat,
// each value moved to the end of its chunk, is read), the pair store of carried
// value blocks ([B*H, max(1, N (N - 1) / 2) * 128, d] bf16, N = ceil(L / 128)), the
// scan's output X ([B*H, L, d] bf16), its LSE ([B*H, L] fp32), the diagonal block's P
// ([B*H, L, 128] bf16) and the max it was formed with ([B*H, L] fp32).
struct VtBlockLayout {
    FwdLayout lay, lay2;
    size_t pairs, x, lse, pdiag, m0, total;
    int N;
    long long pair_rows;  // rows of the pair store per head
};
inline VtBlockLayout vt_block_layout(int B, int H, int L, int d) {
    VtBlockLayout v;
    v.lay = fwd_layout(B, H, L, d, 128, 2);
    const size_t shift = v.lay.total - sizeof(WsHeader);
    v.lay2 = v.lay;
    v.lay2.qhat += shift; v.lay2.khat += shift; v.lay2.un += shift; v.lay2.y += shift; v.lay2.zn += shift;
    v.lay2.cum += shift; v.lay2.kmax += shift; v.lay2.vfac = 0; v.lay2.total += shift;
    v.N = cdiv(L, 128);
    const long long npairs = (long long)v.N * (v.N - 1) / 2;
    v.pair_rows = (npairs > 0 ? npairs : 1) * 128;
    const size_t BH = (size_t)B * H;
    size_t off = v.lay2.total;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 1024); return o; };
    v.pairs = take(BH * (size_t)v.pair_rows * d * 2);
    v.x = take(BH * (size_t)L * d * 2);
    v.lse = take(BH * (size_t)L * sizeof(float));
    v.pdiag = take(BH * (size_t)L * 128 * 2);
    v.m0 = take(BH * (size_t)L * sizeof(float));
    v.total = off;
    return v;
}

// Options of the bf16 tensor-core forward that change no result: no_skip
// visits every key block on the PaTH-FoX path (the far-block stop off).
struct FwdOptions {
    int no_skip;
};

// ----------------------------------------------------------------------------- decode workspace
constexpr int kDecodeRowsPerSplit = 2048;
inline int decode_splits(int n_rows) { return cdiv(n_rows > 0 ? n_rows : 1, kDecodeRowsPerSplit); }
struct DecLayout {
    size_t part_m, part_l, part_o, total;
    int splits;
};
inline DecLayout dec_layout(int B, int H, int n_max, int d) {
    DecLayout s;
    s.splits = decode_splits(n_max);
    const size_t n = (size_t)B * H * s.splits;
    size_t off = sizeof(WsHeader);
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    s.part_m = take(n * sizeof(float));
    s.part_l = take(n * sizeof(float));
    s.part_o = take(n * d * sizeof(float));
    s.total = off;
    return s;
}

// ----------------------------------------------------------------------------- backward workspace
// Chunk size of the backward pass (every d).  With N = ceil(L / C) chunks per
// head and Lp = N * C padded rows (padded rows hold zeros):
//   qbar  : float [BH, Lp, d]   queries walked down through their own chunk
//   khat  : float [BH, Lp, d]   keys walked up to their chunk end
//   pm    : float [BH, N, d, d] chunk transition P_m = H_b ... H_e (row-major)
//   pmt   : float [BH, N, d, d] its transpose (pm and pmt feed the CUDA-core
//           chains only: absent for bf16 at d = 128)
//   khat16, phi, plo : bf16 copies for the tensor-core chains (bf16, d = 128
//           only): khat [BH, Lp, d]; P_m split as hi + lo [BH, N, d, d]
//   delta : float [BH, Lp]      dO_i . o_i
//   cum   : float [BH, Lp]      inclusive cumulative sum of log f (PaTH-FoX)
//   dqbar, dkhat, dvoff : float [BH, Lp, d]  gradients w.r.t. qbar and khat,
//                         and the off-diagonal part of dv
//   dpm   : float [BH, N, d, d] gradient w.r.t. P_m
//   dcrow, dccol, dctot : float [BH, Lp]  FoX: gradient w.r.t. the cumulative
//                         sums (row part, column part, total)
//   pairs : T [BH, N(N-1)/2, 2 C d + 2 C C]  per (query chunk n, key chunk
//           m < n): the transported queries U_{n,m}, the chain gradient
//           G_{n,m-1}, the logit gradient dS_{nm} and the probabilities P_{nm},
//           in the input dtype (bf16 pairs feed the tensor-core reduction)
constexpr int kBwdC = 64;
struct BwdLayout {
    size_t qbar, khat, pm, pmt, khat16, phi, plo, xinv, delta, cum, dqbar, dkhat, dvoff, dpm, dcrow, dccol, dctot, pairs,
        total;
    int Lp, N;
    size_t pair_elems;   // elements per (n, m) pair
    size_t head_pairs;   // N (N - 1) / 2
};
inline BwdLayout bwd_layout(int B, int H, int L, int d, size_t elt) {
    BwdLayout s;
    const int C = kBwdC;
    s.N = cdiv(L, C);
    s.Lp = s.N * C;
    const size_t BH = (size_t)B * H, rows = BH * s.Lp;
    s.pair_elems = 2 * (size_t)C * d + 2 * (size_t)C * C;
    s.head_pairs = (size_t)s.N * (s.N - 1) / 2;
    size_t off = sizeof(WsHeader);
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 1024); return o; };
    s.qbar = take(rows * d * sizeof(float));
    s.khat = take(rows * d * sizeof(float));
    const bool tc = elt == 2 && d == 128;
    s.pm = tc ? 0 : take(BH * s.N * d * d * sizeof(float));
    s.pmt = tc ? 0 : take(BH * s.N * d * d * sizeof(float));
    s.khat16 = tc ? take(rows * d * 2) : 0;
    s.phi = tc ? take(BH * s.N * d * d * 2) : 0;
    s.plo = tc ? take(BH * s.N * d * d * 2) : 0;
    s.xinv = take(BH * s.N * C * C * sizeof(float));  // each chunk's (I + D triu_1 W W^T)^-1, prep -> local
    s.delta = take(rows * sizeof(float));
    s.cum = take(rows * sizeof(float));
    s.dqbar = take(rows * d * sizeof(float));
    s.dkhat = take(rows * d * sizeof(float));
    s.dvoff = take(rows * d * sizeof(float));
    s.dpm = take(BH * s.N * d * d * sizeof(float));
    s.dcrow = take(rows * sizeof(float));
    s.dccol = take(rows * sizeof(float));
    s.dctot = take(rows * sizeof(float));
    s.pairs = take(BH * s.head_pairs * s.pair_elems * elt);
    s.total = off;
    return s;
}

}  // namespace pathattn
