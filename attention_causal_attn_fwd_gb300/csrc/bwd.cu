// Backward pass of PaTH / PaTH-FoX causal attention: dq, dk, dv, dw, dbeta and
// dlog f, in fp32 arithmetic on the CUDA cores.
//
// The forward ("Resumo Técnico: Atenção PaTH", §2 "Mecanismo Central" and
// "Extensões: PaTH-FoX") is s_ij = scale k_j^T H_{j+1} ... H_i q_i (+ c_i - c_j,
// c the cumulative sum of log f), H_s = I - beta_s w_s w_s^T,
// o_i = sum_j softmax_j(s_i.) v_j.  §3 trains it by backpropagation; what
// follows is its chain rule, organised in chunks of C = 64 positions like the
// forward's blockwise scan.  Within chunk m (positions b..e):
//
//   P_m    = H_b ... H_e                       (chunk transition, d x d)
//   qbar_i = H_b ... H_i q_i                   (query walked down its own chunk)
//   khat_j = H_e ... H_{j+1} k_j               (key walked up to its chunk end)
//
// and for a key chunk m below a query chunk n the queries reach chunk m as
// U_{n,n-1} = Qbar_n, U_{n,m-1} = U_{n,m} P_m^T, with S_nm = scale U_{n,m}
// Khat_m^T + bias.  With dS = P o (dO V^T - Delta), Delta_i = dO_i . o_i:
//
//   dV_m     += P_nm^T dO_n
//   dKhat_m  += scale dS_nm^T U_{n,m}
//   G_{n,m}   = scale dS_nm Khat_m + G_{n,m-1} P_m        (G_{n,-1} = 0)
//   dP_m     += G_{n,m-1}^T U_{n,m}
//   dQbar_n   = G_{n,n-1}
//
// and the walks that built qbar, khat, P_m and the diagonal block are then
// reversed inside each chunk.  A transition's gradient dH = g u^T becomes
// dbeta = -(w.g)(w.u) and dw = -beta ((w.u) g + (w.g) u).
//
// Kernels, in stream order:
//   bwd_prep   one CTA per chunk        qbar, khat, Delta and, for the inner
//                                       chunks, P_m = I - W^T A W, all in the
//                                       compact form (fp32 P_m, or hi / lo bf16
//                                       for the tensor-core chains); keeps the
//                                       triangular factor for bwd_local
//   bwd_chain  one CTA per query chunk  U chain down, G chain up; stores U,
//                                       G, dS and P per (n, m) pair; dQbar;
//                                       for bf16 at d = 128 bwd_chain_tc
//                                       (csrc/bwd_tc.cu) runs the chains on
//                                       the tensor cores
//   bwd_reduce one CTA per key chunk    dV_m, dKhat_m, dP_m summed over the
//                                       query chunks (each output owned by
//                                       one CTA, so no global atomics); for
//                                       bf16 at d = 128 bwd_reduce_tc
//                                       (csrc/bwd_tc.cu) does this on the
//                                       tensor cores from the bf16 pair store
//   bwd_local  one CTA per chunk        diagonal block and the within-chunk
//                                       walks in reverse, in the compact form
//                                       (products, with the triangular
//                                       factor that bwd_prep formed); writes
//                                       dq, dk, dv, dw, dbeta
//   bwd_fox_suffix one CTA per head     dlog f_s = sum_{t >= s} dc_t
// The contractions here are register-tiled fp32 GEMMs on shared-memory operands, except
// in bwd_prep and bwd_local for bf16 at d >= 64, where they run as warp-level mma.sync
// (bf16 operands, fp32 accumulation; fp32 operands other than the bf16 inputs enter as
// hi + lo parts).  Nothing here waits on another CTA, so these kernels have no spin
// waits (the tensor-core kernels of csrc/bwd_tc.cu bound every wait).
#include "common.cuh"
#include "ut_prep.cuh"

namespace pathattn {

cudaError_t launch_bwd_chain_tc(const void* dO, const void* v, const void* khat16, const void* phi, const void* plo,
                                void* pairs, const float* qbar, const float* lse, const float* delta,
                                const float* cum, float* dqbar, float* dcrow, float* dccol, int fox, int BH, int L,
                                int Lp, int N, size_t head_pairs, float scale, WsHeader* hdr, cudaStream_t st);
cudaError_t launch_bwd_reduce_tc(const void* dO, const void* pairs, float* dvoff, float* dkhat, float* dpm, int BH,
                                 int L, int Lp, int N, size_t head_pairs, float scale, WsHeader* hdr,
                                 cudaStream_t st);

namespace {

constexpr int kC = kBwdC;
constexpr int kNT = 256;
constexpr int kNTL = 256;  // bwd_local

struct BwdParams {
    const void *q, *k, *v, *w, *o, *dO;
    const float *beta, *lse;
    void *dq, *dk, *dv, *dw;
    float *dbeta, *dlog_f;
    float *qbar, *khat, *pm, *pmt, *xinv, *delta, *cum, *dqbar, *dkhat, *dvoff, *dpm, *dcrow, *dccol, *dctot;
    __nv_bfloat16 *khat16, *phi, *plo;  // tensor-core chains only (else null)
    void* pairs;  // pair store, elements of the input dtype
    int L, Lp, N;
    size_t pair_elems, head_pairs;
    float scale;
    int fox;
};

// Rows [0, rows) of a row-major global array of COLS columns (leading dim lds, rows starting
// on 16-byte boundaries) into shared memory (leading dim ldd) as fp32; rows >= valid read as
// zero.  16-byte loads, several in flight per thread; plain (coherent) loads, since a CTA
// reads back pair data it wrote itself.
template <typename G, int COLS, int NT = kNT>
__device__ __forceinline__ void to_smem_v(float* dst, int ldd, const G* src, int lds, int rows, int valid) {
    constexpr int V = 16 / sizeof(G);
    constexpr int VPR = COLS / V;
    static_assert(COLS % V == 0, "rows must be whole 16-byte vectors");
    const int nvec = rows * VPR;
#pragma unroll 4
    for (int idx = threadIdx.x; idx < nvec; idx += NT) {
        const int r = idx / VPR, cv = idx % VPR;
        Vec16<G> x;
        x.raw = r < valid ? ld_global_v4(src + (size_t)r * lds + cv * V) : make_uint4(0u, 0u, 0u, 0u);
        float* d = dst + r * ldd + cv * V;
#pragma unroll
        for (int j = 0; j < V; ++j) d[j] = x.get(j);
    }
}

// Transposing load: dst[c * ldd + r] = src[r * lds + c] for r < rows (zero for r >= valid),
// c < COLS.  Consecutive threads take consecutive rows of one 16-byte column group, so the
// shared-memory writes of a warp fall in distinct banks.
template <typename G, int COLS, int NT = kNT>
__device__ __forceinline__ void to_smem_t(float* dst, int ldd, const G* src, int lds, int rows, int valid) {
    constexpr int V = 16 / sizeof(G);
    static_assert(COLS % V == 0, "rows must be whole 16-byte vectors");
    const int nvec = rows * (COLS / V);
#pragma unroll 4
    for (int idx = threadIdx.x; idx < nvec; idx += NT) {
        const int r = idx % rows, cv = idx / rows;
        Vec16<G> x;
        x.raw = r < valid ? ld_global_v4(src + (size_t)r * lds + cv * V) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int j = 0; j < V; ++j) dst[(cv * V + j) * ldd + r] = x.get(j);
    }
}
// Transposing store to global memory: dst[r * ldd + c] = src[c * lds + r], r < R, c < COLS
// (R a multiple of 4, lds a multiple of 4 floats).
template <int R, int COLS, typename G>
__device__ __forceinline__ void from_smem_t(G* dst, int ldd, const float* src, int lds) {
    for (int idx = threadIdx.x; idx < R * COLS / 4; idx += kNT) {
        const int c = idx % COLS, r4 = (idx / COLS) * 4;
        const float4 x = *reinterpret_cast<const float4*>(src + c * lds + r4);
        dst[(size_t)r4 * ldd + c] = from_f<G>(x.x);
        dst[(size_t)(r4 + 1) * ldd + c] = from_f<G>(x.y);
        dst[(size_t)(r4 + 2) * ldd + c] = from_f<G>(x.z);
        dst[(size_t)(r4 + 3) * ldd + c] = from_f<G>(x.w);
    }
}

// ------------------------------------------------------------------ register-tiled GEMM on K-major operands
// Thread t owns the contiguous TM x TN output tile at rows m0 = (t / GN) TM, columns
// n0 = (t % GN) TN.  A is read as A[k][m] and B as B[k][n] (K-major in shared memory, leading
// dims and tile offsets multiples of 4 floats), so each k step fetches whole 16-byte vectors:
// one 128-bit shared load per four values.
template <int M, int N> struct VT {
    static constexpr int TOT = M * N / kNT;
    static constexpr int TN = TOT >= 32 ? 8 : (TOT >= 4 ? 4 : 1);
    static constexpr int TM = TOT / TN;
    static constexpr int GN = N / TN, GM = M / TM;
    static_assert(TOT >= 1 && GM * GN == kNT && GM * TM == M && GN * TN == N, "gemm tiling");
    static __device__ __forceinline__ int m0() { return (int)(threadIdx.x / GN) * TM; }
    static __device__ __forceinline__ int n0() { return (int)(threadIdx.x % GN) * TN; }
    using Acc = float[TM][TN];
    static __device__ __forceinline__ void zero(Acc& a) {
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) a[i][j] = 0.f;
    }
};
template <int W>
__device__ __forceinline__ void lds_vec(float (&v)[W], const float* ptr) {
    if constexpr (W % 4 == 0) {
#pragma unroll
        for (int i = 0; i < W; i += 4) {
            const float4 x = *reinterpret_cast<const float4*>(ptr + i);
            v[i] = x.x; v[i + 1] = x.y; v[i + 2] = x.z; v[i + 3] = x.w;
        }
    } else if constexpr (W == 2) {
        const float2 x = *reinterpret_cast<const float2*>(ptr);
        v[0] = x.x; v[1] = x.y;
    } else {
#pragma unroll
        for (int i = 0; i < W; ++i) v[i] = ptr[i];
    }
}
template <int W>
__device__ __forceinline__ void sts_vec(float* ptr, const float (&v)[W]) {
    if constexpr (W % 4 == 0) {
#pragma unroll
        for (int i = 0; i < W; i += 4) *reinterpret_cast<float4*>(ptr + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else if constexpr (W == 2) {
        *reinterpret_cast<float2*>(ptr) = make_float2(v[0], v[1]);
    } else {
#pragma unroll
        for (int i = 0; i < W; ++i) ptr[i] = v[i];
    }
}
// acc += A^T-major product: acc[i][j] += sum_k A[k][m0 + i] B[k][n0 + j]
template <int M, int N, int K>
__device__ __forceinline__ void vgemm(typename VT<M, N>::Acc& acc, const float* A, int lda, const float* B, int ldb) {
    using G = VT<M, N>;
    const float* a = A + G::m0();
    const float* b = B + G::n0();
#pragma unroll 2
    for (int k = 0; k < K; ++k) {
        float av[G::TM], bv[G::TN];
        lds_vec<G::TM>(av, a + k * lda);
        lds_vec<G::TN>(bv, b + k * ldb);
#pragma unroll
        for (int i = 0; i < G::TM; ++i)
#pragma unroll
            for (int j = 0; j < G::TN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
}
// two products of the same shape and depth in one pass
template <int M, int N, int K>
__device__ __forceinline__ void vgemm2(typename VT<M, N>::Acc& c1, const float* A1, int lda1, const float* B1,
                                       int ldb1, typename VT<M, N>::Acc& c2, const float* A2, int lda2,
                                       const float* B2, int ldb2) {
    using G = VT<M, N>;
    const float *a1 = A1 + G::m0(), *b1 = B1 + G::n0(), *a2 = A2 + G::m0(), *b2 = B2 + G::n0();
#pragma unroll 2
    for (int k = 0; k < K; ++k) {
        float av[G::TM], bv[G::TN], aw[G::TM], bw[G::TN];
        lds_vec<G::TM>(av, a1 + k * lda1);
        lds_vec<G::TN>(bv, b1 + k * ldb1);
        lds_vec<G::TM>(aw, a2 + k * lda2);
        lds_vec<G::TN>(bw, b2 + k * ldb2);
#pragma unroll
        for (int i = 0; i < G::TM; ++i)
#pragma unroll
            for (int j = 0; j < G::TN; ++j) {
                c1[i][j] = fmaf(av[i], bv[j], c1[i][j]);
                c2[i][j] = fmaf(aw[i], bw[j], c2[i][j]);
            }
    }
}
// write f * acc to a row-major global array (leading dim ld) at the thread's tile
template <int M, int N, typename E = float>
__device__ __forceinline__ void store_tile(E* dst, int ld, const typename VT<M, N>::Acc& acc, float f) {
    using G = VT<M, N>;
#pragma unroll
    for (int i = 0; i < G::TM; ++i) {
        float v[G::TN];
#pragma unroll
        for (int j = 0; j < G::TN; ++j) v[j] = f * acc[i][j];
        E* d = dst + (size_t)(G::m0() + i) * ld + G::n0();
        if constexpr (sizeof(E) == 4) {
            sts_vec<G::TN>(reinterpret_cast<float*>(d), v);
        } else {
#pragma unroll
            for (int j = 0; j < G::TN; ++j) d[j] = from_f<E>(v[j]);
        }
    }
}
// write acc transposed into shared memory: dst[(n0 + j) * ld + m0 + i] = acc[i][j]
template <int M, int N>
__device__ __forceinline__ void store_tile_t(float* dst, int ld, const typename VT<M, N>::Acc& acc) {
    using G = VT<M, N>;
#pragma unroll
    for (int j = 0; j < G::TN; ++j) {
        float v[G::TM];
#pragma unroll
        for (int i = 0; i < G::TM; ++i) v[i] = acc[i][j];
        sts_vec<G::TM>(dst + (G::n0() + j) * ld + G::m0(), v);
    }
}

// ------------------------------------------------------------------ shared-memory sizes (floats)
template <int D> struct BwdSmem {
    static constexpr int LC = kC + 4, LD = D + 4;  // K-major GEMM operands (16-byte rows)
    static constexpr int RK = (D * LC > kC * LD ? D * LC : kC * LD);
    static constexpr int RV = (D * LC > kC * LC ? D * LC : kC * LC);
    static constexpr int chain = 2 * D * LC + RK + RV + D * LD + 6 * kC;
    static constexpr int reduce = 3 * kC * LD + 2 * kC * LC;
    static constexpr int slot = kC * LC;              // bwd_local: one C x (C + 4) tile
    static constexpr int local = 13 * slot + 6 * kC;  // thirteen slots, six per-position vectors
    static constexpr int prep = 11 * slot + kC;       // bwd_prep: eleven slots and beta
    static_assert(chain * 4 <= 227 * 1024 && local * 4 <= 227 * 1024 && reduce * 4 <= 227 * 1024,
                  "shared memory per CTA");
};

// ------------------------------------------------------------------ bwd_chain
// Pair store layout (floats, per (n, m)): U [C][d], G [C][d], dS [C][C], P [C][C].
template <typename T, int D>
__global__ void __launch_bounds__(kNT) bwd_chain(BwdParams p) {
    using SM = BwdSmem<D>;
    constexpr int C = kC, LC = SM::LC, LD = SM::LD;
    extern __shared__ __align__(16) float smem[];
    float* sUT = smem;             // [D][LC] U^T: the queries reaching key chunk m
    float* sOT = sUT + D * LC;     // [D][LC] dO_n^T; G^T up the chain
    float* sKT = sOT + D * LC;     // [D][LC] khat_m^T (down); khat_m [C][LD] (up)
    float* sVT = sKT + SM::RK;     // [D][LC] v_m^T (down); dS_nm^T [C][LC] (up)
    float* sP = sVT + SM::RV;      // [D][LD] P_m^T (down); P_m (up)
    float* sL = sP + D * LD;       // [C] lse_i
    float* sD = sL + C;            // [C] Delta_i
    float* sCi = sD + C;           // [C] c_i
    float* sCj = sCi + C;          // [C] c_j
    float* sRs = sCj + C;          // [C] FoX row sums of dS
    float* sCs = sRs + C;          // [C] FoX column sums of dS_nm (added to the key chunk's dccol)
    const int n = p.N - 1 - blockIdx.x, bh = blockIdx.y;  // longest chains first
    const int b = n * C, c = min(C, p.L - b);
    const size_t hbase = (size_t)bh * p.L, pbase = (size_t)bh * p.Lp;
    const T* dO = static_cast<const T*>(p.dO);
    const T* v = static_cast<const T*>(p.v);
    const float scale = p.scale;
    to_smem_t<float, D>(sUT, LC, p.qbar + (pbase + b) * D, D, C, C);
    to_smem_t<T, D>(sOT, LC, dO + (hbase + b) * D, D, C, c);
    for (int r = threadIdx.x; r < C; r += kNT) {
        sL[r] = r < c ? p.lse[hbase + b + r] : 0.f;
        sD[r] = p.delta[pbase + b + r];
        sCi[r] = p.fox ? p.cum[pbase + b + r] : 0.f;
        sRs[r] = 0.f;
        sCs[r] = 0.f;
    }
    T* pairs_n = static_cast<T*>(p.pairs) + ((size_t)bh * p.head_pairs + (size_t)n * (n - 1) / 2) * p.pair_elems;
    using GS = VT<C, C>;
    using GU = VT<C, D>;
    for (int m = n - 1; m >= 0; --m) {
        const int bm = m * C;
        T* pr = pairs_n + (size_t)m * p.pair_elems;  // U [C][D], G [C][D], dS [C][C], P [C][C]
        __syncthreads();
        if (p.fox && m < n - 1)  // the previous key chunk's column sums of dS
            for (int j = threadIdx.x; j < C; j += kNT) {
                atomicAdd(p.dccol + pbase + bm + C + j, sCs[j]);
                sCs[j] = 0.f;
            }
        to_smem_t<float, D>(sKT, LC, p.khat + (pbase + bm) * D, D, C, C);
        to_smem_t<T, D>(sVT, LC, v + (hbase + bm) * D, D, C, C);  // key chunks below n are full
        if (m >= 1) to_smem_v<float, D>(sP, LD, p.pmt + ((size_t)bh * p.N + m) * D * D, D, D, D);
        for (int r = threadIdx.x; r < C; r += kNT) sCj[r] = p.fox ? p.cum[pbase + bm + r] : 0.f;
        __syncthreads();
        // S = U khat^T and dO v^T in one pass; probabilities and dS straight from registers
        typename GS::Acc aS, aP;
        GS::zero(aS);
        GS::zero(aP);
        vgemm2<C, C, D>(aS, sUT, LC, sKT, LC, aP, sOT, LC, sVT, LC);
        const int r0 = GS::m0(), j0 = GS::n0();
#pragma unroll
        for (int i = 0; i < GS::TM; ++i) {
            const int r = r0 + i;
            float rs = 0.f;
#pragma unroll
            for (int j = 0; j < GS::TN; ++j) {
                float pij = 0.f, ds = 0.f;
                if (r < c) {
                    pij = __expf(scale * aS[i][j] + sCi[r] - sCj[j0 + j] - sL[r]);
                    ds = pij * (aP[i][j] - sD[r]);
                }
                aS[i][j] = pij;
                aP[i][j] = ds;
                rs += ds;
            }
            if (p.fox) {  // the GN threads of a row are consecutive lanes of one warp
#pragma unroll
                for (int o = 1; o < GS::GN; o <<= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o);
                if (threadIdx.x % GS::GN == 0) sRs[r] += rs;
            }
        }
        if (p.fox)
#pragma unroll
            for (int j = 0; j < GS::TN; ++j) {
                float cs = 0.f;
#pragma unroll
                for (int i = 0; i < GS::TM; ++i) cs += aP[i][j];
                atomicAdd(sCs + j0 + j, cs);
            }
        store_tile<C, C, T>(pr + 2 * C * D, C, aP, 1.f);
        store_tile<C, C, T>(pr + 2 * C * D + C * C, C, aS, 1.f);
        from_smem_t<C, D>(pr, D, sUT, LC);  // U_{n,m}
        if (m >= 1) {  // U <- U P_m^T
            typename GU::Acc aU;
            GU::zero(aU);
            vgemm<C, D, D>(aU, sUT, LC, sP, LD);
            __syncthreads();
            store_tile_t<C, D>(sUT, LC, aU);
        }
    }
    __syncthreads();
    if (p.fox)  // key chunk 0's column sums
        for (int j = threadIdx.x; j < C; j += kNT) atomicAdd(p.dccol + pbase + j, sCs[j]);
    float* sGT = sOT;
    float* sK = sKT;
    float* sST = sVT;
    for (int m = 0; m < n; ++m) {
        const int bm = m * C;
        T* pr = pairs_n + (size_t)m * p.pair_elems;
        __syncthreads();
        to_smem_v<float, D>(sK, LD, p.khat + (pbase + bm) * D, D, C, C);
        to_smem_t<T, C>(sST, LC, pr + 2 * C * D, C, C, C);
        if (m >= 1) {
            to_smem_v<float, D>(sP, LD, p.pm + ((size_t)bh * p.N + m) * D * D, D, D, D);
            from_smem_t<C, D>(pr + C * D, D, sGT, LC);  // G_{n,m-1}
        }
        __syncthreads();
        typename GU::Acc aT, aG;
        GU::zero(aT);
        GU::zero(aG);
        vgemm<C, D, C>(aT, sST, LC, sK, LD);             // dS khat
        if (m >= 1) vgemm<C, D, D>(aG, sGT, LC, sP, LD);  // G P_m
#pragma unroll
        for (int i = 0; i < GU::TM; ++i)
#pragma unroll
            for (int j = 0; j < GU::TN; ++j) aG[i][j] = fmaf(scale, aT[i][j], aG[i][j]);
        __syncthreads();
        store_tile_t<C, D>(sGT, LC, aG);
    }
    __syncthreads();
    from_smem_t<C, D>(p.dqbar + (pbase + b) * D, D, sGT, LC);
    if (p.fox)
        for (int r = threadIdx.x; r < C; r += kNT) p.dcrow[pbase + b + r] = sRs[r];
}

// ------------------------------------------------------------------ bwd_reduce
template <typename T, int D>
__global__ void __launch_bounds__(kNT) bwd_reduce(BwdParams p) {
    using SM = BwdSmem<D>;
    constexpr int C = kC, LC = SM::LC, LD = SM::LD;
    extern __shared__ __align__(16) float smem[];
    float* sU = smem;           // [C][LD] U_{n,m}
    float* sG = sU + C * LD;    // [C][LD] G_{n,m-1}
    float* sO = sG + C * LD;    // [C][LD] dO_n
    float* sS = sO + C * LD;    // [C][LC] dS_nm
    float* sA = sS + C * LC;    // [C][LC] softmax probabilities P_nm
    const int m = blockIdx.x, bh = blockIdx.y, bm = m * C;  // m = 0 has the most query chunks
    const size_t hbase = (size_t)bh * p.L, pbase = (size_t)bh * p.Lp;
    const T* dO = static_cast<const T*>(p.dO);
    using GV = VT<C, D>;
    using GP = VT<D, D>;
    typename GV::Acc accV, accK;
    typename GP::Acc accP;
    GV::zero(accV);
    GV::zero(accK);
    GP::zero(accP);
    for (int n = m + 1; n < p.N; ++n) {
        const int b = n * C, c = min(C, p.L - b);
        const T* pr = static_cast<const T*>(p.pairs) + ((size_t)bh * p.head_pairs + (size_t)n * (n - 1) / 2 + m) * p.pair_elems;
        __syncthreads();
        to_smem_v<T, D>(sU, LD, pr, D, C, C);
        if (m >= 1) to_smem_v<T, D>(sG, LD, pr + C * D, D, C, C);
        to_smem_v<T, D>(sO, LD, dO + (hbase + b) * D, D, C, c);
        to_smem_v<T, C>(sS, LC, pr + 2 * C * D, C, C, C);
        to_smem_v<T, C>(sA, LC, pr + 2 * C * D + C * C, C, C, C);
        __syncthreads();
        vgemm<C, D, C>(accV, sA, LC, sO, LD);             // dV_m  += P^T dO_n
        vgemm<C, D, C>(accK, sS, LC, sU, LD);             // dKhat += dS^T U   (scaled at the end)
        if (m >= 1) vgemm<D, D, C>(accP, sG, LD, sU, LD);  // dP_m  += G^T U
    }
    store_tile<C, D>(p.dvoff + (pbase + bm) * D, D, accV, 1.f);
    store_tile<C, D>(p.dkhat + (pbase + bm) * D, D, accK, p.scale);
    if (m >= 1) store_tile<D, D>(p.dpm + ((size_t)bh * p.N + m) * D * D, D, accP, 1.f);
}

// ------------------------------------------------------------------ bwd_local
// The diagonal block and the within-chunk walks, reversed in the compact ("UT") form of
// "Representação de Transformação UT" (§3) instead of position by position.  For chunk n with
// rows W, Q, K of w, q, k (C rows, padded rows zero, beta = 0 there):
//
//   G = W W^T,  X = (I + D triu_1 G)^{-1} (unit upper triangular),  A = X D,  D = diag(beta)
//   H_{a} ... H_{b} = I - W_{a:b}^T A_{a:b} W_{a:b} for a <= b (a principal block of A), so
//   Qm = tril(Q W^T) (b <= i), Km = striu(K W^T) (a > j),  Y = Qm A^T,  Z = Km A,
//   qbar = Q - Y W,  khat = K - Z W,  P_n = I - W^T A W,
//   S = scale (Q K^T - Y Km^T) + c_i - c_j on j <= i        (the diagonal logits)
//
// Given dQbar (from the chains), dKhat and dP_n (from the per-key-chunk sums) and
// dS = P o (dO V^T - Delta) on the diagonal block, the reverse mode of these products is
//
//   dV  = P^T dO,  dZ = -dKhat W^T,  dY = -dQbar W^T - dSs Km       (dSs = scale dS)
//   dKw = striu(-dSs^T Y + dZ A^T),  dQw = tril(dY A)
//   dA  = Km^T dZ + dY^T Qm - W dP W^T,  dbeta_b += sum_a X_ab dA_ab
//   dM  = -X^T (dA D) X^T,  dG = striu(D dM),  dbeta_a += sum_{b>a} dM_ab G_ab
//   dW  = -Y^T dQbar - Z^T dKhat - A (W dP^T) - A^T (W dP) + dQw^T Q + dKw^T K + (dG + dG^T) W
//   dQ  = dQbar + dSs K + dQw W,   dK = dKhat + dSs^T Q + dKw W
//
// every step a product on shared-memory operands (register-tiled fp32, or mma.sync for bf16 at
// d >= 64); X is formed once, by bwd_prep (its only sequential part, the triangular inverse), and
// read from the workspace here.  Thirteen shared-memory slots of one C x (C + 4) tile each
// hold the operands; a d x C or C x d tile takes two adjacent slots at d = 128 and the d x d
// gradient dP four.  The slot of every matrix and the phase that frees it are listed beside
// the code.

// Thread tiling of an M x N output over the kNTL threads of bwd_local: TM consecutive rows by TN
// consecutive columns per thread.  MM numbers the tiles down the rows first (a warp spans many
// rows and one or two column groups), otherwise across the columns first.
template <int M, int N, bool MM> struct TT {
    static constexpr int TOT = M * N / kNTL;
    static constexpr int TN = TOT >= 32 ? 8 : (TOT >= 4 ? 4 : 1);
    static constexpr int TM = TOT / TN;
    static constexpr int GN = N / TN, GM = M / TM;
    static_assert(TOT >= 1 && GM * GN == kNTL && GM * TM == M && GN * TN == N, "tiling");
    static __device__ __forceinline__ int m0() { return (MM ? (int)threadIdx.x % GM : (int)threadIdx.x / GN) * TM; }
    static __device__ __forceinline__ int n0() { return (MM ? (int)threadIdx.x / GM : (int)threadIdx.x % GN) * TN; }
    using Acc = float[TM][TN];
    static __device__ __forceinline__ void zero(Acc& a) {
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) a[i][j] = 0.f;
    }
};

// acc[i][j] += (or -=) sum_k a(m0 + i, k) b(k, n0 + j).  A is K-major (a(m, k) = A[k lda + m])
// when AK, else row-major (A[m lda + k]); B is K-major (b(k, n) = B[k ldb + n]) when BK, else
// B[n ldb + k].  Four k per step, every shared-memory load 16 bytes wide (or the tile's width).
// A row-major A is read conflict-free with the column-first tiling, a row-major B with the
// row-first one (leading dims of C + 4 floats).  KR states a triangular A (m and k both chunk
// positions): KR = 1 when a(m, k) = 0 for k < m, KR = 2 when a(m, k) = 0 for k > m; the
// thread then runs only the k that can meet its rows (with the column-first tiling a warp holds
// two row groups, so its threads stop together).
template <int M, int N, int K, bool MM, bool AK, bool BK, bool NEG = false, int KR = 0>
__device__ __forceinline__ void mmul(typename TT<M, N, MM>::Acc& acc, const float* A, int lda, const float* B,
                                     int ldb) {
    using G = TT<M, N, MM>;
    constexpr int TM = G::TM, TN = G::TN;
    static_assert(K % 4 == 0, "depth");
    static_assert(KR == 0 || M == K, "a triangular A is square");
    const int m0 = G::m0(), n0 = G::n0();
    const int kb = KR == 1 ? (m0 & ~3) : 0;
    const int ke = KR == 2 ? min(K, (m0 + TM + 3) & ~3) : K;
#pragma unroll 2
    for (int k = kb; k < ke; k += 4) {
        float a[4][TM], b[4][TN];
        if constexpr (AK) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) lds_vec<TM>(a[kk], A + (k + kk) * lda + m0);
        } else {
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const float4 x = *reinterpret_cast<const float4*>(A + (m0 + i) * lda + k);
                a[0][i] = x.x; a[1][i] = x.y; a[2][i] = x.z; a[3][i] = x.w;
            }
        }
        if constexpr (BK) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) lds_vec<TN>(b[kk], B + (k + kk) * ldb + n0);
        } else {
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const float4 x = *reinterpret_cast<const float4*>(B + (n0 + j) * ldb + k);
                b[0][j] = x.x; b[1][j] = x.y; b[2][j] = x.z; b[3][j] = x.w;
            }
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const float av = NEG ? -a[kk][i] : a[kk][i];
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(av, b[kk][j], acc[i][j]);
            }
    }
}

// dst[r ld + col] = f(r, col, acc) over the thread's tile, or dst[col ld + r] when TR
template <int M, int N, bool MM, bool TR, typename F>
__device__ __forceinline__ void mstore(float* dst, int ld, const typename TT<M, N, MM>::Acc& acc, F f) {
    using G = TT<M, N, MM>;
    const int m0 = G::m0(), n0 = G::n0();
    if constexpr (!TR) {
#pragma unroll
        for (int i = 0; i < G::TM; ++i) {
            float v[G::TN];
#pragma unroll
            for (int j = 0; j < G::TN; ++j) v[j] = f(m0 + i, n0 + j, acc[i][j]);
            sts_vec<G::TN>(dst + (m0 + i) * ld + n0, v);
        }
    } else {
#pragma unroll
        for (int j = 0; j < G::TN; ++j) {
            float v[G::TM];
#pragma unroll
            for (int i = 0; i < G::TM; ++i) v[i] = f(m0 + i, n0 + j, acc[i][j]);
            sts_vec<G::TM>(dst + (n0 + j) * ld + m0, v);
        }
    }
}

// A ROWS x COLS block of a row-major global array (leading dim lds; rows >= valid read as zero),
// held in registers between its load and its store to shared memory, so that the load can be
// issued ahead of the phase that frees the destination: load + store_t give the transposed
// layout of to_smem_t, load_r + store_r the row-major one of to_smem_v.
template <typename G, int COLS, int ROWS>
struct TileRegs {
    static constexpr int V = 16 / sizeof(G), NV = ROWS * (COLS / V) / kNTL;
    static_assert(COLS % V == 0 && NV * kNTL == ROWS * (COLS / V), "whole 16-byte vectors per thread");
    uint4 x[NV];
    __device__ __forceinline__ void load(const G* src, int lds, int valid) {
#pragma unroll
        for (int e = 0; e < NV; ++e) {
            const int idx = threadIdx.x + e * kNTL, r = idx % ROWS, cv = idx / ROWS;
            x[e] = r < valid ? ld_global_v4(src + (size_t)r * lds + cv * V) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    // row-major store dst[r ldd + c] of a tile loaded with load_r
    __device__ __forceinline__ void load_r(const G* src, int lds, int valid) {
#pragma unroll
        for (int e = 0; e < NV; ++e) {
            const int idx = threadIdx.x + e * kNTL, r = idx / (COLS / V), cv = idx % (COLS / V);
            x[e] = r < valid ? ld_global_v4(src + (size_t)r * lds + cv * V) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    __device__ __forceinline__ void store_r(float* dst, int ldd) const {
#pragma unroll
        for (int e = 0; e < NV; ++e) {
            const int idx = threadIdx.x + e * kNTL, r = idx / (COLS / V), cv = idx % (COLS / V);
            Vec16<G> v;
            v.raw = x[e];
            float* d = dst + r * ldd + cv * V;
#pragma unroll
            for (int j = 0; j < V; ++j) d[j] = v.get(j);
        }
    }
    __device__ __forceinline__ void store_t(float* dst, int ldd) const {
#pragma unroll
        for (int e = 0; e < NV; ++e) {
            const int idx = threadIdx.x + e * kNTL, r = idx % ROWS, cv = idx / ROWS;
            Vec16<G> v;
            v.raw = x[e];
#pragma unroll
            for (int j = 0; j < V; ++j) dst[(cv * V + j) * ldd + r] = v.get(j);
        }
    }
};

// W consecutive values of a global row as fp32 (16- or 8-byte loads; W a multiple of 4)
template <int W, typename S>
__device__ __forceinline__ void ld_row(float (&v)[W], const S* src) {
    static_assert(W % 4 == 0, "row segment");
    if constexpr (sizeof(S) == 4) {
#pragma unroll
        for (int j = 0; j < W; j += 4) {
            const float4 x = *reinterpret_cast<const float4*>(src + j);
            v[j] = x.x; v[j + 1] = x.y; v[j + 2] = x.z; v[j + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < W; j += 4) {
            const uint2 x = *reinterpret_cast<const uint2*>(src + j);
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.x));
            const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.y));
            v[j] = a.x; v[j + 1] = a.y; v[j + 2] = b.x; v[j + 3] = b.y;
        }
    }
}
// W consecutive values to a global row (W a multiple of 4): fp32 as 16-byte stores, bf16 packed
// into 16-byte (W = 8) or 8-byte stores
template <int W, typename E>
__device__ __forceinline__ void st_row(E* dst, const float (&v)[W]) {
    static_assert(W % 4 == 0, "row segment");
    if constexpr (sizeof(E) == 4) {
#pragma unroll
        for (int j = 0; j < W; j += 4)
            *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
    } else {
        uint32_t u[W / 2];
#pragma unroll
        for (int j = 0; j < W / 2; ++j) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
            u[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        if constexpr (W % 8 == 0) {
#pragma unroll
            for (int j = 0; j < W / 2; j += 4)
                *reinterpret_cast<uint4*>(dst + 2 * j) = make_uint4(u[j], u[j + 1], u[j + 2], u[j + 3]);
        } else {
#pragma unroll
            for (int j = 0; j < W / 2; j += 2) *reinterpret_cast<uint2*>(dst + 2 * j) = make_uint2(u[j], u[j + 1]);
        }
    }
}

// rows r < c of a C x D result to global memory: dst[r][e] = acc + (add ? add[r][e] : 0); the
// addends are all loaded before the first store, and each thread's row segment is stored whole
template <int D, typename E>
__device__ __forceinline__ void mstore_out(E* dst, const typename TT<kC, D, false>::Acc& acc, const float* add,
                                           int c) {
    using G = TT<kC, D, false>;
    constexpr int TN = G::TN;
    const int m0 = G::m0(), n0 = G::n0();
    if constexpr (TN % 4 != 0) {
#pragma unroll
        for (int i = 0; i < G::TM; ++i)
            if (m0 + i < c)
#pragma unroll
                for (int j = 0; j < TN; ++j) {
                    const size_t o = (size_t)(m0 + i) * D + n0 + j;
                    dst[o] = from_f<E>(acc[i][j] + (add ? add[o] : 0.f));
                }
        return;
    } else {
        float v[G::TM][TN];
#pragma unroll
        for (int i = 0; i < G::TM; ++i) {
            const bool ok = add && m0 + i < c;
#pragma unroll
            for (int j = 0; j < TN; j += 4) {
                const float4 x = ok ? *reinterpret_cast<const float4*>(add + (size_t)(m0 + i) * D + n0 + j)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                v[i][j] = acc[i][j] + x.x;
                v[i][j + 1] = acc[i][j + 1] + x.y;
                v[i][j + 2] = acc[i][j + 2] + x.z;
                v[i][j + 3] = acc[i][j + 3] + x.w;
            }
        }
#pragma unroll
        for (int i = 0; i < G::TM; ++i)
            if (m0 + i < c) st_row<TN>(dst + (size_t)(m0 + i) * D + n0, v[i]);
    }
}

// ------------------------------------------------------------------ warp-level bf16 tensor-core products
// mma.sync m16n8k16 (bf16 operands, fp32 accumulation) on fp32 shared-memory operands, for the
// bf16 path.  An operand that holds bf16 values exactly (w, q, k, v, dO) enters as it is; any
// other is split into hi = bf16(x) and lo = bf16(x - hi) and the product takes hi B + lo B (or
// A hi + A lo): what it drops is below 2^-16 of each term.
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ uint32_t pack_bf16(float x0, float x1) {  // x0 in the low half
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 f = __bfloat1622float2(h);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = pack_bf16(x0 - f.x, x1 - f.y);
}

// Warp tiling of an M x N output over the eight warps of a 256-thread CTA: a 2 x 4 grid of warps,
// each owning MT x NT tiles of 16 x 8 in the mma.sync accumulator layout (lane l holds rows
// l / 4 and l / 4 + 8, columns 2 (l % 4) and 2 (l % 4) + 1 of every tile).
template <int M, int N> struct WT {
    static constexpr int WM = 2, WN = 4;
    static constexpr int MT = M / (WM * 16), NT = N / (WN * 8);
    static_assert(MT >= 1 && NT >= 1 && MT * WM * 16 == M && NT * WN * 8 == N, "warp tiling");
    using Acc = float[MT][NT][4];
    static __device__ __forceinline__ int mb() { return (int)(threadIdx.x >> 5) / WN * (M / WM); }
    static __device__ __forceinline__ int nb() { return (int)(threadIdx.x >> 5) % WN * (N / WN); }
    static __device__ __forceinline__ int row(int mt, int i) {
        return mb() + mt * 16 + (int)((threadIdx.x & 31) >> 2) + 8 * (i >> 1);
    }
    static __device__ __forceinline__ int col(int nt, int i) { return nb() + nt * 8 + 2 * (int)(threadIdx.x & 3) + (i & 1); }
    static __device__ __forceinline__ void zero(Acc& a) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) a[mt][nt][i] = 0.f;
    }
};

// acc += sum_k a(m, k) b(k, n) over the warp's tiles, operands fp32 in shared memory with the
// layouts of mmul (AK: a(m, k) = A[k lda + m], else A[m lda + k]; BK: b(k, n) = B[k ldb + n],
// else B[n ldb + k]).  ASPL / BSPL split that operand into hi + lo (both: three products, the
// lo x lo term dropped).  NEG subtracts the product.  KR as in mmul, per warp.  With leading dims
// of 4 mod 32 floats the K-major fragment reads are free of bank conflicts.
template <int M, int N, int K, bool AK, bool BK, bool ASPL, bool BSPL, int KR = 0, bool NEG = false>
__device__ __forceinline__ void mma_mul(typename WT<M, N>::Acc& acc, const float* A, int lda, const float* B,
                                        int ldb) {
    using W = WT<M, N>;
    static_assert(K % 16 == 0, "depth");
    static_assert(KR == 0 || M == K, "a triangular A is square");
    const int g = (threadIdx.x & 31) >> 2, t = threadIdx.x & 3;
    const int mb = W::mb(), nb = W::nb();
    const int kb = KR == 1 ? (mb & ~15) : 0;
    const int ke = KR == 2 ? min(K, mb + M / W::WM) : K;
#pragma unroll 1
    for (int k0 = kb; k0 < ke; k0 += 16) {
        uint32_t ah[W::MT][4], al[W::MT][4], bh[W::NT][2], bl[W::NT][2];
#pragma unroll
        for (int mt = 0; mt < W::MT; ++mt)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int m = mb + mt * 16 + g + 8 * (r & 1), k = k0 + 2 * t + 8 * (r >> 1);
                float x0, x1;
                if constexpr (AK) {
                    x0 = A[k * lda + m];
                    x1 = A[(k + 1) * lda + m];
                } else {
                    const float2 v = *reinterpret_cast<const float2*>(A + m * lda + k);
                    x0 = v.x;
                    x1 = v.y;
                }
                if constexpr (ASPL) split_bf16(x0, x1, ah[mt][r], al[mt][r]);
                else ah[mt][r] = pack_bf16(x0, x1);
                if constexpr (NEG) {  // flip the sign bits of both halves
                    ah[mt][r] ^= 0x80008000u;
                    if constexpr (ASPL) al[mt][r] ^= 0x80008000u;
                }
            }
#pragma unroll
        for (int nt = 0; nt < W::NT; ++nt)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int k = k0 + 2 * t + 8 * r, n = nb + nt * 8 + g;
                float x0, x1;
                if constexpr (BK) {
                    x0 = B[k * ldb + n];
                    x1 = B[(k + 1) * ldb + n];
                } else {
                    const float2 v = *reinterpret_cast<const float2*>(B + n * ldb + k);
                    x0 = v.x;
                    x1 = v.y;
                }
                if constexpr (BSPL) split_bf16(x0, x1, bh[nt][r], bl[nt][r]);
                else bh[nt][r] = pack_bf16(x0, x1);
            }
#pragma unroll
        for (int mt = 0; mt < W::MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < W::NT; ++nt) {
                mma16816(acc[mt][nt], ah[mt], bh[nt]);
                if constexpr (ASPL) mma16816(acc[mt][nt], al[mt], bh[nt]);
                if constexpr (BSPL) mma16816(acc[mt][nt], ah[mt], bl[nt]);
            }
    }
}

// f(row, col, v0, v1) for each pair of adjacent columns (col, col + 1) the lane holds
template <int M, int N, typename F>
__device__ __forceinline__ void frag_pairs(const typename WT<M, N>::Acc& acc, F f) {
    using W = WT<M, N>;
#pragma unroll
    for (int mt = 0; mt < W::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < W::NT; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) f(W::row(mt, 2 * h), W::col(nt, 0), acc[mt][nt][2 * h], acc[mt][nt][2 * h + 1]);
}

// dst[r ld + col] = f(r, col, v) over the lane's elements (dst[col ld + r] when TR)
template <int M, int N, bool TR = false, typename F>
__device__ __forceinline__ void frag_store(float* dst, int ld, const typename WT<M, N>::Acc& acc, F f) {
    frag_pairs<M, N>(acc, [&](int r, int cc, float v0, float v1) {
        const float x0 = f(r, cc, v0), x1 = f(r, cc + 1, v1);
        if constexpr (TR) {
            dst[cc * ld + r] = x0;
            dst[(cc + 1) * ld + r] = x1;
        } else {
            *reinterpret_cast<float2*>(dst + r * ld + cc) = make_float2(x0, x1);
        }
    });
}
template <int M, int N, bool TR = false>
__device__ __forceinline__ void frag_store(float* dst, int ld, const typename WT<M, N>::Acc& acc) {
    frag_store<M, N, TR>(dst, ld, acc, [](int, int, float x) { return x; });
}
// rows r < c of a C x D result to global bf16: dst[r][e] = acc + (add ? add[r][e] : 0); the addends
// are all loaded before the first store
template <int D>
__device__ __forceinline__ void frag_out(__nv_bfloat16* dst, const typename WT<kC, D>::Acc& acc, const float* add,
                                         int c) {
    using W = WT<kC, D>;
    float2 a[W::MT][W::NT][2];
#pragma unroll
    for (int mt = 0; mt < W::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < W::NT; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = W::row(mt, 2 * h);
                a[mt][nt][h] = add && r < c ? *reinterpret_cast<const float2*>(add + (size_t)r * D + W::col(nt, 0))
                                            : make_float2(0.f, 0.f);
            }
#pragma unroll
    for (int mt = 0; mt < W::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < W::NT; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = W::row(mt, 2 * h);
                if (r < c)
                    *reinterpret_cast<__nv_bfloat162*>(dst + (size_t)r * D + W::col(nt, 0)) = __floats2bfloat162_rn(
                        acc[mt][nt][2 * h] + a[mt][nt][h].x, acc[mt][nt][2 * h + 1] + a[mt][nt][h].y);
            }
}

// One doubling merge of the triangular inverse: for each pair of S-row blocks on the diagonal,
// X_12 = -X_11 (D G_12) X_22, written over the X_12 block.  Every thread owns PER elements of
// the pairs' X_12 blocks and sums them side by side over whole blocks (the zeros of the
// triangular X_11 and X_22 add nothing).
template <int C, int LC, int S>
__device__ __forceinline__ void ut_merge(const float* sG, float* sX, const float* sB) {
    constexpr int PER = C * S / (2 * kNTL);
    static_assert(PER >= 1 && PER * 2 * kNTL == C * S, "whole elements per thread");
    int a[PER], bb[PER], kb[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        const int idx = threadIdx.x + e * kNTL, pr = idx / (S * S), rem = idx % (S * S);
        kb[e] = 2 * S * pr;
        a[e] = kb[e] + rem / S;
        bb[e] = kb[e] + S + rem % S;
    }
    float v[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) v[e] = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < S; ++kk)  // T = D G_12 X_22
#pragma unroll
        for (int e = 0; e < PER; ++e)
            v[e] = fmaf(sG[a[e] * LC + kb[e] + S + kk], sX[(kb[e] + S + kk) * LC + bb[e]], v[e]);
#pragma unroll
    for (int e = 0; e < PER; ++e) sX[a[e] * LC + bb[e]] = sB[a[e]] * v[e];
    __syncthreads();
#pragma unroll
    for (int e = 0; e < PER; ++e) v[e] = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < S; ++kk)  // X_12 = -X_11 T
#pragma unroll
        for (int e = 0; e < PER; ++e) v[e] = fmaf(sX[a[e] * LC + kb[e] + kk], sX[(kb[e] + kk) * LC + bb[e]], v[e]);
    __syncthreads();
#pragma unroll
    for (int e = 0; e < PER; ++e) sX[a[e] * LC + bb[e]] = -v[e];
    __syncthreads();
}

// X = (I + D triu_1 G)^{-1} (unit upper triangular) and A = X D, D = diag(beta), for a chunk of
// C = 64 positions: the 16 x 16 diagonal blocks row by row from the bottom (one warp each,
// X_ij = [i == j] - beta_i sum_{i < k <= j} G_ik X_kj), then two doubling merges.  sX must hold
// zeros on entry; the caller synchronises after.
template <int C, int LC>
__device__ __forceinline__ void ut_inverse(const float* sG, float* sX, float* sA, const float* sB) {
    static_assert(C == 64, "two merges after the 16 x 16 blocks");
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (wid < C / 16) {
        const int j = 16 * wid + (lane & 15), h = lane >> 4;
        for (int i = 16 * wid + 15; i >= 16 * wid; --i) {
            float t = 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {  // k = i + 1 + h + 2u <= j, at most eight terms per lane
                const int kk = i + 1 + h + 2 * u;
                if (kk <= j) t = fmaf(sG[i * LC + kk], sX[kk * LC + j], t);
            }
            t += __shfl_xor_sync(0xffffffffu, t, 16);
            if (h == 0 && j >= i) sX[i * LC + j] = (j == i ? 1.f : 0.f) - sB[i] * t;
            __syncwarp();
        }
    }
    __syncthreads();
    ut_merge<C, LC, 16>(sG, sX, sB);
    ut_merge<C, LC, 32>(sG, sX, sB);
    for (int idx = threadIdx.x; idx < C * C; idx += kNTL) {
        const int r = idx / C, cc = idx % C;
        sA[r * LC + cc] = sX[r * LC + cc] * sB[cc];
    }
}

// two consecutive bf16 values of a row as floats
__device__ __forceinline__ float2 to_f2(const __nv_bfloat16* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}

// rows r < C of a C x D result: dst[r][e] = src[r][e] - acc for r < c, 0 for the padded rows
// (fp32, and a bf16 copy when dst16 is set)
template <int D, typename S>
__device__ __forceinline__ void mstore_diff(float* dst, __nv_bfloat16* dst16, const S* src,
                                            const typename TT<kC, D, false>::Acc& acc, int c) {
    using G = TT<kC, D, false>;
    const int m0 = G::m0(), n0 = G::n0();
    static_assert(G::TN % 4 == 0, "row segments of whole 4-vectors");
    float v[G::TM][G::TN];
#pragma unroll
    for (int i = 0; i < G::TM; ++i) {
        if (m0 + i < c) ld_row<G::TN>(v[i], src + (size_t)(m0 + i) * D + n0);
        else
#pragma unroll
            for (int j = 0; j < G::TN; ++j) v[i][j] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < G::TM; ++i) {
        const bool ok = m0 + i < c;
#pragma unroll
        for (int j = 0; j < G::TN; ++j) v[i][j] = ok ? v[i][j] - acc[i][j] : 0.f;
        st_row<G::TN>(dst + (size_t)(m0 + i) * D + n0, v[i]);
        if (dst16) st_row<G::TN>(dst16 + (size_t)(m0 + i) * D + n0, v[i]);
    }
}

// ------------------------------------------------------------------ bwd_prep
// Per chunk, in the compact form of "Representação de Transformação UT" (§3): with G, X and A as
// in bwd_local, Qm = tril(Q W^T), Km = striu(K W^T), Y = Qm A^T and Z = Km A,
//   qbar = Q - Y W  (H_b ... H_i q_i),   khat = K - Z W  (H_e ... H_{j+1} k_j),
//   P_n  = I - W^T (A W) for the inner chunks 1 <= n <= N - 2 (fp32 P and P^T, or hi / lo bf16),
// and Delta_i = dO_i . o_i.  Eleven shared-memory slots as in bwd_local.
template <typename T, int D>
__global__ void __launch_bounds__(kNTL, 1) bwd_prep(BwdParams p) {
    constexpr int C = kC, LC = C + 4, LD = D + 4, U = BwdSmem<D>::slot;
    constexpr bool TC = sizeof(T) == 2 && D >= 64;  // bf16 operands: the products on the tensor cores
    static_assert(C * LD <= 2 * U && D * LC <= 2 * U, "slot sizes");
    extern __shared__ __align__(16) float smem[];
    auto slot = [&](int i) { return smem + i * U; };
    float* sB = smem + 11 * U;  // [C] beta
    const int n = blockIdx.x, bh = blockIdx.y, b = n * C, c = min(C, p.L - b);
    const size_t hrow = (size_t)bh * p.L + b, prow = (size_t)bh * p.Lp + b;
    const T* q = static_cast<const T*>(p.q) + hrow * D;
    const T* k = static_cast<const T*>(p.k) + hrow * D;
    const T* w = static_cast<const T*>(p.w) + hrow * D;
    using GN = TT<C, C, false>;
    using GS = TT<C, C, true>;
    using GR = TT<C, D, false>;
    auto id = [](int, int, float x) { return x; };
    for (int r = threadIdx.x; r < C; r += kNTL) sB[r] = r < c ? p.beta[hrow + r] : 0.f;
    for (int idx = threadIdx.x; idx < U; idx += kNTL) slot(7)[idx] = 0.f;
    to_smem_t<T, D, kNTL>(slot(0), LC, w, D, C, c);  // W^T, slots 0-1
    to_smem_t<T, D, kNTL>(slot(2), LC, q, D, C, c);  // Q^T, slots 2-3
    to_smem_t<T, D, kNTL>(slot(4), LC, k, D, C, c);  // K^T, slots 4-5
    {  // Delta_i = dO_i . o_i: four threads per row, each a quarter of it
        static_assert(kNTL == 4 * C, "four threads per row");
        const int r = threadIdx.x >> 2, part = threadIdx.x & 3;
        float t = 0.f;
        if (r < c) {
            const T* orow = static_cast<const T*>(p.o) + (hrow + r) * D + part * (D / 4);
            const T* grow = static_cast<const T*>(p.dO) + (hrow + r) * D + part * (D / 4);
#pragma unroll
            for (int j = 0; j < D / 4; j += 4) {
                float a[4], g[4];
                ld_row<4>(a, orow + j);
                ld_row<4>(g, grow + j);
                t = fmaf(a[0], g[0], fmaf(a[1], g[1], fmaf(a[2], g[2], fmaf(a[3], g[3], t))));
            }
        }
        t += __shfl_xor_sync(0xffffffffu, t, 1);
        t += __shfl_xor_sync(0xffffffffu, t, 2);
        if (part == 0) p.delta[prow + r] = t;
    }
    __syncthreads();
    if constexpr (TC) {  // G = W W^T, Q W^T, K W^T: bf16 operands, one product each
        using WC = WT<C, C>;
        typename WC::Acc g, qw, kw;
        WC::zero(g);
        WC::zero(qw);
        WC::zero(kw);
        mma_mul<C, C, D, true, true, false, false>(g, slot(0), LC, slot(0), LC);
        mma_mul<C, C, D, true, true, false, false>(qw, slot(2), LC, slot(0), LC);
        mma_mul<C, C, D, true, true, false, false>(kw, slot(4), LC, slot(0), LC);
        __syncthreads();
        float *sG = slot(6), *sQT = slot(2), *sKm = slot(4);
        frag_pairs<C, C>(g, [&](int r, int cc, float v0, float v1) {
            *reinterpret_cast<float2*>(sG + r * LC + cc) = make_float2(v0, v1);
        });
        frag_pairs<C, C>(qw, [&](int r, int cc, float v0, float v1) {  // Qm^T
            sQT[cc * LC + r] = cc <= r ? v0 : 0.f;
            sQT[(cc + 1) * LC + r] = cc + 1 <= r ? v1 : 0.f;
        });
        frag_pairs<C, C>(kw, [&](int r, int cc, float v0, float v1) {  // Km
            *reinterpret_cast<float2*>(sKm + r * LC + cc) = make_float2(cc > r ? v0 : 0.f, cc + 1 > r ? v1 : 0.f);
        });
    } else {
        typename GN::Acc g, qw, kw;
        GN::zero(g);
        GN::zero(qw);
        GN::zero(kw);
        mmul<C, C, D, false, true, true>(g, slot(0), LC, slot(0), LC);   // G = W W^T
        mmul<C, C, D, false, true, true>(qw, slot(2), LC, slot(0), LC);  // Q W^T
        mmul<C, C, D, false, true, true>(kw, slot(4), LC, slot(0), LC);  // K W^T
        __syncthreads();
        mstore<C, C, false, false>(slot(6), LC, g, id);
        mstore<C, C, false, true>(slot(2), LC, qw, [](int i, int bb, float x) { return bb <= i ? x : 0.f; });  // Qm^T
        mstore<C, C, false, false>(slot(4), LC, kw, [](int j, int a, float x) { return a > j ? x : 0.f; });    // Km
    }
    __syncthreads();
    TileRegs<T, TC ? D : 64, C> pw;  // W [C][LD] for slots 0-1, in flight during the inverse
    if constexpr (TC) pw.load_r(w, D, c);
    else to_smem_v<T, D, kNTL>(slot(0), LD, w, D, C, c);
    ut_inverse<C, LC>(slot(6), slot(7), slot(8), sB);  // X -> slot 7, A -> slot 8
    if constexpr (TC) pw.store_r(slot(0), LD);
    __syncthreads();
    {  // X for bwd_local, which needs the same factor
        float* xg = p.xinv + ((size_t)bh * p.N + n) * C * C;
        for (int idx = threadIdx.x; idx < C * C / 4; idx += kNTL) {
            const int r = idx / (C / 4), c4 = (idx % (C / 4)) * 4;
            *reinterpret_cast<float4*>(xg + r * C + c4) = *reinterpret_cast<const float4*>(slot(7) + r * LC + c4);
        }
    }
    if constexpr (TC) {  // fp32 operands: three products each
        typename WT<C, C>::Acc y, z;
        WT<C, C>::zero(y);
        WT<C, C>::zero(z);
        mma_mul<C, C, C, true, false, true, true, 2>(y, slot(2), LC, slot(8), LC);  // Y = Qm A^T
        mma_mul<C, C, C, false, true, true, true, 1>(z, slot(4), LC, slot(8), LC);  // Z = Km A
        frag_store<C, C, true>(slot(3), LC, y);  // Y^T
        frag_store<C, C>(slot(5), LC, z);
    } else {
        typename GS::Acc y;
        GS::zero(y);
        mmul<C, C, C, true, true, false>(y, slot(2), LC, slot(8), LC);  // Y = Qm A^T
        mstore<C, C, true, true>(slot(3), LC, y, id);                   // Y^T
        typename GN::Acc z;
        GN::zero(z);
        mmul<C, C, C, false, false, true, false, 1>(z, slot(4), LC, slot(8), LC);  // Z = Km A
        mstore<C, C, false, false>(slot(5), LC, z, id);
    }
    __syncthreads();
    if constexpr (TC) {  // Y W and Z W (Y, Z split into hi + lo), then qbar = Q - Y W, khat = K - Z W
        using WR = WT<C, D>;
        typename WR::Acc yw, zw;
        WR::zero(yw);
        WR::zero(zw);
        mma_mul<C, D, C, true, true, true, false, 2>(yw, slot(3), LC, slot(0), LD);
        mma_mul<C, D, C, false, true, true, false, 1>(zw, slot(5), LC, slot(0), LD);
        float* qb = p.qbar + prow * D;
        float* kh = p.khat + prow * D;
        __nv_bfloat16* kh16 = p.khat16 ? p.khat16 + prow * D : nullptr;
        // qbar = Q - Y W and khat = K - Z W; the q and k values are all loaded before the first store
        float2 xq[WR::MT][WR::NT][2], xk[WR::MT][WR::NT][2];
#pragma unroll
        for (int mt = 0; mt < WR::MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < WR::NT; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = WR::row(mt, 2 * h), cc = WR::col(nt, 0);
                    const bool ok = r < c;
                    xq[mt][nt][h] = ok ? to_f2(q + (size_t)r * D + cc) : make_float2(0.f, 0.f);
                    xk[mt][nt][h] = ok ? to_f2(k + (size_t)r * D + cc) : make_float2(0.f, 0.f);
                }
#pragma unroll
        for (int mt = 0; mt < WR::MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < WR::NT; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = WR::row(mt, 2 * h), cc = WR::col(nt, 0);
                    const bool ok = r < c;  // padded rows are written as zeros
                    const float2 a = ok ? make_float2(xq[mt][nt][h].x - yw[mt][nt][2 * h], xq[mt][nt][h].y - yw[mt][nt][2 * h + 1])
                                        : make_float2(0.f, 0.f);
                    const float2 b = ok ? make_float2(xk[mt][nt][h].x - zw[mt][nt][2 * h], xk[mt][nt][h].y - zw[mt][nt][2 * h + 1])
                                        : make_float2(0.f, 0.f);
                    *reinterpret_cast<float2*>(qb + (size_t)r * D + cc) = a;
                    *reinterpret_cast<float2*>(kh + (size_t)r * D + cc) = b;
                    if (kh16) *reinterpret_cast<__nv_bfloat162*>(kh16 + (size_t)r * D + cc) = __floats2bfloat162_rn(b.x, b.y);
                }
        if (n < 1 || n > p.N - 2) return;
        typename WR::Acc aw;
        WR::zero(aw);
        mma_mul<C, D, C, false, true, true, false, 1>(aw, slot(8), LC, slot(0), LD);  // A W
        float* sAW = slot(9);  // [C][LD], slots 9-10
        frag_pairs<C, D>(aw, [&](int r, int cc, float v0, float v1) {
            *reinterpret_cast<float2*>(sAW + r * LD + cc) = make_float2(v0, v1);
        });
    } else {
        typename GR::Acc acc;
        GR::zero(acc);
        mmul<C, D, C, false, true, true, false, 2>(acc, slot(3), LC, slot(0), LD);  // Y W
        mstore_diff<D>(p.qbar + prow * D, nullptr, q, acc, c);
        GR::zero(acc);
        mmul<C, D, C, false, false, true, false, 1>(acc, slot(5), LC, slot(0), LD);  // Z W
        mstore_diff<D>(p.khat + prow * D, p.khat16 ? p.khat16 + prow * D : nullptr, k, acc, c);
        if (n < 1 || n > p.N - 2) return;
        typename GR::Acc aw;
        GR::zero(aw);
        mmul<C, D, C, false, false, true, false, 1>(aw, slot(8), LC, slot(0), LD);  // A W
        mstore<C, D, false, false>(slot(9), LD, aw, id);                            // slots 9-10
    }
    __syncthreads();
    const size_t base = ((size_t)bh * p.N + n) * D * D;
    if constexpr (TC) {  // P = I - W^T (A W), A W split into hi + lo
        using WP = WT<D, D>;
        typename WP::Acc pa;
        WP::zero(pa);
        mma_mul<D, D, C, true, true, false, true>(pa, slot(0), LD, slot(9), LD);
        frag_pairs<D, D>(pa, [&](int r, int cc, float v0, float v1) {
            const float x0 = (r == cc ? 1.f : 0.f) - v0, x1 = (r == cc + 1 ? 1.f : 0.f) - v1;
            const size_t o = base + (size_t)r * D + cc;
            if (p.pm) {
                *reinterpret_cast<float2*>(p.pm + o) = make_float2(x0, x1);
                p.pmt[base + (size_t)cc * D + r] = x0;
                p.pmt[base + (size_t)(cc + 1) * D + r] = x1;
            }
            if (p.phi) {
                uint32_t hi, lo;
                split_bf16(x0, x1, hi, lo);
                *reinterpret_cast<uint32_t*>(p.phi + o) = hi;
                *reinterpret_cast<uint32_t*>(p.plo + o) = lo;
            }
        });
        return;
    }
    using GP = TT<D, D, false>;
    typename GP::Acc pa;
    GP::zero(pa);
    mmul<D, D, C, false, true, true>(pa, slot(0), LD, slot(9), LD);  // W^T (A W)
    const int m0 = GP::m0(), n0 = GP::n0();
#pragma unroll
    for (int i = 0; i < GP::TM; ++i)
#pragma unroll
        for (int j = 0; j < GP::TN; ++j) pa[i][j] = (m0 + i == n0 + j ? 1.f : 0.f) - pa[i][j];
    if (p.pm) {  // fp32 P and P^T
#pragma unroll
        for (int i = 0; i < GP::TM; ++i) {
            if constexpr (GP::TN % 4 == 0) st_row<GP::TN>(p.pm + base + (size_t)(m0 + i) * D + n0, pa[i]);
            else
#pragma unroll
                for (int j = 0; j < GP::TN; ++j) p.pm[base + (size_t)(m0 + i) * D + n0 + j] = pa[i][j];
        }
#pragma unroll
        for (int j = 0; j < GP::TN; ++j) {
            float t[GP::TM];
#pragma unroll
            for (int i = 0; i < GP::TM; ++i) t[i] = pa[i][j];
            if constexpr (GP::TM % 4 == 0) st_row<GP::TM>(p.pmt + base + (size_t)(n0 + j) * D + m0, t);
            else
#pragma unroll
                for (int i = 0; i < GP::TM; ++i) p.pmt[base + (size_t)(n0 + j) * D + m0 + i] = t[i];
        }
    }
    if (p.phi) {  // hi + lo bf16 split for the tensor-core chains (d = 128)
#pragma unroll
        for (int i = 0; i < GP::TM; ++i) {
            float lo[GP::TN];
#pragma unroll
            for (int j = 0; j < GP::TN; ++j) lo[j] = pa[i][j] - __bfloat162float(__float2bfloat16_rn(pa[i][j]));
            if constexpr (GP::TN % 4 == 0) {
                st_row<GP::TN>(p.phi + base + (size_t)(m0 + i) * D + n0, pa[i]);
                st_row<GP::TN>(p.plo + base + (size_t)(m0 + i) * D + n0, lo);
            } else {
#pragma unroll
                for (int j = 0; j < GP::TN; ++j) {
                    p.phi[base + (size_t)(m0 + i) * D + n0 + j] = __float2bfloat16_rn(pa[i][j]);
                    p.plo[base + (size_t)(m0 + i) * D + n0 + j] = __float2bfloat16_rn(lo[j]);
                }
            }
        }
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kNTL, 1) bwd_local(BwdParams p) {
    constexpr int C = kC, LC = C + 4, LD = D + 4, U = BwdSmem<D>::slot;
    constexpr int KH = D < 64 ? D : 64, NH = D / KH;  // d x C operands in pieces of KH rows
    constexpr bool TC = sizeof(T) == 2 && D >= 64;  // bf16 operands: most products on the tensor cores
    static_assert(C == 64, "chunks of 64 positions");
    static_assert(C * LD <= 2 * U && D * LC <= 2 * U && D * LD <= 4 * U && KH * LC <= U, "slot sizes");
    extern __shared__ __align__(16) float smem[];
    auto slot = [&](int i) { return smem + i * U; };
    float* sB = smem + 13 * U;  // [C] beta
    float* sC = sB + C;         // [C] c (FoX)
    float* sL = sC + C;         // [C] lse
    float* sDl = sL + C;        // [C] Delta
    float* aB = sDl + C;        // [C] dbeta
    float* aC = aB + C;         // [C] dc (FoX), diagonal part
    const int n = blockIdx.x, bh = blockIdx.y, b = n * C, c = min(C, p.L - b);
    const size_t hrow = (size_t)bh * p.L + b, prow = (size_t)bh * p.Lp + b;
    const T* q = static_cast<const T*>(p.q) + hrow * D;
    const T* k = static_cast<const T*>(p.k) + hrow * D;
    const T* w = static_cast<const T*>(p.w) + hrow * D;
    const T* dO = static_cast<const T*>(p.dO) + hrow * D;
    const bool below = n >= 1;        // query chains from this chunk continue into earlier chunks
    const bool above = n <= p.N - 2;  // later query chunks reach this chunk's keys
    const bool hasP = below && above; // the chunk transition P_n was used
    const float scale = p.scale;
    using GS = TT<C, C, true>;   // C x C, rows first
    using GN = TT<C, C, false>;  // C x C, columns first
    using GR = TT<C, D, false>;  // C x d
    auto id = [](int, int, float x) { return x; };

    for (int r = threadIdx.x; r < C; r += kNTL) {
        sB[r] = r < c ? p.beta[hrow + r] : 0.f;
        sC[r] = p.fox ? p.cum[prow + r] : 0.f;
        sL[r] = r < c ? p.lse[hrow + r] : 0.f;
        sDl[r] = r < c ? p.delta[prow + r] : 0.f;
        aB[r] = 0.f;
        aC[r] = 0.f;
    }
    to_smem_v<float, C, kNTL>(slot(7), LC, p.xinv + ((size_t)bh * p.N + n) * C * C, C, C, C);  // X (bwd_prep) -> slot 7 (until dM)
    to_smem_t<T, D, kNTL>(slot(0), LC, w, D, C, c);  // W^T [D][LC] in slots 0-1 (until the dY phase)
    const float* dP = p.dpm + ((size_t)bh * p.N + n) * D * D;
    if (hasP) to_smem_v<float, D, kNTL>(slot(2), LD, dP, D, D, D);  // dP [D][LD], slots 2-5, read after the inverse
    __syncthreads();
    if constexpr (TC) {  // G = W W^T -> slot 6 (until dM)
        typename WT<C, C>::Acc g;
        WT<C, C>::zero(g);
        mma_mul<C, C, D, true, true, false, false>(g, slot(0), LC, slot(0), LC);
        frag_store<C, C>(slot(6), LC, g);
    } else {
        typename GN::Acc g;
        GN::zero(g);
        mmul<C, C, D, false, true, true>(g, slot(0), LC, slot(0), LC);
        mstore<C, C, false, false>(slot(6), LC, g, id);
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < C * C; idx += kNTL) {  // A = X D -> slot 8 (until dQm)
        const int r = idx / C, cc = idx % C;
        slot(8)[r * LC + cc] = slot(7)[r * LC + cc] * sB[cc];
    }
    __syncthreads();
    typename GR::Acc aW;  // dW, accumulated across the phases (CUDA cores)
    using WD = WT<C, TC ? D : 64>;  // (a valid, unused shape off the tensor-core path)
    typename WD::Acc aWf;             // dW (tensor cores)
    GR::zero(aW);
    WD::zero(aWf);
    using TRg = TileRegs<T, TC ? D : 64, C>;  // (a valid, unused shape off the tensor-core path)
    TRg pq, pk;  // q and k, loaded while the transition's products run (tensor-core path)
    if (hasP) {  // the chunk transition: dW -= A^T (W dP) + A (W dP^T), E = W dP W^T -> slot 9 (until dA)
        if constexpr (TC) {  // R1 = W dP and R2 = W dP^T from the one copy of dP (split into hi + lo)
            pq.load(q, D, c);
            pk.load(k, D, c);
            typename WT<C, D>::Acc r1, r2;
            WT<C, D>::zero(r1);
            WT<C, D>::zero(r2);
            mma_mul<C, D, D, true, true, false, true>(r1, slot(0), LC, slot(2), LD);
            mma_mul<C, D, D, true, false, false, true>(r2, slot(0), LC, slot(2), LD);
            __syncthreads();
            frag_store<C, D>(slot(2), LD, r1);         // R1 [C][LD], slots 2-3
            frag_store<C, D, true>(slot(4), LC, r1);   // R1^T [D][LC], slots 4-5
            frag_store<C, D>(slot(10), LD, r2);        // R2 [C][LD], slots 10-11 (free until Qm^T and Km)
            __syncthreads();
            mma_mul<C, D, C, true, true, true, true, 2, true>(aWf, slot(8), LC, slot(2), LD);    // -= A^T R1
            mma_mul<C, D, C, false, true, true, true, 1, true>(aWf, slot(8), LC, slot(10), LD);  // -= A R2
            typename WT<C, C>::Acc e;  // E = R1 W^T
            WT<C, C>::zero(e);
            mma_mul<C, C, D, true, true, true, false>(e, slot(4), LC, slot(0), LC);
            frag_store<C, C>(slot(9), LC, e);
        } else {
            typename GR::Acc r;
            GR::zero(r);
            mmul<C, D, D, false, true, true>(r, slot(0), LC, slot(2), LD);  // R1 = W dP
            __syncthreads();
            mstore<C, D, false, false>(slot(2), LD, r, id);  // R1 [C][LD], slots 2-3
            mstore<C, D, false, true>(slot(4), LC, r, id);   // R1^T [D][LC], slots 4-5
            __syncthreads();
            mmul<C, D, C, false, true, true, true, 2>(aW, slot(8), LC, slot(2), LD);  // -= A^T R1
            {
                typename GN::Acc e;
                GN::zero(e);
                mmul<C, C, D, false, true, true>(e, slot(4), LC, slot(0), LC);  // E = R1 W^T
                mstore<C, C, false, false>(slot(9), LC, e, id);
            }
            __syncthreads();
            to_smem_t<float, D, kNTL>(slot(2), LD, dP, D, D, D);  // dP^T [D][LD], slots 2-5
            __syncthreads();
            GR::zero(r);
            mmul<C, D, D, false, true, true>(r, slot(0), LC, slot(2), LD);  // R2 = W dP^T
            __syncthreads();
            mstore<C, D, false, false>(slot(2), LD, r, id);
            __syncthreads();
            mmul<C, D, C, false, false, true, true, 1>(aW, slot(8), LC, slot(2), LD);  // -= A R2
        }
    }
    __syncthreads();
    if (TC && hasP) {
        pq.store_t(slot(2), LC);  // Q^T, slots 2-3
        pk.store_t(slot(4), LC);  // K^T, slots 4-5
    } else {
        to_smem_t<T, D, kNTL>(slot(2), LC, q, D, C, c);
        to_smem_t<T, D, kNTL>(slot(4), LC, k, D, C, c);
    }
    __syncthreads();
    typename GS::Acc aS;        // Q K^T - Y Km^T, then the probabilities (CUDA cores)
    typename WT<C, C>::Acc sT;  // Q K^T, then the probabilities (tensor cores)
    GS::zero(aS);
    WT<C, C>::zero(sT);
    if constexpr (TC) {
        typename WT<C, C>::Acc qw, kw;
        WT<C, C>::zero(qw);
        WT<C, C>::zero(kw);
        mma_mul<C, C, D, true, true, false, false>(qw, slot(2), LC, slot(0), LC);
        mma_mul<C, C, D, true, true, false, false>(kw, slot(4), LC, slot(0), LC);
        mma_mul<C, C, D, true, true, false, false>(sT, slot(2), LC, slot(4), LC);
        __syncthreads();
        frag_store<C, C, true>(slot(10), LC, qw, [](int i, int bb, float x) { return bb <= i ? x : 0.f; });  // Qm^T (until dA)
        frag_store<C, C>(slot(11), LC, kw, [](int j, int a, float x) { return a > j ? x : 0.f; });          // Km (until dA)
    } else {
        typename GS::Acc qw, kw;
        GS::zero(qw);
        GS::zero(kw);
        mmul<C, C, D, true, true, true>(qw, slot(2), LC, slot(0), LC);
        mmul<C, C, D, true, true, true>(kw, slot(4), LC, slot(0), LC);
        mmul<C, C, D, true, true, true>(aS, slot(2), LC, slot(4), LC);
        __syncthreads();
        mstore<C, C, true, true>(slot(10), LC, qw, [](int i, int bb, float x) { return bb <= i ? x : 0.f; });  // Qm^T (until dA)
        mstore<C, C, true, false>(slot(11), LC, kw, [](int j, int a, float x) { return a > j ? x : 0.f; });    // Km (until dA)
    }
    __syncthreads();
    if constexpr (TC) {  // fp32 operands: three products each
        typename WT<C, C>::Acc y, z;
        WT<C, C>::zero(y);
        WT<C, C>::zero(z);
        mma_mul<C, C, C, true, false, true, true, 2>(y, slot(10), LC, slot(8), LC);  // Y = Qm A^T
        mma_mul<C, C, C, false, true, true, true, 1>(z, slot(11), LC, slot(8), LC);  // Z = Km A
        frag_store<C, C, true>(slot(12), LC, y);  // Y^T -> slot 12 (until the end)
        frag_store<C, C>(slot(2), LC, z);         // -> slot 2 (until the end)
    } else {
        typename GS::Acc y;
        GS::zero(y);
        mmul<C, C, C, true, true, false>(y, slot(10), LC, slot(8), LC);  // Y = Qm A^T
        mstore<C, C, true, true>(slot(12), LC, y, id);                   // Y^T -> slot 12 (until the end)
        typename GN::Acc z;
        GN::zero(z);
        mmul<C, C, C, false, false, true, false, 1>(z, slot(11), LC, slot(8), LC);  // Z = Km A
        mstore<C, C, false, false>(slot(2), LC, z, id);                   // -> slot 2 (until the end)
    }
    __syncthreads();
    to_smem_t<T, D, kNTL>(slot(0), LC, dO, D, C, c);                                   // dO^T, slots 0-1
    to_smem_t<T, D, kNTL>(slot(4), LC, static_cast<const T*>(p.v) + hrow * D, D, C, c);  // V^T, slots 4-5
    if constexpr (TC) {
        mma_mul<C, C, C, true, false, true, true, 2, true>(sT, slot(12), LC, slot(11), LC);  // -= Y Km^T
        __syncthreads();
        using WC = WT<C, C>;
        typename WC::Acc dp;
        WC::zero(dp);
        mma_mul<C, C, D, true, true, false, false>(dp, slot(0), LC, slot(4), LC);  // dO V^T
        float rs[WC::MT][2], cs[WC::NT][2];
#pragma unroll
        for (int mt = 0; mt < WC::MT; ++mt) rs[mt][0] = rs[mt][1] = 0.f;
#pragma unroll
        for (int nt = 0; nt < WC::NT; ++nt) cs[nt][0] = cs[nt][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < WC::MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < WC::NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = WC::row(mt, i), col = WC::col(nt, i);
                    float pij = 0.f, ds = 0.f;
                    if (r < c && col <= r) {
                        pij = __expf(scale * sT[mt][nt][i] + sC[r] - sC[col] - sL[r]);
                        ds = pij * (dp[mt][nt][i] - sDl[r]);
                    }
                    sT[mt][nt][i] = pij;
                    dp[mt][nt][i] = scale * ds;
                    rs[mt][i >> 1] += ds;
                    cs[nt][i & 1] += ds;
                }
        if (p.fox) {
#pragma unroll
            for (int mt = 0; mt < WC::MT; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) atomicAdd(aC + WC::row(mt, 2 * h), rs[mt][h]);
#pragma unroll
            for (int nt = 0; nt < WC::NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) atomicAdd(aC + WC::col(nt, e), -cs[nt][e]);
        }
        __syncthreads();
        frag_store<C, C>(slot(3), LC, sT);  // P -> slot 3 (until dV)
        frag_store<C, C>(slot(0), LC, dp);  // dSs -> slot 0 (until the end)
    } else {
        mmul<C, C, C, true, true, false, true>(aS, slot(12), LC, slot(11), LC);  // -= Y Km^T
        __syncthreads();
        {
            typename GS::Acc dp;
            GS::zero(dp);
            mmul<C, C, D, true, true, true>(dp, slot(0), LC, slot(4), LC);  // dO V^T
            const int m0 = GS::m0(), n0 = GS::n0();
            float cs[GS::TN];
#pragma unroll
            for (int j = 0; j < GS::TN; ++j) cs[j] = 0.f;
#pragma unroll
            for (int i = 0; i < GS::TM; ++i) {
                const int r = m0 + i;
                float rs = 0.f;
#pragma unroll
                for (int j = 0; j < GS::TN; ++j) {
                    const int col = n0 + j;
                    float pij = 0.f, ds = 0.f;
                    if (r < c && col <= r) {
                        pij = __expf(scale * aS[i][j] + sC[r] - sC[col] - sL[r]);
                        ds = pij * (dp[i][j] - sDl[r]);
                    }
                    aS[i][j] = pij;
                    dp[i][j] = scale * ds;
                    rs += ds;
                    cs[j] += ds;
                }
                if (p.fox) atomicAdd(aC + r, rs);
            }
            if (p.fox)
#pragma unroll
                for (int j = 0; j < GS::TN; ++j) atomicAdd(aC + n0 + j, -cs[j]);
            __syncthreads();
            mstore<C, C, true, false>(slot(3), LC, aS, id);  // P -> slot 3 (until dV)
            mstore<C, C, true, false>(slot(0), LC, dp, id);  // dSs -> slot 0 (until the end)
        }
    }
    to_smem_v<T, D, kNTL>(slot(4), LD, dO, D, C, c);  // dO [C][LD], slots 4-5
    __syncthreads();
    if constexpr (TC) {  // dV = P^T dO (+ the off-diagonal part from the per-key-chunk sums), P split
        typename WT<C, D>::Acc dv;
        WT<C, D>::zero(dv);
        mma_mul<C, D, C, true, true, true, false, 1>(dv, slot(3), LC, slot(4), LD);
        frag_out<D>(reinterpret_cast<__nv_bfloat16*>(p.dv) + hrow * D, dv, above ? p.dvoff + prow * D : nullptr, c);
    } else {
        typename GR::Acc dv;
        GR::zero(dv);
        mmul<C, D, C, false, true, true, false, 1>(dv, slot(3), LC, slot(4), LD);
        mstore_out<D>(static_cast<T*>(p.dv) + hrow * D, dv, above ? p.dvoff + prow * D : nullptr, c);
    }
    __syncthreads();
    if constexpr (TC) {  // dZ = -dKhat W^T and -dQbar W^T on the tensor cores, then dY = -dQbar W^T - dSs Km
        typename WT<C, C>::Acc dz, dy;
        WT<C, C>::zero(dz);
        WT<C, C>::zero(dy);
        // d in pieces of KH rows; piece h + 1 is loaded into registers while piece h's products run
        TileRegs<T, KH, C> rw;
        TileRegs<float, KH, C> rk, rq;
        auto fetch = [&](int h) {
            rw.load(w + h * KH, D, c);
            if (above) rk.load(p.dkhat + prow * D + h * KH, D, C);
            if (below) rq.load(p.dqbar + prow * D + h * KH, D, c);
        };
        auto place = [&]() {
            rw.store_t(slot(1), LC);
            if (above) rk.store_t(slot(3), LC);
            if (below) rq.store_t(slot(4), LC);
        };
        fetch(0);
        place();
        __syncthreads();
#pragma unroll 1
        for (int h = 0; h < NH; ++h) {
            if (h + 1 < NH) fetch(h + 1);
            if (above) mma_mul<C, C, KH, true, true, true, false>(dz, slot(3), LC, slot(1), LC);
            if (below) mma_mul<C, C, KH, true, true, true, false>(dy, slot(4), LC, slot(1), LC);
            __syncthreads();
            if (h + 1 < NH) {
                place();
                __syncthreads();
            }
        }
        mma_mul<C, C, C, false, true, true, true, 2>(dy, slot(0), LC, slot(11), LC);  // + dSs Km
        auto neg = [](int, int, float x) { return -x; };
        frag_store<C, C, true>(slot(1), LC, dz, neg);  // dZ^T -> slot 1 (until dA)
        frag_store<C, C>(slot(3), LC, dy, neg);        // dY -> slot 3 (until dA)
    } else {
        {  // dZ = -dKhat W^T, dY = -dQbar W^T - dSs Km
            typename GN::Acc dz, dy;
            GN::zero(dz);
            GN::zero(dy);
#pragma unroll 1
            for (int h = 0; h < NH; ++h) {
                to_smem_t<T, KH, kNTL>(slot(1), LC, w + h * KH, D, C, c);
                if (above) to_smem_t<float, KH, kNTL>(slot(3), LC, p.dkhat + prow * D + h * KH, D, C, C);
                if (below) to_smem_t<float, KH, kNTL>(slot(4), LC, p.dqbar + prow * D + h * KH, D, C, c);
                __syncthreads();
                if (above) mmul<C, C, KH, false, true, true>(dz, slot(3), LC, slot(1), LC);
                if (below) mmul<C, C, KH, false, true, true>(dy, slot(4), LC, slot(1), LC);
                __syncthreads();
            }
            mmul<C, C, C, false, false, true, false, 2>(dy, slot(0), LC, slot(11), LC);
            mstore<C, C, false, true>(slot(1), LC, dz, [](int, int, float x) { return -x; });   // dZ^T -> slot 1 (until dA)
            mstore<C, C, false, false>(slot(3), LC, dy, [](int, int, float x) { return -x; });  // dY -> slot 3 (until dA)
        }
    }
    __syncthreads();
    if constexpr (TC) {
        typename WT<C, C>::Acc dk, dq;
        WT<C, C>::zero(dk);
        WT<C, C>::zero(dq);
        mma_mul<C, C, C, true, false, true, true, 1, true>(dk, slot(0), LC, slot(12), LC);  // -dSs^T Y
        mma_mul<C, C, C, true, false, true, true>(dk, slot(1), LC, slot(8), LC);           // + dZ A^T
        mma_mul<C, C, C, false, true, true, true>(dq, slot(3), LC, slot(8), LC);           // dY A
        frag_store<C, C>(slot(4), LC, dk, [](int j, int a, float x) { return a > j ? x : 0.f; });   // dKw -> slot 4
        frag_store<C, C>(slot(5), LC, dq, [](int i, int bb, float x) { return bb <= i ? x : 0.f; });  // dQw -> slot 5
    } else {
        typename GS::Acc dk;
        GS::zero(dk);
        mmul<C, C, C, true, true, false, true>(dk, slot(0), LC, slot(12), LC);  // -dSs^T Y
        mmul<C, C, C, true, true, false>(dk, slot(1), LC, slot(8), LC);         // + dZ A^T
        mstore<C, C, true, false>(slot(4), LC, dk, [](int j, int a, float x) { return a > j ? x : 0.f; });  // dKw -> slot 4
        typename GN::Acc dq;
        GN::zero(dq);
        mmul<C, C, C, false, false, true>(dq, slot(3), LC, slot(8), LC);  // dY A
        mstore<C, C, false, false>(slot(5), LC, dq, [](int i, int bb, float x) { return bb <= i ? x : 0.f; });  // dQw -> slot 5
    }
    __syncthreads();
    if constexpr (TC) {  // dA = Km^T dZ + dY^T Qm - E;  dbeta from A = X D;  dX = dA D -> dX^T in slot 8
        using WC = WT<C, C>;
        typename WC::Acc da;
        WC::zero(da);
        mma_mul<C, C, C, true, false, true, true, 2>(da, slot(11), LC, slot(1), LC);
        mma_mul<C, C, C, true, false, true, true>(da, slot(3), LC, slot(10), LC);
        const float* sX = slot(7);
        float cs[WC::NT][2];
#pragma unroll
        for (int nt = 0; nt < WC::NT; ++nt) cs[nt][0] = cs[nt][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < WC::MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < WC::NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = WC::row(mt, i), col = WC::col(nt, i);
                    if (hasP) da[mt][nt][i] -= slot(9)[r * LC + col];
                    cs[nt][i & 1] = fmaf(sX[r * LC + col], da[mt][nt][i], cs[nt][i & 1]);
                }
#pragma unroll
        for (int nt = 0; nt < WC::NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) atomicAdd(aB + WC::col(nt, e), cs[nt][e]);
        frag_store<C, C, true>(slot(8), LC, da, [&](int, int bb, float x) { return x * sB[bb]; });
    } else {
        typename GS::Acc da;
        GS::zero(da);
        mmul<C, C, C, true, true, false>(da, slot(11), LC, slot(1), LC);
        mmul<C, C, C, true, true, false>(da, slot(3), LC, slot(10), LC);
        const int m0 = GS::m0(), n0 = GS::n0();
        const float* sX = slot(7);
#pragma unroll
        for (int j = 0; j < GS::TN; ++j) {
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < GS::TM; ++i) {
                if (hasP) da[i][j] -= slot(9)[(m0 + i) * LC + n0 + j];
                s = fmaf(sX[(m0 + i) * LC + n0 + j], da[i][j], s);
            }
            atomicAdd(aB + n0 + j, s);
        }
        mstore<C, C, true, true>(slot(8), LC, da, [&](int, int bb, float x) { return x * sB[bb]; });
    }
    __syncthreads();
    if constexpr (TC) {  // dM = -X^T (dX X^T);  dG = striu(D dM) stored as dG + dG^T
        using WC = WT<C, C>;
        typename WC::Acc t1, dm;
        WC::zero(t1);
        WC::zero(dm);
        mma_mul<C, C, C, true, false, true, true>(t1, slot(8), LC, slot(7), LC);
        frag_store<C, C>(slot(9), LC, t1);
        __syncthreads();
        mma_mul<C, C, C, true, true, true, true, 2, true>(dm, slot(7), LC, slot(9), LC);
        float* dG = slot(10);
        float rsum[WC::MT][2];
#pragma unroll
        for (int mt = 0; mt < WC::MT; ++mt) rsum[mt][0] = rsum[mt][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < WC::MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < WC::NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int a = WC::row(mt, i), bb = WC::col(nt, i);
                    const float v = dm[mt][nt][i];
                    if (bb > a) {
                        rsum[mt][i >> 1] = fmaf(v, slot(6)[a * LC + bb], rsum[mt][i >> 1]);
                        const float gv = sB[a] * v;
                        dG[a * LC + bb] = gv;
                        dG[bb * LC + a] = gv;
                    } else if (bb == a) {
                        dG[a * LC + a] = 0.f;
                    }
                }
#pragma unroll
        for (int mt = 0; mt < WC::MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) atomicAdd(aB + WC::row(mt, 2 * h), rsum[mt][h]);
    } else {
        typename GS::Acc t1;
        GS::zero(t1);
        mmul<C, C, C, true, true, false>(t1, slot(8), LC, slot(7), LC);
        mstore<C, C, true, false>(slot(9), LC, t1, id);
        __syncthreads();
        typename GN::Acc dm;
        GN::zero(dm);
        mmul<C, C, C, false, true, true, true, 2>(dm, slot(7), LC, slot(9), LC);
        const int m0 = GN::m0(), n0 = GN::n0();
        float* dG = slot(10);
#pragma unroll
        for (int i = 0; i < GN::TM; ++i) {
            const int a = m0 + i;
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < GN::TN; ++j) {
                const int bb = n0 + j;
                if (bb > a) {
                    s = fmaf(dm[i][j], slot(6)[a * LC + bb], s);
                    const float g = sB[a] * dm[i][j];
                    dG[a * LC + bb] = g;
                    dG[bb * LC + a] = g;
                } else if (bb == a) {
                    dG[a * LC + a] = 0.f;
                }
            }
            atomicAdd(aB + a, s);
        }
    }
    __syncthreads();
    if (below) to_smem_v<float, D, kNTL>(slot(6), LD, p.dqbar + prow * D, D, C, c);  // slots 6-7
    if (above) to_smem_v<float, D, kNTL>(slot(8), LD, p.dkhat + prow * D, D, C, C);  // slots 8-9
    __syncthreads();
    if constexpr (TC) {
        pq.load_r(q, D, c);  // q and k for the next phase, in flight meanwhile
        pk.load_r(k, D, c);
        if (below) mma_mul<C, D, C, false, true, true, true, 1, true>(aWf, slot(12), LC, slot(6), LD);  // -= Y^T dQbar
        if (above) mma_mul<C, D, C, true, true, true, true, 2, true>(aWf, slot(2), LC, slot(8), LD);    // -= Z^T dKhat
    } else {
        if (below) mmul<C, D, C, false, false, true, true, 1>(aW, slot(12), LC, slot(6), LD);  // -= Y^T dQbar
        if (above) mmul<C, D, C, false, true, true, true, 2>(aW, slot(2), LC, slot(8), LD);    // -= Z^T dKhat
    }
    __syncthreads();
    if constexpr (TC) {
        pq.store_r(slot(6), LD);
        pk.store_r(slot(8), LD);
    } else {
        to_smem_v<T, D, kNTL>(slot(6), LD, q, D, C, c);
        to_smem_v<T, D, kNTL>(slot(8), LD, k, D, C, c);
    }
    __syncthreads();
    if constexpr (TC) {  // the products with q, k and w on the tensor cores (their partners split)
        using WR = WT<C, D>;
        typename WR::Acc aQ, aK;
        auto& wq = aWf;
        WR::zero(aQ);
        WR::zero(aK);
        pq.load_r(w, D, c);  // w for the last products, in flight meanwhile
        mma_mul<C, D, C, true, true, true, false, 1>(wq, slot(5), LC, slot(6), LD);   // dQw^T Q
        mma_mul<C, D, C, true, true, true, false, 2>(wq, slot(4), LC, slot(8), LD);   // dKw^T K
        mma_mul<C, D, C, false, true, true, false, 2>(aQ, slot(0), LC, slot(8), LD);  // dSs K
        mma_mul<C, D, C, true, true, true, false, 1>(aK, slot(0), LC, slot(6), LD);   // dSs^T Q
        __syncthreads();
        pq.store_r(slot(6), LD);
        __syncthreads();
        mma_mul<C, D, C, true, true, true, false>(wq, slot(10), LC, slot(6), LD);      // (dG + dG^T) W
        mma_mul<C, D, C, false, true, true, false, 2>(aQ, slot(5), LC, slot(6), LD);  // dQw W
        mma_mul<C, D, C, false, true, true, false, 1>(aK, slot(4), LC, slot(6), LD);  // dKw W
        frag_out<D>(reinterpret_cast<__nv_bfloat16*>(p.dq) + hrow * D, aQ, below ? p.dqbar + prow * D : nullptr, c);
        frag_out<D>(reinterpret_cast<__nv_bfloat16*>(p.dk) + hrow * D, aK, above ? p.dkhat + prow * D : nullptr, c);
        frag_out<D>(reinterpret_cast<__nv_bfloat16*>(p.dw) + hrow * D, wq, nullptr, c);
    } else {
        typename GR::Acc aQ, aK;
        GR::zero(aQ);
        GR::zero(aK);
        mmul<C, D, C, false, true, true, false, 1>(aW, slot(5), LC, slot(6), LD);   // += dQw^T Q
        mmul<C, D, C, false, true, true, false, 2>(aW, slot(4), LC, slot(8), LD);   // += dKw^T K
        mmul<C, D, C, false, false, true, false, 2>(aQ, slot(0), LC, slot(8), LD);  // dSs K
        mmul<C, D, C, false, true, true, false, 1>(aK, slot(0), LC, slot(6), LD);   // dSs^T Q
        __syncthreads();
        to_smem_v<T, D, kNTL>(slot(6), LD, w, D, C, c);
        __syncthreads();
        mmul<C, D, C, false, true, true>(aW, slot(10), LC, slot(6), LD);   // += (dG + dG^T) W
        mmul<C, D, C, false, false, true, false, 2>(aQ, slot(5), LC, slot(6), LD);  // += dQw W
        mmul<C, D, C, false, false, true, false, 1>(aK, slot(4), LC, slot(6), LD);  // += dKw W
        mstore_out<D>(static_cast<T*>(p.dq) + hrow * D, aQ, below ? p.dqbar + prow * D : nullptr, c);
        mstore_out<D>(static_cast<T*>(p.dk) + hrow * D, aK, above ? p.dkhat + prow * D : nullptr, c);
        mstore_out<D>(static_cast<T*>(p.dw) + hrow * D, aW, nullptr, c);
    }
    __syncthreads();
    for (int r = threadIdx.x; r < c; r += kNTL) {
        p.dbeta[hrow + r] = aB[r];
        if (p.fox)
            p.dctot[prow + r] = aC[r] + (below ? p.dcrow[prow + r] : 0.f) - (above ? p.dccol[prow + r] : 0.f);
    }
}

// ------------------------------------------------------------------ FoX: dlog f_s = sum_{t >= s} dc_t
__global__ void __launch_bounds__(1024) bwd_fox_suffix(const float* __restrict__ dctot, int L, int Lp,
                                                       float* __restrict__ dlog_f) {
    __shared__ double warp_tot[32];
    __shared__ double carry_s;
    const int bh = blockIdx.x;
    const float* src = dctot + (size_t)bh * Lp;
    float* dst = dlog_f + (size_t)bh * L;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry_s = 0.0;
    __syncthreads();
    for (int base = 0; base < L; base += 1024) {
        const int s = L - 1 - (base + (int)threadIdx.x);  // walks from the end of the head
        double x = s >= 0 ? (double)src[s] : 0.0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) warp_tot[wid] = x;
        __syncthreads();
        if (wid == 0) {
            double t = warp_tot[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const double y = __shfl_up_sync(0xffffffffu, t, off);
                if (lane >= off) t += y;
            }
            warp_tot[lane] = t;
        }
        __syncthreads();
        const double carry = carry_s;
        const double pre = wid > 0 ? warp_tot[wid - 1] : 0.0;
        if (s >= 0) dst[s] = (float)(carry + pre + x);
        __syncthreads();
        if (threadIdx.x == 0) carry_s = carry + warp_tot[31];
        __syncthreads();
    }
}

template <typename T, int D>
cudaError_t launch_bwd_t(const BwdParams& p, int BH, const float* log_f, unsigned char* ws, cudaStream_t st) {
    using S = BwdSmem<D>;
    const size_t b_prep = S::prep * sizeof(float), b_chain = S::chain * sizeof(float),
                 b_reduce = S::reduce * sizeof(float), b_local = S::local * sizeof(float);
    cudaFuncSetAttribute(bwd_prep<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)b_prep);
    cudaFuncSetAttribute(bwd_chain<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)b_chain);
    cudaFuncSetAttribute(bwd_reduce<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)b_reduce);
    cudaFuncSetAttribute(bwd_local<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)b_local);
    if (log_f) {
        fox_cumsum<<<BH, 1024, 0, st>>>(log_f, p.L, p.Lp, p.cum);
        cudaMemsetAsync(p.dccol, 0, (size_t)BH * p.Lp * sizeof(float), st);  // bwd_chain adds column sums
        cudaMemsetAsync(p.dcrow, 0, (size_t)BH * p.Lp * sizeof(float), st);  // bwd_chain_tc adds two halves per row
    }
    bwd_prep<T, D><<<dim3(p.N, BH), kNTL, b_prep, st>>>(p);
    if (p.N >= 2) {
        if constexpr (sizeof(T) == 2 && D == 128) {  // bf16: tensor-core chains (csrc/bwd_tc.cu)
            cudaError_t e = launch_bwd_chain_tc(p.dO, p.v, p.khat16, p.phi, p.plo, p.pairs, p.qbar, p.lse, p.delta,
                                                p.cum, p.dqbar, p.dcrow, p.dccol, p.fox, BH, p.L, p.Lp, p.N,
                                                p.head_pairs, p.scale, reinterpret_cast<WsHeader*>(ws), st);
            if (e != cudaSuccess) return e;
        } else {
            mark_start(st);
            bwd_chain<T, D><<<dim3(p.N - 1, BH), kNT, b_chain, st>>>(p);
            mark_end(st);
        }
        if constexpr (sizeof(T) == 2 && D == 128) {  // bf16 pairs: tensor-core reduction (csrc/bwd_tc.cu)
            cudaError_t e = launch_bwd_reduce_tc(p.dO, p.pairs, p.dvoff, p.dkhat, p.dpm, BH, p.L, p.Lp, p.N,
                                                 p.head_pairs, p.scale, reinterpret_cast<WsHeader*>(ws), st);
            if (e != cudaSuccess) return e;
        } else {
            bwd_reduce<T, D><<<dim3(p.N - 1, BH), kNT, b_reduce, st>>>(p);
        }
    }
    bwd_local<T, D><<<dim3(p.N, BH), kNTL, b_local, st>>>(p);
    if (log_f) bwd_fox_suffix<<<BH, 1024, 0, st>>>(p.dctot, p.L, p.Lp, p.dlog_f);
    return cudaGetLastError();
}

}  // namespace

bool bwd_supported(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

cudaError_t attn_bwd(int dtype, int d, const void* q, const void* k, const void* v, const void* w,
                     const float* beta, const float* log_f, const void* o, const float* lse, const void* dO,
                     void* dq, void* dk, void* dv, void* dw, float* dbeta, float* dlog_f, int BH, int L,
                     float scale, unsigned char* ws, const BwdLayout& lay, cudaStream_t st) {
    BwdParams p;
    p.q = q; p.k = k; p.v = v; p.w = w; p.o = o; p.dO = dO;
    p.beta = beta; p.lse = lse;
    p.dq = dq; p.dk = dk; p.dv = dv; p.dw = dw; p.dbeta = dbeta; p.dlog_f = dlog_f;
    auto f = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
    p.qbar = f(lay.qbar); p.khat = f(lay.khat);
    p.pm = lay.pm ? f(lay.pm) : nullptr;
    p.pmt = lay.pmt ? f(lay.pmt) : nullptr;
    p.xinv = f(lay.xinv);
    p.delta = f(lay.delta); p.cum = f(lay.cum); p.dqbar = f(lay.dqbar); p.dkhat = f(lay.dkhat);
    p.dvoff = f(lay.dvoff); p.dpm = f(lay.dpm); p.dcrow = f(lay.dcrow); p.dccol = f(lay.dccol);
    p.dctot = f(lay.dctot); p.pairs = ws + lay.pairs;
    p.khat16 = lay.khat16 ? reinterpret_cast<__nv_bfloat16*>(ws + lay.khat16) : nullptr;
    p.phi = lay.phi ? reinterpret_cast<__nv_bfloat16*>(ws + lay.phi) : nullptr;
    p.plo = lay.plo ? reinterpret_cast<__nv_bfloat16*>(ws + lay.plo) : nullptr;
    p.L = L; p.Lp = lay.Lp; p.N = lay.N;
    p.pair_elems = lay.pair_elems; p.head_pairs = lay.head_pairs;
    p.scale = scale;
    p.fox = log_f != nullptr;
    cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(WsHeader), st);
    if (e != cudaSuccess) return e;
    const bool bf = dtype == PATH_BF16;
    switch (d) {
        case 16: return bf ? launch_bwd_t<__nv_bfloat16, 16>(p, BH, log_f, ws, st) : launch_bwd_t<float, 16>(p, BH, log_f, ws, st);
        case 32: return bf ? launch_bwd_t<__nv_bfloat16, 32>(p, BH, log_f, ws, st) : launch_bwd_t<float, 32>(p, BH, log_f, ws, st);
        case 64: return bf ? launch_bwd_t<__nv_bfloat16, 64>(p, BH, log_f, ws, st) : launch_bwd_t<float, 64>(p, BH, log_f, ws, st);
        case 128: return bf ? launch_bwd_t<__nv_bfloat16, 128>(p, BH, log_f, ws, st) : launch_bwd_t<float, 128>(p, BH, log_f, ws, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pathattn
