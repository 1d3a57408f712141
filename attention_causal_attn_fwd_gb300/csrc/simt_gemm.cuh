// Small shared-memory GEMM for one thread block (fp32 CUDA-core FMA).
// out(m, n) = sum_k a(m, k) * b(k, n), register-tiled: each of the NT threads
// owns a TM x TN sub-tile with rows strided by M/TM and columns by N/TN, so the
// threads of a warp read consecutive columns of b and broadcast rows of a.
#pragma once

namespace pathattn {

template <int M, int N, int NT>
struct GemmTile {
    static constexpr int TOT = M * N / NT;
    static constexpr int TN = TOT >= 64 ? 8 : (TOT >= 16 ? 4 : (TOT >= 4 ? 2 : 1));
    static constexpr int TM = TOT / TN;
    static constexpr int GN = N / TN;
    static constexpr int GM = M / TM;
    static_assert(M * N % NT == 0 && TOT >= 1, "tile must cover the block");
    static_assert(GM * GN == NT && GM * TM == M && GN * TN == N, "bad gemm tiling");
};

// Accumulates over k in [0, K); `epi(m, n, acc)` runs after a barrier, so it
// may overwrite the operands; a second barrier follows it.
template <int M, int N, int K, int NT, class LA, class LB, class EPI>
__device__ __forceinline__ void block_gemm(const LA& a, const LB& b, const EPI& epi) {
    using G = GemmTile<M, N, NT>;
    const int tm = threadIdx.x / G::GN, tn = threadIdx.x % G::GN;
    float acc[G::TM][G::TN];
#pragma unroll
    for (int i = 0; i < G::TM; ++i)
#pragma unroll
        for (int j = 0; j < G::TN; ++j) acc[i][j] = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < K; ++kk) {
        float av[G::TM], bv[G::TN];
#pragma unroll
        for (int i = 0; i < G::TM; ++i) av[i] = a(tm + i * G::GM, kk);
#pragma unroll
        for (int j = 0; j < G::TN; ++j) bv[j] = b(kk, tn + j * G::GN);
#pragma unroll
        for (int i = 0; i < G::TM; ++i)
#pragma unroll
            for (int j = 0; j < G::TN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < G::TM; ++i)
#pragma unroll
        for (int j = 0; j < G::TN; ++j) epi(tm + i * G::GM, tn + j * G::GN, acc[i][j]);
    __syncthreads();
}

}  // namespace pathattn
