// PaTH forward with value-side transport, on CUDA cores (fp32 arithmetic).
//
// "Resumo Técnico: Por que Transformações Acumuladas Extrapolam?"
// (gist.science/pt/paper/2606.24975), §"Metodologia" 1: the route transport
// P_{j->i} is the product of the per-token steps from source j to query i;
// §"Principais Contribuições" 3 "Proteção do Lado de Valor": the same
// accumulated transport is applied to the values.  With the PaTH steps
// H_s = I - beta_s w_s w_s^T ("Resumo Técnico: Atenção PaTH", §2 "Mecanismo
// Central") the route operator of the logit is H_i ... H_{j+1}, so
//     o_i = sum_j softmax_j(s_i.) H_i ... H_{j+1} v_j,
// with the PaTH(-FoX) logits s_ij = scale k_j^T H_{j+1} ... H_i q_i (+ bias).
//
// Each warp takes a group of kVtRows consecutive query rows and walks their
// keys twice, the rows in lockstep so that every key, w and value row it loads
// serves all of them:
//   1. right to left, each query carried backwards (u <- H_j u): the logits,
//      staged in shared memory and written 32 at a time to the warp's slot of
//      the workspace, and each row's running maximum;
//   2. left to right, each output accumulated along the route
//      (acc <- H_j acc + alpha_ij v_j), which leaves o_i = acc; the weights
//      exp(s_ij - m_i) of 32 keys are formed at once, one per lane.
// A lane holds D/32 consecutive elements of every d-vector.  The per-step dot
// products of all rows are summed over the warp together: each butterfly level
// exchanges half of the values still held, so 2 x 4 sums take 9 shuffles
// instead of 40.  The next two key rows are loaded while the current one is
// processed.  The direct, unblocked form of the operator: a blockwise
// tensor-core version would carry per-chunk d x d route products, which this
// library does not implement.  No waits, no barriers between warps.
#include <algorithm>

#include "common.cuh"

namespace pathattn {

constexpr int kVtRows = 4;                        // query rows per warp
constexpr int kVtWarps = 8;                       // warps per CTA
constexpr int kVtSms = 152;
// Resident CTAs per SM.  Three CTAs cap the walks at 80 registers; at d = 128 that
// spills about 80 bytes a thread and still beats two CTAs without spills (125
// registers), since the walks are latency-bound.
__host__ __device__ constexpr int vt_ctas_per_sm(int) { return 3; }
constexpr size_t kVtScratchCap = size_t(256) << 20;  // logits scratch limit (bytes)

// E consecutive elements of one row, loaded and stored as one vector.
template <typename T, int E> struct alignas(E * sizeof(T)) Frag {
    T x[E];
    __device__ __forceinline__ float get(int e) const { return to_f<T>(x[e]); }
};
template <typename T, int E>
__device__ __forceinline__ Frag<T, E> load_frag(const T* p, bool ok) {
    if (ok) return *reinterpret_cast<const Frag<T, E>*>(p);
    Frag<T, E> z;
#pragma unroll
    for (int e = 0; e < E; ++e) z.x[e] = from_f<T>(0.f);
    return z;
}

// Sums 8 values over the warp; every lane returns the total of value (lane >> 2) & 7.
__device__ __forceinline__ float warp_sum_8(const float (&x)[8], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float y[4], z[2];
#pragma unroll
    for (int v = 0; v < 4; ++v)
        y[v] = (b4 ? x[v + 4] : x[v]) + __shfl_xor_sync(0xffffffffu, b4 ? x[v] : x[v + 4], 16);
#pragma unroll
    for (int v = 0; v < 2; ++v)
        z[v] = (b3 ? y[v + 2] : y[v]) + __shfl_xor_sync(0xffffffffu, b3 ? y[v] : y[v + 2], 8);
    float a = (b2 ? z[1] : z[0]) + __shfl_xor_sync(0xffffffffu, b2 ? z[0] : z[1], 4);
    a += __shfl_xor_sync(0xffffffffu, a, 2);
    a += __shfl_xor_sync(0xffffffffu, a, 1);
    return a;
}
// Sums 4 values over the warp; every lane returns the total of value (lane >> 3) & 3.
__device__ __forceinline__ float warp_sum_4(const float (&x)[4], int lane) {
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

// Launch plan shared by the workspace query and the launch: CTAs, the padded
// logits row (a multiple of 32) and the workspace bytes (header + one slot of
// kVtRows x Lp floats per warp).
struct VtPlan {
    int ctas;
    int Lp;
    size_t bytes;
};
static VtPlan vt_plan(long long BH, int L, int d) {
    VtPlan p;
    p.Lp = cdiv(L, 32) * 32;
    const long long groups = BH * cdiv(L, kVtRows);
    const size_t per_cta = (size_t)kVtWarps * kVtRows * p.Lp * sizeof(float);
    long long ctas = std::min<long long>((groups + kVtWarps - 1) / kVtWarps, (long long)kVtSms * vt_ctas_per_sm(d));
    ctas = std::min<long long>(ctas, std::max<long long>(1, (long long)(kVtScratchCap / per_cta)));
    p.ctas = (int)ctas;
    p.bytes = sizeof(WsHeader) + (size_t)ctas * per_cta;
    return p;
}

// grid (plan.ctas), kVtWarps warps.  Warp gw takes row groups gw, then 2W - 1 - gw,
// then 2W + gw, ... (W warps in all) of the list that runs from the last group of
// every head to the first, so the long rows go first and each warp's share of
// steps comes out nearly equal.
template <typename T, int D, bool FOX>
__global__ void __launch_bounds__(32 * kVtWarps, vt_ctas_per_sm(D)) path_fwd_vt_rows(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, const T* __restrict__ w,
    const float* __restrict__ beta, const float* __restrict__ log_f, T* __restrict__ o, float* __restrict__ lse,
    int BH, int L, int Lp, float scale, WsHeader* hdr, float* __restrict__ scratch, long long scratch_floats) {
    constexpr int E = D >= 32 ? D / 32 : 1;
    constexpr int R = kVtRows;
    static_assert(R == 4, "the shared staging holds one float4 per step");
    __shared__ float4 stage_all[kVtWarps][32];  // [step mod 32][row]: logits, then weights
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kVtWarps + warp;
    const int W = gridDim.x * kVtWarps;
    if (gw == 0 && lane == 0) hdr->status = 0;
    float4* st = stage_all[warp];
    float* slot = scratch + (size_t)gw * R * Lp;
    if (!in_bounds((long long)gw * R * Lp, (long long)R * Lp, scratch_floats, hdr, 225)) return;
    const bool lane_ok = lane * E < D;
    const int col = lane_ok ? lane * E : 0;
    const int r_l = lane >> 3;  // the row whose sums this lane holds after warp_sum_8 / warp_sum_4
    const int ngr = cdiv(L, R);
    const long long G = (long long)BH * ngr;

    for (long long band = 0; band * W < G; ++band) {
        const long long g = band * W + ((band & 1) ? (W - 1 - gw) : gw);
        if (g >= G) continue;
        const int bh = (int)(g % BH);
        const int i0 = (ngr - 1 - (int)(g / BH)) * R;
        const int imax = min(i0 + R, L) - 1;
        // 32-bit offsets from the kernel arguments (B*H*L*D < 2^31) keep the walks' registers low
        const int hr = bh * L;        // the head's first row
        const int ho = hr * D + col;  // element offset of the lane's first column in that row
        // the head's rows lie inside the [B*H, L, D] tensors (checked in the bounds-checked build only)
        if (!in_bounds((long long)hr * D, (long long)L * D, (long long)BH * L * D, hdr, 224)) return;
        int ir[R];  // last key of each row; -1 past the end of the sequence
#pragma unroll
        for (int r = 0; r < R; ++r) ir[r] = i0 + r <= imax ? i0 + r : -1;
        const int il = i0 + r_l <= imax ? i0 + r_l : -1;  // the last key of row r_l

        // walk 1: logits, each query carried backwards through H_i, H_{i-1}, ...
        float u[R][E];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const Frag<T, E> f = load_frag<T, E>(q + ho + (i0 + r) * D, lane_ok && ir[r] >= 0);
#pragma unroll
            for (int e = 0; e < E; ++e) u[r][e] = f.get(e);
        }
        float bias = 0.f, mx = -INFINITY;  // of row r_l: sum_{s=j+1..i} log f_s, running max
        Frag<T, E> kf0 = load_frag<T, E>(k + ho + imax * D, lane_ok);
        Frag<T, E> wf0 = load_frag<T, E>(w + ho + imax * D, lane_ok);
        float bf0 = beta[hr + imax], lf0 = FOX ? log_f[hr + imax] : 0.f;
        const int j1 = max(imax - 1, 0);
        Frag<T, E> kf1 = load_frag<T, E>(k + ho + j1 * D, lane_ok);
        Frag<T, E> wf1 = load_frag<T, E>(w + ho + j1 * D, lane_ok);
        float bf1 = beta[hr + j1], lf1 = FOX ? log_f[hr + j1] : 0.f;
#pragma unroll 2
        for (int j = imax; j >= 0; --j) {
            const Frag<T, E> kc = kf0, wc = wf0;
            const float bj = bf0, lfj = lf0;
            kf0 = kf1;
            wf0 = wf1;
            bf0 = bf1;
            lf0 = lf1;
            const int jn = max(j - 2, 0);
            kf1 = load_frag<T, E>(k + ho + jn * D, lane_ok);
            wf1 = load_frag<T, E>(w + ho + jn * D, lane_ok);
            bf1 = beta[hr + jn];
            if (FOX) lf1 = log_f[hr + jn];
            float x[2 * R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float a = 0.f, b = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    a = fmaf(kc.get(e), u[r][e], a);
                    b = fmaf(wc.get(e), u[r][e], b);
                }
                x[2 * r] = a;
                x[2 * r + 1] = b;
            }
            const float sum = warp_sum_8(x, lane);  // lanes 8r..8r+3: k_j . u_r; 8r+4..8r+7: w_j . u_r
            const float s = fmaf(scale, sum, bias);
            if (j <= il) {
                mx = fmaxf(mx, s);
                if (FOX) bias += lfj;
            }
            if ((lane & 7) == 0) reinterpret_cast<float*>(&st[j & 31])[r_l] = s;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float t = j <= ir[r] ? bj * __shfl_sync(0xffffffffu, sum, 8 * r + 4) : 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) u[r][e] = fmaf(-t, wc.get(e), u[r][e]);
            }
            if ((j & 31) == 0) {  // logits j .. j+31 of every row to the slot
                __syncwarp();
                const float4 sv = st[lane];
                slot[0 * Lp + j + lane] = sv.x;
                slot[1 * Lp + j + lane] = sv.y;
                slot[2 * Lp + j + lane] = sv.z;
                slot[3 * Lp + j + lane] = sv.w;
                __syncwarp();
            }
        }
        float m[R];
#pragma unroll
        for (int r = 0; r < R; ++r) m[r] = __shfl_sync(0xffffffffu, mx, 8 * r);

        // walk 2: the outputs carried forward along the route
        float acc[R][E], lsum[R], sn[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            lsum[r] = 0.f;
            sn[r] = slot[r * Lp + lane];  // same lane wrote it
#pragma unroll
            for (int e = 0; e < E; ++e) acc[r][e] = 0.f;
        }
        wf0 = load_frag<T, E>(w + ho, lane_ok);
        Frag<T, E> vf0 = load_frag<T, E>(v + ho, lane_ok);
        bf0 = beta[hr];
        const int j2 = min(1, imax);
        wf1 = load_frag<T, E>(w + ho + j2 * D, lane_ok);
        Frag<T, E> vf1 = load_frag<T, E>(v + ho + j2 * D, lane_ok);
        bf1 = beta[hr + j2];
#pragma unroll 2
        for (int j = 0; j <= imax; ++j) {
            if ((j & 31) == 0) {  // weights of keys j .. j+31, one per lane
                float ew[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    ew[r] = j + lane <= ir[r] ? expf(sn[r] - m[r]) : 0.f;
                    lsum[r] += ew[r];
                    if (j + 32 <= imax) sn[r] = slot[r * Lp + j + 32 + lane];
                }
                __syncwarp();
                st[lane] = make_float4(ew[0], ew[1], ew[2], ew[3]);
                __syncwarp();
            }
            const Frag<T, E> wc = wf0, vc = vf0;
            const float bj = bf0;
            wf0 = wf1;
            vf0 = vf1;
            bf0 = bf1;
            const int jn = min(j + 2, imax);
            wf1 = load_frag<T, E>(w + ho + jn * D, lane_ok);
            vf1 = load_frag<T, E>(v + ho + jn * D, lane_ok);
            bf1 = beta[hr + jn];
            const float4 a4 = st[j & 31];
            const float a[R] = {a4.x, a4.y, a4.z, a4.w};
            float x[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float p = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) p = fmaf(wc.get(e), acc[r][e], p);
                x[r] = p;
            }
            const float sum = warp_sum_4(x, lane);  // lanes 8r..8r+7: w_j . acc_r
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float t = j <= ir[r] ? bj * __shfl_sync(0xffffffffu, sum, 8 * r) : 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[r][e] = fmaf(a[r], vc.get(e), fmaf(-t, wc.get(e), acc[r][e]));
            }
        }
        const float ltot = warp_sum_4(lsum, lane);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float l = __shfl_sync(0xffffffffu, ltot, 8 * r);
            if (ir[r] < 0) continue;
            const float inv_l = 1.f / l;
            if (lane_ok) {
                Frag<T, E> f;
#pragma unroll
                for (int e = 0; e < E; ++e) f.x[e] = from_f<T>(acc[r][e] * inv_l);
                *reinterpret_cast<Frag<T, E>*>(o + ho + (i0 + r) * D) = f;
            }
            if (lse && lane == 0) lse[hr + i0 + r] = m[r] + logf(l);
        }
        __syncwarp();  // the next group's staging writes come after every lane's reads
    }
}

bool fwd_vt_supported(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

cudaError_t fwd_tc_vt_bf16(const void* q, const void* k, const void* v, const void* w, const float* beta,
                           const float* log_f, void* o, float* lse, int BH, int L, float scale, unsigned char* ws,
                           const VtBlockLayout& vl, cudaStream_t st);

// bf16 at d = 128 runs the blockwise form (csrc/fwd_tc.cu, fwd_tc_vt_bf16: the UT prep
// and the scan on the tensor cores, the value chains and the diagonal walks of
// csrc/fwd_vt_block.cu) while its workspace, dominated by the pair store of O(L^2 d)
// bytes per head, stays under 64 GB; every other case runs the row walks above.
constexpr size_t kVtBlockCap = size_t(64) << 30;
static bool vt_blockwise(int dtype, int d, long long BH, int L, VtBlockLayout* out) {
    if (dtype != PATH_BF16 || d != 128 || BH > 65535) return false;
    const VtBlockLayout v = vt_block_layout(1, (int)BH, L, 128);
    if (v.total > kVtBlockCap) return false;
    if (out) *out = v;
    return true;
}

size_t fwd_vt_workspace_bytes(long long BH, int L, int d, int dtype) {
    VtBlockLayout vl;
    if (vt_blockwise(dtype, d, BH, L, &vl)) return vl.total;
    return vt_plan(BH, L, d).bytes;
}

template <typename T, int D, bool FOX>
static cudaError_t launch_vt(const void* q, const void* k, const void* v, const void* w, const float* beta,
                             const float* log_f, void* o, float* lse, int BH, int L, float scale, unsigned char* ws,
                             cudaStream_t st) {
    const VtPlan p = vt_plan(BH, L, D);
    const long long scratch_floats = (long long)((p.bytes - sizeof(WsHeader)) / sizeof(float));
    mark_start(st);
    path_fwd_vt_rows<T, D, FOX><<<p.ctas, 32 * kVtWarps, 0, st>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), static_cast<const T*>(w),
        beta, log_f, static_cast<T*>(o), lse, BH, L, p.Lp, scale, reinterpret_cast<WsHeader*>(ws),
        reinterpret_cast<float*>(ws + sizeof(WsHeader)), scratch_floats);
    mark_end(st);
    return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t launch_vt_f(const void* q, const void* k, const void* v, const void* w, const float* beta,
                               const float* log_f, void* o, float* lse, int BH, int L, float scale,
                               unsigned char* ws, cudaStream_t st) {
    if (log_f) return launch_vt<T, D, true>(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, st);
    return launch_vt<T, D, false>(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, st);
}

template <typename T>
static cudaError_t launch_vt_d(int d, const void* q, const void* k, const void* v, const void* w, const float* beta,
                               const float* log_f, void* o, float* lse, int BH, int L, float scale,
                               unsigned char* ws, cudaStream_t st) {
    switch (d) {
        case 16: return launch_vt_f<T, 16>(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, st);
        case 32: return launch_vt_f<T, 32>(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, st);
        case 64: return launch_vt_f<T, 64>(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, st);
        case 128: return launch_vt_f<T, 128>(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t fwd_vt(int dtype, int d, const void* q, const void* k, const void* v, const void* w, const float* beta,
                   const float* log_f, void* o, float* lse, int BH, int L, float scale, unsigned char* ws,
                   cudaStream_t st) {
    VtBlockLayout vl;
    if (vt_blockwise(dtype, d, BH, L, &vl))
        return fwd_tc_vt_bf16(q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, vl, st);
    if (dtype == PATH_F32) return launch_vt_d<float>(d, q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, st);
    return launch_vt_d<__nv_bfloat16>(d, q, k, v, w, beta, log_f, o, lse, BH, L, scale, ws, st);
}

}  // namespace pathattn
