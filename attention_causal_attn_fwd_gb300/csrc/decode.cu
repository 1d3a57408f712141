// PaTH decode on GB300: in-place key transport fused with split-K one-query
// attention ("Resumo Técnico: Atenção PaTH", gist.science/pt/paper/2505.16381,
// §3 "Inferência": the historical keys are updated in place with the current
// step's transition H_t = I - beta_t w_t w_t^T, after which decoding is
// ordinary attention over the cache, as in FlashDecoding).
//
// The step is HBM-bound: every cached key row is read, transported, written
// back and scored, and every value row is read — 3 * n * d * sizeof(T) bytes
// per head.  Each row is d * sizeof(T) bytes, moved as 16-byte vectors: LPR
// lanes per row, 32 / LPR rows per warp, several rows per lane in flight.
#include "common.cuh"

namespace pathattn {

template <typename T, int D>
struct DecGeom {
    static constexpr int EPL = 16 / sizeof(T);  // elements per lane (one 16-byte vector)
    static constexpr int LPR = D / EPL;          // lanes per row
    static constexpr int RPW = 32 / LPR;         // rows per warp
    static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "row must be 16..512 bytes");
};

template <int LPR>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// k <- k - beta (w.k) w  in fp32, rounded to T; returns the rounded vector.
template <typename T, int D>
__device__ __forceinline__ Vec16<T> transport(const Vec16<T>& kv, const float* wv, float beta) {
    using G = DecGeom<T, D>;
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < G::EPL; ++e) part = fmaf(wv[e], kv.get(e), part);
    const float t = beta * group_sum<G::LPR>(part);
    Vec16<T> out;
#pragma unroll
    for (int e = 0; e < G::EPL; ++e) out.set(e, fmaf(-t, wv[e], kv.get(e)));
    return out;
}

constexpr int kDecNT = 256;
constexpr int kDecUnroll = 8;

// grid (splits, B*H).  Split s covers cache rows [s*R, min((s+1)*R, n_cached+1));
// row n_cached is the new token.  Writes per-split (m, l, o) in log2 units.
// VT: value-side transport ("Resumo Técnico: Por que Transformações Acumuladas
// Extrapolam?", §"Principais Contribuições" 3): the cached values are carried
// along the same route as the keys, v~_j <- H_t v~_j in place, and the step
// attends to the stored (transported) values.  The value transport needs a
// few more registers; VT builds are held to 128 (two CTAs per SM, the memory
// parallelism the step depends on) at the cost of a 12-byte spill.
template <typename T, int D, bool VT = false>
__global__ void __launch_bounds__(kDecNT, VT ? 2 : 0) decode_update_score(
    const T* __restrict__ q_t, const T* __restrict__ k_t, const T* __restrict__ v_t, const T* __restrict__ w_t,
    const float* __restrict__ beta_t, T* __restrict__ kcache, T* __restrict__ vcache, int n_cached, int n_max,
    float scale_log2, float* __restrict__ part_m, float* __restrict__ part_l, float* __restrict__ part_o,
    WsHeader* hdr) {
    using G = DecGeom<T, D>;
    constexpr int NW = kDecNT / 32;
    constexpr int NG = NW * G::RPW;  // row groups per CTA
    __shared__ float s_m[NG], s_l[NG];
    __shared__ float s_o[NG][D + 1];

    const int split = blockIdx.x, bh = blockIdx.y, nsplit = gridDim.x;
    if (split == 0 && bh == 0 && threadIdx.x == 0) hdr->status = 0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane / G::LPR, li = lane % G::LPR;
    const int grp = warp * G::RPW + sub;
    const int total = n_cached + 1;
    const int j0 = split * kDecodeRowsPerSplit;
    const int j1 = min(j0 + kDecodeRowsPerSplit, total);

    const size_t hv = (size_t)bh * D + li * G::EPL;  // this lane's slice of a [B,H,D] vector
    const long long n_bh = gridDim.y, n_cache = (long long)gridDim.y * n_max * D;
    const bool hv_ok = in_bounds((long long)hv, G::EPL, n_bh * D, hdr, 220);
    float wv[G::EPL], qv[G::EPL];
    {
        Vec16<T> a, b;
        a.raw = hv_ok ? ld_global_v4(w_t + hv) : make_uint4(0, 0, 0, 0);
        b.raw = hv_ok ? ld_global_v4(q_t + hv) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int e = 0; e < G::EPL; ++e) {
            wv[e] = a.get(e);
            qv[e] = b.get(e);
        }
    }
    const float beta = beta_t[bh];
    T* kh = kcache + (size_t)bh * n_max * D + li * G::EPL;
    T* vh = vcache + (size_t)bh * n_max * D + li * G::EPL;

    float m = -INFINITY, l = 0.f, acc[G::EPL];
#pragma unroll
    for (int e = 0; e < G::EPL; ++e) acc[e] = 0.f;

    constexpr int STRIDE = NG;  // rows between consecutive rows of one group
    // The trip count must be warp-uniform (the row reductions shuffle across
    // the whole warp), so the loop runs on the warp's first row and each group
    // masks its own rows.
    for (int wbase = j0 + warp * G::RPW; wbase < j1; wbase += STRIDE * kDecUnroll) {
        const int base = wbase + sub;
        Vec16<T> kvec[kDecUnroll], vvec[kDecUnroll];
#pragma unroll
        for (int u = 0; u < kDecUnroll; ++u) {
            const int j = base + u * STRIDE;
            const bool row_ok = j < j1 && in_bounds(((long long)bh * n_max + j) * D + li * G::EPL, G::EPL, n_cache, hdr, 221);
            if (row_ok) {
                if (j < n_cached) {
                    kvec[u].raw = ld_global_stream_v4(kh + (size_t)j * D);
                    vvec[u].raw = ld_global_stream_v4(vh + (size_t)j * D);
                } else {  // the new token: appended untransported
                    kvec[u].raw = hv_ok ? ld_global_v4(k_t + hv) : make_uint4(0, 0, 0, 0);
                    vvec[u].raw = hv_ok ? ld_global_v4(v_t + hv) : make_uint4(0, 0, 0, 0);
                }
            } else {
                kvec[u].raw = make_uint4(0, 0, 0, 0);
                vvec[u].raw = make_uint4(0, 0, 0, 0);
            }
        }
        float s[kDecUnroll];
        float mx = m;
#pragma unroll
        for (int u = 0; u < kDecUnroll; ++u) {
            const int j = base + u * STRIDE;
            const Vec16<T> tr = transport<T, D>(kvec[u], wv, beta);  // all lanes shuffle
            const Vec16<T> kn = (j < n_cached) ? tr : kvec[u];
            if (VT) {
                const Vec16<T> trv = transport<T, D>(vvec[u], wv, beta);  // all lanes shuffle
                if (j < n_cached) vvec[u] = trv;
            }
            if (j < j1 && in_bounds(((long long)bh * n_max + j) * D + li * G::EPL, G::EPL, n_cache, hdr, 222)) {
                st_global_v4(kh + (size_t)j * D, kn.raw);
                if (VT || j == n_cached) st_global_v4(vh + (size_t)j * D, vvec[u].raw);
            }
            float part = 0.f;
#pragma unroll
            for (int e = 0; e < G::EPL; ++e) part = fmaf(qv[e], kn.get(e), part);
            const float dotp = group_sum<G::LPR>(part);  // all lanes shuffle
            s[u] = j < j1 ? dotp * scale_log2 : -INFINITY;
            mx = fmaxf(mx, s[u]);
        }
        if (mx != -INFINITY) {  // false only when none of this group's rows is valid
            const float corr = exp2f(m - mx);
            l *= corr;
#pragma unroll
            for (int e = 0; e < G::EPL; ++e) acc[e] *= corr;
#pragma unroll
            for (int u = 0; u < kDecUnroll; ++u) {
                const float p = exp2f(s[u] - mx);
                l += p;
#pragma unroll
                for (int e = 0; e < G::EPL; ++e) acc[e] = fmaf(p, vvec[u].get(e), acc[e]);
            }
            m = mx;
        }
    }

    if (li == 0) {
        s_m[grp] = m;
        s_l[grp] = l;
    }
#pragma unroll
    for (int e = 0; e < G::EPL; ++e) s_o[grp][li * G::EPL + e] = acc[e];
    __syncthreads();
    float M = -INFINITY;
    for (int g = 0; g < NG; ++g) M = fmaxf(M, s_m[g]);
    const size_t pi = (size_t)bh * nsplit + split;
    for (int c = threadIdx.x; c < D; c += kDecNT) {
        float o = 0.f;
        for (int g = 0; g < NG; ++g)
            if (s_m[g] != -INFINITY) o += s_o[g][c] * exp2f(s_m[g] - M);
        if (in_bounds((long long)pi * D + c, 1, (long long)gridDim.y * nsplit * D, hdr, 223)) part_o[pi * D + c] = o;
    }
    if (threadIdx.x == 0) {
        float L = 0.f;
        for (int g = 0; g < NG; ++g)
            if (s_m[g] != -INFINITY) L += s_l[g] * exp2f(s_m[g] - M);
        part_m[pi] = M;
        part_l[pi] = L;
    }
}

// grid B*H, block D threads: log-sum-exp merge of the split partials.
template <typename T, int D>
__global__ void __launch_bounds__(128) decode_combine(const float* __restrict__ part_m,
                                                     const float* __restrict__ part_l,
                                                     const float* __restrict__ part_o, int nsplit,
                                                     T* __restrict__ o_t, float* __restrict__ lse_t) {
    const int bh = blockIdx.x;
    const float* pm = part_m + (size_t)bh * nsplit;
    const float* pl = part_l + (size_t)bh * nsplit;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, pm[s]);
    float L = 0.f;
    for (int s = 0; s < nsplit; ++s) L += pl[s] * exp2f(pm[s] - M);
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < nsplit; ++s) acc += part_o[((size_t)bh * nsplit + s) * D + c] * exp2f(pm[s] - M);
        o_t[(size_t)bh * D + c] = from_f<T>(acc / L);
    }
    if (lse_t && threadIdx.x == 0) lse_t[bh] = (M + log2f(L)) * 0.6931471805599453f;
}

// The in-place transport alone: grid (splits, B*H).
template <typename T, int D>
__global__ void __launch_bounds__(kDecNT) kcache_update(T* __restrict__ kcache, int n_cached, int n_max,
                                                        const T* __restrict__ w_t,
                                                        const float* __restrict__ beta_t) {
    using G = DecGeom<T, D>;
    constexpr int NG = (kDecNT / 32) * G::RPW;
    const int split = blockIdx.x, bh = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane / G::LPR, li = lane % G::LPR;
    const int j0 = split * kDecodeRowsPerSplit;
    const int j1 = min(j0 + kDecodeRowsPerSplit, n_cached);
    float wv[G::EPL];
    {
        Vec16<T> a;
        a.raw = ld_global_v4(w_t + (size_t)bh * D + li * G::EPL);
#pragma unroll
        for (int e = 0; e < G::EPL; ++e) wv[e] = a.get(e);
    }
    const float beta = beta_t[bh];
    T* kh = kcache + (size_t)bh * n_max * D + li * G::EPL;
    for (int wbase = j0 + warp * G::RPW; wbase < j1; wbase += NG * kDecUnroll) {  // warp-uniform trip count
        const int base = wbase + sub;
        Vec16<T> kvec[kDecUnroll];
#pragma unroll
        for (int u = 0; u < kDecUnroll; ++u) {
            const int j = base + u * NG;
            kvec[u].raw = j < j1 ? ld_global_stream_v4(kh + (size_t)j * D) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kDecUnroll; ++u) {
            const int j = base + u * NG;
            Vec16<T> kn = transport<T, D>(kvec[u], wv, beta);
            if (j < j1) st_global_v4(kh + (size_t)j * D, kn.raw);
        }
    }
}

// ----------------------------------------------------------------------------- host launchers
template <typename T, int D>
static cudaError_t launch_decode_t(const void* q_t, const void* k_t, const void* v_t, const void* w_t,
                                   const float* beta_t, void* kcache, void* vcache, int n_cached, int n_max,
                                   void* o_t, float* lse_t, int BH, float scale, unsigned char* ws,
                                   const DecLayout& lay, bool vt, cudaStream_t st) {
    const int nsplit = decode_splits(n_cached + 1);
    float* pm = reinterpret_cast<float*>(ws + lay.part_m);
    float* pl = reinterpret_cast<float*>(ws + lay.part_l);
    float* po = reinterpret_cast<float*>(ws + lay.part_o);
    auto kern = vt ? decode_update_score<T, D, true> : decode_update_score<T, D, false>;
    mark_start(st);
    kern<<<dim3(nsplit, BH), kDecNT, 0, st>>>(
        static_cast<const T*>(q_t), static_cast<const T*>(k_t), static_cast<const T*>(v_t),
        static_cast<const T*>(w_t), beta_t, static_cast<T*>(kcache), static_cast<T*>(vcache), n_cached, n_max,
        scale * 1.4426950408889634f, pm, pl, po, reinterpret_cast<WsHeader*>(ws));
    mark_end(st);
    decode_combine<T, D><<<BH, D < 128 ? D : 128, 0, st>>>(pm, pl, po, nsplit, static_cast<T*>(o_t), lse_t);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_decode_d(int d, const void* q_t, const void* k_t, const void* v_t, const void* w_t,
                                   const float* beta_t, void* kc, void* vc, int n_cached, int n_max, void* o_t,
                                   float* lse_t, int BH, float scale, unsigned char* ws, const DecLayout& lay,
                                   bool vt, cudaStream_t st) {
    switch (d) {
        case 16: return launch_decode_t<T, 16>(q_t, k_t, v_t, w_t, beta_t, kc, vc, n_cached, n_max, o_t, lse_t, BH, scale, ws, lay, vt, st);
        case 32: return launch_decode_t<T, 32>(q_t, k_t, v_t, w_t, beta_t, kc, vc, n_cached, n_max, o_t, lse_t, BH, scale, ws, lay, vt, st);
        case 64: return launch_decode_t<T, 64>(q_t, k_t, v_t, w_t, beta_t, kc, vc, n_cached, n_max, o_t, lse_t, BH, scale, ws, lay, vt, st);
        case 128: return launch_decode_t<T, 128>(q_t, k_t, v_t, w_t, beta_t, kc, vc, n_cached, n_max, o_t, lse_t, BH, scale, ws, lay, vt, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t decode_step(int dtype, int d, const void* q_t, const void* k_t, const void* v_t, const void* w_t,
                        const float* beta_t, void* kc, void* vc, int n_cached, int n_max, void* o_t, float* lse_t,
                        int BH, float scale, unsigned char* ws, const DecLayout& lay, bool vt, cudaStream_t st) {
    if (dtype == PATH_F32)
        return launch_decode_d<float>(d, q_t, k_t, v_t, w_t, beta_t, kc, vc, n_cached, n_max, o_t, lse_t, BH, scale, ws, lay, vt, st);
    return launch_decode_d<__nv_bfloat16>(d, q_t, k_t, v_t, w_t, beta_t, kc, vc, n_cached, n_max, o_t, lse_t, BH, scale, ws, lay, vt, st);
}

template <typename T>
static cudaError_t launch_update_t(int d, void* kc, int n_cached, int n_max, const void* w_t, const float* beta_t,
                                   int BH, cudaStream_t st) {
    if (n_cached == 0) return cudaSuccess;
    const dim3 grid(decode_splits(n_cached), BH);
    T* k = static_cast<T*>(kc);
    const T* w = static_cast<const T*>(w_t);
    switch (d) {
        case 16: kcache_update<T, 16><<<grid, kDecNT, 0, st>>>(k, n_cached, n_max, w, beta_t); break;
        case 32: kcache_update<T, 32><<<grid, kDecNT, 0, st>>>(k, n_cached, n_max, w, beta_t); break;
        case 64: kcache_update<T, 64><<<grid, kDecNT, 0, st>>>(k, n_cached, n_max, w, beta_t); break;
        case 128: kcache_update<T, 128><<<grid, kDecNT, 0, st>>>(k, n_cached, n_max, w, beta_t); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t kcache_update_launch(int dtype, int d, void* kc, int n_cached, int n_max, const void* w_t,
                                 const float* beta_t, int BH, cudaStream_t st) {
    if (dtype == PATH_F32) return launch_update_t<float>(d, kc, n_cached, n_max, w_t, beta_t, BH, st);
    return launch_update_t<__nv_bfloat16>(d, kc, n_cached, n_max, w_t, beta_t, BH, st);
}

}  // namespace pathattn

// ----------------------------------------------------------------------------- allocation-free decode step
// Scratch for path_decode_step_noalloc: the split-K partials and the status
// header live in this file-scope device array instead of a caller workspace.
// Every GPU that loads the library holds it until the process exits.
#include <cuda.h>

#include <cstdio>
#include <mutex>

namespace pathattn {

static __device__ __align__(256) unsigned char g_decode_scratch[PATH_DECODE_NOALLOC_SCRATCH_BYTES];

// Unique id of the current device's primary context (driver entry points
// fetched through the runtime, so the library does not link libcuda).  It
// changes when the context is destroyed and recreated (cudaDeviceReset), which
// unloads the module and with it the array.
static bool current_context_id(unsigned long long* id) {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    if (!get_current || !get_id) {
        void* a = nullptr;
        void* b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) != cudaSuccess ||
            qa != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) != cudaSuccess ||
            qb != cudaDriverEntryPointSuccess)
            return false;
        get_current = reinterpret_cast<GetCurrent>(a);
        get_id = reinterpret_cast<GetId>(b);
    }
    CUcontext ctx = nullptr;
    return get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr && get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_decode_scratch for the current device, looked up once per
// device (and again after the device's context has been reset).  In host code
// the array's name is only a host-side stand-in, so the kernels are given this
// address instead.
static int noalloc_scratch_address(unsigned char** out) {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    static unsigned long long ctx_id[kMaxDevices] = {};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return PATH_ERR_CUDA;
    if (dev >= kMaxDevices) return PATH_ERR_UNSUPPORTED;
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);  // false while no context is current on this thread
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] || !have_id || ctx_id[dev] != id) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || p == nullptr) {
            std::fprintf(stderr, "pathattn: cudaGetSymbolAddress for the decode scratch failed: %s\n",
                         cudaGetErrorString(e));
            return PATH_ERR_CUDA;
        }
        // the lookup made the device's context current: record which one the address belongs to
        if (!current_context_id(&id)) return PATH_ERR_CUDA;
        addr[dev] = p;
        ctx_id[dev] = id;
    }
    *out = static_cast<unsigned char*>(addr[dev]);
    return PATH_OK;
}

static bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace pathattn

extern "C" int path_decode_step_noalloc(const void* q_t, const void* k_t, const void* v_t, const void* w_t,
                                        const float* beta_t, void* kcache, void* vcache, int n_cached, int n_max,
                                        void* o_t, float* lse_t, int B, int H, int d, float scale, int dtype,
                                        path_stream_t stream) {
    using namespace pathattn;
    if (B < 1 || H < 1 || n_max < 1 || n_cached < 0) return PATH_ERR_INVALID;
    if (n_cached + 1 > n_max) return PATH_ERR_INVALID;
    if (dtype != PATH_F32 && dtype != PATH_BF16) return PATH_ERR_UNSUPPORTED;
    if (d != 16 && d != 32 && d != 64 && d != 128) return PATH_ERR_UNSUPPORTED;
    if ((long long)B * H > 65535) return PATH_ERR_UNSUPPORTED;
    if (!q_t || !k_t || !v_t || !w_t || !beta_t || !kcache || !vcache || !o_t) return PATH_ERR_INVALID;
    const void* ptrs[] = {q_t, k_t, v_t, w_t, kcache, vcache, o_t};
    for (const void* p : ptrs)
        if (!al16(p)) return PATH_ERR_INVALID;
    const DecLayout lay = dec_layout(B, H, n_max, d);
    if (lay.total > (size_t)PATH_DECODE_NOALLOC_SCRATCH_BYTES) {
        std::fprintf(stderr,
                     "pathattn: path_decode_step_noalloc needs %zu bytes of scratch for B=%d H=%d n_max=%d d=%d, "
                     "more than its built-in %zu bytes; use path_decode_step with a caller workspace\n",
                     lay.total, B, H, n_max, d, (size_t)PATH_DECODE_NOALLOC_SCRATCH_BYTES);
        return PATH_ERR_WORKSPACE;
    }
    unsigned char* ws = nullptr;
    const int rc = noalloc_scratch_address(&ws);
    if (rc != PATH_OK) return rc;
    const cudaError_t e = decode_step(dtype, d, q_t, k_t, v_t, w_t, beta_t, kcache, vcache, n_cached, n_max, o_t,
                                      lse_t, B * H, scale, ws, lay, false, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PATH_OK : PATH_ERR_CUDA;
}
