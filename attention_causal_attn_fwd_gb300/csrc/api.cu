// C ABI of libpathattn.so (declarations and contracts in include/path_attn.h).
// Host side only: argument validation, workspace carve-up and kernel dispatch.
// Nothing here allocates device memory; every launch goes to the caller's stream.
#include <atomic>
#include <cstddef>
#include <cstdio>

#include "common.cuh"

namespace pathattn {
int simt_chunk(int d);
cudaError_t fwd_simt_f32(const void* q, const void* k, const void* v, const void* w, const float* beta,
                         const float* log_f, const float* rel_bias, int H, void* o, float* lse, int BH, int L, int d,
                         float scale, unsigned char* ws, const FwdLayout& lay, cudaStream_t st);
int tc_chunk(int d);
bool tc_supported(int d);
cudaError_t fwd_tc_bf16(const void* q, const void* k, const void* v, const void* w, const float* beta,
                        const float* log_f, const float* rel_bias, int H, void* o, float* lse, int BH, int L, int d,
                        float scale, unsigned char* ws, const FwdLayout& lay, int fault_mask, const FwdOptions& opt,
                        cudaStream_t st);
cudaError_t prefill_kcache(int dtype, int C, int d, const void* k, const void* w, const float* beta, void* kcache,
                           int BH, int L, int n_max, unsigned char* ws, const FwdLayout& lay, cudaStream_t st);
cudaError_t decode_step(int dtype, int d, const void* q_t, const void* k_t, const void* v_t, const void* w_t,
                        const float* beta_t, void* kc, void* vc, int n_cached, int n_max, void* o_t, float* lse_t,
                        int BH, float scale, unsigned char* ws, const DecLayout& lay, bool vt, cudaStream_t st);
bool fwd_vt_supported(int d);
size_t fwd_vt_workspace_bytes(long long BH, int L, int d, int dtype);
cudaError_t fwd_vt(int dtype, int d, const void* q, const void* k, const void* v, const void* w, const float* beta,
                   const float* log_f, void* o, float* lse, int BH, int L, float scale, unsigned char* ws,
                   cudaStream_t st);
bool bwd_supported(int d);
cudaError_t attn_bwd(int dtype, int d, const void* q, const void* k, const void* v, const void* w,
                     const float* beta, const float* log_f, const void* o, const float* lse, const void* dO,
                     void* dq, void* dk, void* dv, void* dw, float* dbeta, float* dlog_f, int BH, int L,
                     float scale, unsigned char* ws, const BwdLayout& lay, cudaStream_t st);
cudaError_t kcache_update_launch(int dtype, int d, void* kc, int n_cached, int n_max, const void* w_t,
                                 const float* beta_t, int BH, cudaStream_t st);

static std::atomic<int> g_fault_mask{0};
static std::atomic<int> g_fox_no_skip{0};
static std::atomic<void*> g_ev_start{nullptr}, g_ev_end{nullptr};

void timing_events(cudaEvent_t* start, cudaEvent_t* end) {
    *start = static_cast<cudaEvent_t>(g_ev_start.load());
    *end = static_cast<cudaEvent_t>(g_ev_end.load());
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static size_t elt_size(int dtype) { return dtype == PATH_F32 ? 4 : 2; }

static bool fwd_d_ok(int d, int dtype) {
    if (dtype == PATH_F32) return d == 16 || d == 32 || d == 64 || d == 128;
    if (dtype == PATH_BF16) return tc_supported(d);
    return false;
}
static int fwd_chunk(int d, int dtype) { return dtype == PATH_F32 ? simt_chunk(d) : tc_chunk(d); }
static bool dec_d_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

// extra: 0 plain, 1 FoX (bias = log forget gates), 2 relative-position bias table
static int fwd_common(const void* q, const void* k, const void* v, const void* w, const float* beta,
                      const float* bias, int extra, void* o, float* lse, int B, int H, int L, int d, int dtype,
                      int causal, float scale, void* ws, size_t ws_bytes, cudaStream_t st) {
    const bool fox = extra == 1, rel = extra == 2;
    if (B < 1 || H < 1 || L < 1 || d < 1) return PATH_ERR_INVALID;
    if (dtype != PATH_F32 && dtype != PATH_BF16) return PATH_ERR_UNSUPPORTED;
    if (!causal) return PATH_ERR_UNSUPPORTED;
    if (!fwd_d_ok(d, dtype)) return PATH_ERR_UNSUPPORTED;
    if ((long long)B * H * L > (1ll << 31) / 256 || (long long)B * H > 65535) return PATH_ERR_UNSUPPORTED;
    if (!q || !k || !v || !w || !beta || !o || (extra != 0 && !bias)) return PATH_ERR_INVALID;
    const void* ptrs[] = {q, k, v, w, beta, o};
    for (const void* p : ptrs)
        if (!aligned16(p)) return PATH_ERR_INVALID;
    if ((extra != 0 && !aligned16(bias)) || (lse && !aligned16(lse))) return PATH_ERR_INVALID;
    const FwdLayout lay = fwd_layout(B, H, L, d, fwd_chunk(d, dtype), elt_size(dtype));
    if (!ws || ws_bytes < lay.total || !aligned16(ws)) return PATH_ERR_WORKSPACE;
    unsigned char* wsb = static_cast<unsigned char*>(ws);
    cudaError_t e;
    const float* log_f = fox ? bias : nullptr;
    const float* rel_bias = rel ? bias : nullptr;
    if (dtype == PATH_F32)
        e = fwd_simt_f32(q, k, v, w, beta, log_f, rel_bias, H, o, lse, B * H, L, d, scale, wsb, lay, st);
    else
        e = fwd_tc_bf16(q, k, v, w, beta, log_f, rel_bias, H, o, lse, B * H, L, d, scale, wsb, lay,
                        g_fault_mask.load(), FwdOptions{g_fox_no_skip.load()}, st);
    if (e != cudaSuccess) {
        std::fprintf(stderr, "pathattn: forward launch failed: %s\n", cudaGetErrorString(e));
        return PATH_ERR_CUDA;
    }
    return PATH_OK;
}

}  // namespace pathattn

using namespace pathattn;

extern "C" {

int path_version(void) { return (0 << 16) | 1; }

const char* path_status_string(int code) {
    switch (code) {
        case PATH_OK: return "ok";
        case PATH_ERR_INVALID: return "invalid argument";
        case PATH_ERR_UNSUPPORTED: return "unsupported request";
        case PATH_ERR_CUDA: return "CUDA runtime error";
        case PATH_ERR_TIMEOUT: return "device-side wait timed out";
        case PATH_ERR_WORKSPACE: return "workspace missing or too small";
        case PATH_ERR_BOUNDS: return "device-side index check failed";
        default: return "unknown status";
    }
}

size_t path_attn_workspace_bytes(int B, int H, int L, int d, int dtype) {
    if (B < 1 || H < 1 || L < 1 || !fwd_d_ok(d, dtype)) return 0;
    return fwd_layout(B, H, L, d, fwd_chunk(d, dtype), elt_size(dtype)).total;
}

int path_attn_fwd(const void* q, const void* k, const void* v, const void* w, const float* beta, void* o,
                  float* lse, int B, int H, int L, int d, int dtype, int causal, float scale, void* workspace,
                  size_t workspace_bytes, path_stream_t stream) {
    return fwd_common(q, k, v, w, beta, nullptr, 0, o, lse, B, H, L, d, dtype, causal, scale, workspace,
                      workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int path_attn_fwd_fox(const void* q, const void* k, const void* v, const void* w, const float* beta,
                      const float* log_f, void* o, float* lse, int B, int H, int L, int d, int dtype, int causal,
                      float scale, void* workspace, size_t workspace_bytes, path_stream_t stream) {
    return fwd_common(q, k, v, w, beta, log_f, 1, o, lse, B, H, L, d, dtype, causal, scale, workspace,
                      workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int path_attn_fwd_relbias(const void* q, const void* k, const void* v, const void* w, const float* beta,
                          const float* rel_bias, void* o, float* lse, int B, int H, int L, int d, int dtype,
                          int causal, float scale, void* workspace, size_t workspace_bytes, path_stream_t stream) {
    return fwd_common(q, k, v, w, beta, rel_bias, 2, o, lse, B, H, L, d, dtype, causal, scale, workspace,
                      workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

size_t path_prefill_workspace_bytes(int B, int H, int L, int d, int dtype) {
    if (B < 1 || H < 1 || L < 1 || !fwd_d_ok(d, dtype)) return 0;
    return fwd_layout(B, H, L, d, fwd_chunk(d, dtype), elt_size(dtype), true).total;
}

int path_prefill_kcache(const void* k, const void* w, const float* beta, void* kcache, int B, int H, int L,
                        int n_max, int d, int dtype, void* workspace, size_t workspace_bytes, path_stream_t stream) {
    if (B < 1 || H < 1 || L < 1 || n_max < L) return PATH_ERR_INVALID;
    if (dtype != PATH_F32 && dtype != PATH_BF16) return PATH_ERR_UNSUPPORTED;
    if (!fwd_d_ok(d, dtype)) return PATH_ERR_UNSUPPORTED;
    if ((long long)B * H > 65535 || (long long)B * H * L > (1ll << 31) / 256) return PATH_ERR_UNSUPPORTED;
    if (!k || !w || !beta || !kcache) return PATH_ERR_INVALID;
    if (!aligned16(k) || !aligned16(w) || !aligned16(beta) || !aligned16(kcache)) return PATH_ERR_INVALID;
    const FwdLayout lay = fwd_layout(B, H, L, d, fwd_chunk(d, dtype), elt_size(dtype), true);
    if (!workspace || workspace_bytes < lay.total || !aligned16(workspace)) return PATH_ERR_WORKSPACE;
    cudaError_t e = prefill_kcache(dtype, fwd_chunk(d, dtype), d, k, w, beta, kcache, B * H, L, n_max,
                                   static_cast<unsigned char*>(workspace), lay, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        std::fprintf(stderr, "pathattn: prefill launch failed: %s\n", cudaGetErrorString(e));
        return PATH_ERR_CUDA;
    }
    return PATH_OK;
}

size_t path_attn_bwd_workspace_bytes(int B, int H, int L, int d, int dtype) {
    if (B < 1 || H < 1 || L < 1 || (long long)B * H > 65535 || !bwd_supported(d)) return 0;
    if (dtype != PATH_F32 && dtype != PATH_BF16) return 0;
    return bwd_layout(B, H, L, d, elt_size(dtype)).total;
}

int path_attn_bwd(const void* q, const void* k, const void* v, const void* w, const float* beta,
                  const float* log_f, const void* o, const float* lse, const void* dO, void* dq, void* dk,
                  void* dv, void* dw, float* dbeta, float* dlog_f, int B, int H, int L, int d, int dtype,
                  int causal, float scale, void* workspace, size_t workspace_bytes, path_stream_t stream) {
    if (B < 1 || H < 1 || L < 1 || d < 1) return PATH_ERR_INVALID;
    if (dtype != PATH_F32 && dtype != PATH_BF16) return PATH_ERR_UNSUPPORTED;
    if (!causal) return PATH_ERR_UNSUPPORTED;
    if (!bwd_supported(d) || (long long)B * H > 65535) return PATH_ERR_UNSUPPORTED;
    if ((long long)B * H * L > (1ll << 31) / 256) return PATH_ERR_UNSUPPORTED;
    if (!q || !k || !v || !w || !beta || !o || !lse || !dO || !dq || !dk || !dv || !dw || !dbeta)
        return PATH_ERR_INVALID;
    if (log_f && !dlog_f) return PATH_ERR_INVALID;
    const void* ptrs[] = {q, k, v, w, beta, o, lse, dO, dq, dk, dv, dw, dbeta};
    for (const void* p : ptrs)
        if (!aligned16(p)) return PATH_ERR_INVALID;
    if (log_f && (!aligned16(log_f) || !aligned16(dlog_f))) return PATH_ERR_INVALID;
    const BwdLayout lay = bwd_layout(B, H, L, d, elt_size(dtype));
    if (!workspace || workspace_bytes < lay.total || !aligned16(workspace)) return PATH_ERR_WORKSPACE;
    cudaError_t e = attn_bwd(dtype, d, q, k, v, w, beta, log_f, o, lse, dO, dq, dk, dv, dw, dbeta,
                             log_f ? dlog_f : nullptr, B * H, L, scale, static_cast<unsigned char*>(workspace), lay,
                             reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        std::fprintf(stderr, "pathattn: backward launch failed: %s\n", cudaGetErrorString(e));
        return PATH_ERR_CUDA;
    }
    return PATH_OK;
}

size_t path_decode_workspace_bytes(int B, int H, int n_max, int d) {
    if (B < 1 || H < 1 || n_max < 1 || !dec_d_ok(d)) return 0;
    return dec_layout(B, H, n_max, d).total;
}

int path_kcache_update(void* kcache, int B, int H, int n_cached, int n_max, int d, const void* w_t,
                       const float* beta_t, int dtype, path_stream_t stream) {
    if (B < 1 || H < 1 || n_max < 1 || n_cached < 0 || n_cached > n_max) return PATH_ERR_INVALID;
    if (dtype != PATH_F32 && dtype != PATH_BF16) return PATH_ERR_UNSUPPORTED;
    if (!dec_d_ok(d) || (long long)B * H > 65535) return PATH_ERR_UNSUPPORTED;
    if (!kcache || !w_t || !beta_t) return PATH_ERR_INVALID;
    if (!aligned16(kcache) || !aligned16(w_t)) return PATH_ERR_INVALID;
    cudaError_t e = kcache_update_launch(dtype, d, kcache, n_cached, n_max, w_t, beta_t, B * H,
                                         reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PATH_OK : PATH_ERR_CUDA;
}

static int decode_common(const void* q_t, const void* k_t, const void* v_t, const void* w_t, const float* beta_t,
                         void* kcache, void* vcache, int n_cached, int n_max, void* o_t, float* lse_t, int B, int H,
                         int d, float scale, int dtype, void* workspace, size_t workspace_bytes, bool vt,
                         path_stream_t stream) {
    if (B < 1 || H < 1 || n_max < 1 || n_cached < 0) return PATH_ERR_INVALID;
    if (n_cached + 1 > n_max) return PATH_ERR_INVALID;
    if (dtype != PATH_F32 && dtype != PATH_BF16) return PATH_ERR_UNSUPPORTED;
    if (!dec_d_ok(d) || (long long)B * H > 65535) return PATH_ERR_UNSUPPORTED;
    if (!q_t || !k_t || !v_t || !w_t || !beta_t || !kcache || !vcache || !o_t) return PATH_ERR_INVALID;
    const void* ptrs[] = {q_t, k_t, v_t, w_t, kcache, vcache, o_t};
    for (const void* p : ptrs)
        if (!aligned16(p)) return PATH_ERR_INVALID;
    const DecLayout lay = dec_layout(B, H, n_max, d);
    if (!workspace || workspace_bytes < lay.total || !aligned16(workspace)) return PATH_ERR_WORKSPACE;
    cudaError_t e = decode_step(dtype, d, q_t, k_t, v_t, w_t, beta_t, kcache, vcache, n_cached, n_max, o_t, lse_t,
                                B * H, scale, static_cast<unsigned char*>(workspace), lay, vt,
                                reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PATH_OK : PATH_ERR_CUDA;
}

int path_decode_step(const void* q_t, const void* k_t, const void* v_t, const void* w_t, const float* beta_t,
                     void* kcache, void* vcache, int n_cached, int n_max, void* o_t, float* lse_t, int B, int H,
                     int d, float scale, int dtype, void* workspace, size_t workspace_bytes,
                     path_stream_t stream) {
    return decode_common(q_t, k_t, v_t, w_t, beta_t, kcache, vcache, n_cached, n_max, o_t, lse_t, B, H, d, scale,
                         dtype, workspace, workspace_bytes, false, stream);
}

int path_decode_step_vt(const void* q_t, const void* k_t, const void* v_t, const void* w_t, const float* beta_t,
                        void* kcache, void* vcache, int n_cached, int n_max, void* o_t, float* lse_t, int B, int H,
                        int d, float scale, int dtype, void* workspace, size_t workspace_bytes,
                        path_stream_t stream) {
    return decode_common(q_t, k_t, v_t, w_t, beta_t, kcache, vcache, n_cached, n_max, o_t, lse_t, B, H, d, scale,
                         dtype, workspace, workspace_bytes, true, stream);
}

size_t path_attn_fwd_vt_workspace_bytes(int B, int H, int L, int d, int dtype) {
    if (B < 1 || H < 1 || L < 1 || (long long)B * H > 65535 || !fwd_vt_supported(d)) return 0;
    if ((long long)B * H * L > (1ll << 31) / 256) return 0;
    if (dtype != PATH_F32 && dtype != PATH_BF16) return 0;
    return fwd_vt_workspace_bytes((long long)B * H, L, d, dtype);
}

int path_attn_fwd_vt(const void* q, const void* k, const void* v, const void* w, const float* beta,
                     const float* log_f, void* o, float* lse, int B, int H, int L, int d, int dtype, int causal,
                     float scale, void* workspace, size_t workspace_bytes, path_stream_t stream) {
    if (B < 1 || H < 1 || L < 1 || d < 1) return PATH_ERR_INVALID;
    if (dtype != PATH_F32 && dtype != PATH_BF16) return PATH_ERR_UNSUPPORTED;
    if (!causal || !fwd_vt_supported(d) || (long long)B * H > 65535) return PATH_ERR_UNSUPPORTED;
    if ((long long)B * H * L > (1ll << 31) / 256) return PATH_ERR_UNSUPPORTED;
    if (!q || !k || !v || !w || !beta || !o) return PATH_ERR_INVALID;
    const void* ptrs[] = {q, k, v, w, beta, o};
    for (const void* p : ptrs)
        if (!aligned16(p)) return PATH_ERR_INVALID;
    if ((log_f && !aligned16(log_f)) || (lse && !aligned16(lse))) return PATH_ERR_INVALID;
    if (!workspace || workspace_bytes < fwd_vt_workspace_bytes((long long)B * H, L, d, dtype) || !aligned16(workspace))
        return PATH_ERR_WORKSPACE;
    cudaError_t e = fwd_vt(dtype, d, q, k, v, w, beta, log_f, o, lse, B * H, L, scale,
                           static_cast<unsigned char*>(workspace), reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        std::fprintf(stderr, "pathattn: value-transport forward launch failed: %s\n", cudaGetErrorString(e));
        return PATH_ERR_CUDA;
    }
    return PATH_OK;
}

int path_get_status(const void* workspace, path_stream_t stream) {
    if (!workspace) return PATH_ERR_INVALID;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int status = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return PATH_ERR_CUDA;
    if (cudaMemcpyAsync(&status, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return PATH_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return PATH_ERR_CUDA;
    return status;
}

long long path_fwd_visited_blocks(const void* workspace, path_stream_t stream) {
    if (!workspace) return -1;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    unsigned visited = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
    if (cudaMemcpyAsync(&visited, static_cast<const unsigned char*>(workspace) + offsetof(WsHeader, visited),
                        sizeof(unsigned), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return -1;
    if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
    return (long long)visited;
}

void path_debug_set_fox_skip(int enabled) { g_fox_no_skip.store(enabled ? 0 : 1); }

void path_debug_set_fault(int mask) { g_fault_mask.store(mask); }

void path_debug_set_timing_events(void* ev_start, void* ev_end) {
    g_ev_start.store(ev_end ? ev_start : nullptr);
    g_ev_end.store(ev_start ? ev_end : nullptr);
}

}  // extern "C"
