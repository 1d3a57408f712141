/*
 * path_attn.h — C ABI of libpathattn.so: PaTH causal attention (forward,
 * PaTH-FoX forward, decode with in-place key transport) on GB300 (sm_103a).
 *
 * The operation ("Resumo Técnico: Atenção PaTH", gist.science/pt/paper/2505.16381):
 *   §2 "Mecanismo Central", attention-logit equation: for each head and query i,
 *       s_ij = scale * k_j^T (H_{j+1} H_{j+2} ... H_i) q_i        for j <= i,
 *       o_i  = sum_j softmax_j(s_i.) v_j,
 *   §2 "Mecanismo Central", transition equation: H_s = I - beta_s w_s w_s^T.
 *   The product is ascending (H_{j+1} leftmost) and empty (= I) at j = i.
 *   §2 "Extensões: PaTH-FoX": adds the forget-gate bias sum_{s=j+1..i} log f_s,
 *   unscaled, to s_ij.
 *   §3 "Inferência": decoding applies the current step's H_t in place to every
 *   cached key, so the cache holds transported keys and attention over it is
 *   ordinary one-query attention.
 *
 * Conventions shared by every entry point
 *   - Pointers named q, k, v, w, o, kcache, vcache, *_t, beta*, log_f, lse and
 *     workspace are DEVICE pointers.  The caller owns every buffer; the library
 *     never allocates, frees, or keeps a pointer after the call returns.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).  A returned PATH_OK means "validated and
 *     launched", not "finished".
 *   - Argument errors (null pointer, bad size, unsupported d or dtype,
 *     misaligned pointer, too-small workspace) are returned synchronously
 *     before anything is launched.  A launch error reported by the CUDA
 *     runtime is returned as PATH_ERR_CUDA.  Errors detected on the device
 *     (a bounded wait that expired) are written to the status word at the
 *     start of the workspace and read back with path_get_status().
 *   - dtype PATH_F32: q, k, v, w, o, caches are float; arithmetic is fp32
 *     (no TF32).  dtype PATH_BF16: those tensors are bfloat16; products are
 *     taken on bf16 tensor cores with fp32 accumulation, softmax in fp32.
 *     beta, log_f and lse are always float.
 *   - Preconditions that are NOT checked: beta in [0, 2] and |w| = 1.  The
 *     library neither clips beta nor normalises w; values are used as given.
 *   - All device pointers must be 16-byte aligned.
 */
#ifndef PATH_ATTN_H
#define PATH_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* path_stream_t; /* identical to cudaStream_t */

enum path_status {
    PATH_OK = 0,
    PATH_ERR_INVALID = 1,     /* bad pointer, size, alignment or capacity */
    PATH_ERR_UNSUPPORTED = 2, /* valid request outside what is implemented (non-causal, d, dtype) */
    PATH_ERR_CUDA = 3,        /* the CUDA runtime reported an error */
    PATH_ERR_TIMEOUT = 4,     /* a device-side bounded wait expired (read via path_get_status) */
    PATH_ERR_WORKSPACE = 5,   /* workspace null or smaller than the *_workspace_bytes() value */
    PATH_ERR_BOUNDS = 6       /* a device-side index check failed (bounds-checked builds only, read via
                                 path_get_status; the normal build has no such checks) */
};

enum path_dtype { PATH_F32 = 0, PATH_BF16 = 1 };

/* Library version, (major << 16) | minor. */
int path_version(void);

/* Human-readable name of a path_status code (static storage). */
const char* path_status_string(int code);

/*
 * Workspace size in bytes for path_attn_fwd / path_attn_fwd_fox with these
 * sizes.  The workspace holds the per-chunk UT-transform products (the
 * boundary-adjusted queries and keys, and the chunk factors used by the
 * right-to-left scan) and a status word.  Returns 0 for unsupported sizes.
 */
size_t path_attn_workspace_bytes(int B, int H, int L, int d, int dtype);

/*
 * PaTH causal attention forward (§2 "Mecanismo Central"; computed blockwise as
 * in §3 "Algoritmo Estilo FlashAttention": per-chunk UT transform
 * (§3 "Representação de Transformação UT"), boundary-adjusted queries and keys,
 * and a right-to-left scan over key/value blocks, never forming the L x L
 * matrix).
 *
 *   q, k, v, w : [B, H, L, d] row-major (element (b,h,i,c) at ((b*H+h)*L+i)*d+c)
 *   beta       : [B, H, L] float
 *   o          : [B, H, L, d], same dtype as q (written)
 *   lse        : [B, H, L] float, natural-log log-sum-exp of the scaled logits
 *                per query (written), or NULL
 *   B, H >= 1, B*H <= 65535; L >= 1; d in {16, 32, 64, 128} for PATH_F32, {64, 128}
 *   for PATH_BF16
 *   causal     : must be 1 (the PaTH product is defined only for j <= i);
 *                0 returns PATH_ERR_UNSUPPORTED
 *   scale      : multiplies k_j^T(...)q_i (typically 1/sqrt(d))
 *   workspace  : >= path_attn_workspace_bytes(B,H,L,d,dtype) bytes, device,
 *                16-byte aligned, contents need not be initialised
 *
 * o may not alias any input.  The workspace must not be used by another call
 * that can run concurrently.
 */
int path_attn_fwd(const void* q, const void* k, const void* v, const void* w, const float* beta,
                  void* o, float* lse, int B, int H, int L, int d, int dtype, int causal, float scale,
                  void* workspace, size_t workspace_bytes, path_stream_t stream);

/*
 * PaTH-FoX forward (§2 "Extensões: PaTH-FoX"): as path_attn_fwd, with the
 * forget-gate bias  sum_{s=j+1..i} log_f[s]  added unscaled to the scaled
 * logit of (i, j).  log_f: [B, H, L] float (log of the forget gate, <= 0).
 * The bf16 tensor-core path stops a query tile's scan once every key further
 * left provably has weight exactly 0 in fp32 (bias plus a bound on the
 * transported logit); the bound assumes the unchecked preconditions above
 * (beta in [0, 2], |w| = 1, up to bf16 rounding of w) and log_f <= 0.
 */
int path_attn_fwd_fox(const void* q, const void* k, const void* v, const void* w, const float* beta,
                      const float* log_f, void* o, float* lse, int B, int H, int L, int d, int dtype,
                      int causal, float scale, void* workspace, size_t workspace_bytes,
                      path_stream_t stream);

/*
 * PaTH forward with a relative-position bias: as path_attn_fwd, with
 * rel_bias[h*L + (i - j)] added unscaled to the scaled logit of (i, j).  This
 * is the additive positional prior of "Resumo Técnico: Mecanismo de Atenção
 * Bayesiana (BAM)", §"Solução Proposta: GGD-BAM" (b_ij = -|(j - i - mu)/alpha|^p,
 * a function of i - j with per-head parameters), or ALiBi's -slope (i - j),
 * applied on top of the PaTH logits.
 *   rel_bias : [H, L] float, device, shared by every batch entry; entry
 *              (h, delta) is the bias at distance delta = i - j.  Values must
 *              be finite (not checked).
 * Everything else as path_attn_fwd (same workspace size).
 */
int path_attn_fwd_relbias(const void* q, const void* k, const void* v, const void* w, const float* beta,
                          const float* rel_bias, void* o, float* lse, int B, int H, int L, int d, int dtype,
                          int causal, float scale, void* workspace, size_t workspace_bytes,
                          path_stream_t stream);

/*
 * Workspace size in bytes for path_attn_bwd.  The backward keeps, per head and
 * per pair (query chunk n, key chunk m < n) of 64-position chunks, the queries
 * transported to chunk m, the chain gradient, the logit gradient and the softmax
 * probabilities in the input dtype, so it grows as B*H*L^2 (about 11.5 GB for
 * bf16 at B=8, H=12, L=4096, d=128; about twice that for fp32).  Returns 0 for
 * unsupported sizes.
 */
size_t path_attn_bwd_workspace_bytes(int B, int H, int L, int d, int dtype);

/*
 * Gradients of PaTH (log_f == NULL) or PaTH-FoX causal attention with respect to
 * every input: the chain rule of the forward of §2 "Mecanismo Central" (logit and
 * transition equations) and "Extensões: PaTH-FoX", which §3 "Treinamento e
 * Inferência Eficientes" trains by backpropagation.  For a loss with gradient dO
 * with respect to o:
 *   q, k, v, w, beta, log_f : the forward's inputs (as path_attn_fwd_fox; log_f
 *                             may be NULL for plain PaTH)
 *   o, lse : the forward's outputs for these inputs (lse is required)
 *   dO     : [B, H, L, d], same dtype as q
 *   dq, dk, dv, dw : [B, H, L, d], same dtype as q (written)
 *   dbeta  : [B, H, L] float (written)
 *   dlog_f : [B, H, L] float (written); required when log_f is given, ignored
 *            otherwise
 *   d in {16, 32, 64, 128} for PATH_F32 and PATH_BF16; B*H <= 65535; causal = 1
 *   workspace : >= path_attn_bwd_workspace_bytes(B,H,L,d,dtype) bytes, device,
 *            16-byte aligned, contents need not be initialised
 * Arithmetic: fp32 inputs run in fp32 on the CUDA cores.  bf16 inputs at d = 128
 * run the query-side chunk chains and the per-key-chunk sums on the tensor cores
 * (bf16 operands, fp32 accumulation; the carried states enter as hi + lo bf16
 * parts).  The within-chunk parts (qbar, khat, the chunk transitions, the
 * diagonal block and the reverse of the within-chunk products) are products of
 * the compact ("UT") form: for bf16 at d >= 64 on the tensor cores (fp32
 * operands other than q, k, v, w, dO enter as hi + lo bf16 parts), otherwise in
 * fp32 on the CUDA cores.  Gradients are rounded to the input dtype (nearest
 * even) on store.  dbeta and dlog_f at position 0 are exactly zero (those enter
 * no logit).  Repeated calls agree to rounding in dbeta and dlog_f, not bit for
 * bit (their partial sums are added into shared- and global-memory accumulators
 * in an order that depends on scheduling); dq, dk, dv and dw repeat exactly.
 * Outputs may not alias inputs.  Argument errors return before any launch.  The
 * tensor-core kernels bound every wait; an expiry sets PATH_ERR_TIMEOUT in the
 * workspace status word (read it with path_get_status), which otherwise stays
 * PATH_OK.
 */
int path_attn_bwd(const void* q, const void* k, const void* v, const void* w, const float* beta,
                  const float* log_f, const void* o, const float* lse, const void* dO, void* dq, void* dk,
                  void* dv, void* dw, float* dbeta, float* dlog_f, int B, int H, int L, int d, int dtype,
                  int causal, float scale, void* workspace, size_t workspace_bytes, path_stream_t stream);

/*
 * Workspace size in bytes for path_decode_step (split-K partial results and a
 * status word) for caches of capacity n_max.  Returns 0 for unsupported sizes.
 */
size_t path_decode_workspace_bytes(int B, int H, int n_max, int d);

/*
 * Workspace size in bytes for path_prefill_kcache (the UT-prep products plus
 * the key-side chunk factors).  Returns 0 for unsupported sizes.
 */
size_t path_prefill_workspace_bytes(int B, int H, int L, int d, int dtype);

/*
 * Prefill -> decode hand-off (§3 "Inferência"): writes the transported key
 * cache of a prompt of L tokens,
 *     kcache[b,h,j,:] = H_{L-1} ... H_{j+1} k[b,h,j,:]      for j < L,
 * i.e. the cache that token-by-token path_decode_step calls from an empty
 * cache would leave, so that decoding continues with n_cached = L.  Computed
 * per chunk from the UT representation (§3 "Representação de Transformação
 * UT"): keys transported to their chunk end, then through every later chunk.
 *   k, w   : [B, H, L, d] (dtype);  beta : [B, H, L] float
 *   kcache : [B, H, n_max, d] (dtype), n_max >= L; rows >= L are not touched.
 *            The value cache is the caller's copy of v (values are not transported).
 *   d      : as for path_attn_fwd;  workspace >= path_prefill_workspace_bytes(...)
 */
int path_prefill_kcache(const void* k, const void* w, const float* beta, void* kcache, int B, int H, int L,
                        int n_max, int d, int dtype, void* workspace, size_t workspace_bytes, path_stream_t stream);

/*
 * In-place key transport alone (§3 "Inferência"): for every head and every
 * cached row j < n_cached,
 *     kcache[b,h,j,:] <- (I - beta_t[b,h] w_t[b,h] w_t[b,h]^T) kcache[b,h,j,:]
 * computed in fp32 and stored in the cache dtype (round to nearest even).
 *   kcache : [B, H, n_max, d] (updated in place); 0 <= n_cached <= n_max; B*H <= 65535
 *   w_t    : [B, H, d] cache dtype;  beta_t : [B, H] float
 *   d in {16, 32, 64, 128}
 */
int path_kcache_update(void* kcache, int B, int H, int n_cached, int n_max, int d, const void* w_t,
                       const float* beta_t, int dtype, path_stream_t stream);

/*
 * One decode step for every head (§3 "Inferência"; one-query attention over
 * the cache as in FlashDecoding, split over the key axis and merged by
 * log-sum-exp):
 *   1. kcache[j] <- H_t kcache[j] for j < n_cached   (fp32 math, stored in cache dtype)
 *   2. kcache[n_cached] <- k_t, vcache[n_cached] <- v_t   (the new key is not transported)
 *   3. o_t = softmax_j(scale * q_t . kcache[j]) vcache[j] over j = 0..n_cached,
 *      scoring each key with the value just stored.
 *   q_t, k_t, v_t, w_t : [B, H, d] cache dtype;  beta_t : [B, H] float
 *   kcache, vcache     : [B, H, n_max, d]; requires n_cached + 1 <= n_max and
 *                        B*H <= 65535 (else PATH_ERR_UNSUPPORTED)
 *                        (else PATH_ERR_INVALID); 0 <= n_cached
 *   o_t                : [B, H, d] cache dtype (written);  lse_t : [B, H] float or NULL
 *   workspace          : >= path_decode_workspace_bytes(B, H, n_max, d) bytes
 *   d in {16, 32, 64, 128}
 * The caller advances n_cached by one after each step.
 */
int path_decode_step(const void* q_t, const void* k_t, const void* v_t, const void* w_t,
                     const float* beta_t, void* kcache, void* vcache, int n_cached, int n_max, void* o_t,
                     float* lse_t, int B, int H, int d, float scale, int dtype, void* workspace,
                     size_t workspace_bytes, path_stream_t stream);

/*
 * One decode step with value-side transport ("Resumo Técnico: Por que
 * Transformações Acumuladas Extrapolam?", §"Metodologia" 1 route transport
 * P_{j->i}, §"Principais Contribuições" 3 "Proteção do Lado de Valor": the
 * accumulated route transport applied to the values as well as the keys).  As
 * path_decode_step, with the value cache transported in place alongside the
 * keys:
 *   1. kcache[j] <- H_t kcache[j] and vcache[j] <- H_t vcache[j] for j < n_cached
 *      (fp32 math, stored in the cache dtype)
 *   2. kcache[n_cached] <- k_t, vcache[n_cached] <- v_t (untransported)
 *   3. o_t = softmax_j(scale * q_t . kcache[j]) vcache[j], scoring and summing
 *      the values just stored.
 * The value cache therefore holds v~_j = H_{t-1} ... H_{j+1} v_j; after a prompt
 * of L tokens it is what path_prefill_kcache computes with v in place of k.
 * Arguments, sizes, workspace and errors as path_decode_step.
 */
int path_decode_step_vt(const void* q_t, const void* k_t, const void* v_t, const void* w_t,
                        const float* beta_t, void* kcache, void* vcache, int n_cached, int n_max, void* o_t,
                        float* lse_t, int B, int H, int d, float scale, int dtype, void* workspace,
                        size_t workspace_bytes, path_stream_t stream);

/*
 * Workspace size in bytes for path_attn_fwd_vt.  For bf16 at d = 128 (the
 * blockwise form below) it holds two forward layouts, the pair store of carried
 * value blocks, B*H * max(1, N (N - 1) / 2) * 128 * d bf16 with N = ceil(L / 128),
 * and the scan's output and LSE; otherwise the status header plus a logits
 * scratch of 16 * ceil(L / 32) * 32 bytes per warp (at most 256 MB; past that
 * fewer warps run).  Returns 0 for unsupported sizes.
 */
size_t path_attn_fwd_vt_workspace_bytes(int B, int H, int L, int d, int dtype);

/*
 * PaTH (log_f == NULL) or PaTH-FoX forward with value-side transport (the
 * operator of path_decode_step_vt over a whole sequence):
 *     o_i = sum_j softmax_j(s_i.) H_i ... H_{j+1} v_j
 * with the logits s_ij of path_attn_fwd / path_attn_fwd_fox (lse is theirs too).
 * Arguments as path_attn_fwd_fox (log_f nullable); d in {16, 32, 64, 128} for
 * PATH_F32 and PATH_BF16, B*H <= 65535, B*H*L <= 2^23.  `workspace` holds at
 * least path_attn_fwd_vt_workspace_bytes(B, H, L, d, dtype) bytes (else
 * PATH_ERR_WORKSPACE); its contents need no initialisation.
 * bf16 at d = 128 (while that workspace stays under 64 GB) runs blockwise: the
 * UT prep of the keys and, with v in the key slot, of the values (each value
 * moved to the end of its chunk); per key chunk m a chain carrying its values
 * through every later chunk transition (CUDA cores, fp32, stored bf16 per
 * (query chunk, key chunk) pair); the tensor-core scan with those blocks as its
 * values and a zero diagonal; and per row the walks of the diagonal chunk, which
 * carry the scan's output through the row's own chunk and add the diagonal's
 * terms.  Every other case runs on CUDA cores in fp32: each warp takes four
 * consecutive query rows and walks their keys twice (the logits right to left
 * into its workspace slot, then the outputs left to right).  Results are
 * rounded to the input dtype.
 */
int path_attn_fwd_vt(const void* q, const void* k, const void* v, const void* w, const float* beta,
                     const float* log_f, void* o, float* lse, int B, int H, int L, int d, int dtype, int causal,
                     float scale, void* workspace, size_t workspace_bytes, path_stream_t stream);

/*
 * Status of the most recent call that used `workspace` (each call clears the
 * word when it starts).  Synchronises `stream` first.  Returns a path_status
 * code: PATH_OK, PATH_ERR_TIMEOUT if a device-side bounded wait expired, or
 * PATH_ERR_CUDA if the synchronisation or read failed.
 */
int path_get_status(const void* workspace, path_stream_t stream);

/*
 * Number of (query tile, key block) pairs, diagonal blocks included, that the
 * most recent bf16 forward on `workspace` (path_attn_fwd, path_attn_fwd_fox or
 * path_attn_fwd_relbias with dtype PATH_BF16) visited, summed over every head.
 * Query tiles and key blocks are 128 positions, so a full causal pass visits
 * B*H*N*(N+1)/2 of them with N = ceil(L/128); PaTH-FoX visits fewer when its
 * far-block stop applies (§2 "Extensões: PaTH-FoX" workloads, §4 "Extrapolação
 * de Comprimento").  Synchronises `stream` first.  Returns -1 if `workspace` is
 * NULL or the read fails; the value is meaningless after an fp32 forward.
 */
long long path_fwd_visited_blocks(const void* workspace, path_stream_t stream);

/*
 * Test switch for the PaTH-FoX far-block stop of the bf16 forward: 0 makes
 * later calls visit every key block, non-zero (the default) restores the stop.
 * The stop only skips blocks whose every weight is exactly zero in fp32, so
 * both settings give bit-identical outputs for inputs that meet the
 * preconditions (beta in [0, 2], |w| = 1, log f <= 0); the switch exists to
 * test that.
 * It is process-wide and not synchronised with calls already enqueued.
 */
void path_debug_set_fox_skip(int enabled);

/*
 * Test hook for the device-side failure path.  A non-zero mask makes the next
 * bf16 forward launches skip one producer signal on purpose, so that the
 * consumer's bounded wait expires and the call reports PATH_ERR_TIMEOUT
 * through path_get_status() instead of hanging.  0 (the default) disables it.
 */
void path_debug_set_fault(int mask);

/*
 * Measurement hook.  When both are non-NULL, every later forward or decode
 * call records `ev_start` (a cudaEvent_t) on its stream immediately before
 * launching its dominant kernel (the scan kernel of the forward, the fused
 * update + score kernel of decode) and `ev_end` immediately after it, so the
 * caller can time that kernel alone with cudaEventElapsedTime.  Pass NULL,
 * NULL to stop.  The events are not owned by the library.
 */
void path_debug_set_timing_events(void* ev_start, void* ev_end);

/*
 * Allocation-free decode step.  The paper has no counterpart: this entry point
 * exists for callers that cannot allocate device memory when they decode, for
 * instance a runtime whose device memory is wholly owned by another allocator,
 * or a latency-critical serving loop that must never call cudaMalloc (which can
 * fail, and can synchronise the device) once it is running.  It computes
 * exactly what path_decode_step computes, with the same arguments except the
 * workspace: the split-K scratch is a fixed device array inside the library,
 * PATH_DECODE_NOALLOC_SCRATCH_BYTES bytes, held by every GPU that loads the
 * library until the process exits.
 *   - Scratch needed is path_decode_workspace_bytes(B, H, n_max, d); sizes that
 *     need more than PATH_DECODE_NOALLOC_SCRATCH_BYTES are rejected with
 *     PATH_ERR_WORKSPACE (and a message on stderr) before anything is launched.
 *     The 8 MiB covers B*H = 768 heads of d = 128 up to n_max = 43008.
 *   - The first call on each device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.  The address is tied to the device's context: after a
 *     cudaDeviceReset the next call looks it up again (so, again, outside any
 *     capture).
 *   - No call allocates or frees memory.  All calls share the one array, which
 *     keeps the previous call's contents; everything a step reads from it is
 *     written earlier in the same step.  Calls that can overlap on the GPU (two
 *     streams, or two host threads on one device) race on the array: order them.
 *   - Launch errors are returned; there is no device-side status to read with
 *     path_get_status (the decode kernels have no waits that can expire).
 */
#define PATH_DECODE_NOALLOC_SCRATCH_BYTES (8u << 20)
int path_decode_step_noalloc(const void* q_t, const void* k_t, const void* v_t, const void* w_t,
                             const float* beta_t, void* kcache, void* vcache, int n_cached, int n_max,
                             void* o_t, float* lse_t, int B, int H, int d, float scale, int dtype,
                             path_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* PATH_ATTN_H */
