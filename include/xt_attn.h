/*
 * xt_attn.h -- C ABI of the GB300 (sm_103a) causal grouped-query attention
 * core: per-head QK-RMSNorm, rotate_half RoPE and causal GQA scaled-dot-
 * product attention, forward and backward.
 *
 * What the operation is (web pages, cited by title and section):
 *  - xtrain "Phase T9: Export to xserv", architecture-diff table and
 *    Decision 1: y = x * rsqrt(mean(x^2) + eps) * gamma over every
 *    [head_dim] vector of Q and of K (one [head_dim] gamma per tensor, shared
 *    by all heads), applied before rotate_half RoPE with
 *    freq_i = theta^(-2i/head_dim) and position = token row; scores scaled
 *    by 1/sqrt(head_dim); causal masking.
 *  - Mint project report 5.4.1-5.4.2 (the rotation of the pair
 *    (i, i + head_dim/2) by the angle pos * theta^(-2i/head_dim)), 5.3.1
 *    (max-subtracted softmax and P V), 5.5.2 (RMSNorm backward).
 *  - xtrain "Phase T5: Tiny Transformer", Key Design Decisions: additive
 *    -1e9 mask above the diagonal (key j is visible to query t iff j <= t).
 *  - xtrain "Phase T15: GQA", "What is GQA": query head qh reads key/value
 *    head qh / (n_heads / n_kv_heads); Decision 2: the gradient of a shared
 *    key/value head is the sum of its group's query-head gradients, formed
 *    deterministically (no atomics).
 *  - xtrain "Phase T12: bf16 mixed precision", precision table: bf16
 *    activations in and out, fp32 accumulation, norm / softmax / RoPE in fp32.
 *
 * Layouts (all row-major and contiguous; B batch, S sequence, H = n_heads,
 * G = n_kv_heads, D = head_dim):
 *    q, out, dout, dq  [B, S, H, D]  element type `dtype`
 *    k, v, dk, dv      [B, S, G, D]  element type `dtype`
 *    q_hat             [B, H, S, D]  `dtype`  (Q after norm + RoPE)
 *    k_hat             [B, G, S, D]  `dtype`  (K after norm + RoPE)
 *    lse               [B, H, S]     fp32, natural-log log-sum-exp of the
 *                                    scaled, masked scores of each query row
 *    rstd_q / rstd_k   [B, S, H] / [B, S, G]  fp32, 1/sqrt(mean(x^2)+eps)
 *    gamma_q, gamma_k, dgamma_q, dgamma_k   [D] fp32
 *
 * Ownership and execution: every pointer is a device allocation owned by the
 * caller, 16-byte aligned. The library never allocates, frees or
 * synchronizes; XT_OK means the work was enqueued on `stream` (a
 * cudaStream_t; NULL = the legacy default stream) and results are valid once
 * that stream reaches the enqueued point. Scratch memory is the caller's
 * `workspace`, sized by xt_attn_workspace_bytes(). dgamma_q and dgamma_k are
 * overwritten, not accumulated. Forward and backward are deterministic:
 * identical inputs give bitwise identical outputs.
 *
 * Supported shapes: B, S, H, G >= 1, H % G == 0, H + G <= 8192; dtype
 * XT_BF16 with head_dim 32, 64 or 128 (tensor-core path), dtype XT_F32 with
 * head_dim a multiple of 8 up to 128 and B * H <= 65535 (fp32 CUDA-core
 * path). Every tensor must hold fewer than 2^31 elements.
 *
 * Errors: calls validate their arguments on the host before any launch and
 * return an xt_status; no call aborts the process. XT_ECUDA reports a launch
 * or CUDA API failure (xt_last_cuda_error() gives the cudaError_t); it is not
 * cleared or hidden. Kernels that wait on barriers give up after a bounded
 * number of polls and raise a device-side error word, which
 * xt_attn_check() reads back (as XT_ETIMEOUT).
 */
#ifndef XT_ATTN_H
#define XT_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { XT_F32 = 0, XT_BF16 = 1 } xt_dtype;

typedef enum {
    XT_OK = 0,
    XT_EINVAL = 1,        /* bad size, null pointer, H % G != 0, bad eps/theta   */
    XT_EUNSUPPORTED = 2,  /* valid but unsupported (dtype, head_dim) pair         */
    XT_ECUDA = 3,         /* a CUDA call or kernel launch failed                  */
    XT_EWORKSPACE = 4,    /* workspace pointer null or workspace_bytes too small  */
    XT_ETIMEOUT = 5       /* a kernel gave up waiting on a barrier (device flag)  */
} xt_status;

/* Bytes of scratch the forward (backward = 0) or backward (backward != 0)
 * call needs for this problem; 0 on invalid arguments. The forward's scratch
 * is the RoPE table, S * head_dim/2 (cos, sin) fp32 pairs (rounded up to 256
 * bytes); the backward's holds that table too, plus Dlt [B, H, S] and
 * dgamma partial rows of head_dim floats. In fp32 it also holds fp32 dQhat
 * and dKhat and 2 * 1024 partial rows. In bf16 the tensor-core kernels finish
 * dq and dk themselves: one q partial row per (b, head, 128-row query tile)
 * and one k partial row per (b, kv head, 128-row key tile); except that for
 * problems whose key/value heads carry far more work than there are blocks to
 * share it (few kv heads and long sequences, e.g. MQA) the dK/dV work of the
 * longest key tiles is split over several thread blocks, and the scratch
 * then holds their fp32 partials, fp32 dKhat and 1024 k partial rows. The
 * size depends on the current device's SM count (which decides the split). */
size_t xt_attn_workspace_bytes(int B, int S, int n_heads, int n_kv_heads, int head_dim,
                               int dtype, int backward);

/* Forward: out = causal GQA SDPA(rope(norm(q)), rope(norm(k)), v) with scale
 * 1/sqrt(head_dim). Also writes what the backward needs: lse, q_hat, k_hat,
 * rstd_q, rstd_k. `eps` is the RMSNorm epsilon (added to mean(x^2) inside the
 * square root), `theta` the RoPE base. `workspace` must hold at least
 * xt_attn_workspace_bytes(..., backward = 0) bytes (else XT_EWORKSPACE). */
int xt_attn_fwd(int B, int S, int n_heads, int n_kv_heads, int head_dim,
                double eps, double theta,
                const void *q, const void *k, const void *v,
                const float *gamma_q, const float *gamma_k, int dtype,
                void *out, float *lse, void *q_hat, void *k_hat,
                float *rstd_q, float *rstd_k,
                void *workspace, size_t workspace_bytes, void *stream);

/* Backward for upstream gradient dout: writes dq, dk, dv (input layouts and
 * dtype) and dgamma_q, dgamma_k (overwritten). q, k, v, gammas and the saved
 * tensors are those of the matching xt_attn_fwd call. The gradient of each
 * shared key/value head is the sum over its group's query heads, formed in a
 * fixed order inside one thread block. */
int xt_attn_bwd(int B, int S, int n_heads, int n_kv_heads, int head_dim,
                double eps, double theta,
                const void *q, const void *k, const void *v,
                const float *gamma_q, const float *gamma_k, int dtype,
                const void *out, const float *lse, const void *q_hat, const void *k_hat,
                const float *rstd_q, const float *rstd_k, const void *dout,
                void *dq, void *dk, void *dv, float *dgamma_q, float *dgamma_k,
                void *workspace, size_t workspace_bytes, void *stream);

/* Backward without a workspace: identical in arguments and results to
 * xt_attn_bwd, but its scratch memory is a fixed 16 MiB array that this
 * library keeps in device memory (no counterpart on the pages: it exists for
 * callers that cannot allocate device memory themselves, e.g. a host
 * application whose own memory pool exposes no allocation hook to plugins, or
 * a latency-critical loop where cudaMalloc is not allowed). The call itself
 * allocates and frees nothing.
 *  - Limit: problems whose xt_attn_workspace_bytes(..., backward=1) exceeds
 *    16 MiB (16777216 bytes) are refused with XT_EWORKSPACE before any launch.
 *  - Every GPU that loads the library holds the 16 MiB array until the
 *    process exits.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, on the current device); make that first call
 *    before any stream capture begins.
 *  - All calls share the one array, which keeps the previous call's contents
 *    (a call that completes writes every scratch byte it reads, so nothing
 *    needs clearing). Calls whose GPU work overlaps in time -- on different
 *    streams, or from different host threads -- race on the array: serialize
 *    them.
 *  - After a call that xt_attn_check() reports as XT_ETIMEOUT, the contents of
 *    dq, dk, dv, dgamma_q and dgamma_k are unspecified (a kernel that gave up
 *    leaves its part of the scratch unwritten, and a later one may read the
 *    previous call's). */
int xt_attn_bwd_noalloc(int B, int S, int n_heads, int n_kv_heads, int head_dim,
                        double eps, double theta,
                        const void *q, const void *k, const void *v,
                        const float *gamma_q, const float *gamma_k, int dtype,
                        const void *out, const float *lse, const void *q_hat, const void *k_hat,
                        const float *rstd_q, const float *rstd_k, const void *dout,
                        void *dq, void *dk, void *dv, float *dgamma_q, float *dgamma_k,
                        void *stream);

/* ------------------------------------------------------- packed batches
 * Variable-length samples packed into one row dimension (Mint project
 * report, 8.2, forward pass of a chat batch: the batch is flattened to
 * [total] rows, RoPE numbers the positions inside each sample, and a
 * block-causal mask hides every other sample's rows entirely and, inside a
 * sample, the later rows). Sample s holds rows cu_seqlens[s] ..
 * cu_seqlens[s+1]-1; its rows sit at positions 0, 1, ... for RoPE and attend
 * causally to the rows of the same sample only. The operation per sample is
 * exactly xt_attn_fwd / xt_attn_bwd with B = 1, S = its length.
 *
 * Layouts: the batched ones with B = 1 and S = total:
 *    q, out, dout, dq  [total, H, D];  k, v, dk, dv  [total, G, D]
 *    q_hat [H, total, D];  k_hat [G, total, D];  lse [H, total]
 *    rstd_q [total, H];  rstd_k [total, G]
 * cu_seqlens: int32 [nseq + 1] in device memory (4-byte aligned), with
 * 0 = cu[0] <= cu[1] <= ... <= cu[nseq] = total (empty samples allowed) and
 * every cu[s+1] - cu[s] <= max_seqlen; 0 < max_seqlen <= total, nseq >= 1.
 * Offsets are read on the device: the host checks nseq, max_seqlen and the
 * pointer (XT_EINVAL), and a device-side check of the offsets raises the
 * error word, which xt_attn_check() reports as XT_EINVAL (accesses stay in
 * bounds either way; results are then unspecified).
 * Workspace: xt_attn_varlen_workspace_bytes() for the same total, nseq and
 * max_seqlen (the forward's RoPE table has one row per packed row; the bf16
 * backward keeps one dgamma_q partial row per (sample, head, 128-row query
 * tile of max_seqlen)); 0 for invalid sizes. Grids are sized by max_seqlen: a
 * short sample's blocks past its end exit at once. dtype XT_F32 needs nseq * n_heads <= 65535.
 * Deterministic, like the batched calls. */
size_t xt_attn_varlen_workspace_bytes(int total, int nseq, int max_seqlen, int n_heads,
                                      int n_kv_heads, int head_dim, int dtype, int backward);

int xt_attn_fwd_varlen(int total, int nseq, int max_seqlen, int n_heads, int n_kv_heads,
                       int head_dim, double eps, double theta, const int *cu_seqlens,
                       const void *q, const void *k, const void *v,
                       const float *gamma_q, const float *gamma_k, int dtype,
                       void *out, float *lse, void *q_hat, void *k_hat,
                       float *rstd_q, float *rstd_k,
                       void *workspace, size_t workspace_bytes, void *stream);

int xt_attn_bwd_varlen(int total, int nseq, int max_seqlen, int n_heads, int n_kv_heads,
                       int head_dim, double eps, double theta, const int *cu_seqlens,
                       const void *q, const void *k, const void *v,
                       const float *gamma_q, const float *gamma_k, int dtype,
                       const void *out, const float *lse, const void *q_hat, const void *k_hat,
                       const float *rstd_q, const float *rstd_k, const void *dout,
                       void *dq, void *dk, void *dv, float *dgamma_q, float *dgamma_k,
                       void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------- decode
 * One decode step against a key/value cache (Mint project report, 10.3 "KV
 * cache": the new token computes its own q, k, v, appends k and v to the
 * cache, and its query attends over every cached key, all of which are at or
 * before it, so the mask is implicit; the page states this equals the
 * full-sequence attention at that row).
 *
 * For each batch element b, with p = pos[b] (device memory, int32 [B]):
 *  - k_cache[b, g, p, :] = rope(norm(k[b, g]) * gamma_k, p) and
 *    v_cache[b, g, p, :] = v[b, g] for every kv head g (the rows the
 *    training forward writes to k_hat, and v, at position p);
 *  - out[b, h] = sum_{j <= p} softmax_j(q_hat . k_cache[b, h/group, j] /
 *    sqrt(head_dim)) v_cache[b, h/group, j] with q_hat = rope(norm(q[b, h]) *
 *    gamma_q, p), and lse[b, h] its natural-log log-sum-exp.
 * Rows 0..p-1 of the caches must hold the earlier tokens (e.g. the k_hat of a
 * training-style forward over the prompt, and v transposed to the cache
 * layout); rows after p are not read.
 *
 * Layouts: q [B, H, D], k and v [B, G, D] (the new token; input dtype),
 * k_cache and v_cache [B, G, S_max, D] (head-major, dtype), out [B, H, D]
 * (dtype), lse [B, H] fp32, gamma_q / gamma_k [D] fp32. Same dtype and
 * head_dim rules as xt_attn_fwd. The workspace must hold
 * xt_attn_decode_workspace_bytes() bytes. A position outside [0, S_max) is
 * detected on the device: that batch element is skipped and xt_attn_check()
 * reports XT_EINVAL. Deterministic: the key splits are merged in a fixed
 * order. */
size_t xt_attn_decode_workspace_bytes(int B, int S_max, int n_heads, int n_kv_heads, int head_dim,
                                      int dtype);
int xt_attn_decode(int B, int S_max, int n_heads, int n_kv_heads, int head_dim,
                   double eps, double theta, const int *pos,
                   const void *q, const void *k, const void *v,
                   const float *gamma_q, const float *gamma_k, int dtype,
                   void *k_cache, void *v_cache, void *out, float *lse,
                   void *workspace, size_t workspace_bytes, void *stream);

/* Synchronizes `stream`, then reads and clears the device error word of the
 * current device: XT_OK, XT_ETIMEOUT (a bounded wait ran out), XT_EINVAL (a
 * decode position was out of range) or XT_ECUDA. */
int xt_attn_check(void *stream);

/* Human-readable name of an xt_status value (static storage). */
const char *xt_status_str(int status);

/* The cudaError_t behind the most recent XT_ECUDA on this thread (0 if none). */
int xt_last_cuda_error(void);

/* Per-kernel timing, for measurement: when enabled, every launch the library
 * makes is bracketed by CUDA events recorded on the launch stream, and
 * xt_timing_query() sums their elapsed times (it synchronizes on those
 * events). Disabled by default; enabling costs two event records per launch.
 * Kernel ids run from 0 to xt_kernel_count()-1. */
int xt_timing_enable(int on);
int xt_timing_reset(void);
int xt_timing_query(int kernel_id, double *total_ms, long *launches);
int xt_kernel_count(void);
const char *xt_kernel_name(int kernel_id);

/* Fault injection for the timeout path, for tests. The pages have no
 * counterpart; it exercises what the Mint project report 9.7 (error
 * handling) asks of GPU failures: they surface at a check point as an error
 * and are neither swallowed nor left to hang the process. kernel_mask selects bf16
 * tensor-core kernels: 1 the forward attention, 2 the dK/dV kernel, 4 the dQ
 * kernel (0 = off, the default). Each CTA of a selected kernel launched while
 * the mask is set makes its MMA-issuing thread wait, before its first MMA, on
 * a barrier that nothing arrives on; after 20 ms the wait gives up and the CTA
 * takes the same path as any timed-out wait: it raises the device error word,
 * sets its abort flag so that its other warps stop waiting, lets every copy
 * and MMA it issued land, frees its tensor memory and exits. The call that
 * launched it returns XT_OK (the work was enqueued); xt_attn_check() then
 * reports XT_ETIMEOUT and clears the word, and that call's outputs are
 * unspecified. The mask is process-wide and read at launch time. Returns
 * XT_EINVAL for bits outside 1|2|4. */
int xt_test_inject_stall(int kernel_mask);

#ifdef __cplusplus
}
#endif

#endif /* XT_ATTN_H */
