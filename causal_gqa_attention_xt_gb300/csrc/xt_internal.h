// xt_internal.h -- declarations shared by the library's translation units.
// Host-side launchers return cudaError_t; the C ABI in xt_api.cu validates
// arguments, lays out the workspace and times launches.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace xt {

// Kernel ids for the per-launch timing hooks (xt_timing_*).
enum KernelId {
    KID_PROLOGUE = 0,     // QK-RMSNorm + RoPE of Q and K
    KID_FWD_SIMT,         // fp32 CUDA-core flash forward
    KID_FWD_TC,           // bf16 tcgen05 flash forward
    KID_BWD_PRE,          // Dlt = rowsum(dO * O)
    KID_BWD_DQ_SIMT,      // fp32 CUDA-core dQhat
    KID_BWD_DKDV_SIMT,    // fp32 CUDA-core dKhat, dV (group sum in-block)
    KID_BWD_DQ_TC,        // bf16 tcgen05 dQhat
    KID_BWD_DKDV_TC,      // bf16 tcgen05 dKhat, dV (group sum in-block)
    KID_BWD_EPILOGUE,     // RoPE^-1 + RMSNorm backward, dgamma partials
    KID_DGAMMA_REDUCE,    // fixed-order sum of dgamma partials
    KID_ROPE_TABLE,       // cos/sin table of the RoPE angles
    KID_DECODE_ROWS,      // decode: the new token's rows normed, rotated, cached
    KID_DECODE_ATTN,      // decode: split attention over the cache
    KID_DECODE_COMBINE,   // decode: fixed-order merge of the splits
    KID_DKDV_REDUCE,      // fixed-order sum of split dK/dV tiles' chunk partials
    KID_COUNT
};

// B planes of S rows. A packed batch is B = 1, S = total rows, with the
// samples' row offsets cu [units + 1] (device) and the longest sample max_len;
// a plain batch has cu = nullptr, units = B, max_len = S.
struct Problem {
    int B, S, H, G, D;
    float eps;
    double theta;
    int dtype;  // 0 = fp32, 1 = bf16
    const int *cu;
    int units, max_len;
    int group() const { return H / G; }
};

// Error word bits: a bounded wait ran out; a decode position was out of
// range; packed-batch offsets were not 0 = cu[0] <= ... <= cu[n] = total
// with every sample at most max_len rows.
enum : unsigned int { ERR_TIMEOUT = 1u, ERR_BADPOS = 2u, ERR_BADSEQ = 4u };

// Kernels that xt_test_inject_stall can make stall (bit mask), and the mask
// currently set (0 in normal operation).
enum : int { STALL_FWD_TC = 1, STALL_DKDV_TC = 2, STALL_DQ_TC = 4, STALL_ALL = 7 };
int test_stall_mask();

// ---- norm / RoPE kernels (xt_normrope.cu) ----
// Persistent grids: at most this many CTAs, which bounds the number of
// per-CTA dgamma partials the backward epilogue writes.
constexpr int kMaxNormParts = 1024;
// n_heads + n_kv_heads limit: every warp of those grids (8 per CTA) must be
// able to own one head chunk of a position.
constexpr int kMaxHeads = 8 * kMaxNormParts;
// cos/sin table [S][D/2] of (cos, sin) float pairs, filled by launch_rope_table
// and read by the prologue and the epilogue.
// A packed batch gets one table row per packed row (its position inside its
// sample); that launch also checks the offsets (ERR_BADSEQ).
size_t rope_table_bytes(const Problem &p);
cudaError_t launch_rope_table(const Problem &p, void *tab, unsigned int *err, cudaStream_t st);
cudaError_t launch_prologue(const Problem &p, const void *q, const void *k, const float *gq,
                            const float *gk, const void *tab, void *qhat, void *khat,
                            float *rstd_q, float *rstd_k, unsigned int *err, cudaStream_t st);
cudaError_t launch_bwd_pre(const Problem &p, const void *out, const void *dout, float *dlt,
                           unsigned int *err, cudaStream_t st);
// Writes the number of dgamma partial rows it produced (<= kMaxNormParts) to *nparts.
// dqhat == nullptr: the k rows only (dq and its dgamma partials come from the
// bf16 dQ kernel); part_q is then untouched.
cudaError_t launch_epilogue(const Problem &p, const float *dqhat, const float *dkhat,
                            const void *q, const void *k, const float *gq, const float *gk,
                            const float *rstd_q, const float *rstd_k, const void *tab, void *dq,
                            void *dk, float *part_q, float *part_k, int *nparts,
                            unsigned int *err, cudaStream_t st);
cudaError_t launch_dgamma_reduce(const Problem &p, const float *part_q, const float *part_k,
                                 int nparts_q, int nparts_k, float *dgq, float *dgk,
                                 cudaStream_t st);

// ---- decode step against a key/value cache (xt_decode.cu) ----
// Problem::S is the cache capacity S_max. The workspace holds the fp32 q rows
// and the per-split partials.
struct DecodePlan {
    int nsplit, L, nhc;   // key splits, keys per split, query-head chunks per kv head
    int units, grid;      // work units (b, kv head, head chunk, split); CTAs of the attention kernel
    size_t off_qhat, off_o, off_ml, total;
};
DecodePlan decode_plan(const Problem &p);
cudaError_t launch_decode_rows(const Problem &p, const int *pos, const void *q, const void *k,
                               const void *v, const float *gq, const float *gk, float *qhat,
                               void *kc, void *vc, unsigned int *err, cudaStream_t st);
cudaError_t launch_decode_attn(const Problem &p, const DecodePlan &d, const int *pos,
                               const float *qhat, const void *kc, const void *vc, float *part_o,
                               float *part_ml, unsigned int *err, cudaStream_t st);
cudaError_t launch_decode_combine(const Problem &p, const DecodePlan &d, const float *part_o,
                                  const float *part_ml, void *out, float *lse, cudaStream_t st);

// ---- TMA tensor maps and the SM count (xt_tmap.cu) ----
// Multiprocessors of the current device (queried once per device).
int sm_count();

// Launches `kernel` as a programmatic dependent of the previous launch on the
// stream: it may be scheduled before that grid ends; the kernel waits for it
// (pdl_enter, griddepcontrol) before touching memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
// swizzle_bytes: 128 or 64 (the smem row width of the box, see tc::Atoms).
cudaError_t encode_tmap_bf16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                             const uint64_t *strides_bytes, const uint32_t *box,
                             int swizzle_bytes);
cudaError_t encode_tmap_f32(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                            const uint64_t *strides_bytes, const uint32_t *box,
                            int swizzle_bytes);

// ---- bf16 tcgen05 kernels ----
// The bf16 backward kernels finish dq and dk themselves (RoPE backward and
// RMSNorm backward of each owned row) and write one dgamma partial row of D
// floats per CTA (CTAs past a short sample write zeros): the dQ kernel
// dq_part_count(p) rows of dgamma_q; the dK/dV kernel, when dkdv_part_bytes(p)
// is 0 (no split key tiles), dk_part_count(p) rows of dgamma_k (with split
// tiles it writes fp32 dKhat and the k-row epilogue finishes dk).
struct RowEpilogue {
    const void *x;          // [.., S, heads, D] bf16 forward input (q or k)
    const float *gamma;     // [D]
    const float *rstd;      // [.., S, heads]
    const void *tab;        // RoPE table (float2 [rows, D/2])
    void *out;              // [.., S, heads, D] bf16: dq or dk
    float *part;            // dgamma partial rows
};
size_t dq_part_count(const Problem &p);
size_t dk_part_count(const Problem &p);

cudaError_t launch_fwd_tc(const Problem &p, const void *qhat, const void *khat, const void *v,
                          void *out, float *lse, unsigned int *err, cudaStream_t st);
// part: fp32 scratch of dkdv_part_bytes(p) for the chunk partials of key
// tiles whose work is split over several CTAs (none when that is 0);
// launch_dkdv_reduce then sums them in chunk order into dkhat and dv.
size_t dkdv_part_bytes(const Problem &p);
cudaError_t launch_bwd_dkdv_tc(const Problem &p, const void *qhat, const void *khat,
                               const void *v, const void *dout, const float *lse,
                               const float *dlt, float *dkhat, void *dv, float *part,
                               const RowEpilogue &ek, unsigned int *err, cudaStream_t st);
cudaError_t launch_dkdv_reduce(const Problem &p, const float *part, float *dkhat, void *dv,
                               cudaStream_t st);
// The bf16 dQ kernel also computes Dlt = rowsum(dO o O) of its rows and writes
// it to dlt, for the dK/dV kernel launched after it.
cudaError_t launch_bwd_dq_tc(const Problem &p, const void *qhat, const void *khat, const void *v,
                             const void *dout, const void *out, const float *lse, float *dlt,
                             const RowEpilogue &ep, unsigned int *err, cudaStream_t st);

// ---- fp32 CUDA-core flash kernels (xt_simt.cu) ----
cudaError_t launch_fwd_simt(const Problem &p, const void *qhat, const void *khat, const void *v,
                            void *out, float *lse, cudaStream_t st);
cudaError_t launch_bwd_dq_simt(const Problem &p, const void *qhat, const void *khat,
                               const void *v, const void *dout, const float *lse,
                               const float *dlt, float *dqhat, cudaStream_t st);
cudaError_t launch_bwd_dkdv_simt(const Problem &p, const void *qhat, const void *khat,
                                 const void *v, const void *dout, const float *lse,
                                 const float *dlt, float *dkhat, void *dv, cudaStream_t st);

}  // namespace xt
