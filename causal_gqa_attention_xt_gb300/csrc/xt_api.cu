// xt_api.cu -- the C ABI declared in include/xt_attn.h: host-side argument
// validation, workspace layout, kernel dispatch and per-launch timing.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/xt_attn.h"
#include "xt_internal.h"

namespace xt {

// Device error word raised by kernels whose bounded barrier waits run out.
__device__ unsigned int g_error_word;

namespace {

thread_local int g_last_cuda_error = 0;
std::atomic<int> g_stall_mask{0};

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return XT_ECUDA;
}

// ---------------------------------------------------------------- timing
struct PendingTiming {
    int kid;
    cudaEvent_t start, stop;
};

struct Timing {
    std::mutex mu;
    bool on = false;
    std::vector<PendingTiming> pending;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> free_pairs;
    double total_ms[KID_COUNT] = {};
    long launches[KID_COUNT] = {};
} g_timing;

const char *kKernelNames[KID_COUNT] = {
    "prologue_qknorm_rope", "fwd_simt_f32", "fwd_tcgen05_bf16", "bwd_pre_dlt",
    "bwd_dq_simt_f32",      "bwd_dkdv_simt_f32", "bwd_dq_tcgen05_bf16",
    "bwd_dkdv_tcgen05_bf16", "bwd_epilogue_rope_norm", "bwd_dgamma_reduce",
    "rope_table", "decode_rows", "decode_attn", "decode_combine", "bwd_dkdv_reduce"};

void drain_locked() {
    for (auto &p : g_timing.pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(p.stop) == cudaSuccess &&
            cudaEventElapsedTime(&ms, p.start, p.stop) == cudaSuccess) {
            g_timing.total_ms[p.kid] += ms;
            g_timing.launches[p.kid] += 1;
        }
        g_timing.free_pairs.push_back({p.start, p.stop});
    }
    g_timing.pending.clear();
}

// Runs one launcher; when timing is on, brackets it with events on `st`.
template <typename F>
int timed_launch(int kid, cudaStream_t st, F &&launch) {
    cudaEvent_t a = nullptr, b = nullptr;
    bool on;
    {
        std::lock_guard<std::mutex> lk(g_timing.mu);
        on = g_timing.on;
        if (on) {
            if (!g_timing.free_pairs.empty()) {
                a = g_timing.free_pairs.back().first;
                b = g_timing.free_pairs.back().second;
                g_timing.free_pairs.pop_back();
            } else {
                if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess)
                    return cuda_fail(cudaGetLastError());
            }
        }
    }
    if (on && cudaEventRecord(a, st) != cudaSuccess) return cuda_fail(cudaGetLastError());
    cudaError_t e = launch();
    if (e != cudaSuccess) return cuda_fail(e);
    if (on) {
        if (cudaEventRecord(b, st) != cudaSuccess) return cuda_fail(cudaGetLastError());
        std::lock_guard<std::mutex> lk(g_timing.mu);
        g_timing.pending.push_back({kid, a, b});
    }
    return XT_OK;
}

// ---------------------------------------------------------------- validation
bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

int validate_shape(int B, int S, int H, int G, int D, int dtype) {
    if (B <= 0 || S <= 0 || H <= 0 || G <= 0 || D <= 0) return XT_EINVAL;
    if (H % G != 0) return XT_EINVAL;
    if (D % 2 != 0) return XT_EINVAL;
    if (dtype != XT_F32 && dtype != XT_BF16) return XT_EINVAL;
    const double big = (double)B * (double)S * (double)H * (double)D;
    if (big >= 2147483648.0) return XT_EINVAL;
    if (dtype == XT_BF16 && D != 32 && D != 64 && D != 128) return XT_EUNSUPPORTED;
    if (dtype == XT_F32 && (D % 8 != 0 || D > 128)) return XT_EUNSUPPORTED;
    if (H + G > kMaxHeads) return XT_EUNSUPPORTED;
    if (dtype == XT_F32 && (long)B * H > 65535) return XT_EUNSUPPORTED;   // grid.y of the fp32 path
    return XT_OK;
}

int validate_scalars(double eps, double theta) {
    if (!(eps >= 0.0) || !isfinite(eps)) return XT_EINVAL;
    if (!(theta > 0.0) || !isfinite(theta)) return XT_EINVAL;
    return XT_OK;
}

size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

// Forward scratch: the RoPE cos/sin table.
size_t fwd_workspace(const Problem &p) { return align_up(rope_table_bytes(p)); }

// Backward scratch: the RoPE cos/sin table, Dlt, fp32 dQhat and dKhat where
// a separate epilogue finishes dq / dk (fp32 problems; dk of bf16 problems
// with split dK/dV tiles), the dgamma partials (the epilogue's, at most
// kMaxNormParts rows, or one row per CTA of the bf16 kernels that finish
// their rows themselves) and the split dK/dV partials.
struct BwdWorkspace {
    size_t off_tab, off_dlt, off_dqhat, off_dkhat, off_part_q, off_part_k, off_dkdv, total;
};

BwdWorkspace bwd_layout(const Problem &p) {
    BwdWorkspace w = {};
    size_t o = 0;
    w.off_tab = o;    o = align_up(o + rope_table_bytes(p));
    w.off_dlt = o;    o = align_up(o + sizeof(float) * (size_t)p.B * p.H * p.S);
    // bf16: the dQ kernel finishes dq itself (no fp32 dQhat), one dgamma_q
    // partial per CTA of it; likewise the dK/dV kernel for dk unless it splits
    const bool tc = p.dtype == XT_BF16;
    const bool fuse_k = tc && dkdv_part_bytes(p) == 0;
    w.off_dqhat = o;  o = align_up(o + (tc ? 0 : sizeof(float) * (size_t)p.B * p.H * p.S * p.D));
    w.off_dkhat = o;
    o = align_up(o + (fuse_k ? 0 : sizeof(float) * (size_t)p.B * p.G * p.S * p.D));
    w.off_part_q = o;
    o = align_up(o + sizeof(float) * (tc ? dq_part_count(p) : (size_t)kMaxNormParts) * p.D);
    w.off_part_k = o;
    o = align_up(o + sizeof(float) * (fuse_k ? dk_part_count(p) : (size_t)kMaxNormParts) * p.D);
    w.off_dkdv = o;   o = align_up(o + (p.dtype == XT_BF16 ? dkdv_part_bytes(p) : 0));
    w.total = o;
    return w;
}

unsigned int *error_word_ptr() {
    // device address of g_error_word on the current device (cached per device)
    static unsigned int *cache[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_error_word) != cudaSuccess) return nullptr;
        cache[dev] = (unsigned int *)ptr;
    }
    return cache[dev];
}

Problem make_problem(int B, int S, int H, int G, int D, double eps, double theta, int dtype) {
    Problem p;
    p.B = B; p.S = S; p.H = H; p.G = G; p.D = D;
    p.eps = (float)eps; p.theta = theta; p.dtype = dtype;
    p.cu = nullptr; p.units = B; p.max_len = S;
    return p;
}

// A packed batch: one plane of `total` rows holding nseq samples.
Problem make_packed_problem(int total, int nseq, int max_seqlen, const int *cu, int H, int G,
                            int D, double eps, double theta, int dtype) {
    Problem p = make_problem(1, total, H, G, D, eps, theta, dtype);
    p.cu = cu; p.units = nseq; p.max_len = max_seqlen;
    return p;
}

int validate_packed(int total, int nseq, int max_seqlen, const int *cu, int H, int dtype) {
    if (nseq <= 0 || max_seqlen <= 0 || max_seqlen > total) return XT_EINVAL;
    if (cu == nullptr || ((uintptr_t)cu & 3u) != 0) return XT_EINVAL;
    if (dtype == XT_F32 && (long)nseq * H > 65535) return XT_EUNSUPPORTED;
    return XT_OK;
}

// The forward pipeline: RoPE table, prologue, attention.
int run_fwd(const Problem &p, const void *q, const void *k, const void *v, const float *gamma_q,
            const float *gamma_k, void *out, float *lse, void *q_hat, void *k_hat, float *rstd_q,
            float *rstd_k, void *workspace, size_t workspace_bytes, void *stream) {
    const void *ptrs[] = {q, k, v, gamma_q, gamma_k, out, lse, q_hat, k_hat, rstd_q, rstd_k};
    for (const void *ptr : ptrs)
        if (ptr == nullptr || !aligned16(ptr)) return XT_EINVAL;
    if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < fwd_workspace(p))
        return XT_EWORKSPACE;
    void *tab = workspace;
    cudaStream_t s = (cudaStream_t)stream;
    unsigned int *err = error_word_ptr();
    if (!err) return cuda_fail(cudaGetLastError());
    int st = timed_launch(KID_ROPE_TABLE, s, [&] { return launch_rope_table(p, tab, err, s); });
    if (st != XT_OK) return st;
    st = timed_launch(KID_PROLOGUE, s, [&] {
        return launch_prologue(p, q, k, gamma_q, gamma_k, tab, q_hat, k_hat, rstd_q, rstd_k, err,
                               s);
    });
    if (st != XT_OK) return st;
    if (p.dtype == XT_BF16) {
        return timed_launch(KID_FWD_TC, s, [&] {
            return launch_fwd_tc(p, q_hat, k_hat, v, out, lse, err, s);
        });
    }
    return timed_launch(KID_FWD_SIMT, s, [&] {
        return launch_fwd_simt(p, q_hat, k_hat, v, out, lse, s);
    });
}

// The backward pipeline: RoPE table; bf16: dQ (which also writes Dlt), dK/dV
// (+ chunk reduce for split key tiles); fp32: Dlt, dK/dV, dQ; then the row
// epilogue where the attention kernels do not finish the rows themselves (fp32
// problems; k rows of split bf16 problems) and the dgamma reduce.
int run_bwd(const Problem &p, const void *q, const void *k, const void *v, const float *gamma_q,
            const float *gamma_k, const void *out, const float *lse, const void *q_hat,
            const void *k_hat, const float *rstd_q, const float *rstd_k, const void *dout,
            void *dq, void *dk, void *dv, float *dgamma_q, float *dgamma_k, void *workspace,
            size_t workspace_bytes, void *stream) {
    const void *ptrs[] = {q, k, v, gamma_q, gamma_k, out, lse, q_hat, k_hat, rstd_q, rstd_k,
                          dout, dq, dk, dv, dgamma_q, dgamma_k};
    for (const void *ptr : ptrs)
        if (ptr == nullptr || !aligned16(ptr)) return XT_EINVAL;
    const BwdWorkspace w = bwd_layout(p);
    if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < w.total)
        return XT_EWORKSPACE;
    char *ws = (char *)workspace;
    void *tab = ws + w.off_tab;
    float *dlt = (float *)(ws + w.off_dlt);
    float *dqhat = (float *)(ws + w.off_dqhat);
    float *dkhat = (float *)(ws + w.off_dkhat);
    float *part_q = (float *)(ws + w.off_part_q);
    float *part_k = (float *)(ws + w.off_part_k);
    cudaStream_t s = (cudaStream_t)stream;
    unsigned int *err = error_word_ptr();
    if (!err) return cuda_fail(cudaGetLastError());

    int st = timed_launch(KID_ROPE_TABLE, s, [&] { return launch_rope_table(p, tab, err, s); });
    if (st != XT_OK) return st;
    const bool tc = p.dtype == XT_BF16;
    const bool fuse_k = tc && dkdv_part_bytes(p) == 0;   // the dK/dV kernel finishes dk
    if (!tc) {
        st = timed_launch(KID_BWD_PRE, s, [&] {
            return launch_bwd_pre(p, out, dout, dlt, err, s);
        });
        if (st != XT_OK) return st;
    }
    if (tc) {
        // dQ first: it also writes Dlt, which the dK/dV kernel reads
        const RowEpilogue ep = {q, gamma_q, rstd_q, tab, dq, part_q};
        st = timed_launch(KID_BWD_DQ_TC, s, [&] {
            return launch_bwd_dq_tc(p, q_hat, k_hat, v, dout, out, lse, dlt, ep, err, s);
        });
        if (st != XT_OK) return st;
        float *part_dkdv = (float *)(ws + w.off_dkdv);
        const RowEpilogue ek = {k, gamma_k, rstd_k, tab, dk, part_k};
        st = timed_launch(KID_BWD_DKDV_TC, s, [&] {
            return launch_bwd_dkdv_tc(p, q_hat, k_hat, v, dout, lse, dlt, dkhat, dv, part_dkdv,
                                      ek, err, s);
        });
        if (st != XT_OK) return st;
        if (dkdv_part_bytes(p) > 0) {
            st = timed_launch(KID_DKDV_REDUCE, s, [&] {
                return launch_dkdv_reduce(p, part_dkdv, dkhat, dv, s);
            });
            if (st != XT_OK) return st;
        }
    } else {
        st = timed_launch(KID_BWD_DKDV_SIMT, s, [&] {
            return launch_bwd_dkdv_simt(p, q_hat, k_hat, v, dout, lse, dlt, dkhat, dv, s);
        });
        if (st != XT_OK) return st;
        st = timed_launch(KID_BWD_DQ_SIMT, s, [&] {
            return launch_bwd_dq_simt(p, q_hat, k_hat, v, dout, lse, dlt, dqhat, s);
        });
        if (st != XT_OK) return st;
    }
    int nparts = 0;
    if (!fuse_k) {   // k rows (and, for fp32, q rows) not finished by the attention kernels
        st = timed_launch(KID_BWD_EPILOGUE, s, [&] {
            return launch_epilogue(p, tc ? nullptr : dqhat, dkhat, q, k, gamma_q, gamma_k,
                                   rstd_q, rstd_k, tab, dq, dk, part_q, part_k, &nparts, err, s);
        });
        if (st != XT_OK) return st;
    }
    const int nparts_q = tc ? (int)dq_part_count(p) : nparts;
    const int nparts_k = fuse_k ? (int)dk_part_count(p) : nparts;
    return timed_launch(KID_DGAMMA_REDUCE, s, [&] {
        return launch_dgamma_reduce(p, part_q, part_k, nparts_q, nparts_k, dgamma_q, dgamma_k, s);
    });
}

}  // namespace

int test_stall_mask() { return g_stall_mask.load(std::memory_order_relaxed); }

}  // namespace xt

using namespace xt;

extern "C" {

size_t xt_attn_workspace_bytes(int B, int S, int n_heads, int n_kv_heads, int head_dim,
                               int dtype, int backward) {
    if (validate_shape(B, S, n_heads, n_kv_heads, head_dim, dtype) != XT_OK) return 0;
    const Problem p = make_problem(B, S, n_heads, n_kv_heads, head_dim, 0.0, 1.0, dtype);
    return backward ? bwd_layout(p).total : fwd_workspace(p);
}

int xt_attn_fwd(int B, int S, int n_heads, int n_kv_heads, int head_dim, double eps,
                double theta, const void *q, const void *k, const void *v,
                const float *gamma_q, const float *gamma_k, int dtype, void *out, float *lse,
                void *q_hat, void *k_hat, float *rstd_q, float *rstd_k, void *workspace,
                size_t workspace_bytes, void *stream) {
    int st = validate_shape(B, S, n_heads, n_kv_heads, head_dim, dtype);
    if (st != XT_OK) return st;
    if ((st = validate_scalars(eps, theta)) != XT_OK) return st;
    const Problem p = make_problem(B, S, n_heads, n_kv_heads, head_dim, eps, theta, dtype);
    return run_fwd(p, q, k, v, gamma_q, gamma_k, out, lse, q_hat, k_hat, rstd_q, rstd_k,
                   workspace, workspace_bytes, stream);
}

int xt_attn_bwd(int B, int S, int n_heads, int n_kv_heads, int head_dim, double eps,
                double theta, const void *q, const void *k, const void *v,
                const float *gamma_q, const float *gamma_k, int dtype, const void *out,
                const float *lse, const void *q_hat, const void *k_hat, const float *rstd_q,
                const float *rstd_k, const void *dout, void *dq, void *dk, void *dv,
                float *dgamma_q, float *dgamma_k, void *workspace, size_t workspace_bytes,
                void *stream) {
    int st = validate_shape(B, S, n_heads, n_kv_heads, head_dim, dtype);
    if (st != XT_OK) return st;
    if ((st = validate_scalars(eps, theta)) != XT_OK) return st;
    const Problem p = make_problem(B, S, n_heads, n_kv_heads, head_dim, eps, theta, dtype);
    return run_bwd(p, q, k, v, gamma_q, gamma_k, out, lse, q_hat, k_hat, rstd_q, rstd_k, dout,
                   dq, dk, dv, dgamma_q, dgamma_k, workspace, workspace_bytes, stream);
}

size_t xt_attn_varlen_workspace_bytes(int total, int nseq, int max_seqlen, int n_heads,
                                      int n_kv_heads, int head_dim, int dtype, int backward) {
    if (validate_shape(1, total, n_heads, n_kv_heads, head_dim, dtype) != XT_OK) return 0;
    if (nseq <= 0 || max_seqlen <= 0 || max_seqlen > total) return 0;
    // the sizes depend on the offsets only through nseq and max_seqlen
    const Problem p = make_packed_problem(total, nseq, max_seqlen, nullptr, n_heads, n_kv_heads,
                                          head_dim, 0.0, 1.0, dtype);
    return backward ? bwd_layout(p).total : fwd_workspace(p);
}

int xt_attn_fwd_varlen(int total, int nseq, int max_seqlen, int n_heads, int n_kv_heads,
                       int head_dim, double eps, double theta, const int *cu_seqlens,
                       const void *q, const void *k, const void *v, const float *gamma_q,
                       const float *gamma_k, int dtype, void *out, float *lse, void *q_hat,
                       void *k_hat, float *rstd_q, float *rstd_k, void *workspace,
                       size_t workspace_bytes, void *stream) {
    int st = validate_shape(1, total, n_heads, n_kv_heads, head_dim, dtype);
    if (st != XT_OK) return st;
    if ((st = validate_scalars(eps, theta)) != XT_OK) return st;
    if ((st = validate_packed(total, nseq, max_seqlen, cu_seqlens, n_heads, dtype)) != XT_OK)
        return st;
    const Problem p = make_packed_problem(total, nseq, max_seqlen, cu_seqlens, n_heads,
                                          n_kv_heads, head_dim, eps, theta, dtype);
    return run_fwd(p, q, k, v, gamma_q, gamma_k, out, lse, q_hat, k_hat, rstd_q, rstd_k,
                   workspace, workspace_bytes, stream);
}

int xt_attn_bwd_varlen(int total, int nseq, int max_seqlen, int n_heads, int n_kv_heads,
                       int head_dim, double eps, double theta, const int *cu_seqlens,
                       const void *q, const void *k, const void *v, const float *gamma_q,
                       const float *gamma_k, int dtype, const void *out, const float *lse,
                       const void *q_hat, const void *k_hat, const float *rstd_q,
                       const float *rstd_k, const void *dout, void *dq, void *dk, void *dv,
                       float *dgamma_q, float *dgamma_k, void *workspace, size_t workspace_bytes,
                       void *stream) {
    int st = validate_shape(1, total, n_heads, n_kv_heads, head_dim, dtype);
    if (st != XT_OK) return st;
    if ((st = validate_scalars(eps, theta)) != XT_OK) return st;
    if ((st = validate_packed(total, nseq, max_seqlen, cu_seqlens, n_heads, dtype)) != XT_OK)
        return st;
    const Problem p = make_packed_problem(total, nseq, max_seqlen, cu_seqlens, n_heads,
                                          n_kv_heads, head_dim, eps, theta, dtype);
    return run_bwd(p, q, k, v, gamma_q, gamma_k, out, lse, q_hat, k_hat, rstd_q, rstd_k, dout,
                   dq, dk, dv, dgamma_q, dgamma_k, workspace, workspace_bytes, stream);
}

size_t xt_attn_decode_workspace_bytes(int B, int S_max, int n_heads, int n_kv_heads,
                                      int head_dim, int dtype) {
    if (validate_shape(B, S_max, n_heads, n_kv_heads, head_dim, dtype) != XT_OK) return 0;
    return decode_plan(make_problem(B, S_max, n_heads, n_kv_heads, head_dim, 0.0, 1.0, dtype)).total;
}

int xt_attn_decode(int B, int S_max, int n_heads, int n_kv_heads, int head_dim, double eps,
                   double theta, const int *pos, const void *q, const void *k, const void *v,
                   const float *gamma_q, const float *gamma_k, int dtype, void *k_cache,
                   void *v_cache, void *out, float *lse, void *workspace, size_t workspace_bytes,
                   void *stream) {
    int st = validate_shape(B, S_max, n_heads, n_kv_heads, head_dim, dtype);
    if (st != XT_OK) return st;
    if ((st = validate_scalars(eps, theta)) != XT_OK) return st;
    if (pos == nullptr || ((uintptr_t)pos & 3u) != 0) return XT_EINVAL;
    const void *ptrs[] = {q, k, v, gamma_q, gamma_k, k_cache, v_cache, out, lse};
    for (const void *ptr : ptrs)
        if (ptr == nullptr || !aligned16(ptr)) return XT_EINVAL;
    const Problem p = make_problem(B, S_max, n_heads, n_kv_heads, head_dim, eps, theta, dtype);
    const DecodePlan d = decode_plan(p);
    if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < d.total)
        return XT_EWORKSPACE;
    char *ws = (char *)workspace;
    float *qhat = (float *)(ws + d.off_qhat);
    float *part_o = (float *)(ws + d.off_o);
    float *part_ml = (float *)(ws + d.off_ml);
    cudaStream_t s = (cudaStream_t)stream;
    unsigned int *err = error_word_ptr();
    if (!err) return cuda_fail(cudaGetLastError());
    st = timed_launch(KID_DECODE_ROWS, s, [&] {
        return launch_decode_rows(p, pos, q, k, v, gamma_q, gamma_k, qhat, k_cache, v_cache, err, s);
    });
    if (st != XT_OK) return st;
    st = timed_launch(KID_DECODE_ATTN, s, [&] {
        return launch_decode_attn(p, d, pos, qhat, k_cache, v_cache, part_o, part_ml, err, s);
    });
    if (st != XT_OK) return st;
    return timed_launch(KID_DECODE_COMBINE, s, [&] {
        return launch_decode_combine(p, d, part_o, part_ml, out, lse, s);
    });
}

int xt_attn_check(void *stream) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word));
    if (e != cudaSuccess) return cuda_fail(e);
    if (word != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
        if (e != cudaSuccess) return cuda_fail(e);
        return (word & ERR_TIMEOUT) ? XT_ETIMEOUT : XT_EINVAL;
    }
    return XT_OK;
}

const char *xt_status_str(int status) {
    switch (status) {
        case XT_OK: return "ok";
        case XT_EINVAL: return "invalid argument";
        case XT_EUNSUPPORTED: return "unsupported dtype/head_dim combination";
        case XT_ECUDA: return "CUDA error";
        case XT_EWORKSPACE: return "workspace missing or too small";
        case XT_ETIMEOUT: return "a kernel timed out waiting on a barrier";
        default: return "unknown status";
    }
}

int xt_last_cuda_error(void) { return g_last_cuda_error; }

int xt_timing_enable(int on) {
    std::lock_guard<std::mutex> lk(g_timing.mu);
    g_timing.on = on != 0;
    return XT_OK;
}

int xt_timing_reset(void) {
    std::lock_guard<std::mutex> lk(g_timing.mu);
    drain_locked();
    for (int i = 0; i < KID_COUNT; ++i) { g_timing.total_ms[i] = 0.0; g_timing.launches[i] = 0; }
    return XT_OK;
}

int xt_timing_query(int kernel_id, double *total_ms, long *launches) {
    if (kernel_id < 0 || kernel_id >= KID_COUNT || !total_ms || !launches) return XT_EINVAL;
    std::lock_guard<std::mutex> lk(g_timing.mu);
    drain_locked();
    *total_ms = g_timing.total_ms[kernel_id];
    *launches = g_timing.launches[kernel_id];
    return XT_OK;
}

int xt_test_inject_stall(int kernel_mask) {
    if (kernel_mask < 0 || (kernel_mask & ~STALL_ALL) != 0) return XT_EINVAL;
    g_stall_mask.store(kernel_mask, std::memory_order_relaxed);
    return XT_OK;
}

int xt_kernel_count(void) { return KID_COUNT; }

const char *xt_kernel_name(int kernel_id) {
    if (kernel_id < 0 || kernel_id >= KID_COUNT) return "";
    return kKernelNames[kernel_id];
}

}  // extern "C"
