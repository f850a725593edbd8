// xt_simt.cu -- fp32 CUDA-core flash attention, forward and backward.
//
// This is the path for dtype fp32: TF32 tensor cores cannot meet a 1e-4
// relative error, so the contractions run as FFMA. Everything is computed in
// fp32 from inputs of type T.
//
// Operation (web pages): xtrain "Phase T5: Tiny Transformer", multi-head
// layout pipeline (per-head 2D SDPA, scores = q k^T / sqrt(hd) + causal mask,
// softmax, P V); Mint project report 5.3.1 (max-subtracted softmax);
// xtrain "Phase T15: GQA" ("What is GQA": query head qh reads kv head
// qh/group; Decision 2: a kv head's gradient is the in-order sum over its
// group). The masked keys (j > t) are skipped: the pages' -1e9 additive mask
// makes their probabilities exactly zero in fp32.
//
// Online softmax in the log2 domain: s2 = (q.k) * log2(e)/sqrt(D), running
// max m2 and sum l; lse = (m2 + log2 l) * ln 2 (natural log).
//
// Block shapes: 32 query (or key) rows per block, 8 warps, each warp owns 4
// rows; a lane owns head-dim elements lane + 32c (c < 4, D <= 128); tiles of
// 32 keys (or queries) are staged in shared memory as fp32.
#include "xt_common.cuh"
#include "xt_internal.h"

namespace xt {

namespace {

constexpr int kBR = 32;       // rows per block
constexpr int kBC = 32;       // columns (keys or queries) per tile
constexpr int kWarps = 8;
constexpr int kRowsPerWarp = kBR / kWarps;

template <typename T>
__device__ __forceinline__ void stage_tile(float *dst, int ld, const T *src, size_t src_row_stride,
                                           int row0, int nrows_valid, int D) {
    for (int e = threadIdx.x; e < kBC * D; e += blockDim.x) {
        int r = e / D, d = e - r * D;
        dst[r * ld + d] = (r < nrows_valid) ? to_f32(src[(size_t)(row0 + r) * src_row_stride + d]) : 0.f;
    }
}

// ---------------------------------------------------------------- forward
template <typename T>
__global__ void __launch_bounds__(256)
k_fwd_simt(const T *__restrict__ qhat, const T *__restrict__ khat, const T *__restrict__ v,
           T *__restrict__ out, float *__restrict__ lse, const SeqRows sr, int H, int G, int D) {
    extern __shared__ float sm[];
    const int ldk = D + 1;
    float *Qs = sm;                    // [32][D]
    float *Ks = Qs + kBR * D;          // [32][D+1]
    float *Vs = Ks + kBC * ldk;        // [32][D]
    const int bh = blockIdx.y, unit = bh / H, h = bh - unit * H, g = h / (H / G);
    const SeqSpan sp = seq_span(sr, unit);
    const int S = sp.len;
    const int q0 = blockIdx.x * kBR;
    if (q0 >= S) return;   // a packed sample shorter than this block's rows
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float sl2 = kLog2e * rsqrtf((float)D);
    const size_t qrow0 = ((size_t)sp.plane * H + h) * sr.S + sp.start;   // [.., H, S, ..] rows
    const size_t trow0 = (size_t)sp.plane * sr.S + sp.start;              // [.., S, heads, ..] rows

    const T *qsrc = qhat + qrow0 * D;
    const T *ksrc = khat + (((size_t)sp.plane * G + g) * sr.S + sp.start) * D;
    const T *vsrc = v + (trow0 * G + g) * D;   // row stride G*D
    stage_tile<T>(Qs, D, qsrc, D, q0, min(kBR, S - q0), D);

    float m[kRowsPerWarp], l[kRowsPerWarp], o[kRowsPerWarp][4];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        m[r] = -INFINITY; l[r] = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) o[r][c] = 0.f;
    }
    const int last = min(q0 + kBR, S) - 1;
    for (int j0 = 0; j0 <= last; j0 += kBC) {
        __syncthreads();
        stage_tile<T>(Ks, ldk, ksrc, D, j0, min(kBC, S - j0), D);
        stage_tile<T>(Vs, D, vsrc, (size_t)G * D, j0, min(kBC, S - j0), D);
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const int row = warp * kRowsPerWarp + r, t = q0 + row;
            if (t >= S) continue;                       // warp-uniform
            const int j = j0 + lane;
            float s = -INFINITY;
            if (j <= t) {
                float acc = 0.f;
                for (int d = 0; d < D; ++d) acc += Qs[row * D + d] * Ks[lane * ldk + d];
                s = acc * sl2;
            }
            const float mn = fmaxf(m[r], warp_max(s));
            const float p = (j <= t) ? exp2f(s - mn) : 0.f;
            const float alpha = exp2f(m[r] - mn);
            l[r] = l[r] * alpha + warp_sum(p);
            m[r] = mn;
#pragma unroll
            for (int c = 0; c < 4; ++c) o[r][c] *= alpha;
            for (int jj = 0; jj < kBC; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int d = lane + 32 * c;
                    if (d < D) o[r][c] += pj * Vs[jj * D + d];
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int t = q0 + warp * kRowsPerWarp + r;
        if (t >= S) continue;
        const float inv = 1.0f / l[r];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int d = lane + 32 * c;
            if (d < D) out[((trow0 + t) * H + h) * D + d] = from_f32<T>(o[r][c] * inv);
        }
        if (lane == 0) lse[qrow0 + t] = (m[r] + log2f(l[r])) * kLn2;
    }
}

// ---------------------------------------------------------------- dQhat
template <typename T>
__global__ void __launch_bounds__(256)
k_dq_simt(const T *__restrict__ qhat, const T *__restrict__ khat, const T *__restrict__ v,
          const T *__restrict__ dout, const float *__restrict__ lse, const float *__restrict__ dlt,
          float *__restrict__ dqhat, const SeqRows sr, int H, int G, int D) {
    extern __shared__ float sm[];
    const int ld = D + 1;
    float *Qs = sm;                 // [32][D]
    float *dOs = Qs + kBR * D;      // [32][D]
    float *Ks = dOs + kBR * D;      // [32][D+1]
    float *Vs = Ks + kBC * ld;      // [32][D+1]
    const int bh = blockIdx.y, unit = bh / H, h = bh - unit * H, g = h / (H / G);
    const SeqSpan sp = seq_span(sr, unit);
    const int S = sp.len;
    const int q0 = blockIdx.x * kBR;
    if (q0 >= S) return;   // a packed sample shorter than this block's rows
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float scale = rsqrtf((float)D);
    const float sl2 = kLog2e * scale;
    const size_t qrow0 = ((size_t)sp.plane * H + h) * sr.S + sp.start;
    const size_t trow0 = (size_t)sp.plane * sr.S + sp.start;

    stage_tile<T>(Qs, D, qhat + qrow0 * D, D, q0, min(kBR, S - q0), D);
    stage_tile<T>(dOs, D, dout + (trow0 * H + h) * D, (size_t)H * D, q0, min(kBR, S - q0), D);
    const T *ksrc = khat + (((size_t)sp.plane * G + g) * sr.S + sp.start) * D;
    const T *vsrc = v + (trow0 * G + g) * D;

    float lse2[kRowsPerWarp], dl[kRowsPerWarp], acc[kRowsPerWarp][4];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int t = q0 + warp * kRowsPerWarp + r;
        lse2[r] = t < S ? lse[qrow0 + t] * kLog2e : 0.f;
        dl[r] = t < S ? dlt[qrow0 + t] : 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
    }
    const int last = min(q0 + kBR, S) - 1;
    for (int j0 = 0; j0 <= last; j0 += kBC) {
        __syncthreads();
        stage_tile<T>(Ks, ld, ksrc, D, j0, min(kBC, S - j0), D);
        stage_tile<T>(Vs, ld, vsrc, (size_t)G * D, j0, min(kBC, S - j0), D);
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const int row = warp * kRowsPerWarp + r, t = q0 + row;
            if (t >= S) continue;
            const int j = j0 + lane;
            float ds = 0.f;
            if (j <= t) {
                float s = 0.f, dp = 0.f;
                for (int d = 0; d < D; ++d) {
                    s += Qs[row * D + d] * Ks[lane * ld + d];
                    dp += dOs[row * D + d] * Vs[lane * ld + d];
                }
                const float p = exp2f(s * sl2 - lse2[r]);
                ds = p * (dp - dl[r]);
            }
            for (int jj = 0; jj < kBC; ++jj) {
                const float dsj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int d = lane + 32 * c;
                    if (d < D) acc[r][c] += dsj * Ks[jj * ld + d];
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int t = q0 + warp * kRowsPerWarp + r;
        if (t >= S) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int d = lane + 32 * c;
            if (d < D) dqhat[(qrow0 + t) * D + d] = acc[r][c] * scale;
        }
    }
}

// ---------------------------------------------------------------- dKhat, dV
// Block = (b, kv head g, 32 key rows). It loops over the group's query heads
// r = 0..group-1 in order and, for each, over the query tiles at or after its
// keys, so the group sum of xtrain T15 Decision 2 happens in registers in a
// fixed order (no atomics).
template <typename T>
__global__ void __launch_bounds__(256)
k_dkdv_simt(const T *__restrict__ qhat, const T *__restrict__ khat, const T *__restrict__ v,
            const T *__restrict__ dout, const float *__restrict__ lse,
            const float *__restrict__ dlt, float *__restrict__ dkhat, T *__restrict__ dv,
            const SeqRows sr, int H, int G, int D) {
    extern __shared__ float sm[];
    const int ld = D + 1;
    float *Ks = sm;                 // [32][D+1] own key rows
    float *Vs = Ks + kBR * ld;      // [32][D+1]
    float *Qs = Vs + kBR * ld;      // [32][D+1] query tile
    float *dOs = Qs + kBC * ld;     // [32][D+1]
    float *lse2s = dOs + kBC * ld;  // [32]
    float *dls = lse2s + kBC;       // [32]
    const int bg = blockIdx.y, unit = bg / G, g = bg - unit * G, group = H / G;
    const SeqSpan sp = seq_span(sr, unit);
    const int S = sp.len;
    const int j0 = blockIdx.x * kBR;
    if (j0 >= S) return;   // a packed sample shorter than this block's rows
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float scale = rsqrtf((float)D);
    const float sl2 = kLog2e * scale;
    const size_t krow0 = ((size_t)sp.plane * G + g) * sr.S + sp.start;
    const size_t trow0 = (size_t)sp.plane * sr.S + sp.start;

    stage_tile<T>(Ks, ld, khat + krow0 * D, D, j0, min(kBR, S - j0), D);
    stage_tile<T>(Vs, ld, v + (trow0 * G + g) * D, (size_t)G * D, j0, min(kBR, S - j0), D);

    float dk[kRowsPerWarp][4], dvv[kRowsPerWarp][4];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) { dk[r][c] = 0.f; dvv[r][c] = 0.f; }

    for (int rr = 0; rr < group; ++rr) {
        const int h = g * group + rr;
        const size_t qrow0 = ((size_t)sp.plane * H + h) * sr.S + sp.start;
        const T *qsrc = qhat + qrow0 * D;
        const T *dsrc = dout + (trow0 * H + h) * D;
        for (int t0 = j0; t0 < S; t0 += kBC) {
            __syncthreads();
            const int nv = min(kBC, S - t0);
            stage_tile<T>(Qs, ld, qsrc, D, t0, nv, D);
            stage_tile<T>(dOs, ld, dsrc, (size_t)H * D, t0, nv, D);
            if (threadIdx.x < kBC) {
                const int t = t0 + threadIdx.x;
                lse2s[threadIdx.x] = t < S ? lse[qrow0 + t] * kLog2e : 0.f;
                dls[threadIdx.x] = t < S ? dlt[qrow0 + t] : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                const int row = warp * kRowsPerWarp + r, j = j0 + row;
                if (j >= S) continue;
                const int t = t0 + lane;
                float p = 0.f, ds = 0.f;
                if (t < S && t >= j) {
                    float s = 0.f, dp = 0.f;
                    for (int d = 0; d < D; ++d) {
                        s += Qs[lane * ld + d] * Ks[row * ld + d];
                        dp += dOs[lane * ld + d] * Vs[row * ld + d];
                    }
                    p = exp2f(s * sl2 - lse2s[lane]);
                    ds = p * (dp - dls[lane]);
                }
                for (int tt = 0; tt < kBC; ++tt) {
                    const float pt = __shfl_sync(0xffffffffu, p, tt);
                    const float dst = __shfl_sync(0xffffffffu, ds, tt);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int d = lane + 32 * c;
                        if (d < D) {
                            dvv[r][c] += pt * dOs[tt * ld + d];
                            dk[r][c] += dst * Qs[tt * ld + d];
                        }
                    }
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int j = j0 + warp * kRowsPerWarp + r;
        if (j >= S) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int d = lane + 32 * c;
            if (d < D) {
                dkhat[(krow0 + j) * D + d] = dk[r][c] * scale;
                dv[((trow0 + j) * G + g) * D + d] = from_f32<T>(dvv[r][c]);
            }
        }
    }
}

template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t launch_fwd_simt(const Problem &p, const void *qhat, const void *khat, const void *v,
                            void *out, float *lse, cudaStream_t st) {
    dim3 grid((p.max_len + kBR - 1) / kBR, p.units * p.H);
    size_t smem = sizeof(float) * (kBR * p.D + kBC * (p.D + 1) + kBC * p.D);
    cudaError_t e;
    if (p.dtype == 1) {
        if ((e = allow_smem(k_fwd_simt<bf16>, smem)) != cudaSuccess) return e;
        k_fwd_simt<bf16><<<grid, 256, smem, st>>>((const bf16 *)qhat, (const bf16 *)khat,
                                                  (const bf16 *)v, (bf16 *)out, lse,
                                                  SeqRows{p.cu, p.S, p.max_len}, p.H, p.G, p.D);
    } else {
        if ((e = allow_smem(k_fwd_simt<float>, smem)) != cudaSuccess) return e;
        k_fwd_simt<float><<<grid, 256, smem, st>>>((const float *)qhat, (const float *)khat,
                                                   (const float *)v, (float *)out, lse,
                                                   SeqRows{p.cu, p.S, p.max_len}, p.H, p.G, p.D);
    }
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq_simt(const Problem &p, const void *qhat, const void *khat,
                               const void *v, const void *dout, const float *lse,
                               const float *dlt, float *dqhat, cudaStream_t st) {
    dim3 grid((p.max_len + kBR - 1) / kBR, p.units * p.H);
    size_t smem = sizeof(float) * (2 * kBR * p.D + 2 * kBC * (p.D + 1));
    cudaError_t e;
    if (p.dtype == 1) {
        if ((e = allow_smem(k_dq_simt<bf16>, smem)) != cudaSuccess) return e;
        k_dq_simt<bf16><<<grid, 256, smem, st>>>((const bf16 *)qhat, (const bf16 *)khat,
                                                 (const bf16 *)v, (const bf16 *)dout, lse, dlt,
                                                 dqhat, SeqRows{p.cu, p.S, p.max_len}, p.H,
                                                 p.G, p.D);
    } else {
        if ((e = allow_smem(k_dq_simt<float>, smem)) != cudaSuccess) return e;
        k_dq_simt<float><<<grid, 256, smem, st>>>((const float *)qhat, (const float *)khat,
                                                  (const float *)v, (const float *)dout, lse,
                                                  dlt, dqhat, SeqRows{p.cu, p.S, p.max_len},
                                                  p.H, p.G, p.D);
    }
    return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv_simt(const Problem &p, const void *qhat, const void *khat,
                                 const void *v, const void *dout, const float *lse,
                                 const float *dlt, float *dkhat, void *dv, cudaStream_t st) {
    dim3 grid((p.max_len + kBR - 1) / kBR, p.units * p.G);
    size_t smem = sizeof(float) * (4 * kBR * (p.D + 1) + 2 * kBC);
    cudaError_t e;
    if (p.dtype == 1) {
        if ((e = allow_smem(k_dkdv_simt<bf16>, smem)) != cudaSuccess) return e;
        k_dkdv_simt<bf16><<<grid, 256, smem, st>>>((const bf16 *)qhat, (const bf16 *)khat,
                                                   (const bf16 *)v, (const bf16 *)dout, lse, dlt,
                                                   dkhat, (bf16 *)dv,
                                                   SeqRows{p.cu, p.S, p.max_len}, p.H, p.G, p.D);
    } else {
        if ((e = allow_smem(k_dkdv_simt<float>, smem)) != cudaSuccess) return e;
        k_dkdv_simt<float><<<grid, 256, smem, st>>>((const float *)qhat, (const float *)khat,
                                                    (const float *)v, (const float *)dout, lse,
                                                    dlt, dkhat, (float *)dv,
                                                    SeqRows{p.cu, p.S, p.max_len}, p.H, p.G, p.D);
    }
    return cudaGetLastError();
}

}  // namespace xt
