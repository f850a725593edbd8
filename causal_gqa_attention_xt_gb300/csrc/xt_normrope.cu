// xt_normrope.cu -- HBM-bound kernels around the attention:
//   * prologue: per-head QK-RMSNorm followed by rotate_half RoPE (forward);
//   * bwd_pre:  Dlt = rowsum(dO * O) for the softmax backward;
//   * epilogue: RoPE backward (rotation by the negative angle) and RMSNorm
//               backward, with per-block dgamma partials;
//   * dgamma_reduce: fixed-order sum of those partials.
//
// The operations (web pages): xtrain "Phase T9: Export to xserv",
// architecture-diff table and Decision 1 (norm over each [head_dim] vector of
// Q and K with one shared [head_dim] gamma, then rotate_half RoPE with
// freq = theta^(-2i/hd) and pos = token row); Mint project report 5.4.1-5.4.4
// (pair (i, i + hd/2), x' = x cos - y sin, y' = x sin + y cos; backward =
// rotation by the negative angle) and 5.5.1-5.5.2 (RMSNorm forward and
// backward, dgamma summed over rows); xtrain "Phase T12: bf16 mixed
// precision" (norm and RoPE computed in fp32 on bf16 activations).
//
// Layout of work: one block takes kRowsPerBlock consecutive positions of one
// batch element and every q and k head at those positions, so the cos/sin of
// those positions are computed once per block into shared memory. A row of D
// elements is handled by tpr = D / (2 * VEC) lanes, each owning VEC elements of
// the first half and the VEC matching elements of the second half (the RoPE
// pair), read and written with 16-byte accesses.
#include "xt_common.cuh"
#include "xt_internal.h"

namespace xt {

namespace {

constexpr int kThreads = 256;

__host__ __device__ inline int pow2_at_least(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

// cos/sin of angle (s * theta^(-2i/D)) for the block's positions, i < D/2.
// The angle is formed in double (position times the host's double inverse
// frequency, as in the pages' formula) and reduced by 2*pi in double before
// an fp32 sincos, so that large positions keep their accuracy.
__device__ void rope_table(float *cs, float *sn, int s0, int ns, int D, const RopeFreqs &fr) {
    const int half = D / 2;
    const double two_pi = 6.283185307179586476925;
    for (int e = threadIdx.x; e < ns * half; e += blockDim.x) {
        int si = e / half, i = e - si * half;
        double ang = (double)(s0 + si) * fr.inv_freq[i];
        double turns = rint(ang * (1.0 / two_pi));
        float red = (float)fma(-turns, two_pi, ang);
        float sv, cv;
        sincosf(red, &sv, &cv);
        cs[e] = cv;
        sn[e] = sv;
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
k_prologue(const T *__restrict__ q, const T *__restrict__ k, const float *__restrict__ gq,
           const float *__restrict__ gk, T *__restrict__ qhat, T *__restrict__ khat,
           float *__restrict__ rstd_q, float *__restrict__ rstd_k, int S, int H, int G, int D,
           float eps, const RopeFreqs fr) {
    constexpr int VEC = 16 / sizeof(T);
    extern __shared__ float smem[];
    const int half = D / 2;
    const int blocks_s = (S + kRowsPerBlock - 1) / kRowsPerBlock;
    const int b = blockIdx.x / blocks_s;
    const int s0 = (blockIdx.x - b * blocks_s) * kRowsPerBlock;
    const int ns = min(kRowsPerBlock, S - s0);
    float *cs = smem, *sn = smem + kRowsPerBlock * half;
    rope_table(cs, sn, s0, ns, D, fr);
    __syncthreads();

    const int chunks = half / VEC;             // lanes that carry data
    const int tpr = pow2_at_least(chunks);     // lanes per row (power of two)
    const int c = threadIdx.x & (tpr - 1);
    const int rows_per_iter = kThreads / tpr;
    const int NH = H + G;
    const int nrows = ns * NH;
    const float inv_d = 1.0f / (float)D;
    for (int rr = threadIdx.x / tpr; rr < ((nrows + rows_per_iter - 1) / rows_per_iter) * rows_per_iter;
         rr += rows_per_iter) {
        const bool row_ok = rr < nrows;
        const bool lane_ok = row_ok && c < chunks;
        int si = 0, head = 0;
        if (row_ok) { si = rr / NH; head = rr - si * NH; }
        const int s = s0 + si;
        const bool isq = head < H;
        const T *x = isq ? q + (((size_t)b * S + s) * H + head) * D
                         : k + (((size_t)b * S + s) * G + (head - H)) * D;
        const float *gamma = isq ? gq : gk;
        float lo[VEC], hi[VEC];
        float ss = 0.f;
        if (lane_ok) {
            load16<T>(x + c * VEC, lo);
            load16<T>(x + half + c * VEC, hi);
#pragma unroll
            for (int e = 0; e < VEC; ++e) ss += lo[e] * lo[e] + hi[e] * hi[e];
        }
        ss = group_sum(ss, tpr);
        const float r = 1.0f / sqrtf(ss * inv_d + eps);
        if (lane_ok) {
            float olo[VEC], ohi[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int i = c * VEC + e;
                const float ylo = lo[e] * r * gamma[i];
                const float yhi = hi[e] * r * gamma[half + i];
                const float cv = cs[si * half + i], sv = sn[si * half + i];
                olo[e] = ylo * cv - yhi * sv;
                ohi[e] = ylo * sv + yhi * cv;
            }
            T *y = isq ? qhat + (((size_t)b * H + head) * S + s) * D
                       : khat + (((size_t)b * G + (head - H)) * S + s) * D;
            store16<T>(y + c * VEC, olo);
            store16<T>(y + half + c * VEC, ohi);
            if (c == 0) {
                if (isq) rstd_q[((size_t)b * S + s) * H + head] = r;
                else rstd_k[((size_t)b * S + s) * G + (head - H)] = r;
            }
        }
    }
}

// Dlt[b, h, s] = sum_d dO[b, s, h, d] * O[b, s, h, d]
template <typename T>
__global__ void __launch_bounds__(kThreads)
k_bwd_pre(const T *__restrict__ out, const T *__restrict__ dout, float *__restrict__ dlt,
          int S, int H, int D, long rows) {
    constexpr int VEC = 16 / sizeof(T);
    const int chunks = D / VEC;
    const int tpr = pow2_at_least(chunks);
    const int c = threadIdx.x & (tpr - 1);
    const long rows_per_grid = (long)gridDim.x * (kThreads / tpr);
    for (long row = (long)blockIdx.x * (kThreads / tpr) + threadIdx.x / tpr;
         row < ((rows + rows_per_grid - 1) / rows_per_grid) * rows_per_grid; row += rows_per_grid) {
        float acc = 0.f;
        if (row < rows && c < chunks) {
            float a[VEC], g[VEC];
            load16<T>(out + row * D + c * VEC, a);
            load16<T>(dout + row * D + c * VEC, g);
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc += a[e] * g[e];
        }
        acc = group_sum(acc, tpr);
        if (row < rows && c == 0) {
            const long bs = row / H;
            const int h = (int)(row - bs * H);
            const long b = bs / S;
            const int s = (int)(bs - b * S);
            dlt[((size_t)b * H + h) * S + s] = acc;
        }
    }
}

// dq = RMSNorm_bwd(RoPE_bwd(dqhat)), likewise dk; per-block dgamma partials.
template <typename T>
__global__ void __launch_bounds__(kThreads)
k_epilogue(const float *__restrict__ dqhat, const float *__restrict__ dkhat,
           const T *__restrict__ q, const T *__restrict__ k, const float *__restrict__ gq,
           const float *__restrict__ gk, const float *__restrict__ rstd_q,
           const float *__restrict__ rstd_k, T *__restrict__ dq, T *__restrict__ dk,
           float *__restrict__ part_q, float *__restrict__ part_k, int S, int H, int G, int D,
           const RopeFreqs fr) {
    constexpr int VEC = 16 / sizeof(T);
    extern __shared__ float smem[];
    const int half = D / 2;
    const int blocks_s = (S + kRowsPerBlock - 1) / kRowsPerBlock;
    const int b = blockIdx.x / blocks_s;
    const int s0 = (blockIdx.x - b * blocks_s) * kRowsPerBlock;
    const int ns = min(kRowsPerBlock, S - s0);
    float *cs = smem, *sn = smem + kRowsPerBlock * half;
    const int chunks = half / VEC;
    const int tpr = pow2_at_least(chunks);
    const int rows_per_iter = kThreads / tpr;
    float *red = smem + 2 * kRowsPerBlock * half;   // [rows_per_iter][D]
    rope_table(cs, sn, s0, ns, D, fr);
    __syncthreads();

    const int c = threadIdx.x & (tpr - 1);
    const int NH = H + G;
    const int nrows = ns * NH;
    const float inv_d = 1.0f / (float)D;
    float accq[2 * VEC], acck[2 * VEC];
#pragma unroll
    for (int e = 0; e < 2 * VEC; ++e) { accq[e] = 0.f; acck[e] = 0.f; }

    for (int rr = threadIdx.x / tpr; rr < ((nrows + rows_per_iter - 1) / rows_per_iter) * rows_per_iter;
         rr += rows_per_iter) {
        const bool row_ok = rr < nrows;
        const bool lane_ok = row_ok && c < chunks;
        int si = 0, head = 0;
        if (row_ok) { si = rr / NH; head = rr - si * NH; }
        const int s = s0 + si;
        const bool isq = head < H;
        const int hh = isq ? head : head - H;
        const int NHx = isq ? H : G;
        const T *x = (isq ? q : k) + (((size_t)b * S + s) * NHx + hh) * D;
        const float *g = (isq ? dqhat : dkhat) + (((size_t)b * NHx + hh) * S + s) * D;
        const float *gamma = isq ? gq : gk;
        float r = 0.f;
        if (row_ok) r = isq ? rstd_q[((size_t)b * S + s) * H + hh] : rstd_k[((size_t)b * S + s) * G + hh];
        float xl[VEC], xh[VEC], dyl[VEC], dyh[VEC];
        float dot = 0.f;
        if (lane_ok) {
            float gl[VEC], gh[VEC];
            load16<T>(x + c * VEC, xl);
            load16<T>(x + half + c * VEC, xh);
            *reinterpret_cast<float4 *>(gl) = *reinterpret_cast<const float4 *>(g + c * VEC);
            *reinterpret_cast<float4 *>(gh) = *reinterpret_cast<const float4 *>(g + half + c * VEC);
            if constexpr (VEC == 8) {
                *reinterpret_cast<float4 *>(gl + 4) = *reinterpret_cast<const float4 *>(g + c * VEC + 4);
                *reinterpret_cast<float4 *>(gh + 4) = *reinterpret_cast<const float4 *>(g + half + c * VEC + 4);
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int i = c * VEC + e;
                const float cv = cs[si * half + i], sv = sn[si * half + i];
                // rotation by the negative angle
                dyl[e] = gl[e] * cv + gh[e] * sv;
                dyh[e] = gh[e] * cv - gl[e] * sv;
                dot += gamma[i] * dyl[e] * xl[e] + gamma[half + i] * dyh[e] * xh[e];
            }
        }
        dot = group_sum(dot, tpr);
        if (lane_ok) {
            const float corr = dot * r * r * r * inv_d;
            float ol[VEC], oh[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int i = c * VEC + e;
                ol[e] = gamma[i] * dyl[e] * r - xl[e] * corr;
                oh[e] = gamma[half + i] * dyh[e] * r - xh[e] * corr;
                if (isq) { accq[e] += dyl[e] * xl[e] * r; accq[VEC + e] += dyh[e] * xh[e] * r; }
                else { acck[e] += dyl[e] * xl[e] * r; acck[VEC + e] += dyh[e] * xh[e] * r; }
            }
            T *dst = (isq ? dq : dk) + (((size_t)b * S + s) * NHx + hh) * D;
            store16<T>(dst + c * VEC, ol);
            store16<T>(dst + half + c * VEC, oh);
        }
    }
    // Fixed-order block reduction of the dgamma partials: row-slot major.
    const int slot = threadIdx.x / tpr;
    for (int pass = 0; pass < 2; ++pass) {
        const float *acc = pass == 0 ? accq : acck;
        __syncthreads();
        if (c < chunks) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                red[slot * D + c * VEC + e] = acc[e];
                red[slot * D + half + c * VEC + e] = acc[VEC + e];
            }
        }
        __syncthreads();
        for (int d = threadIdx.x; d < D; d += kThreads) {
            float sum = 0.f;
            for (int sl = 0; sl < rows_per_iter; ++sl) sum += red[sl * D + d];
            (pass == 0 ? part_q : part_k)[(size_t)blockIdx.x * D + d] = sum;
        }
    }
}

__global__ void k_dgamma_reduce(const float *__restrict__ part_q, const float *__restrict__ part_k,
                                int nparts, int D, float *__restrict__ dgq, float *__restrict__ dgk) {
    const float *part = blockIdx.x == 0 ? part_q : part_k;
    float *out = blockIdx.x == 0 ? dgq : dgk;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float sum = 0.f;
        for (int p = 0; p < nparts; ++p) sum += part[(size_t)p * D + d];
        out[d] = sum;
    }
}

size_t table_smem(int D) { return sizeof(float) * 2 * kRowsPerBlock * (D / 2); }

}  // namespace

RopeFreqs rope_freqs(const Problem &p) {
    RopeFreqs f;
    for (int i = 0; i < kMaxHalfDim; ++i)
        f.inv_freq[i] = (i < p.D / 2) ? pow(p.theta, -2.0 * (double)i / (double)p.D) : 0.0;
    return f;
}

cudaError_t launch_prologue(const Problem &p, const void *q, const void *k, const float *gq,
                            const float *gk, void *qhat, void *khat, float *rstd_q,
                            float *rstd_k, cudaStream_t st) {
    dim3 grid(normrope_blocks(p));
    size_t smem = table_smem(p.D);
    if (p.dtype == 1)
        k_prologue<bf16><<<grid, kThreads, smem, st>>>(
            (const bf16 *)q, (const bf16 *)k, gq, gk, (bf16 *)qhat, (bf16 *)khat, rstd_q, rstd_k,
            p.S, p.H, p.G, p.D, p.eps, rope_freqs(p));
    else
        k_prologue<float><<<grid, kThreads, smem, st>>>(
            (const float *)q, (const float *)k, gq, gk, (float *)qhat, (float *)khat, rstd_q,
            rstd_k, p.S, p.H, p.G, p.D, p.eps, rope_freqs(p));
    return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const Problem &p, const void *out, const void *dout, float *dlt,
                           cudaStream_t st) {
    long rows = (long)p.B * p.S * p.H;
    int blocks = (int)((rows + 255) / 256);
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (p.dtype == 1)
        k_bwd_pre<bf16><<<blocks, kThreads, 0, st>>>((const bf16 *)out, (const bf16 *)dout, dlt,
                                                     p.S, p.H, p.D, rows);
    else
        k_bwd_pre<float><<<blocks, kThreads, 0, st>>>((const float *)out, (const float *)dout,
                                                      dlt, p.S, p.H, p.D, rows);
    return cudaGetLastError();
}

cudaError_t launch_epilogue(const Problem &p, const float *dqhat, const float *dkhat,
                            const void *q, const void *k, const float *gq, const float *gk,
                            const float *rstd_q, const float *rstd_k, void *dq, void *dk,
                            float *part_q, float *part_k, cudaStream_t st) {
    dim3 grid(normrope_blocks(p));
    const int vec = p.dtype == 1 ? 8 : 4;
    const int tpr = pow2_at_least((p.D / 2) / vec);
    size_t smem = table_smem(p.D) + sizeof(float) * (kThreads / tpr) * p.D;
    if (p.dtype == 1)
        k_epilogue<bf16><<<grid, kThreads, smem, st>>>(
            dqhat, dkhat, (const bf16 *)q, (const bf16 *)k, gq, gk, rstd_q, rstd_k, (bf16 *)dq,
            (bf16 *)dk, part_q, part_k, p.S, p.H, p.G, p.D, rope_freqs(p));
    else
        k_epilogue<float><<<grid, kThreads, smem, st>>>(
            dqhat, dkhat, (const float *)q, (const float *)k, gq, gk, rstd_q, rstd_k,
            (float *)dq, (float *)dk, part_q, part_k, p.S, p.H, p.G, p.D, rope_freqs(p));
    return cudaGetLastError();
}

cudaError_t launch_dgamma_reduce(const Problem &p, const float *part_q, const float *part_k,
                                 int nparts, float *dgq, float *dgk, cudaStream_t st) {
    k_dgamma_reduce<<<2, 128, 0, st>>>(part_q, part_k, nparts, p.D, dgq, dgk);
    return cudaGetLastError();
}

}  // namespace xt
