// xt_decode.cu -- one decode step of the attention core against a key/value
// cache (Mint project report, 10.3 "KV cache"): the new token of each batch
// element, at position pos[b], computes its own q, k, v; its k and v are
// appended to the cache; its query attends over every cached key, all of which
// are at or before the new position (so the causal mask is implicit):
// s_j = q^R . k^R_j / sqrt(D) for j = 0..pos, p = softmax(s), a = sum_j p_j v_j,
// which the page states equals the full-sequence attention at that row. The
// new q and k rows are normed and rotated exactly as in training (xtrain
// "Phase T9: Export to xserv", Decision 1 and architecture-diff table), and
// query head h reads kv head h / (H / G) (xtrain "Phase T15: GQA").
//
// Caches are head-major, [B, G, S_max, D] (the layout of the training
// forward's k_hat), so a kv head's cached rows are one contiguous run.
//
// Three kernels (the work is a matrix-vector product per kv head, bound by
// reading the cache from HBM, so it runs on the CUDA cores):
//  * k_decode_rows: one warp per new row: q heads normed + rotated into an
//    fp32 scratch (rounded through the storage type, as the training forward
//    rounds q_hat), k heads normed + rotated into the k cache at row pos[b], v
//    rows copied into the v cache. A position outside [0, S_max) raises an
//    error bit (reported as XT_EINVAL by xt_attn_check) and the batch element
//    is skipped.
//  * k_decode_attn: grid (kv head x chunk of <= 16 of its query heads, key
//    split). A CTA streams its split's cached rows, 64 keys per tile, through
//    a 2-stage shared-memory ring filled by bulk asynchronous copies; one
//    thread per (head, key) forms the score over D, one warp per head keeps
//    the running max and sum, one thread per (head, column) accumulates P V.
//    It writes the split's partial (max, sum, unnormalised output).
//  * k_decode_combine: per (b, h), the splits merged in split order, so the
//    result does not depend on scheduling: m = max m_s, l = sum l_s 2^(m_s-m),
//    o = sum o_s 2^(m_s-m) / l; lse = (m + log2 l) ln 2 (natural log).
#include "xt_common.cuh"
#include "xt_internal.h"
#include "xt_rope.cuh"
#include "xt_tc.cuh"

namespace xt {

namespace {

using tc::bulk_load;
using tc::mbar_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;

constexpr int kDecThreads = 256;
constexpr int kDecKeys = 64;        // keys per staged tile
constexpr int kDecHeads = 16;       // query heads per CTA (a chunk of the group)
constexpr int kDecStages = 2;
constexpr int kDecAcc = kDecHeads * 128 / kDecThreads;   // outputs per thread (D <= 128)

// ---------------------------------------------------------------- new rows
template <typename T>
__global__ void __launch_bounds__(256)
k_decode_rows(const int *__restrict__ pos, const T *__restrict__ q, const T *__restrict__ k,
              const T *__restrict__ v, const float *__restrict__ gq, const float *__restrict__ gk,
              float *__restrict__ qhat, T *__restrict__ kc, T *__restrict__ vc, int S_max, int H,
              int G, int D, float eps, const __grid_constant__ RopeConsts rc, unsigned int *err) {
    const int b = blockIdx.y;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);   // H q rows, G k rows, G v rows
    const int lane = threadIdx.x & 31;
    if (row >= H + 2 * G) return;
    const int p = pos[b];
    if (p < 0 || p >= S_max) {
        if (row == 0 && lane == 0) atomicOr(err, ERR_BADPOS);
        return;
    }
    if (row >= H + G) {   // v row: into the cache as it is
        const int g = row - H - G;
        const T *src = v + ((size_t)b * G + g) * D;
        T *dst = vc + (((size_t)b * G + g) * S_max + p) * D;
        for (int d = lane; d < D; d += 32) dst[d] = src[d];
        return;
    }
    const bool isq = row < H;
    const int hh = isq ? row : row - H;
    const T *x = isq ? q + ((size_t)b * H + hh) * D : k + ((size_t)b * G + hh) * D;
    const float *gamma = isq ? gq : gk;
    const int half = D / 2;
    // lane holds the RoPE pairs (i, i + D/2) for i = lane and lane + 32
    float lo[2], hi[2];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int i = lane + 32 * j;
        lo[j] = 0.f;
        hi[j] = 0.f;
        if (i < half) {
            lo[j] = to_f32(x[i]);
            hi[j] = to_f32(x[i + half]);
        }
        ss = fmaf(lo[j], lo[j], fmaf(hi[j], hi[j], ss));
    }
    ss = warp_sum(ss);
    const float r = rsqrtf(fmaf(ss, 1.0f / (float)D, eps));
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int i = lane + 32 * j;
        if (i >= half) continue;
        const float ylo = lo[j] * (r * gamma[i]);
        const float yhi = hi[j] * (r * gamma[i + half]);
        const float2 cs = rope_cos_sin(p, rc.fhi[i], rc.flo[i], rc.fd[i]);
        const float olo = ylo * cs.x - yhi * cs.y;
        const float ohi = ylo * cs.y + yhi * cs.x;
        if (isq) {
            float *dst = qhat + ((size_t)b * H + hh) * D;
            dst[i] = to_f32(from_f32<T>(olo));
            dst[i + half] = to_f32(from_f32<T>(ohi));
        } else {
            T *dst = kc + (((size_t)b * G + hh) * S_max + p) * D;
            dst[i] = from_f32<T>(olo);
            dst[i + half] = from_f32<T>(ohi);
        }
    }
}

// ---------------------------------------------------------------- attention
template <typename T>
__global__ void __launch_bounds__(kDecThreads, 2)
k_decode_attn(const int *__restrict__ pos, const float *__restrict__ qhat,
              const T *__restrict__ kc, const T *__restrict__ vc, float *__restrict__ part_o,
              float *__restrict__ part_ml, int B, int S_max, int H, int G, int D, int L, int nhc,
              unsigned int *err) {
    constexpr int VEC = 16 / sizeof(T);
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t full[kDecStages];
    __shared__ float m_run[kDecHeads], l_run[kDecHeads], alpha[kDecHeads];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hc = blockIdx.x % nhc;
    const int bg = blockIdx.x / nhc;
    const int g = bg % G, b = bg / G;
    const int split = blockIdx.y;
    const int group = H / G;
    const int h0 = g * group + hc * kDecHeads;
    const int nh = min(kDecHeads, group - hc * kDecHeads);
    const int rowb = D * (int)sizeof(T);
    const int tile_bytes = kDecKeys * rowb;
    unsigned char *ring = smem;                                         // [stage][K | V]
    float *qs = reinterpret_cast<float *>(smem + kDecStages * 2 * tile_bytes);   // [head][D]
    float *sp = qs + kDecHeads * D;                                     // [head][key]

    const int p = pos[b];
    const bool valid = p >= 0 && p < S_max;
    const int k0 = split * L;
    const int k1 = valid ? min(k0 + L, p + 1) : k0;                     // keys [k0, k1)
    const int ntiles = k1 > k0 ? (k1 - k0 + kDecKeys - 1) / kDecKeys : 0;
    const size_t crow0 = ((size_t)b * G + g) * S_max;

    if (tid == 0) {
        for (int st = 0; st < kDecStages; ++st) mbar_init(&full[st], 1);
        tc::fence_barrier_init();
    }
    for (int e = tid; e < nh * D; e += kDecThreads) qs[e] = qhat[((size_t)b * H + h0) * D + e];
    if (tid < kDecHeads) {
        m_run[tid] = -INFINITY;
        l_run[tid] = 0.f;
    }
    __syncthreads();
    auto issue = [&](int i) {   // thread 0
        const int st = i % kDecStages;
        const int ks = k0 + i * kDecKeys, n = min(kDecKeys, k1 - ks);
        unsigned char *base = ring + st * 2 * tile_bytes;
        mbar_expect_tx(&full[st], (uint32_t)(2 * n * rowb));
        bulk_load(base, kc + (crow0 + ks) * D, (uint32_t)(n * rowb), &full[st]);
        bulk_load(base + tile_bytes, vc + (crow0 + ks) * D, (uint32_t)(n * rowb), &full[st]);
    };
    if (tid == 0)
        for (int i = 0; i < ntiles && i < kDecStages; ++i) issue(i);

    float acc[kDecAcc];
#pragma unroll
    for (int r = 0; r < kDecAcc; ++r) acc[r] = 0.f;
    const float sl2 = kLog2e * rsqrtf((float)D);
    const int nch = D / VEC;
    bool ok = true;
    for (int i = 0; i < ntiles; ++i) {
        const int st = i % kDecStages;
        const int n = min(kDecKeys, k1 - (k0 + i * kDecKeys));
        ok = mbar_wait(&full[st], (uint32_t)((i / kDecStages) & 1), nullptr);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(err, ERR_TIMEOUT);
                for (int j = i; j < ntiles && j < i + kDecStages; ++j)
                    mbar_wait(&full[j % kDecStages], (uint32_t)((j / kDecStages) & 1), nullptr);
            }
            return;
        }
        const unsigned char *base = ring + st * 2 * tile_bytes;
        const T *Kt = reinterpret_cast<const T *>(base);
        const T *Vt = reinterpret_cast<const T *>(base + tile_bytes);
        // scores in the log2 domain, one thread per (head, key); the 16-byte
        // chunks are visited in a lane-rotated order so that the 8 lanes of a
        // quarter warp read 8 different bank groups of their 8 rows
        for (int e = tid; e < nh * kDecKeys; e += kDecThreads) {
            const int hh = e / kDecKeys, key = e - hh * kDecKeys;
            float s = -INFINITY;
            if (key < n) {
                const T *kr = Kt + (size_t)key * D;
                const float *qr = qs + hh * D;
                float a0 = 0.f, a1 = 0.f;
                for (int c0 = 0; c0 < nch; ++c0) {
                    const int c = (c0 + lane) % nch;
                    float kv[VEC];
                    load16<T>(kr + c * VEC, kv);
#pragma unroll
                    for (int x = 0; x < VEC; x += 2) {
                        a0 = fmaf(qr[c * VEC + x], kv[x], a0);
                        a1 = fmaf(qr[c * VEC + x + 1], kv[x + 1], a1);
                    }
                }
                s = (a0 + a1) * sl2;
            }
            sp[hh * kDecKeys + key] = s;
        }
        __syncthreads();
        // online softmax, one warp per head
        for (int hh = warp; hh < nh; hh += kDecThreads / 32) {
            const float s0 = sp[hh * kDecKeys + lane], s1 = sp[hh * kDecKeys + 32 + lane];
            const float mo = m_run[hh];
            const float mn = fmaxf(mo, warp_max(fmaxf(s0, s1)));   // finite: every tile has a key
            const float p0 = exp2f(s0 - mn), p1 = exp2f(s1 - mn);
            const float lt = warp_sum(p0 + p1);
            sp[hh * kDecKeys + lane] = p0;
            sp[hh * kDecKeys + 32 + lane] = p1;
            __syncwarp();
            if (lane == 0) {
                const float a = exp2f(mo - mn);   // 0 on the first tile
                alpha[hh] = a;
                m_run[hh] = mn;
                l_run[hh] = l_run[hh] * a + lt;
            }
        }
        __syncthreads();
        // O = alpha O + P V, one thread per (head, column)
#pragma unroll
        for (int r = 0; r < kDecAcc; ++r) {
            const int o = tid + kDecThreads * r;
            if (o < nh * D) {
                const int hh = o / D, d = o - hh * D;
                const float *pr = sp + hh * kDecKeys;
                float a = acc[r] * alpha[hh];
                for (int key = 0; key < n; ++key) a = fmaf(pr[key], to_f32(Vt[(size_t)key * D + d]), a);
                acc[r] = a;
            }
        }
        __syncthreads();   // the stage is free
        if (tid == 0 && i + kDecStages < ntiles) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(i + kDecStages);
        }
    }
    // partials of this split (m in the log2 domain; o unnormalised)
    const size_t pbase = (size_t)split * B + b;
#pragma unroll
    for (int r = 0; r < kDecAcc; ++r) {
        const int o = tid + kDecThreads * r;
        if (o < nh * D) part_o[(pbase * H + h0) * D + o] = acc[r];
    }
    if (tid < nh) {
        part_ml[((pbase * H) + h0 + tid) * 2] = m_run[tid];
        part_ml[((pbase * H) + h0 + tid) * 2 + 1] = l_run[tid];
    }
}

// ---------------------------------------------------------------- combine
template <typename T>
__global__ void __launch_bounds__(128)
k_decode_combine(const float *__restrict__ part_o, const float *__restrict__ part_ml,
                 T *__restrict__ out, float *__restrict__ lse, int B, int H, int D, int nsplit) {
    const int bh = blockIdx.x;   // b * H + h
    float m = -INFINITY;
    for (int s = 0; s < nsplit; ++s)
        if (part_ml[((size_t)s * B * H + bh) * 2 + 1] > 0.f)
            m = fmaxf(m, part_ml[((size_t)s * B * H + bh) * 2]);
    float l = 0.f;
    for (int s = 0; s < nsplit; ++s) {
        const float ls = part_ml[((size_t)s * B * H + bh) * 2 + 1];
        if (ls > 0.f) l += ls * exp2f(part_ml[((size_t)s * B * H + bh) * 2] - m);
    }
    const float inv_l = l > 0.f ? 1.0f / l : 0.f;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float o = 0.f;
        for (int s = 0; s < nsplit; ++s) {
            const float ls = part_ml[((size_t)s * B * H + bh) * 2 + 1];
            if (ls > 0.f)
                o += part_o[((size_t)s * B * H + bh) * D + d] *
                     exp2f(part_ml[((size_t)s * B * H + bh) * 2] - m);
        }
        out[(size_t)bh * D + d] = from_f32<T>(o * inv_l);
    }
    if (threadIdx.x == 0) lse[bh] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

DecodePlan decode_plan(const Problem &p) {
    DecodePlan d = {};
    const int group = p.H / p.G;
    d.nhc = (group + kDecHeads - 1) / kDecHeads;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        sms = 148;
    const long units = (long)p.B * p.G * d.nhc;
    const long tiles = (p.S + kDecKeys - 1) / kDecKeys;
    long ns = (2L * sms + units - 1) / units;   // about two CTAs per SM
    if (ns > tiles) ns = tiles;
    if (ns < 1) ns = 1;
    const long per = (tiles + ns - 1) / ns;
    d.L = (int)(per * kDecKeys);
    d.nsplit = (int)((p.S + d.L - 1) / d.L);
    const size_t align = 256;
    auto up = [&](size_t x) { return (x + align - 1) & ~(align - 1); };
    d.off_qhat = 0;
    d.off_o = up(sizeof(float) * (size_t)p.B * p.H * p.D);
    d.off_ml = d.off_o + up(sizeof(float) * (size_t)d.nsplit * p.B * p.H * p.D);
    d.total = d.off_ml + up(sizeof(float) * 2 * (size_t)d.nsplit * p.B * p.H);
    return d;
}

cudaError_t launch_decode_rows(const Problem &p, const int *pos, const void *q, const void *k,
                               const void *v, const float *gq, const float *gk, float *qhat,
                               void *kc, void *vc, unsigned int *err, cudaStream_t st) {
    dim3 grid((p.H + 2 * p.G + 7) / 8, p.B);
    const RopeConsts rc = make_rope_consts(p.theta, p.D);
    if (p.dtype == 1)
        k_decode_rows<bf16><<<grid, 256, 0, st>>>(pos, (const bf16 *)q, (const bf16 *)k,
                                                  (const bf16 *)v, gq, gk, qhat, (bf16 *)kc,
                                                  (bf16 *)vc, p.S, p.H, p.G, p.D, p.eps, rc, err);
    else
        k_decode_rows<float><<<grid, 256, 0, st>>>(pos, (const float *)q, (const float *)k,
                                                   (const float *)v, gq, gk, qhat, (float *)kc,
                                                   (float *)vc, p.S, p.H, p.G, p.D, p.eps, rc, err);
    return cudaGetLastError();
}

cudaError_t launch_decode_attn(const Problem &p, const DecodePlan &d, const int *pos,
                               const float *qhat, const void *kc, const void *vc, float *part_o,
                               float *part_ml, unsigned int *err, cudaStream_t st) {
    const size_t es = p.dtype == 1 ? 2 : 4;
    const size_t smem = (size_t)kDecStages * 2 * kDecKeys * p.D * es +
                        sizeof(float) * kDecHeads * (p.D + kDecKeys);
    dim3 grid((unsigned)((long)p.B * p.G * d.nhc), (unsigned)d.nsplit);
    cudaError_t e;
    if (p.dtype == 1) {
        if ((e = set_smem(k_decode_attn<bf16>, smem)) != cudaSuccess) return e;
        k_decode_attn<bf16><<<grid, kDecThreads, smem, st>>>(pos, qhat, (const bf16 *)kc,
                                                             (const bf16 *)vc, part_o, part_ml, p.B,
                                                             p.S, p.H, p.G, p.D, d.L, d.nhc, err);
    } else {
        if ((e = set_smem(k_decode_attn<float>, smem)) != cudaSuccess) return e;
        k_decode_attn<float><<<grid, kDecThreads, smem, st>>>(pos, qhat, (const float *)kc,
                                                              (const float *)vc, part_o, part_ml,
                                                              p.B, p.S, p.H, p.G, p.D, d.L, d.nhc,
                                                              err);
    }
    return cudaGetLastError();
}

cudaError_t launch_decode_combine(const Problem &p, const DecodePlan &d, const float *part_o,
                                  const float *part_ml, void *out, float *lse, cudaStream_t st) {
    const unsigned grid = (unsigned)((long)p.B * p.H);
    if (p.dtype == 1)
        k_decode_combine<bf16><<<grid, 128, 0, st>>>(part_o, part_ml, (bf16 *)out, lse, p.B, p.H,
                                                     p.D, d.nsplit);
    else
        k_decode_combine<float><<<grid, 128, 0, st>>>(part_o, part_ml, (float *)out, lse, p.B,
                                                      p.H, p.D, d.nsplit);
    return cudaGetLastError();
}

}  // namespace xt
