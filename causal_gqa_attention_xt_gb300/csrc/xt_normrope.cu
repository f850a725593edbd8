// xt_normrope.cu -- HBM-bound kernels around the attention:
//   * rope_table: cos/sin of every (position, frequency) pair, once per call;
//   * prologue: per-head QK-RMSNorm followed by rotate_half RoPE (forward);
//   * bwd_pre:  Dlt = rowsum(dO * O) for the softmax backward;
//   * epilogue: RoPE backward (rotation by the negative angle) and RMSNorm
//               backward, with per-CTA dgamma partials;
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
// Data movement. The three row kernels are persistent grids (two CTAs of
// eight warps per SM). Every warp runs its own pipeline over "units": one
// position of one batch element times a chunk of HC heads, all q heads or all
// k heads (for bwd_pre: of O and dO). Warp w of the grid takes units w,
// w + W, w + 2W, ... (W = warps in the grid). A unit's inputs are a few
// contiguous runs of global memory -- the chunk's rows from the
// [B, S, heads, D] tensors, one row per head from the [B, heads, S, D] ones,
// the position's cos/sin row, the rows' rstd words -- which the warp's lanes
// copy with bulk asynchronous copies (cp.async.bulk; 4-byte cp.async for the
// rstd words) into one of its NS shared-memory stages, completion counted on
// that stage's mbarrier. While the warp computes one unit from shared memory,
// the copies of its next NS - 1 units are in flight; no barrier couples the
// warps. A row of D elements is handled by tpr lanes, each owning VEC
// elements of the first half of the row and the VEC matching elements of the
// second half (the RoPE pair); a warp-iteration covers 32 / tpr heads.
//
// RoPE angles: xt_rope.cuh (one table per call, read by the prologue and the
// epilogue).
#include <algorithm>
#include "xt_common.cuh"
#include "xt_internal.h"
#include "xt_rope.cuh"
#include "xt_tc.cuh"

namespace xt {

namespace {

using tc::bulk_load;
using tc::cp_async4;
using tc::cp_async_mbar_arrive;
using tc::mbar_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;
using tc::mbar_wait_sleep;

constexpr int kWarps = 8;                    // warps per CTA, each its own pipeline
constexpr int kThreads = 32 * kWarps;
constexpr int kCtasPerSm = 2;

__host__ __device__ inline int pow2_at_least(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

constexpr size_t align128(size_t x) { return (x + 127) & ~(size_t)127; }
constexpr size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

// n / d for 0 <= n < 2^31 by a multiply-high and a shift (Granlund and
// Montgomery, division by run-time invariant integers, round-up multiplier).
struct FastDiv {
    uint32_t d, m, s;
};

FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d;
    f.s = 0;
    while ((1ull << f.s) < d) ++f.s;
    f.m = (uint32_t)((((1ull << 32) * ((1ull << f.s) - d)) / d) + 1);
    return f;
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f) {
    return (__umulhi(f.m, n) + n) >> f.s;
}

// ---------------------------------------------------------------- RoPE table
// tab[s * half + i] = (cos, sin) of pos(s) * theta^(-2i/D), s < S, i < half,
// where pos(s) = s, or for a packed batch (cu set) the row's position inside
// its sample (Mint report 8.2: positions restart in every sample), s - cu[u]
// for the last sample u with cu[u] <= s. Block 0 also checks the offsets.
__global__ void __launch_bounds__(256)
k_rope_table(float2 *__restrict__ tab, int S, int half, const int *__restrict__ cu, int units,
             int max_len, unsigned int *err, const __grid_constant__ RopeConsts rc) {
    pdl_enter();
    __shared__ float fhi[kRopeMaxHalf], flo[kRopeMaxHalf];
    __shared__ double fd[kRopeMaxHalf];
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        fhi[i] = rc.fhi[i];
        flo[i] = rc.flo[i];
        fd[i] = rc.fd[i];
    }
    if (cu != nullptr && blockIdx.x == 0) {
        for (int u = threadIdx.x; u < units; u += blockDim.x) {
            const int a = cu[u], b = cu[u + 1];
            if ((u == 0 && a != 0) || b < a || b - a > max_len || (u == units - 1 && b != S))
                atomicOr(err, ERR_BADSEQ);
        }
    }
    __syncthreads();
    const long n = (long)S * half;
    for (long e = (long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (long)gridDim.x * blockDim.x) {
        const int s = (int)(e / half), i = (int)(e - (long)s * half);
        int pos = s;
        if (cu != nullptr) {
            int lo = 0, hi = units;   // cu[lo] <= s < cu[hi] for well-formed offsets
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (cu[mid] <= s) lo = mid;
                else hi = mid;
            }
            pos = max(0, s - cu[lo]);
        }
        tab[e] = rope_cos_sin(pos, fhi[i], flo[i], fd[i]);
    }
}

// ---------------------------------------------------------------- units
// Units: u = (b * SG + sg) * (nqc + nkc) + chunk; chunk < nqc are q-head chunks
// of HC heads, the rest k-head chunks; position group sg holds positions
// [P sg, P sg + P) (P = 1 unless one chunk covers all heads of each tensor, when a
// unit may take several positions: their rows are contiguous then).
struct UnitGeo {
    int HC;           // heads per unit
    int nqc, nkc;     // chunks over the q heads and over the k heads
    int P;            // positions per unit
    int units;        // B * SG * (nqc + nkc), SG = ceil(S / P)
    FastDiv fd_chunks, fd_S;   // fd_S divides by SG
    int y_off;        // stage offset of the second input's rows
    int r_off;        // stage offset of the rstd words
    int t_off;        // stage offset of the cos/sin row
    int stage_bytes;
};

struct Unit {
    int b, s;         // batch element, first position
    int np;           // positions [s, s + np)
    int h0, nh;       // heads [h0, h0 + nh) of q (isq) or of k
    bool isq;
};

__device__ __forceinline__ Unit decode_unit(uint32_t u, const UnitGeo &g, int H, int G, int S) {
    Unit t;
    const uint32_t bs = fdiv(u, g.fd_chunks);
    const int ch = (int)(u - bs * (uint32_t)(g.nqc + g.nkc));
    t.b = (int)fdiv(bs, g.fd_S);
    const int sg = (int)(bs - (uint32_t)t.b * g.fd_S.d);
    t.s = sg * g.P;
    t.np = g.P == 1 ? 1 : min(g.P, S - t.s);
    t.isq = ch < g.nqc;
    t.h0 = (t.isq ? ch : ch - g.nqc) * g.HC;
    t.nh = min(g.HC, (t.isq ? H : G) - t.h0);
    return t;
}

// Fixed-chunk assignment: warp w of the grid takes units w, w + nw,
// w + 2 nw, ... with nw the number of warps rounded down to a multiple of the
// chunks per position, so that all of a warp's units have the same chunk
// (same tensor, same heads); warps at or past nw take none. Balanced when the
// chunks are of equal size.
__device__ __forceinline__ void warp_units_fixed(const UnitGeo &g, uint32_t &first,
                                                 uint32_t &stride) {
    const uint32_t nch = (uint32_t)(g.nqc + g.nkc);
    stride = (gridDim.x * kWarps) / nch * nch;
    first = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (first >= stride) first = 0xffffffffu;   // idle warp
}

// Per-warp pipeline over units first, first + stride, ... < units through NS
// stages of `stage_bytes` at `ring`, with one mbarrier per stage in `full`.
// issue(u, buf, bar) is run by all 32 lanes and starts the copies of unit u;
// process(u, buf) computes it once they have landed. Returns false if a wait
// ran out (the error word is raised and the copies in flight are let land).
template <int NS, class Issue, class Process>
__device__ bool warp_pipeline(uint64_t *full, unsigned char *ring, int stage_bytes, uint32_t first,
                              uint32_t stride, uint32_t units, unsigned int *err, Issue issue,
                              Process process) {
    const int lane = threadIdx.x & 31;
    if (first >= units) return true;
    if (lane == 0)
        for (int k = 0; k < NS; ++k) mbar_init(&full[k], 1);
    __syncwarp();
    if (lane == 0) tc::fence_barrier_init();
    __syncwarp();
#pragma unroll
    for (int k = 0; k < NS; ++k) {
        const uint32_t u = first + k * stride;
        if (u < units) issue(u, ring + (size_t)k * stage_bytes, &full[k]);
    }
    int it = 0;
    for (uint32_t u = first; u < units; u += stride, ++it) {
        const int st = it % NS;
        const bool ok = mbar_wait_sleep(&full[st], (uint32_t)((it / NS) & 1));
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) {
                atomicOr(err, ERR_TIMEOUT);
                for (int k = 0; k < NS; ++k)
                    if (u + k * stride < units)
                        mbar_wait(&full[(it + k) % NS], (uint32_t)(((it + k) / NS) & 1), nullptr);
            }
            __syncwarp();
            return false;
        }
        process(u, ring + (size_t)st * stage_bytes);
        const uint32_t un = u + NS * stride;
        if (un < units) {
            // the reads of this stage (generic proxy) come before the copies
            // that overwrite it (async proxy)
            __syncwarp();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(un, ring + (size_t)st * stage_bytes, &full[st]);
        }
    }
    return true;
}

template <int N>
__device__ __forceinline__ void load_f32(const float *p, float *dst) {
#pragma unroll
    for (int v = 0; v < N / 4; ++v) {
        const float4 x = *reinterpret_cast<const float4 *>(p + 4 * v);
        dst[4 * v] = x.x; dst[4 * v + 1] = x.y; dst[4 * v + 2] = x.z; dst[4 * v + 3] = x.w;
    }
}

template <int N>
__device__ __forceinline__ void ldg_f32(const float *p, float *dst) {
#pragma unroll
    for (int v = 0; v < N / 4; ++v) {
        const float4 x = __ldg(reinterpret_cast<const float4 *>(p + 4 * v));
        dst[4 * v] = x.x; dst[4 * v + 1] = x.y; dst[4 * v + 2] = x.z; dst[4 * v + 3] = x.w;
    }
}

// cos/sin of the N pairs starting at tb (N even): cv[e], sv[e].
template <int N>
__device__ __forceinline__ void load_cs(const float2 *tb, float *cv, float *sv) {
#pragma unroll
    for (int v = 0; v < N / 2; ++v) {
        const float4 x = *reinterpret_cast<const float4 *>(tb + 2 * v);
        cv[2 * v] = x.x; sv[2 * v] = x.y; cv[2 * v + 1] = x.z; sv[2 * v + 1] = x.w;
    }
}

// Shared memory of a CTA: [kWarps * NS mbarriers][kWarps rings of NS stages]
template <int NS>
constexpr size_t ring_offset() { return align128(sizeof(uint64_t) * kWarps * NS); }

// ---------------------------------------------------------------- prologue
// q_hat = rope(rmsnorm(q) * gamma_q), k_hat likewise; rstd saved.
constexpr int kStagesPro = 3;

template <typename T>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
k_prologue(const T *__restrict__ q, const T *__restrict__ k, const float *__restrict__ gq,
           const float *__restrict__ gk, const float2 *__restrict__ tab, T *__restrict__ qhat,
           T *__restrict__ khat, float *__restrict__ rstd_q, float *__restrict__ rstd_k, int S,
           int H, int G, int D, float eps, const UnitGeo geo, unsigned int *err) {
    pdl_enter();
    constexpr int VEC = 16 / sizeof(T);
    constexpr int NS = kStagesPro;
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem) + warp * NS;
    unsigned char *ring = smem + ring_offset<NS>() + (size_t)warp * NS * geo.stage_bytes;
    const int half = D / 2;
    const uint32_t xrow = (uint32_t)D * sizeof(T);
    const uint32_t trow = (uint32_t)half * sizeof(float2);
    const int chunks = half / VEC;
    const int tpr = pow2_at_least(chunks);
    const int c = lane & (tpr - 1);
    const int sub = lane / tpr, rpi = 32 / tpr;   // row within an iteration, rows per iteration
    const bool lane_has = c < chunks;
    const int cc = lane_has ? c : 0;              // clamped column group for the loads
    const float inv_d = 1.0f / (float)D;

    // a unit's rows (np positions x nh heads, contiguous in q / k: with np > 1 the
    // chunk holds all heads) and its np table rows
    auto issue = [&](uint32_t u, unsigned char *buf, uint64_t *bar) {
        const Unit t = decode_unit(u, geo, H, G, S);
        const uint32_t xb = (uint32_t)(t.np * t.nh) * xrow;
        if (lane == 0) {
            mbar_expect_tx(bar, xb + (uint32_t)t.np * trow);
            const T *x = t.isq ? q + (((size_t)t.b * S + t.s) * H + t.h0) * D
                               : k + (((size_t)t.b * S + t.s) * G + t.h0) * D;
            bulk_load(buf, x, xb, bar);
            bulk_load(buf + geo.t_off, tab + (size_t)t.s * half, (uint32_t)t.np * trow, bar);
        }
    };
    auto process = [&](uint32_t u, const unsigned char *buf) {
        const Unit t = decode_unit(u, geo, H, G, S);
        const int NH = t.isq ? H : G;
        float glo[VEC], ghi[VEC], cv[VEC], sv[VEC];
        const float *gamma = t.isq ? gq : gk;
        ldg_f32<VEC>(gamma + cc * VEC, glo);
        ldg_f32<VEC>(gamma + half + cc * VEC, ghi);
        const float2 *tb = reinterpret_cast<const float2 *>(buf + geo.t_off) + cc * VEC;
        if (geo.P == 1) load_cs<VEC>(tb, cv, sv);
        T *obase = (t.isq ? qhat : khat) + (((size_t)t.b * NH + t.h0) * S + t.s) * D;
        float *rbase = (t.isq ? rstd_q : rstd_k) + ((size_t)t.b * S + t.s) * NH + t.h0;
        const int nrow = t.np * t.nh;   // row l: position l / nh of the unit, head l % nh
        for (int l0 = 0; l0 < nrow; l0 += rpi) {
            const int l = l0 + sub;
            const bool ok = l < nrow && lane_has;
            const int lc = min(l, nrow - 1);
            const int pp = geo.P == 1 ? 0 : lc / t.nh, lh = lc - pp * t.nh;
            if (geo.P != 1) load_cs<VEC>(tb + (size_t)pp * half, cv, sv);
            const T *x = reinterpret_cast<const T *>(buf + (size_t)lc * xrow);
            float lo[VEC], hi[VEC];
            load16<T>(x + cc * VEC, lo);
            load16<T>(x + half + cc * VEC, hi);
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                s0 = fmaf(lo[e], lo[e], fmaf(hi[e], hi[e], s0));
                s1 = fmaf(lo[e + 1], lo[e + 1], fmaf(hi[e + 1], hi[e + 1], s1));
            }
            const float ss = group_sum(lane_has ? s0 + s1 : 0.f, tpr);
            const float r = rsqrtf(fmaf(ss, inv_d, eps));
            float olo[VEC], ohi[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float ylo = lo[e] * (r * glo[e]);
                const float yhi = hi[e] * (r * ghi[e]);
                olo[e] = ylo * cv[e] - yhi * sv[e];
                ohi[e] = ylo * sv[e] + yhi * cv[e];
            }
            if (ok) {
                T *y = obase + ((size_t)lh * S + pp) * D;
                store16<T>(y + c * VEC, olo);
                store16<T>(y + half + c * VEC, ohi);
                if (c == 0) rbase[(size_t)pp * NH + lh] = r;
            }
        }
    };
    // Warp w takes units w, w + stride, ... With q and k chunks alternating in the
    // unit order, an even stride would give each warp one kind only, and the warps
    // with the (smaller) k units would finish early and leave fewer copies in flight
    // for the rest of the kernel; an odd stride gives every warp both kinds in turn.
    const uint32_t gw = blockIdx.x * kWarps + warp, nw = gridDim.x * kWarps;
    const uint32_t stride = ((geo.nqc + geo.nkc) % 2 == 0 && nw % 2 == 0 && nw > 1) ? nw - 1 : nw;
    warp_pipeline<NS>(full, ring, geo.stage_bytes, gw < stride ? gw : 0xffffffffu, stride,
                      (uint32_t)geo.units, err, issue, process);
}

// ---------------------------------------------------------------- bwd_pre
// Dlt[b, h, s] = sum_d dO[b, s, h, d] * O[b, s, h, d].
constexpr int kStagesPre = 3;

template <typename T>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
k_bwd_pre(const T *__restrict__ out, const T *__restrict__ dout, float *__restrict__ dlt, int S,
          int H, int D, const UnitGeo geo, unsigned int *err) {
    constexpr int VEC = 16 / sizeof(T);
    constexpr int NS = kStagesPre;
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem) + warp * NS;
    unsigned char *ring = smem + ring_offset<NS>() + (size_t)warp * NS * geo.stage_bytes;
    const uint32_t xrow = (uint32_t)D * sizeof(T);
    const int chunks = D / VEC;
    const int tpr = pow2_at_least(chunks);
    const int c = lane & (tpr - 1);
    const int sub = lane / tpr, rpi = 32 / tpr;
    const bool lane_has = c < chunks;
    const int cc = lane_has ? c : 0;

    auto issue = [&](uint32_t u, unsigned char *buf, uint64_t *bar) {
        const Unit t = decode_unit(u, geo, H, 0, S);
        const uint32_t nb = (uint32_t)t.nh * xrow;
        const size_t off = (((size_t)t.b * S + t.s) * H + t.h0) * D;
        if (lane == 0) {
            mbar_expect_tx(bar, 2 * nb);
            bulk_load(buf, out + off, nb, bar);
            bulk_load(buf + geo.y_off, dout + off, nb, bar);
        }
    };
    auto process = [&](uint32_t u, const unsigned char *buf) {
        const Unit t = decode_unit(u, geo, H, 0, S);
        float *dbase = dlt + ((size_t)t.b * H + t.h0) * S + t.s;
        for (int lh0 = 0; lh0 < t.nh; lh0 += rpi) {
            const int lh = lh0 + sub;
            const size_t ro = (size_t)min(lh, t.nh - 1) * xrow;
            float a[VEC], g[VEC];
            load16<T>(reinterpret_cast<const T *>(buf + ro) + cc * VEC, a);
            load16<T>(reinterpret_cast<const T *>(buf + geo.y_off + ro) + cc * VEC, g);
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
                a0 = fmaf(a[e], g[e], a0);
                a1 = fmaf(a[e + 1], g[e + 1], a1);
            }
            const float acc = group_sum(lane_has ? a0 + a1 : 0.f, tpr);
            if (lh < t.nh && c == 0) dbase[(size_t)lh * S] = acc;
        }
    };
    const uint32_t gw = blockIdx.x * kWarps + warp, nw = gridDim.x * kWarps;
    warp_pipeline<NS>(full, ring, geo.stage_bytes, gw, nw, (uint32_t)geo.units, err, issue,
                      process);
}

// ---------------------------------------------------------------- epilogue
// dq = RMSNorm_bwd(RoPE_bwd(dqhat)), likewise dk; one dgamma partial per CTA.
// With dqhat == nullptr (bf16: the dQ kernel finishes dq itself) the units
// cover the k heads only.
constexpr int kStagesEpi = 2;

template <typename T>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
k_epilogue(const float *__restrict__ dqhat, const float *__restrict__ dkhat,
           const T *__restrict__ q, const T *__restrict__ k, const float *__restrict__ gq,
           const float *__restrict__ gk, const float *__restrict__ rstd_q,
           const float *__restrict__ rstd_k, const float2 *__restrict__ tab,
           T *__restrict__ dq, T *__restrict__ dk, float *__restrict__ part_q,
           float *__restrict__ part_k, int S, int H, int G, int D, const UnitGeo geo,
           unsigned int *err) {
    pdl_enter();
    constexpr int VEC = 16 / sizeof(T);
    constexpr int NS = kStagesEpi;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int any_failed;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem) + warp * NS;
    unsigned char *ring = smem + ring_offset<NS>() + (size_t)warp * NS * geo.stage_bytes;
    const int half = D / 2;
    const uint32_t xrow = (uint32_t)D * sizeof(T);
    const uint32_t yrow = (uint32_t)D * sizeof(float);
    const uint32_t trow = (uint32_t)half * sizeof(float2);
    const int chunks = half / VEC;
    const int tpr = pow2_at_least(chunks);
    const int c = lane & (tpr - 1);
    const int sub = lane / tpr, rpi = 32 / tpr;
    const bool lane_has = c < chunks;
    const int cc = lane_has ? c : 0;
    const float inv_d = 1.0f / (float)D;
    if (threadIdx.x == 0) any_failed = 0;
    uint32_t gw, nw;
    warp_units_fixed(geo, gw, nw);
    // every unit of this warp has the same chunk: one gamma, one set of
    // dgamma accumulators (for that tensor)
    const bool wq = gw < nw && (int)(gw % (uint32_t)(geo.nqc + geo.nkc)) < geo.nqc;
    float gml[VEC], gmh[VEC];
    ldg_f32<VEC>((wq ? gq : gk) + cc * VEC, gml);
    ldg_f32<VEC>((wq ? gq : gk) + half + cc * VEC, gmh);
    float acc[2 * VEC];
#pragma unroll
    for (int e = 0; e < 2 * VEC; ++e) acc[e] = 0.f;

    // Stage: x rows [lh], dyhat rows [lh] (one copy per head: dqhat/dkhat are
    // [B, heads, S, D]), rstd [lh], the position's cos/sin row.
    auto issue = [&](uint32_t u, unsigned char *buf, uint64_t *bar) {
        const Unit t = decode_unit(u, geo, H, G, S);
        const int NH = t.isq ? H : G;
        const size_t bs = (size_t)t.b * S + t.s;
        if (lane < t.nh)
            cp_async4(reinterpret_cast<float *>(buf + geo.r_off) + lane,
                      (t.isq ? rstd_q : rstd_k) + bs * NH + t.h0 + lane);
        cp_async_mbar_arrive(bar);   // one pending arrival until this lane's copy lands
        __syncwarp();
        const uint32_t xb = (uint32_t)t.nh * xrow;
        if (lane == 0) {
            mbar_expect_tx(bar, xb + (uint32_t)t.nh * yrow + trow);
            bulk_load(buf, (t.isq ? q : k) + (bs * NH + t.h0) * D, xb, bar);
            bulk_load(buf + geo.t_off, tab + (size_t)t.s * half, trow, bar);
        }
        __syncwarp();
        const float *dy = (t.isq ? dqhat : dkhat) + (((size_t)t.b * NH + t.h0) * S + t.s) * D;
        if (lane < t.nh)
            bulk_load(buf + geo.y_off + (size_t)lane * yrow, dy + (size_t)lane * S * D, yrow, bar);
    };
    auto process = [&](uint32_t u, const unsigned char *buf) {
        const Unit t = decode_unit(u, geo, H, G, S);
        const int NH = t.isq ? H : G;
        float cv[VEC], sv[VEC];
        load_cs<VEC>(reinterpret_cast<const float2 *>(buf + geo.t_off) + cc * VEC, cv, sv);
        T *obase = (t.isq ? dq : dk) + (((size_t)t.b * S + t.s) * NH + t.h0) * D;
        const float *rbuf = reinterpret_cast<const float *>(buf + geo.r_off);
        for (int lh0 = 0; lh0 < t.nh; lh0 += rpi) {
            const int lh = lh0 + sub;
            const bool ok = lh < t.nh && lane_has;
            const int lr = min(lh, t.nh - 1);
            const T *xr = reinterpret_cast<const T *>(buf + (size_t)lr * xrow);
            const float *yr = reinterpret_cast<const float *>(buf + geo.y_off + (size_t)lr * yrow);
            float xl[VEC], xh[VEC], gl[VEC], gh[VEC];
            load16<T>(xr + cc * VEC, xl);
            load16<T>(xr + half + cc * VEC, xh);
            load_f32<VEC>(yr + cc * VEC, gl);
            load_f32<VEC>(yr + half + cc * VEC, gh);
            const float r = rbuf[lr];
            float dyl[VEC], dyh[VEC];
            float d0 = 0.f, d1 = 0.f;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                // rotation by the negative angle
                dyl[e] = gl[e] * cv[e] + gh[e] * sv[e];
                dyh[e] = gh[e] * cv[e] - gl[e] * sv[e];
                d0 = fmaf(gml[e] * dyl[e], xl[e], d0);
                d1 = fmaf(gmh[e] * dyh[e], xh[e], d1);
            }
            const float dot = group_sum(lane_has ? d0 + d1 : 0.f, tpr);
            const float corr = dot * r * r * r * inv_d;
            float ol[VEC], oh[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                ol[e] = gml[e] * dyl[e] * r - xl[e] * corr;
                oh[e] = gmh[e] * dyh[e] * r - xh[e] * corr;
            }
            if (ok) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    acc[e] += dyl[e] * xl[e] * r;
                    acc[VEC + e] += dyh[e] * xh[e] * r;
                }
                T *dst = obase + (size_t)lh * D;
                store16<T>(dst + c * VEC, ol);
                store16<T>(dst + half + c * VEC, oh);
            }
        }
    };
    const bool ok = warp_pipeline<NS>(full, ring, geo.stage_bytes, gw, nw, (uint32_t)geo.units,
                                      err, issue, process);
    if (!ok && lane == 0) any_failed = 1;

    // Fixed-order reduction of the dgamma terms: over the rows a thread slot
    // (warp, sub) handled, then over the slots in order. Every copy has landed
    // once all warps are here, so the rings can hold the [slots][D] scratch.
    __syncthreads();
    if (any_failed) return;
    float *red = reinterpret_cast<float *>(smem + ring_offset<NS>());
    const int nslots = kWarps * rpi, slot = warp * rpi + sub;
    for (int pass = geo.nqc > 0 ? 0 : 1; pass < 2; ++pass) {   // pass 0: q, pass 1: k
        const bool mine = (pass == 0) == wq;
        if (pass) __syncthreads();
        if (lane_has) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                red[slot * D + c * VEC + e] = mine ? acc[e] : 0.f;
                red[slot * D + half + c * VEC + e] = mine ? acc[VEC + e] : 0.f;
            }
        }
        __syncthreads();
        for (int d = threadIdx.x; d < D; d += kThreads) {
            float sum = 0.f;
            for (int sl = 0; sl < nslots; ++sl) sum += red[sl * D + d];
            (pass == 0 ? part_q : part_k)[(size_t)blockIdx.x * D + d] = sum;
        }
    }
}

// dgamma[d] = sum over partials p of part[p][d], in a fixed association:
// slice s (of 128) sums p = s, s+128, s+256, ... in order, then slices
// 0..127 are added in order. Block (x = 8-column group, y = q or k), 1024
// threads: thread = (slice, column); a warp reads 4 partial rows x 32 bytes.
__global__ void __launch_bounds__(1024)
k_dgamma_reduce(const float *__restrict__ part_q, const float *__restrict__ part_k,
                int nparts_q, int nparts_k, int D, float *__restrict__ dgq, float *__restrict__ dgk) {
    pdl_enter();
    constexpr int kCols = 8, kSlices = 128;
    __shared__ float red[kSlices][kCols + 1];
    const float *part = blockIdx.y == 0 ? part_q : part_k;
    const int nparts = blockIdx.y == 0 ? nparts_q : nparts_k;
    float *out = blockIdx.y == 0 ? dgq : dgk;
    const int c = threadIdx.x % kCols, slice = threadIdx.x / kCols;
    const int d = blockIdx.x * kCols + c;
    float sum = 0.f;
    if (d < D) {
        // eight loads in flight, added in the same order as one at a time
        int p = slice;
        for (; p + kSlices * 7 < nparts; p += kSlices * 8) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = part[(size_t)(p + kSlices * u) * D + d];
#pragma unroll
            for (int u = 0; u < 8; ++u) sum += v[u];
        }
        for (; p < nparts; p += kSlices) sum += part[(size_t)p * D + d];
    }
    red[slice][c] = sum;
    __syncthreads();
    if (slice == 0 && d < D) {
        float total = 0.f;
        for (int sl = 0; sl < kSlices; ++sl) total += red[sl][c];
        out[d] = total;
    }
}

// ---------------------------------------------------------------- host side

// Units over H q heads and G k heads (G = 0: q only), one position each. A
// stage holds HC rows of x_row + y_row + r_row bytes (and a cos/sin row with
// a table); HC is the largest multiple of `rpi` (rows per warp-iteration)
// whose rows fit `row_budget` bytes, at most max(H, G) rounded up to rpi, and
// at most 32 (one copy per lane).
UnitGeo make_geo(const Problem &p, int H, int G, size_t x_row, size_t y_row, size_t r_row,
                 bool table, int rpi, size_t row_budget, bool group_positions = false) {
    UnitGeo g = {};
    const size_t row = x_row + y_row + r_row;
    const int hmax = H > G ? H : G;
    int hc = (int)(row_budget / row) / rpi * rpi;
    if (hc < rpi) hc = rpi;
    const int cap = (hmax + rpi - 1) / rpi * rpi;
    if (hc > cap) hc = cap;
    if (hc > 32) hc = 32;
    g.HC = hc;
    g.nqc = (H + hc - 1) / hc;
    g.nkc = G > 0 ? (G + hc - 1) / hc : 0;
    // several positions per unit when one chunk holds all heads of each tensor and
    // a position's rows are small (the unit's copies stay near the row budget)
    g.P = 1;
    if (group_positions && g.nqc <= 1 && g.nkc <= 1) {
        const size_t pos_bytes = (size_t)hc * (x_row + y_row + r_row);   // as the stage is laid out
        g.P = (int)std::max<size_t>(1, std::min<size_t>(8, row_budget / pos_bytes));
    }
    const int SG = (p.S + g.P - 1) / g.P;
    g.units = p.B * SG * (g.nqc + g.nkc);
    g.fd_chunks = make_fastdiv((uint32_t)(g.nqc + g.nkc));
    g.fd_S = make_fastdiv((uint32_t)SG);
    g.y_off = (int)align16((size_t)hc * x_row * g.P);
    g.r_off = (int)align16(g.y_off + (size_t)hc * y_row * g.P);
    g.t_off = (int)align16(g.r_off + (size_t)hc * r_row * g.P);
    g.stage_bytes =
        (int)align128(g.t_off + (table ? (size_t)g.P * (p.D / 2) * sizeof(float2) : 0));
    return g;
}

// CTAs: enough warps for the units, at most kCtasPerSm per SM and
// kMaxNormParts, at least one warp per head chunk of a position.
int persistent_grid(const UnitGeo &geo) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        sms = 1;
    int g = kCtasPerSm * sms;
    if (g > kMaxNormParts) g = kMaxNormParts;
    const int need = (geo.units + kWarps - 1) / kWarps;
    if (need < g) g = need;
    const int min_ctas = (geo.nqc + geo.nkc + kWarps - 1) / kWarps;
    return g < min_ctas ? min_ctas : g;
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

int rows_per_iter(int D, int dtype, bool halves) {
    const int vec = dtype == 1 ? 8 : 4;
    const int chunks = (halves ? D / 2 : D) / vec;
    return 32 / pow2_at_least(chunks);
}

}  // namespace

size_t rope_table_bytes(const Problem &p) { return (size_t)p.S * (p.D / 2) * sizeof(float2); }

cudaError_t launch_rope_table(const Problem &p, void *tab, unsigned int *err, cudaStream_t st) {
    const long n = (long)p.S * (p.D / 2);
    long blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    return launch_dependent(k_rope_table, dim3((unsigned)blocks), dim3(256), 0, st, (float2 *)tab,
                            p.S, p.D / 2, p.cu, p.units, p.max_len, err, rope_consts(p.theta, p.D));
}

cudaError_t launch_prologue(const Problem &p, const void *q, const void *k, const float *gq,
                            const float *gk, const void *tab, void *qhat, void *khat,
                            float *rstd_q, float *rstd_k, unsigned int *err, cudaStream_t st) {
    const size_t es = p.dtype == 1 ? 2 : 4;
    const UnitGeo geo = make_geo(p, p.H, p.G, (size_t)p.D * es, 0, 0, true,
                                 rows_per_iter(p.D, p.dtype, true), 4096, true);
    const size_t smem = ring_offset<kStagesPro>() + (size_t)kWarps * kStagesPro * geo.stage_bytes;
    const int grid = persistent_grid(geo);
    cudaError_t e;
    if (p.dtype == 1) {
        if ((e = set_smem(k_prologue<bf16>, smem)) != cudaSuccess) return e;
        return launch_dependent(k_prologue<bf16>, dim3(grid), dim3(kThreads), smem, st,
                                (const bf16 *)q, (const bf16 *)k, gq, gk, (const float2 *)tab,
                                (bf16 *)qhat, (bf16 *)khat, rstd_q, rstd_k, p.S, p.H, p.G, p.D,
                                p.eps, geo, err);
    }
    if ((e = set_smem(k_prologue<float>, smem)) != cudaSuccess) return e;
    return launch_dependent(k_prologue<float>, dim3(grid), dim3(kThreads), smem, st,
                            (const float *)q, (const float *)k, gq, gk, (const float2 *)tab,
                            (float *)qhat, (float *)khat, rstd_q, rstd_k, p.S, p.H, p.G, p.D, p.eps,
                            geo, err);
}

cudaError_t launch_bwd_pre(const Problem &p, const void *out, const void *dout, float *dlt,
                           unsigned int *err, cudaStream_t st) {
    const size_t es = p.dtype == 1 ? 2 : 4;
    const size_t xrow = (size_t)p.D * es;
    const UnitGeo geo = make_geo(p, p.H, 0, xrow, xrow, 0, false,
                                 rows_per_iter(p.D, p.dtype, false), 4096);
    const size_t smem = ring_offset<kStagesPre>() + (size_t)kWarps * kStagesPre * geo.stage_bytes;
    const int grid = persistent_grid(geo);
    cudaError_t e;
    if (p.dtype == 1) {
        if ((e = set_smem(k_bwd_pre<bf16>, smem)) != cudaSuccess) return e;
        k_bwd_pre<bf16><<<grid, kThreads, smem, st>>>((const bf16 *)out, (const bf16 *)dout, dlt,
                                                      p.S, p.H, p.D, geo, err);
    } else {
        if ((e = set_smem(k_bwd_pre<float>, smem)) != cudaSuccess) return e;
        k_bwd_pre<float><<<grid, kThreads, smem, st>>>((const float *)out, (const float *)dout,
                                                       dlt, p.S, p.H, p.D, geo, err);
    }
    return cudaGetLastError();
}

cudaError_t launch_epilogue(const Problem &p, const float *dqhat, const float *dkhat,
                            const void *q, const void *k, const float *gq, const float *gk,
                            const float *rstd_q, const float *rstd_k, const void *tab, void *dq,
                            void *dk, float *part_q, float *part_k, int *nparts,
                            unsigned int *err, cudaStream_t st) {
    const size_t es = p.dtype == 1 ? 2 : 4;
    const int rpi = rows_per_iter(p.D, p.dtype, true);
    const UnitGeo geo = make_geo(p, dqhat ? p.H : 0, p.G, (size_t)p.D * es,
                                 (size_t)p.D * sizeof(float), sizeof(float), true, rpi, 6400);
    size_t ring = (size_t)kWarps * kStagesEpi * geo.stage_bytes;
    const size_t red = (size_t)kWarps * rpi * p.D * sizeof(float);
    if (ring < red) ring = red;
    const size_t smem = ring_offset<kStagesEpi>() + ring;
    const int grid = persistent_grid(geo);
    *nparts = grid;
    cudaError_t e;
    if (p.dtype == 1) {
        if ((e = set_smem(k_epilogue<bf16>, smem)) != cudaSuccess) return e;
        e = launch_dependent(k_epilogue<bf16>, dim3(grid), dim3(kThreads), smem, st, dqhat, dkhat,
                             (const bf16 *)q, (const bf16 *)k, gq, gk, rstd_q, rstd_k,
                             (const float2 *)tab, (bf16 *)dq, (bf16 *)dk, part_q, part_k, p.S, p.H,
                             p.G, p.D, geo, err);
        if (e != cudaSuccess) return e;
    } else {
        if ((e = set_smem(k_epilogue<float>, smem)) != cudaSuccess) return e;
        e = launch_dependent(k_epilogue<float>, dim3(grid), dim3(kThreads), smem, st, dqhat,
                             dkhat, (const float *)q, (const float *)k, gq, gk, rstd_q, rstd_k,
                             (const float2 *)tab, (float *)dq, (float *)dk, part_q, part_k, p.S,
                             p.H, p.G, p.D, geo, err);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_dgamma_reduce(const Problem &p, const float *part_q, const float *part_k,
                                 int nparts_q, int nparts_k, float *dgq, float *dgk,
                                 cudaStream_t st) {
    return launch_dependent(k_dgamma_reduce, dim3((p.D + 7) / 8, 2), dim3(1024), 0, st, part_q,
                            part_k, nparts_q, nparts_k, p.D, dgq, dgk);
}

}  // namespace xt
