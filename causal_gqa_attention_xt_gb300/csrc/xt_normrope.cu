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
// Data movement. The three row kernels are persistent grids (two CTAs per
// SM) that walk "units": P consecutive positions of one batch element times a
// chunk of HC heads, all q heads or all k heads. P makes a head's run in the
// [B, heads, S, D] tensors about kRunBytes long, HC fills the stage budget.
// A producer warp copies each unit's inputs -- one run per position from the
// [B, S, heads, D] tensors, one run per head from the [B, heads, S, D] ones,
// the unit's rows of the cos/sin table -- into a ring of kStages shared-memory
// buffers with bulk asynchronous copies (cp.async.bulk, byte count on a
// "full" mbarrier). Eight consumer warps read the staged rows, compute in
// fp32, store results with 16-byte stores and release the buffer on an
// "empty" mbarrier; no CTA-wide barrier is taken per unit. A row of D
// elements is handled by tpr lanes, each owning VEC elements of the first
// half of the row and the VEC matching elements of the second half (the RoPE
// pair); gamma for those elements stays in registers for the whole unit.
//
// RoPE angles (rope_table): for positions below 2^21 the product pos * f is
// formed in fp32 with f = theta^(-2i/D) split as hi + lo and the rounding
// error of pos * hi recovered exactly by an fma, then reduced by 2*pi with
// Cody and Waite's three-constant scheme; beyond 2^21 product and reduction
// are done in double. The reduced angle (|r| <= pi + small, within a few fp32
// ulps) goes to the fp32 sincosf.
#include "xt_common.cuh"
#include "xt_internal.h"
#include "xt_tc.cuh"

namespace xt {

namespace {

using tc::bulk_load;
using tc::cp_async4;
using tc::cp_async_mbar_arrive;
using tc::mbar_arrive;
using tc::mbar_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;    // + the producer warp
constexpr int kStages = 3;                   // ring depth
constexpr int kCtasPerSm = 2;
constexpr size_t kStageBudget = 28 * 1024;   // staged bytes per unit (rows + table)
constexpr size_t kRunBytes = 2048;           // target run per head in [B, heads, S, D]
constexpr int kRopeFp32Limit = 1 << 21;      // positions with the fp32 angle path

// 2*pi = kC1 + kC2 + kC3 (Cody-Waite): kC1 has 5 significant bits, so k * kC1
// is exact for |k| < 2^19; kC2 and kC3 carry the rest.
constexpr double kTwoPi = 6.283185307179586476925;
constexpr float kC1 = 6.25f;
constexpr float kC2 = (float)(kTwoPi - 6.25);
constexpr float kC3 = (float)((kTwoPi - 6.25) - (double)kC2);
constexpr float kInvTwoPi = (float)(1.0 / kTwoPi);

__host__ __device__ inline int pow2_at_least(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

constexpr size_t align128(size_t x) { return (x + 127) & ~(size_t)127; }
constexpr size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

// ---------------------------------------------------------------- RoPE table
// Inverse frequencies theta^(-2i/D), formed on the host in double; fhi + flo
// is that double to ~48 bits.
constexpr int kMaxHalf = 64;   // D / 2 for D <= 128
struct RopeConsts {
    float fhi[kMaxHalf], flo[kMaxHalf];
    double fd[kMaxHalf];
};

// tab[s * half + i] = (cos, sin) of s * theta^(-2i/D), s < S, i < half.
__global__ void __launch_bounds__(256)
k_rope_table(float2 *__restrict__ tab, int S, int half, const __grid_constant__ RopeConsts rc) {
    const long n = (long)S * half;
    for (long e = (long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (long)gridDim.x * blockDim.x) {
        const int s = (int)(e / half), i = (int)(e - (long)s * half);
        float red;
        if (s < kRopeFp32Limit) {
            const float fs = (float)s;   // exact
            const float hi = rc.fhi[i];
            const float p = __fmul_rn(fs, hi);
            const float tail = fmaf(fs, rc.flo[i], fmaf(fs, hi, -p));   // s * f - p
            const float k = rintf(p * kInvTwoPi);
            float r = fmaf(-k, kC1, p);   // exact
            r = fmaf(-k, kC2, r);
            red = __fadd_rn(r, fmaf(-k, kC3, tail));
        } else {
            const double ang = (double)s * rc.fd[i];
            red = (float)fma(-rint(ang * (1.0 / kTwoPi)), kTwoPi, ang);
        }
        float sv, cv;
        sincosf(red, &sv, &cv);
        tab[e] = make_float2(cv, sv);
    }
}

// ---------------------------------------------------------------- units
// How the rows of a problem are cut into units.
struct UnitGeo {
    int P;            // positions per unit
    int HC;           // heads per unit (all q or all k)
    int nsb;          // position blocks per batch element
    int nqc, nkc;     // head chunks over the q heads and over the k heads
    int units;        // B * nsb * (nqc + nkc)
    int y_off;        // ring-buffer offset of the second input
    int r_off;        // ring-buffer offset of the staged rstd values
    int t_off;        // ring-buffer offset of the cos/sin rows
    int stage_bytes;  // one ring buffer
};

struct Unit {
    int b, s0, np;    // batch element, first position, number of positions
    int h0, nh;       // heads [h0, h0 + nh) of q (isq) or of k
    bool isq;
};

__device__ __forceinline__ Unit decode_unit(int u, const UnitGeo &g, int S, int H, int G) {
    Unit t;
    const int nhc = g.nqc + g.nkc;
    const int ch = u % nhc;
    const int r = u / nhc;
    const int sb = r % g.nsb;
    t.b = r / g.nsb;
    t.s0 = sb * g.P;
    t.np = min(g.P, S - t.s0);
    t.isq = ch < g.nqc;
    t.h0 = (t.isq ? ch : ch - g.nqc) * g.HC;
    t.nh = min(g.HC, (t.isq ? H : G) - t.h0);
    return t;
}

// Shared memory: [RingCtl][ring: kStages buffers]
struct alignas(16) RingCtl {
    uint64_t full[kStages];    // producer's copies landed (1 arrival + bytes)
    uint64_t empty[kStages];   // consumer warps done with the buffer (kConsumerWarps)
    int abort_flag;
};

__device__ __forceinline__ void ring_init(RingCtl *c) {
    if (threadIdx.x == 0) {
        for (int st = 0; st < kStages; ++st) {
            mbar_init(&c->full[st], 1);
            mbar_init(&c->empty[st], kConsumerWarps);
        }
        c->abort_flag = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();
}

__device__ __forceinline__ void raise_timeout(RingCtl *c, unsigned int *err) {
    atomicOr(err, ERR_TIMEOUT);
    *(volatile int *)&c->abort_flag = 1;
}

// Producer warp: units blockIdx.x, blockIdx.x + gridDim.x, ... ; issue(u, buf,
// bar) is run by all 32 lanes and starts the copies of unit u into buf.
template <class Issue>
__device__ void produce(RingCtl *c, unsigned char *ring, int stage_bytes, int units,
                        unsigned int *err, Issue issue) {
    const int lane = threadIdx.x & 31;
    int it = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++it) {
        const int st = it % kStages;
        if (it >= kStages) {
            const bool ok = mbar_wait(&c->empty[st], (uint32_t)(((it / kStages) - 1) & 1),
                                      &c->abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0 && !*(volatile int *)&c->abort_flag) raise_timeout(c, err);
                break;
            }
        }
        issue(u, ring + (size_t)st * stage_bytes, &c->full[st]);
    }
    // After an abort, let the copies still in flight land before the CTA exits.
    if (lane == 0 && *(volatile int *)&c->abort_flag)
        for (int k = 1; k <= kStages && it - k >= 0; ++k)
            mbar_wait(&c->full[(it - k) % kStages], (uint32_t)(((it - k) / kStages) & 1), nullptr);
}

// Consumer warps: process(u, buf) on every unit of this CTA, then release.
template <class Process>
__device__ void consume(RingCtl *c, unsigned char *ring, int stage_bytes, int units,
                        unsigned int *err, Process process) {
    const int lane = threadIdx.x & 31;
    int it = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++it) {
        const int st = it % kStages;
        const bool ok = mbar_wait(&c->full[st], (uint32_t)((it / kStages) & 1), &c->abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0 && !*(volatile int *)&c->abort_flag) raise_timeout(c, err);
            break;
        }
        process(u, ring + (size_t)st * stage_bytes);
        __syncwarp();
        if (lane == 0) mbar_arrive(&c->empty[st]);
    }
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

// cos/sin of the N pairs starting at tb (N even): c[e], s[e].
template <int N>
__device__ __forceinline__ void load_cs(const float2 *tb, float *cv, float *sv) {
#pragma unroll
    for (int v = 0; v < N / 2; ++v) {
        const float4 x = *reinterpret_cast<const float4 *>(tb + 2 * v);
        cv[2 * v] = x.x; sv[2 * v] = x.y; cv[2 * v + 1] = x.z; sv[2 * v + 1] = x.w;
    }
}

// Copies of a unit's x rows from a [B, S, heads, D] tensor (one run of nh rows
// per position, into buf rows [pos][lh]) and of its cos/sin rows; copy j is
// issued by lane j % 32.
template <typename T>
__device__ __forceinline__ void issue_x_and_table(const Unit &t, const T *x, int S, int NH,
                                                  int D, const float2 *tab, int t_off,
                                                  unsigned char *buf, uint64_t *bar, int lane) {
    const uint32_t xrow = (uint32_t)D * sizeof(T);
    const uint32_t trow = (uint32_t)(D / 2) * sizeof(float2);
    for (int j = lane; j <= t.np; j += 32) {
        if (j < t.np)
            bulk_load(buf + (size_t)j * t.nh * xrow,
                      x + (((size_t)t.b * S + t.s0 + j) * NH + t.h0) * D, t.nh * xrow, bar);
        else
            bulk_load(buf + t_off, tab + (size_t)t.s0 * (D / 2), t.np * trow, bar);
    }
}

// ---------------------------------------------------------------- prologue
// q_hat = rope(rmsnorm(q) * gamma_q), k_hat likewise; rstd saved.
template <typename T>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
k_prologue(const T *__restrict__ q, const T *__restrict__ k, const float *__restrict__ gq,
           const float *__restrict__ gk, const float2 *__restrict__ tab, T *__restrict__ qhat,
           T *__restrict__ khat, float *__restrict__ rstd_q, float *__restrict__ rstd_k, int S,
           int H, int G, int D, float eps, const UnitGeo geo, unsigned int *err) {
    constexpr int VEC = 16 / sizeof(T);
    extern __shared__ __align__(128) unsigned char smem[];
    RingCtl *ctl = reinterpret_cast<RingCtl *>(smem);
    unsigned char *ring = smem + align128(sizeof(RingCtl));
    ring_init(ctl);
    const int half = D / 2;
    const uint32_t xrow = (uint32_t)D * sizeof(T);

    if (threadIdx.x >= kConsumers) {
        const int lane = threadIdx.x & 31;
        produce(ctl, ring, geo.stage_bytes, geo.units, err,
                [&](int u, unsigned char *buf, uint64_t *bar) {
                    const Unit t = decode_unit(u, geo, S, H, G);
                    if (lane == 0)
                        mbar_expect_tx(bar, (uint32_t)(t.np * t.nh) * xrow +
                                                (uint32_t)t.np * half * sizeof(float2));
                    __syncwarp();
                    issue_x_and_table<T>(t, t.isq ? q : k, S, t.isq ? H : G, D, tab, geo.t_off,
                                         buf, bar, lane);
                });
        return;
    }

    const int chunks = half / VEC;
    const int tpr = pow2_at_least(chunks);
    const int c = threadIdx.x & (tpr - 1);
    const int slot = threadIdx.x / tpr, nslots = kConsumers / tpr;
    const bool lane_has = c < chunks;
    const float inv_d = 1.0f / (float)D;

    consume(ctl, ring, geo.stage_bytes, geo.units, err, [&](int u, const unsigned char *buf) {
        const Unit t = decode_unit(u, geo, S, H, G);
        const int NH = t.isq ? H : G;
        float glo[VEC], ghi[VEC];
        if (lane_has) {
            const float *gamma = t.isq ? gq : gk;
            ldg_f32<VEC>(gamma + c * VEC, glo);
            ldg_f32<VEC>(gamma + half + c * VEC, ghi);
        }
        T *obase = (t.isq ? qhat : khat) + (((size_t)t.b * NH + t.h0) * S + t.s0) * D;
        float *rbase = (t.isq ? rstd_q : rstd_k) + ((size_t)t.b * S + t.s0) * NH + t.h0;
        const float2 *tb0 = reinterpret_cast<const float2 *>(buf + geo.t_off) + c * VEC;
        const int nrows = t.np * t.nh;
        const int lim = ((nrows + nslots - 1) / nslots) * nslots;   // warp-uniform trip count
        int pos = slot / t.nh, lh = slot - pos * t.nh;
        const int dpos = nslots / t.nh, dlh = nslots - dpos * t.nh;
        for (int rr = slot; rr < lim; rr += nslots) {
            const bool row_ok = rr < nrows;
            const bool lane_ok = row_ok && lane_has;
            float lo[VEC], hi[VEC];
            float ss = 0.f;
            if (lane_ok) {
                const T *x = reinterpret_cast<const T *>(buf + (size_t)rr * xrow);
                load16<T>(x + c * VEC, lo);
                load16<T>(x + half + c * VEC, hi);
#pragma unroll
                for (int e = 0; e < VEC; ++e) ss = fmaf(lo[e], lo[e], fmaf(hi[e], hi[e], ss));
            }
            ss = group_sum(ss, tpr);
            const float r = rsqrtf(fmaf(ss, inv_d, eps));
            if (lane_ok) {
                float cv[VEC], sv[VEC];
                load_cs<VEC>(tb0 + pos * half, cv, sv);
                float olo[VEC], ohi[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float ylo = lo[e] * (r * glo[e]);
                    const float yhi = hi[e] * (r * ghi[e]);
                    olo[e] = ylo * cv[e] - yhi * sv[e];
                    ohi[e] = ylo * sv[e] + yhi * cv[e];
                }
                T *y = obase + ((size_t)lh * S + pos) * D;
                store16<T>(y + c * VEC, olo);
                store16<T>(y + half + c * VEC, ohi);
                if (c == 0) rbase[(size_t)pos * NH + lh] = r;
            }
            lh += dlh;
            pos += dpos;
            if (lh >= t.nh) { lh -= t.nh; ++pos; }
        }
    });
}

// ---------------------------------------------------------------- bwd_pre
// Dlt[b, h, s] = sum_d dO[b, s, h, d] * O[b, s, h, d]. Units are whole
// positions (or one position and a chunk of heads), contiguous in O and dO.
template <typename T>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
k_bwd_pre(const T *__restrict__ out, const T *__restrict__ dout, float *__restrict__ dlt, int S,
          int H, int D, const UnitGeo geo, unsigned int *err) {
    constexpr int VEC = 16 / sizeof(T);
    extern __shared__ __align__(128) unsigned char smem[];
    RingCtl *ctl = reinterpret_cast<RingCtl *>(smem);
    unsigned char *ring = smem + align128(sizeof(RingCtl));
    ring_init(ctl);
    const uint32_t xrow = (uint32_t)D * sizeof(T);

    if (threadIdx.x >= kConsumers) {
        const int lane = threadIdx.x & 31;
        produce(ctl, ring, geo.stage_bytes, geo.units, err,
                [&](int u, unsigned char *buf, uint64_t *bar) {
                    if (lane != 0) return;
                    const Unit t = decode_unit(u, geo, S, H, 0);
                    const uint32_t nb = (uint32_t)(t.np * t.nh) * xrow;
                    const size_t off = (((size_t)t.b * S + t.s0) * H + t.h0) * D;
                    mbar_expect_tx(bar, 2 * nb);
                    bulk_load(buf, out + off, nb, bar);
                    bulk_load(buf + geo.y_off, dout + off, nb, bar);
                });
        return;
    }

    const int chunks = D / VEC;
    const int tpr = pow2_at_least(chunks);
    const int c = threadIdx.x & (tpr - 1);
    const int slot = threadIdx.x / tpr, nslots = kConsumers / tpr;

    consume(ctl, ring, geo.stage_bytes, geo.units, err, [&](int u, const unsigned char *buf) {
        const Unit t = decode_unit(u, geo, S, H, 0);
        const int nrows = t.np * t.nh;
        const int lim = ((nrows + nslots - 1) / nslots) * nslots;
        float *dbase = dlt + ((size_t)t.b * H + t.h0) * S + t.s0;
        int pos = slot / t.nh, lh = slot - pos * t.nh;
        const int dpos = nslots / t.nh, dlh = nslots - dpos * t.nh;
        for (int rr = slot; rr < lim; rr += nslots) {
            const bool row_ok = rr < nrows;
            float acc = 0.f;
            if (row_ok && c < chunks) {
                float a[VEC], g[VEC];
                load16<T>(reinterpret_cast<const T *>(buf + (size_t)rr * xrow) + c * VEC, a);
                load16<T>(reinterpret_cast<const T *>(buf + geo.y_off + (size_t)rr * xrow) +
                              c * VEC, g);
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc = fmaf(a[e], g[e], acc);
            }
            acc = group_sum(acc, tpr);
            if (row_ok && c == 0) dbase[(size_t)lh * S + pos] = acc;
            lh += dlh;
            pos += dpos;
            if (lh >= t.nh) { lh -= t.nh; ++pos; }
        }
    });
}

// ---------------------------------------------------------------- epilogue
// dq = RMSNorm_bwd(RoPE_bwd(dqhat)), likewise dk; one dgamma partial per CTA.
template <typename T>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
k_epilogue(const float *__restrict__ dqhat, const float *__restrict__ dkhat,
           const T *__restrict__ q, const T *__restrict__ k, const float *__restrict__ gq,
           const float *__restrict__ gk, const float *__restrict__ rstd_q,
           const float *__restrict__ rstd_k, const float2 *__restrict__ tab,
           T *__restrict__ dq, T *__restrict__ dk, float *__restrict__ part_q,
           float *__restrict__ part_k, int S, int H, int G, int D, const UnitGeo geo,
           unsigned int *err) {
    constexpr int VEC = 16 / sizeof(T);
    extern __shared__ __align__(128) unsigned char smem[];
    RingCtl *ctl = reinterpret_cast<RingCtl *>(smem);
    unsigned char *ring = smem + align128(sizeof(RingCtl));
    ring_init(ctl);
    const int half = D / 2;
    const uint32_t xrow = (uint32_t)D * sizeof(T);
    const uint32_t yrow = (uint32_t)D * sizeof(float);

    const int chunks = half / VEC;
    const int tpr = pow2_at_least(chunks);
    const int c = threadIdx.x & (tpr - 1);
    const int slot = threadIdx.x / tpr, nslots = kConsumers / tpr;
    const bool lane_has = c < chunks;
    float accq[2 * VEC], acck[2 * VEC];
#pragma unroll
    for (int e = 0; e < 2 * VEC; ++e) { accq[e] = 0.f; acck[e] = 0.f; }

    // Ring buffer: x rows [pos][lh], then dyhat rows [lh][pos] (one run per
    // head: dqhat/dkhat are [B, heads, S, D]), rstd [pos][lh], cos/sin rows.
    if (threadIdx.x >= kConsumers) {
        const int lane = threadIdx.x & 31;
        produce(ctl, ring, geo.stage_bytes, geo.units, err,
                [&](int u, unsigned char *buf, uint64_t *bar) {
                    const Unit t = decode_unit(u, geo, S, H, G);
                    const int NH = t.isq ? H : G;
                    const float *rs = (t.isq ? rstd_q : rstd_k) +
                                      ((size_t)t.b * S + t.s0) * NH + t.h0;
                    float *rbuf = reinterpret_cast<float *>(buf + geo.r_off);
                    for (int rr = lane; rr < t.np * t.nh; rr += 32) {
                        const int pos = rr / t.nh;
                        cp_async4(rbuf + rr, rs + (size_t)pos * NH + (rr - pos * t.nh));
                    }
                    cp_async_mbar_arrive(bar);   // one pending arrival until this lane's copies land
                    __syncwarp();
                    const uint32_t hb = (uint32_t)t.np * yrow;
                    if (lane == 0)
                        mbar_expect_tx(bar, (uint32_t)(t.np * t.nh) * xrow + (uint32_t)t.nh * hb +
                                                (uint32_t)t.np * half * sizeof(float2));
                    __syncwarp();
                    issue_x_and_table<T>(t, t.isq ? q : k, S, NH, D, tab, geo.t_off, buf, bar,
                                         lane);
                    const float *dy = (t.isq ? dqhat : dkhat) +
                                      (((size_t)t.b * NH + t.h0) * S + t.s0) * D;
                    for (int lh = lane; lh < t.nh; lh += 32)
                        bulk_load(buf + geo.y_off + (size_t)lh * hb, dy + (size_t)lh * S * D, hb,
                                  bar);
                });
    } else {
        const float inv_d = 1.0f / (float)D;
        consume(ctl, ring, geo.stage_bytes, geo.units, err, [&](int u, const unsigned char *buf) {
            const Unit t = decode_unit(u, geo, S, H, G);
            const int NH = t.isq ? H : G;
            float gml[VEC], gmh[VEC];
            if (lane_has) {
                const float *gamma = t.isq ? gq : gk;
                ldg_f32<VEC>(gamma + c * VEC, gml);
                ldg_f32<VEC>(gamma + half + c * VEC, gmh);
            }
            T *obase = (t.isq ? dq : dk) + (((size_t)t.b * S + t.s0) * NH + t.h0) * D;
            const float *rbuf = reinterpret_cast<const float *>(buf + geo.r_off);
            const float2 *tb0 = reinterpret_cast<const float2 *>(buf + geo.t_off) + c * VEC;
            const int nrows = t.np * t.nh;
            const int lim = ((nrows + nslots - 1) / nslots) * nslots;
            int pos = slot / t.nh, lh = slot - pos * t.nh;
            const int dpos = nslots / t.nh, dlh = nslots - dpos * t.nh;
            for (int rr = slot; rr < lim; rr += nslots) {
                const bool row_ok = rr < nrows;
                const bool lane_ok = row_ok && lane_has;
                float xl[VEC], xh[VEC], dyl[VEC], dyh[VEC];
                float r = 0.f, dot = 0.f;
                if (lane_ok) {
                    const T *xr = reinterpret_cast<const T *>(buf + (size_t)rr * xrow);
                    load16<T>(xr + c * VEC, xl);
                    load16<T>(xr + half + c * VEC, xh);
                    const float *yr = reinterpret_cast<const float *>(
                        buf + geo.y_off + (size_t)(lh * t.np + pos) * yrow);
                    float gl[VEC], gh[VEC], cv[VEC], sv[VEC];
                    load_f32<VEC>(yr + c * VEC, gl);
                    load_f32<VEC>(yr + half + c * VEC, gh);
                    load_cs<VEC>(tb0 + pos * half, cv, sv);
                    r = rbuf[rr];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        // rotation by the negative angle
                        dyl[e] = gl[e] * cv[e] + gh[e] * sv[e];
                        dyh[e] = gh[e] * cv[e] - gl[e] * sv[e];
                        dot += gml[e] * dyl[e] * xl[e] + gmh[e] * dyh[e] * xh[e];
                    }
                }
                dot = group_sum(dot, tpr);
                if (lane_ok) {
                    const float corr = dot * r * r * r * inv_d;
                    float ol[VEC], oh[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        ol[e] = gml[e] * dyl[e] * r - xl[e] * corr;
                        oh[e] = gmh[e] * dyh[e] * r - xh[e] * corr;
                        if (t.isq) {   // uniform per unit; keeps both arrays in registers
                            accq[e] += dyl[e] * xl[e] * r;
                            accq[VEC + e] += dyh[e] * xh[e] * r;
                        } else {
                            acck[e] += dyl[e] * xl[e] * r;
                            acck[VEC + e] += dyh[e] * xh[e] * r;
                        }
                    }
                    T *dst = obase + ((size_t)pos * NH + lh) * D;
                    store16<T>(dst + c * VEC, ol);
                    store16<T>(dst + half + c * VEC, oh);
                }
                lh += dlh;
                pos += dpos;
                if (lh >= t.nh) { lh -= t.nh; ++pos; }
            }
        });
    }

    // Fixed-order reduction of the dgamma terms over the consumer row slots.
    // Every copy has landed once all threads are here (the consumers waited
    // for each unit), so the ring can hold the [nslots][D] scratch.
    __syncthreads();
    if (*(volatile int *)&ctl->abort_flag) return;
    float *red = reinterpret_cast<float *>(ring);
    for (int pass = 0; pass < 2; ++pass) {
        const float *acc = pass == 0 ? accq : acck;
        if (pass) __syncthreads();
        if (threadIdx.x < kConsumers && lane_has) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                red[slot * D + c * VEC + e] = acc[e];
                red[slot * D + half + c * VEC + e] = acc[VEC + e];
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
// slice s (of 32) sums p = s, s+32, s+64, ... in order, then slices 0..31 are
// added in order. Block (x = 32-column group, y = q or k), 1024 threads.
__global__ void __launch_bounds__(1024)
k_dgamma_reduce(const float *__restrict__ part_q, const float *__restrict__ part_k,
                int nparts_q, int nparts_k, int D, float *__restrict__ dgq, float *__restrict__ dgk) {
    __shared__ float red[32][33];
    const float *part = blockIdx.y == 0 ? part_q : part_k;
    const int nparts = blockIdx.y == 0 ? nparts_q : nparts_k;
    float *out = blockIdx.y == 0 ? dgq : dgk;
    const int c = threadIdx.x & 31, slice = threadIdx.x >> 5;
    const int d = blockIdx.x * 32 + c;
    float sum = 0.f;
    if (d < D)
        for (int p = slice; p < nparts; p += 32) sum += part[(size_t)p * D + d];
    red[slice][c] = sum;
    __syncthreads();
    if (slice == 0 && d < D) {
        float total = 0.f;
        for (int sl = 0; sl < 32; ++sl) total += red[sl][c];
        out[d] = total;
    }
}

// ---------------------------------------------------------------- host side
RopeConsts rope_consts(const Problem &p) {
    RopeConsts f = {};
    for (int i = 0; i < p.D / 2 && i < kMaxHalf; ++i) {
        const double v = pow(p.theta, -2.0 * (double)i / (double)p.D);
        f.fd[i] = v;
        f.fhi[i] = (float)v;
        f.flo[i] = (float)(v - (double)f.fhi[i]);
    }
    return f;
}

int gcd_int(int a, int b) {
    while (b) { const int t = a % b; a = b; b = t; }
    return a;
}

// Units over H q heads and G k heads (G = 0: q only). Per row the ring stages
// x_row bytes of the first input, y_row of the second and r_row of rstd; with
// a table, each unit also stages its positions' cos/sin rows.
//  run_row > 0: each head's P rows are also a run of P * run_row bytes in a
//    [B, heads, S, D] tensor: P makes that run about kRunBytes, HC fills the
//    budget, rounded down to a divisor of gcd(H, G) when that loses at most
//    half of it (equal units).
//  run_row == 0: units are whole positions (all H heads, contiguous in the
//    [B, S, H, D] inputs), or one position and a chunk of its heads when a
//    position alone exceeds the budget.
UnitGeo make_geo(const Problem &p, int H, int G, size_t x_row, size_t y_row, size_t r_row,
                 size_t run_row, bool table) {
    UnitGeo g = {};
    const size_t row = x_row + y_row + r_row;
    const size_t trow = table ? (size_t)(p.D / 2) * sizeof(float2) : 0;
    const int hmax = H > G ? H : G;
    size_t P = 1, HC = 1;
    if (run_row > 0) {
        P = kRunBytes / run_row;
        if (P > (size_t)p.S) P = (size_t)p.S;
        if (P < 1) P = 1;
        while (P > 1 && P * (row + trow) > kStageBudget) P /= 2;
        size_t hc_max = (kStageBudget - P * trow) / (P * row);
        if (hc_max < 1) hc_max = 1;
        if (hc_max > (size_t)hmax) hc_max = (size_t)hmax;
        HC = hc_max;
        const int hdiv = G > 0 ? gcd_int(H, G) : H;
        size_t d = hc_max < (size_t)hdiv ? hc_max : (size_t)hdiv;
        while (d > 1 && hdiv % d != 0) --d;
        if (2 * d >= hc_max) HC = d;
    } else {
        const size_t per_pos = (size_t)H * row;
        if (per_pos <= kStageBudget) {
            P = kStageBudget / per_pos;
            if (P > (size_t)p.S) P = (size_t)p.S;
            HC = (size_t)H;
        } else {
            P = 1;
            HC = kStageBudget / row;
            if (HC < 1) HC = 1;
        }
    }
    g.P = (int)P;
    g.HC = (int)HC;
    g.nsb = (p.S + g.P - 1) / g.P;
    g.nqc = (H + g.HC - 1) / g.HC;
    g.nkc = G > 0 ? (G + g.HC - 1) / g.HC : 0;
    g.units = p.B * g.nsb * (g.nqc + g.nkc);
    const size_t rows = P * HC;
    g.y_off = (int)align16(rows * x_row);
    g.r_off = (int)align16(g.y_off + rows * y_row);
    g.t_off = (int)align16(g.r_off + rows * r_row);
    g.stage_bytes = (int)align128(g.t_off + P * trow);
    return g;
}

int persistent_grid(int units) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        sms = 1;
    int g = kCtasPerSm * sms;
    if (g > kMaxNormParts) g = kMaxNormParts;
    return units < g ? units : g;
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

size_t ring_smem(const UnitGeo &g, size_t min_ring) {
    size_t ring = (size_t)kStages * g.stage_bytes;
    if (ring < min_ring) ring = min_ring;
    return align128(sizeof(RingCtl)) + ring;
}

}  // namespace

size_t rope_table_bytes(const Problem &p) { return (size_t)p.S * (p.D / 2) * sizeof(float2); }

cudaError_t launch_rope_table(const Problem &p, void *tab, cudaStream_t st) {
    const long n = (long)p.S * (p.D / 2);
    long blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    k_rope_table<<<(unsigned)blocks, 256, 0, st>>>((float2 *)tab, p.S, p.D / 2, rope_consts(p));
    return cudaGetLastError();
}

cudaError_t launch_prologue(const Problem &p, const void *q, const void *k, const float *gq,
                            const float *gk, const void *tab, void *qhat, void *khat,
                            float *rstd_q, float *rstd_k, unsigned int *err, cudaStream_t st) {
    const size_t es = p.dtype == 1 ? 2 : 4;
    const size_t xrow = (size_t)p.D * es;
    const UnitGeo geo = make_geo(p, p.H, p.G, xrow, 0, 0, xrow, true);
    const size_t smem = ring_smem(geo, 0);
    const int grid = persistent_grid(geo.units);
    cudaError_t e;
    if (p.dtype == 1) {
        if ((e = set_smem(k_prologue<bf16>, smem)) != cudaSuccess) return e;
        k_prologue<bf16><<<grid, kThreads, smem, st>>>(
            (const bf16 *)q, (const bf16 *)k, gq, gk, (const float2 *)tab, (bf16 *)qhat,
            (bf16 *)khat, rstd_q, rstd_k, p.S, p.H, p.G, p.D, p.eps, geo, err);
    } else {
        if ((e = set_smem(k_prologue<float>, smem)) != cudaSuccess) return e;
        k_prologue<float><<<grid, kThreads, smem, st>>>(
            (const float *)q, (const float *)k, gq, gk, (const float2 *)tab, (float *)qhat,
            (float *)khat, rstd_q, rstd_k, p.S, p.H, p.G, p.D, p.eps, geo, err);
    }
    return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const Problem &p, const void *out, const void *dout, float *dlt,
                           unsigned int *err, cudaStream_t st) {
    const size_t es = p.dtype == 1 ? 2 : 4;
    const size_t xrow = (size_t)p.D * es;
    const UnitGeo geo = make_geo(p, p.H, 0, xrow, xrow, 0, 0, false);
    const size_t smem = ring_smem(geo, 0);
    const int grid = persistent_grid(geo.units);
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
    const size_t xrow = (size_t)p.D * es;
    const size_t yrow = (size_t)p.D * sizeof(float);
    const UnitGeo geo = make_geo(p, p.H, p.G, xrow, yrow, sizeof(float), yrow, true);
    const int vec = p.dtype == 1 ? 8 : 4;
    const int tpr = pow2_at_least((p.D / 2) / vec);
    const size_t red_bytes = (size_t)(kConsumers / tpr) * p.D * sizeof(float);
    const size_t smem = ring_smem(geo, red_bytes);
    const int grid = persistent_grid(geo.units);
    *nparts = grid;
    cudaError_t e;
    if (p.dtype == 1) {
        if ((e = set_smem(k_epilogue<bf16>, smem)) != cudaSuccess) return e;
        k_epilogue<bf16><<<grid, kThreads, smem, st>>>(
            dqhat, dkhat, (const bf16 *)q, (const bf16 *)k, gq, gk, rstd_q, rstd_k,
            (const float2 *)tab, (bf16 *)dq, (bf16 *)dk, part_q, part_k, p.S, p.H, p.G, p.D, geo,
            err);
    } else {
        if ((e = set_smem(k_epilogue<float>, smem)) != cudaSuccess) return e;
        k_epilogue<float><<<grid, kThreads, smem, st>>>(
            dqhat, dkhat, (const float *)q, (const float *)k, gq, gk, rstd_q, rstd_k,
            (const float2 *)tab, (float *)dq, (float *)dk, part_q, part_k, p.S, p.H, p.G, p.D,
            geo, err);
    }
    return cudaGetLastError();
}

cudaError_t launch_dgamma_reduce(const Problem &p, const float *part_q, const float *part_k,
                                 int nparts_q, int nparts_k, float *dgq, float *dgk,
                                 cudaStream_t st) {
    k_dgamma_reduce<<<dim3((p.D + 31) / 32, 2), 1024, 0, st>>>(part_q, part_k, nparts_q, nparts_k,
                                                               p.D, dgq, dgk);
    return cudaGetLastError();
}

}  // namespace xt
