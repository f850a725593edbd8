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
// reading the cache from HBM, so it runs on the CUDA cores), the second and
// third launched as programmatic dependents of the one before, so each is
// launched while its predecessor still runs and waits for it on the device:
//  * k_decode_rows: one warp per new row: q heads normed + rotated into an
//    fp32 scratch (rounded through the storage type, as the training forward
//    rounds q_hat), k heads normed + rotated into the k cache at row pos[b], v
//    rows copied into the v cache. A position outside [0, S_max) raises an
//    error bit (reported as XT_EINVAL by xt_attn_check) and the batch element
//    is skipped.
//  * k_decode_attn: work unit = (b, kv head, chunk of <= 4 of its query
//    heads, key split); a CTA's warps run units independently, each on its own
//    ring of 3 shared-memory stages (a stage = 16 cached K-hat rows and the same
//    V rows, two bulk asynchronous copies) that its lane 0 refills as soon as
//    the warp is done with a stage, running ahead across unit boundaries.
//    Lanes: lane / 8 picks one key of each group of four, lane % 8 the 16-byte
//    chunks lane % 8, lane % 8 + 8, ... of the row, so a quarter warp reads one
//    row's 128 contiguous bytes (no bank conflicts). The four heads' partial
//    dot products are summed over the 8 lanes of a key by a transposing
//    butterfly (each step halves the values a lane carries), the online softmax
//    runs on the result (one (key, head pair) per lane), and P V accumulates
//    in registers (4 heads x the lane's columns), fp32 pairs through the packed
//    fp32 FMA. It writes the unit's partial (max, sum, unnormalised output).
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
using tc::mbar_wait_sleep;

constexpr int kDecKT = 16;   // keys per stage: four passes of four keys
constexpr int kDecHP = 4;    // query heads per work unit
constexpr int kDecNS = 3;    // stages per warp

// Warps per CTA: one CTA per SM with 3 stages per warp, 192 KB of stages at
// D = 128 (8 KB stages in bf16, 16 KB in fp32).
template <typename T> __host__ __device__ constexpr int dec_warps() { return sizeof(T) == 2 ? 8 : 4; }

// ---------------------------------------------------------------- new rows
template <typename T>
__global__ void __launch_bounds__(256)
k_decode_rows(const int *__restrict__ pos, const T *__restrict__ q, const T *__restrict__ k,
              const T *__restrict__ v, const float *__restrict__ gq, const float *__restrict__ gk,
              float *__restrict__ qhat, T *__restrict__ kc, T *__restrict__ vc, int S_max, int H,
              int G, int D, float eps, const __grid_constant__ RopeConsts rc, unsigned int *err) {
    // the attention kernel may launch now; it waits for this grid before reading
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
template <typename T, int DP>
struct DecLane {
    static constexpr int VEC = 16 / (int)sizeof(T);   // elements per 16-byte chunk
    static constexpr int CPL = DP / VEC / 8;          // chunks per lane
    static constexpr int P2 = CPL * VEC / 2;          // fp32 pairs per lane
};

// a += b * c on two fp32 lanes at once (the packed fp32 FMA of sm_100 on)
__device__ __forceinline__ void fma2(float2 &a, const float2 b, const float2 c) {
    asm("{\n .reg .b64 ra, rb, rc;\n"
        " mov.b64 ra, {%0, %1};\n mov.b64 rb, {%2, %3};\n mov.b64 rc, {%4, %5};\n"
        " fma.rn.f32x2 ra, rb, rc, ra;\n mov.b64 {%0, %1}, ra;\n}\n"
        : "+f"(a.x), "+f"(a.y)
        : "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
}

// 16 bytes of shared memory as fp32 pairs (bf16 widened exactly)
template <typename T>
__device__ __forceinline__ void lds_pairs(const T *p, float2 *dst) {
    const uint4 r = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    if constexpr (sizeof(T) == 4) {
        dst[0] = make_float2(__uint_as_float(w[0]), __uint_as_float(w[1]));
        dst[1] = make_float2(__uint_as_float(w[2]), __uint_as_float(w[3]));
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            dst[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
    }
}

struct DecUnit {
    int b, g, hc, split, k0, k1, nt;   // keys [k0, k1) in nt stages
};

__device__ __forceinline__ DecUnit dec_unit(int u, const int *pos, int S_max, int G, int L,
                                            int nsplit, int nhc) {
    DecUnit U;
    U.hc = u % nhc;
    const int t = u / nhc;
    U.split = t % nsplit;
    const int bg = t / nsplit;
    U.g = bg % G;
    U.b = bg / G;
    const int p = pos[U.b];
    U.k0 = U.split * L;
    U.k1 = (p >= 0 && p < S_max) ? min(U.k0 + L, p + 1) : U.k0;
    U.nt = U.k1 > U.k0 ? (U.k1 - U.k0 + kDecKT - 1) / kDecKT : 0;
    return U;
}

__device__ __forceinline__ float2 f2add(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 shfl_xor2(float2 v, int m) {
    return make_float2(__shfl_xor_sync(0xffffffffu, v.x, m), __shfl_xor_sync(0xffffffffu, v.y, m));
}

// FULL: D == DP (every lane chunk lies inside the row)
template <typename T, int DP, bool FULL>
__global__ void __launch_bounds__(dec_warps<T>() * 32, 1)
k_decode_attn(const int *__restrict__ pos, const float *__restrict__ qhat,
              const T *__restrict__ kc, const T *__restrict__ vc, float *__restrict__ part_o,
              float *__restrict__ part_ml, int B, int S_max, int H, int G, int D, int L,
              int nsplit, int nhc, int units, unsigned int *err) {
    using LG = DecLane<T, DP>;
    constexpr int VEC = LG::VEC, CPL = LG::CPL, P2 = LG::P2;
    constexpr int HP = kDecHP, KT = kDecKT, NS = kDecNS, WARPS = dec_warps<T>();
    constexpr unsigned FULLMASK = 0xffffffffu;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t full[WARPS][NS];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = warp * (int)gridDim.x + (int)blockIdx.x;   // units spread over CTAs first
    const int TW = (int)gridDim.x * WARPS;
    // the merge kernel may launch now (it waits for this grid); this grid waits
    // for the new-rows grid before it reads q-hat or the caches
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (gw >= units) return;
    const int kq = lane >> 3, j = lane & 7;
    const int group = H / G;
    const int rowe = D;                                        // elements per cached row
    const uint32_t rowb = (uint32_t)(D * (int)sizeof(T));
    const uint32_t stage_bytes = 2u * KT * rowb;
    unsigned char *ring = smem + (size_t)warp * NS * stage_bytes;
    uint64_t *bar = full[warp];
    if (lane == 0) {
        for (int st = 0; st < NS; ++st) mbar_init(&bar[st], 1);
        tc::fence_barrier_init();
    }
    __syncwarp();

    // Producer: every lane steps through the warp's (unit, stage) sequence;
    // lane 0 issues the copies.
    int pu = gw, pt = 0, issued = 0;
    DecUnit PU = dec_unit(pu, pos, S_max, G, L, nsplit, nhc);
    auto produce = [&]() {
        while (pu < units && pt >= PU.nt) {
            pu += TW;
            pt = 0;
            if (pu < units) PU = dec_unit(pu, pos, S_max, G, L, nsplit, nhc);
        }
        if (pu >= units) return;
        if (lane == 0) {
            const int st = issued % NS;
            const int ks = PU.k0 + pt * KT;
            const uint32_t bytes = (uint32_t)min(KT, PU.k1 - ks) * rowb;
            unsigned char *dst = ring + (size_t)st * stage_bytes;
            const size_t row = ((size_t)PU.b * G + PU.g) * S_max + ks;
            mbar_expect_tx(&bar[st], 2u * bytes);
            bulk_load(dst, kc + row * rowe, bytes, &bar[st]);
            bulk_load(dst + (size_t)KT * rowb, vc + row * rowe, bytes, &bar[st]);
        }
        ++pt;
        ++issued;
    };
#pragma unroll 1
    for (int i = 0; i < NS; ++i) produce();

    const float sl2 = kLog2e * rsqrtf((float)D);
    bool dv[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) dv[c] = FULL || (j + 8 * c) * VEC < D;
    const bool b2 = (j & 4) != 0, b1 = (j & 2) != 0, b0 = (j & 1) != 0;
    const bool c0 = (lane & 8) != 0, c1 = (lane & 16) != 0;
    int x = 0;   // stages consumed

#pragma unroll 1
    for (int u = gw; u < units; u += TW) {
        const DecUnit U = dec_unit(u, pos, S_max, G, L, nsplit, nhc);
        const int h0 = U.g * group + U.hc * HP;
        const int nh = min(HP, group - U.hc * HP);
        // this lane's columns of the unit's (pre-scaled) query rows
        float2 q2[HP][P2];
#pragma unroll
        for (int h = 0; h < HP; ++h)
#pragma unroll
            for (int c = 0; c < CPL; ++c)
#pragma unroll
                for (int e = 0; e < VEC / 2; ++e) {
                    float2 v = make_float2(0.f, 0.f);
                    if (h < nh && dv[c]) {
                        const float2 r = *reinterpret_cast<const float2 *>(
                            qhat + ((size_t)U.b * H + h0 + h) * D + (j + 8 * c) * VEC + 2 * e);
                        v = make_float2(r.x * sl2, r.y * sl2);
                    }
                    q2[h][c * (VEC / 2) + e] = v;
                }
        float2 o2[HP][P2];
#pragma unroll
        for (int h = 0; h < HP; ++h)
#pragma unroll
            for (int e = 0; e < P2; ++e) o2[h][e] = make_float2(0.f, 0.f);
        // running max and (lane-partial) sum of this lane's two heads 2*b0, 2*b0+1
        float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

#pragma unroll 1
        for (int t = 0; t < U.nt; ++t, ++x) {
            const int st = x % NS;
            const bool ok = __all_sync(FULLMASK, mbar_wait_sleep(&bar[st], (uint32_t)((x / NS) & 1)));
            if (!ok) {
                if (lane == 0) {
                    atomicOr(err, ERR_TIMEOUT);
                    for (int y = x; y < issued; ++y)   // let the copies in flight land
                        mbar_wait_sleep(&bar[y % NS], (uint32_t)((y / NS) & 1));
                }
                __syncwarp();
                return;
            }
            const T *Kt = reinterpret_cast<const T *>(ring + (size_t)st * stage_bytes);
            const T *Vt = Kt + (size_t)KT * rowe;
            const int n = min(KT, U.k1 - (U.k0 + t * KT));

            // partial scores: key 4*pass + kq, heads 0..3, over this lane's chunks
            float sc[4 * HP];
#pragma unroll
            for (int pass = 0; pass < 4; ++pass) {
                const int key = 4 * pass + kq;
                float2 a[HP];
#pragma unroll
                for (int h = 0; h < HP; ++h) a[h] = make_float2(0.f, 0.f);
                if (key < n) {
#pragma unroll
                    for (int c = 0; c < CPL; ++c) {
                        if (!dv[c]) continue;
                        float2 kv[VEC / 2];
                        lds_pairs<T>(Kt + (size_t)key * rowe + (j + 8 * c) * VEC, kv);
#pragma unroll
                        for (int e = 0; e < VEC / 2; ++e)
#pragma unroll
                            for (int h = 0; h < HP; ++h) fma2(a[h], q2[h][c * (VEC / 2) + e], kv[e]);
                    }
                }
#pragma unroll
                for (int h = 0; h < HP; ++h) sc[pass * HP + h] = a[h].x + a[h].y;
            }
            // sum over the key's 8 lanes, halving the carried values per step:
            // afterwards this lane holds key 4*(j>>1) + kq, heads 2*b0 + {0,1}
            float r8[8], r4[4], r2[2];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float snd = b2 ? sc[i] : sc[i + 8], kp = b2 ? sc[i + 8] : sc[i];
                r8[i] = kp + __shfl_xor_sync(FULLMASK, snd, 4);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float snd = b1 ? r8[i] : r8[i + 4], kp = b1 ? r8[i + 4] : r8[i];
                r4[i] = kp + __shfl_xor_sync(FULLMASK, snd, 2);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float snd = b0 ? r4[i] : r4[i + 2], kp = b0 ? r4[i + 2] : r4[i];
                r2[i] = kp + __shfl_xor_sync(FULLMASK, snd, 1);
            }
            // online softmax (log2 domain) over the stage's keys
            const bool kvalid = 4 * (j >> 1) + kq < n;
            float s0 = kvalid ? r2[0] : -INFINITY, s1 = kvalid ? r2[1] : -INFINITY;
            float t0 = s0, t1 = s1;
#pragma unroll
            for (int o = 2; o <= 16; o <<= 1) {
                t0 = fmaxf(t0, __shfl_xor_sync(FULLMASK, t0, o));
                t1 = fmaxf(t1, __shfl_xor_sync(FULLMASK, t1, o));
            }
            const float mn0 = fmaxf(m_run[0], t0), mn1 = fmaxf(m_run[1], t1);
            const float al0 = exp2f(m_run[0] - mn0), al1 = exp2f(m_run[1] - mn1);
            m_run[0] = mn0;
            m_run[1] = mn1;
            const float p0 = exp2f(s0 - mn0), p1 = exp2f(s1 - mn1);
            l_run[0] = fmaf(l_run[0], al0, p0);
            l_run[1] = fmaf(l_run[1], al1, p1);
            const float ax0 = __shfl_xor_sync(FULLMASK, al0, 1);
            const float ax1 = __shfl_xor_sync(FULLMASK, al1, 1);
            const float alpha[HP] = {b0 ? ax0 : al0, b0 ? ax1 : al1, b0 ? al0 : ax0,
                                     b0 ? al1 : ax1};
            if (!(alpha[0] == 1.f && alpha[1] == 1.f && alpha[2] == 1.f && alpha[3] == 1.f)) {
#pragma unroll
                for (int h = 0; h < HP; ++h)
#pragma unroll
                    for (int e = 0; e < P2; ++e) {
                        o2[h][e].x *= alpha[h];
                        o2[h][e].y *= alpha[h];
                    }
            }
            // O += P V: key 4*pass + kq, its probabilities from the lanes holding them
#pragma unroll
            for (int pass = 0; pass < 4; ++pass) {
                const int key = 4 * pass + kq;
                const int src = (kq << 3) | (2 * pass);
                const float ph[HP] = {__shfl_sync(FULLMASK, p0, src), __shfl_sync(FULLMASK, p1, src),
                                      __shfl_sync(FULLMASK, p0, src + 1),
                                      __shfl_sync(FULLMASK, p1, src + 1)};
                if (key < n) {
#pragma unroll
                    for (int c = 0; c < CPL; ++c) {
                        if (!dv[c]) continue;
                        float2 vv[VEC / 2];
                        lds_pairs<T>(Vt + (size_t)key * rowe + (j + 8 * c) * VEC, vv);
#pragma unroll
                        for (int e = 0; e < VEC / 2; ++e)
#pragma unroll
                            for (int h = 0; h < HP; ++h)
                                fma2(o2[h][c * (VEC / 2) + e], make_float2(ph[h], ph[h]), vv[e]);
                    }
                }
            }
            __syncwarp();   // the stage is free: refill it
            if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            produce();
        }

        // the unit's partial: sum the four key slots (lane bits 3, 4), halving
        // the carried heads per step; this lane ends with head 2*c0 + c1
        float2 h2[2][P2], h1[P2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int e = 0; e < P2; ++e) {
                const float2 snd = c0 ? o2[hh][e] : o2[hh + 2][e];
                const float2 kp = c0 ? o2[hh + 2][e] : o2[hh][e];
                h2[hh][e] = f2add(kp, shfl_xor2(snd, 8));
            }
#pragma unroll
        for (int e = 0; e < P2; ++e) {
            const float2 snd = c1 ? h2[0][e] : h2[1][e];
            const float2 kp = c1 ? h2[1][e] : h2[0][e];
            h1[e] = f2add(kp, shfl_xor2(snd, 16));
        }
        float lt0 = l_run[0], lt1 = l_run[1];
#pragma unroll
        for (int o = 2; o <= 16; o <<= 1) {
            lt0 += __shfl_xor_sync(FULLMASK, lt0, o);
            lt1 += __shfl_xor_sync(FULLMASK, lt1, o);
        }
        const size_t pbase = ((size_t)U.split * B + U.b) * H + h0;
        const int hw = 2 * (int)c0 + (int)c1;
        if (hw < nh) {
            float *dst = part_o + (pbase + hw) * D;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                if (!dv[c]) continue;
#pragma unroll
                for (int e = 0; e < VEC / 2; e += 2)
                    *reinterpret_cast<float4 *>(dst + (j + 8 * c) * VEC + 2 * e) =
                        make_float4(h1[c * (VEC / 2) + e].x, h1[c * (VEC / 2) + e].y,
                                    h1[c * (VEC / 2) + e + 1].x, h1[c * (VEC / 2) + e + 1].y);
            }
        }
        if (lane < 2) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int h = 2 * lane + k;
                if (h < nh) {
                    part_ml[(pbase + h) * 2] = m_run[k];
                    part_ml[(pbase + h) * 2 + 1] = k ? lt1 : lt0;
                }
            }
        }
    }
}

// ---------------------------------------------------------------- combine
template <typename T>
__global__ void __launch_bounds__(128)
k_decode_combine(const float *__restrict__ part_o, const float *__restrict__ part_ml,
                 T *__restrict__ out, float *__restrict__ lse, int B, int H, int D, int nsplit) {
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the attention grid's partials
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
    d.nhc = (group + kDecHP - 1) / kDecHP;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        sms = 148;
    // Key splits: each SM runs its units side by side, one per warp, and is
    // bound by the bytes it streams once about four warps stream at once, so
    // the step takes about max(ceil(units / SMs), 4) * (stages per unit + a
    // fixed cost of two stages); take the split count that minimises that
    // (ties: more, shorter units).
    const long base = (long)p.B * p.G * d.nhc;
    const long tiles = (p.S + kDecKT - 1) / kDecKT;
    long best_cost = -1, best_per = tiles, best_ns = 1;
    for (long ns = 1; ns <= tiles && ns <= 1024; ++ns) {
        const long per = (tiles + ns - 1) / ns;
        const long nse = (tiles + per - 1) / per;
        if (nse != ns) continue;
        const long units = base * nse;
        if (units > (1L << 30)) break;
        const long cost = std::max<long>((units + sms - 1) / sms, 4) * (per + 2);
        if (best_cost < 0 || cost <= best_cost) {
            best_cost = cost;
            best_per = per;
            best_ns = nse;
        }
    }
    d.L = (int)(best_per * kDecKT);
    d.nsplit = (int)best_ns;
    d.units = (int)(base * best_ns);
    // units go to the CTAs first (warp w of CTA c runs units w * grid + c, ...),
    // so every SM gets a share even when the units fill only part of the warps
    d.grid = std::min(sms, d.units);
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
    const RopeConsts &rc = rope_consts(p.theta, p.D);
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

template <typename T, int DP, bool FULL>
cudaError_t run_decode_attn(const Problem &p, const DecodePlan &d, const int *pos,
                            const float *qhat, const void *kc, const void *vc, float *part_o,
                            float *part_ml, unsigned int *err, cudaStream_t st) {
    constexpr int warps = dec_warps<T>();
    const size_t smem = (size_t)warps * kDecNS * 2 * kDecKT * p.D * sizeof(T);
    auto kern = k_decode_attn<T, DP, FULL>;
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, dim3(d.grid), dim3(warps * 32), smem, st, pos, qhat,
                            (const T *)kc, (const T *)vc, part_o, part_ml, p.B, p.S, p.H, p.G, p.D,
                            d.L, d.nsplit, d.nhc, d.units, err);
}

cudaError_t launch_decode_attn(const Problem &p, const DecodePlan &d, const int *pos,
                               const float *qhat, const void *kc, const void *vc, float *part_o,
                               float *part_ml, unsigned int *err, cudaStream_t st) {
    if (p.dtype == 1) {
        if (p.D == 128)
            return run_decode_attn<bf16, 128, true>(p, d, pos, qhat, kc, vc, part_o, part_ml, err,
                                                    st);
        if (p.D == 64)
            return run_decode_attn<bf16, 64, true>(p, d, pos, qhat, kc, vc, part_o, part_ml, err,
                                                   st);
        return run_decode_attn<bf16, 64, false>(p, d, pos, qhat, kc, vc, part_o, part_ml, err, st);
    }
    if (p.D > 64)
        return run_decode_attn<float, 128, false>(p, d, pos, qhat, kc, vc, part_o, part_ml, err, st);
    if (p.D > 32)
        return run_decode_attn<float, 64, false>(p, d, pos, qhat, kc, vc, part_o, part_ml, err, st);
    return run_decode_attn<float, 32, false>(p, d, pos, qhat, kc, vc, part_o, part_ml, err, st);
}

cudaError_t launch_decode_combine(const Problem &p, const DecodePlan &d, const float *part_o,
                                  const float *part_ml, void *out, float *lse, cudaStream_t st) {
    const dim3 grid((unsigned)((long)p.B * p.H));
    if (p.dtype == 1)
        return launch_dependent(k_decode_combine<bf16>, grid, dim3(128), 0, st, part_o, part_ml,
                                (bf16 *)out, lse, p.B, p.H, p.D, d.nsplit);
    return launch_dependent(k_decode_combine<float>, grid, dim3(128), 0, st, part_o, part_ml,
                            (float *)out, lse, p.B, p.H, p.D, d.nsplit);
}

}  // namespace xt
