// xt_bwd_tc.cu -- bf16 causal GQA flash backward on sm_103a tensor cores.
//
// Operation (web pages): the backward of the per-head causal SDPA of xtrain
// "Phase T5: Tiny Transformer" (scores = q k^T / sqrt(hd) + mask, softmax,
// P V), using the softmax Jacobian dS = P o (dP - Dlt), Dlt = rowsum(dO o O)
// (the pages name only a fused softmax backward); xtrain "Phase T15: GQA",
// Decision 2: the gradient of a shared kv head is the in-order sum over its
// group's query heads, formed without atomics; xtrain "Phase T12: bf16
// mixed precision" (bf16 operands, fp32 accumulation).
//
// Two kernels, both deterministic:
//  * k_bwd_dkdv_tc: a CTA owns 128 key rows of one (batch, kv head) and walks
//    the group's query heads r = 0..group-1 in order, each over the 64-row
//    query tiles at or after its keys, accumulating dV += P^T dO and
//    dKhat += dS^T Qhat in TMEM: the group sum happens inside the CTA.
//  * k_bwd_dq_tc: a CTA owns 128 query rows of one (batch, head) and walks
//    the 64-row key tiles at or before them, accumulating dQhat += dS Khat.
// Both recompute S from the saved Qhat, Khat and lse. For each streamed
// 64-row tile the MMA warp issues S (or S^T) and dP (or dP^T) into one of two
// TMEM buffers; the softmax warps (thread = one owned row) turn them into P
// and dS, written back as bf16 over the columns they have read, and the MMA
// warp consumes those as the A operand of TS MMAs. With two buffers the S/dP
// MMAs of tile t+1 overlap the softmax of tile t.
//
// Warps: 0-3 softmax + epilogue (thread = owned row = TMEM lane), 4 TMA
// producer, 5 TMEM allocator + MMA issuer.
// TMEM (512 columns): buffer b at [128b, 128b+128) with S (or S^T) in its
// first 64 columns and dP (or dP^T) in the next 64; accumulators at 256
// (and 384).
#include "xt_common.cuh"
#include "xt_internal.h"
#include "xt_tc.cuh"

namespace xt {

namespace {

using namespace tc;

constexpr int kOwn = 128;          // owned rows per CTA (MMA M)
constexpr int kStream = 64;        // rows per streamed tile (N of the S / dP MMAs)
constexpr int kThreadsBwd = 192;
constexpr int kStages = 3;

template <int D> struct BwdCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kOwnTile = kChunks * 16384;     // 128 rows x D bf16
    static constexpr int kStreamTile = kChunks * 8192;   // 64 rows x D bf16
    // a stage holds two streamed tiles and (dK/dV kernel) 2 x 64 row statistics
    static constexpr int kStageBytes = 2 * kStreamTile + 1024;
    static constexpr int kSmemBytes = 2 * kOwnTile + kStages * kStageBytes + 1024;
};

struct BwdBarriers {
    uint64_t own_full;
    uint64_t st_full[kStages], st_empty[kStages];
    uint64_t s_full[2], p_full[2], s_free[2];
    uint64_t acc_done;
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ void raise_error_b(unsigned int *err, volatile int *abort_flag) {
    atomicOr(err, ERR_TIMEOUT);
    *abort_flag = 1;
}

__device__ __forceinline__ void init_bwd_barriers(BwdBarriers &bars, uint32_t st_full_count) {
    bars.abort_flag = 0;
    mbar_init(&bars.own_full, 1);
    for (int s = 0; s < kStages; ++s) {
        mbar_init(&bars.st_full[s], st_full_count);
        mbar_init(&bars.st_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
        mbar_init(&bars.s_full[i], 1);
        mbar_init(&bars.p_full[i], 128);
        mbar_init(&bars.s_free[i], 1);
    }
    mbar_init(&bars.acc_done, 1);
    mbar_init(&bars.drain, 1);
    fence_barrier_init();
}

// K-major operand descriptors (128B swizzle, 8-row groups 1024 B apart):
// k-step kk of 16 elements inside 64-column chunks of `chunk_bytes`.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int kk, uint32_t chunk_bytes) {
    return smem_desc(base + (kk >> 2) * chunk_bytes + (kk & 3) * 32, 16, 1024, kSwizzle128B);
}

// MN-major B operand: k-step kk of 16 rows (2048 B), N spread over 64-column
// chunks `chunk_bytes` apart.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int kk, uint32_t chunk_bytes) {
    return smem_desc(base + kk * 2048, chunk_bytes, 1024, kSwizzle128B);
}

// ---------------------------------------------------------------------------
// dKhat, dV
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreadsBwd, 1)
k_bwd_dkdv_tc(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
              const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
              const float *__restrict__ lse, const float *__restrict__ dlt,
              float *__restrict__ dkhat, bf16 *__restrict__ dv, int S, int H, int G,
              int n_kvt, unsigned int *err) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ BwdBarriers bars;
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sK = smem;
    uint8_t *sV = smem + C::kOwnTile;
    uint8_t *sStage = smem + 2 * C::kOwnTile;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BG = gridDim.x / n_kvt;
    const int j = (int)(blockIdx.x / BG);          // key tile, longest first
    const int bg = blockIdx.x % BG;
    const int b = bg / G, g = bg - b * G, group = H / G;
    const int n_q64 = (S + kStream - 1) / kStream;
    const int u0 = 2 * j;                           // first query tile at/after the keys
    const int nU = n_q64 - u0;
    const int T = group * nU;
    volatile int *abort_flag = &bars.abort_flag;

    if (threadIdx.x == 0) init_bwd_barriers(bars, 2);
    if (warp == 5) {
        tmem_alloc(&bars.tmem_base, 512);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&map_k);
            tma_prefetch_desc(&map_v);
            tma_prefetch_desc(&map_q);
            tma_prefetch_desc(&map_do);
            mbar_expect_tx(&bars.own_full, 2 * C::kOwnTile);
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_3d(sK + c * 16384, &map_k, &bars.own_full, c * 64, j * kOwn, bg);
                tma_load_4d(sV + c * 16384, &map_v, &bars.own_full, c * 64, g, j * kOwn, b);
            }
        }
        int issued = 0;
        for (int t = 0; t < T; ++t) {
            const int st = t % kStages;
            bool ok = true;
            if (t >= kStages && lane == 0)
                ok = mbar_wait(&bars.st_empty[st], ((t / kStages) - 1) & 1, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0 && !*abort_flag) raise_error_b(err, abort_flag);
                break;
            }
            const int r = t / nU, u = u0 + (t - r * nU);
            const int h = g * group + r;
            uint8_t *base = sStage + st * C::kStageBytes;
            if (lane == 0) {
                mbar_expect_tx(&bars.st_full[st], 2 * C::kStreamTile);
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_3d(base + c * 8192, &map_q, &bars.st_full[st], c * 64, u * kStream,
                                b * H + h);
                    tma_load_4d(base + C::kStreamTile + c * 8192, &map_do, &bars.st_full[st],
                                c * 64, h, u * kStream, b);
                }
            }
            float *sl = reinterpret_cast<float *>(base + 2 * C::kStreamTile);
            const size_t row0 = ((size_t)b * H + h) * S;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int k = lane + 32 * e, q = u * kStream + k;
                sl[k] = q < S ? lse[row0 + q] * kLog2e : 0.f;
                sl[64 + k] = q < S ? dlt[row0 + q] : 0.f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.st_full[st]);
            issued = t + 1;
        }
        if (lane == 0) {
            // drain: every copy issued by this CTA lands before it exits
            mbar_wait(&bars.own_full, 0, nullptr);
            for (int t = max(0, issued - kStages); t < issued; ++t)
                mbar_wait(&bars.st_full[t % kStages], (t / kStages) & 1, nullptr);
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16_f32(kOwn, kStream, 0, 0);
            const uint32_t idesc_acc = idesc_bf16_f32(kOwn, D, 0, 1);
            const uint32_t aK = smem_u32(sK), aV = smem_u32(sV);
            bool ok = mbar_wait(&bars.own_full, 0, abort_flag);
            for (int t = 0; ok && t <= T; ++t) {
                if (t < T) {
                    const int st = t % kStages, buf = t & 1;
                    if (!(ok = mbar_wait(&bars.st_full[st], (t / kStages) & 1, abort_flag))) break;
                    if (t >= 2 && !(ok = mbar_wait(&bars.s_free[buf], ((t >> 1) - 1) & 1, abort_flag)))
                        break;
                    tc_fence_after();
                    const uint32_t aQ = smem_u32(sStage + st * C::kStageBytes);
                    const uint32_t aDO = aQ + C::kStreamTile;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)      // S^T = Khat Qhat^T
                        mma_ss(tmem + 128 * buf, kmajor_desc(aK, kk, 16384),
                               kmajor_desc(aQ, kk, 8192), idesc_s, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)      // dP^T = V dO^T
                        mma_ss(tmem + 128 * buf + 64, kmajor_desc(aV, kk, 16384),
                               kmajor_desc(aDO, kk, 8192), idesc_s, kk > 0);
                    mma_commit(&bars.s_full[buf]);
                }
                if (t >= 1) {
                    const int tp = t - 1, bp = tp & 1, stp = tp % kStages;
                    if (!(ok = mbar_wait(&bars.p_full[bp], (tp >> 1) & 1, abort_flag))) break;
                    tc_fence_after();
                    const uint32_t aQ = smem_u32(sStage + stp * C::kStageBytes);
                    const uint32_t aDO = aQ + C::kStreamTile;
#pragma unroll
                    for (int kk = 0; kk < kStream / 16; ++kk)   // dV += P^T dO
                        mma_ts(tmem + 256, tmem + 128 * bp + kk * 8,
                               mnmajor_desc(aDO, kk, 8192), idesc_acc, (tp > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < kStream / 16; ++kk)   // dKhat += dS^T Qhat
                        mma_ts(tmem + 384, tmem + 128 * bp + 64 + kk * 8,
                               mnmajor_desc(aQ, kk, 8192), idesc_acc, (tp > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&bars.s_free[bp]);
                    mma_commit(&bars.st_empty[stp]);
                }
            }
            if (ok) mma_commit(&bars.acc_done);
            else if (!*abort_flag) raise_error_b(err, abort_flag);
            mma_commit(&bars.drain);
            mbar_wait(&bars.drain, 0, nullptr);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int r = warp * 32 + lane;                 // owned key row = TMEM lane
        const int kp = j * kOwn + r;                    // key position
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const float sl2 = kLog2e * rsqrtf((float)D);
        bool ok = true;
        for (int t = 0; t < T; ++t) {
            const int buf = t & 1, st = t % kStages;
            ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full[buf], (t >> 1) & 1, abort_flag) &&
                                             mbar_wait(&bars.st_full[st], (t / kStages) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            const int u = u0 + (t % nU);
            const int q0 = u * kStream;
            const float *sl = reinterpret_cast<const float *>(sStage + st * C::kStageBytes +
                                                              2 * C::kStreamTile);
            const uint32_t tS = tmem + 128 * buf + lane_off;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t s[32], dp[32], pp[16], dd[16];
                tmem_ld32_sync(tS + 32 * c, s);
                tmem_ld32_sync(tS + 64 + 32 * c, dp);
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float pv[2], dsv[2];
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        const int col = 32 * c + e + x, q = q0 + col;
                        const float p = (q >= kp && q < S)
                                            ? fast_exp2(__uint_as_float(s[e + x]) * sl2 - sl[col])
                                            : 0.f;
                        pv[x] = p;
                        dsv[x] = p * (__uint_as_float(dp[e + x]) - sl[64 + col]);
                    }
                    pp[e >> 1] = pack_bf16x2(pv[0], pv[1]);
                    dd[e >> 1] = pack_bf16x2(dsv[0], dsv[1]);
                }
                tmem_st16_sync(tS + 16 * c, pp);
                tmem_st16_sync(tS + 64 + 16 * c, dd);
            }
            tc_fence_before();
            mbar_arrive(&bars.p_full[buf]);
        }
        if (ok) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars.acc_done, 0, abort_flag));
            if (ok) {
                tc_fence_after();
                const float scale = rsqrtf((float)D);
                bf16 *dvrow = dv + (((size_t)b * S + kp) * G + g) * D;
                float *dkrow = dkhat + ((size_t)bg * S + kp) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t a[32];
                    tmem_ld32_sync(tmem + 256 + lane_off + 32 * c, a);
                    if (kp < S) {
#pragma unroll
                        for (int q8 = 0; q8 < 4; ++q8) {
                            uint4 v4;
                            v4.x = pack_bf16x2(__uint_as_float(a[q8 * 8 + 0]), __uint_as_float(a[q8 * 8 + 1]));
                            v4.y = pack_bf16x2(__uint_as_float(a[q8 * 8 + 2]), __uint_as_float(a[q8 * 8 + 3]));
                            v4.z = pack_bf16x2(__uint_as_float(a[q8 * 8 + 4]), __uint_as_float(a[q8 * 8 + 5]));
                            v4.w = pack_bf16x2(__uint_as_float(a[q8 * 8 + 6]), __uint_as_float(a[q8 * 8 + 7]));
                            *reinterpret_cast<uint4 *>(dvrow + 32 * c + 8 * q8) = v4;
                        }
                    }
                    tmem_ld32_sync(tmem + 384 + lane_off + 32 * c, a);
                    if (kp < S) {
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4) {
                            float4 f;
                            f.x = __uint_as_float(a[q4 * 4 + 0]) * scale;
                            f.y = __uint_as_float(a[q4 * 4 + 1]) * scale;
                            f.z = __uint_as_float(a[q4 * 4 + 2]) * scale;
                            f.w = __uint_as_float(a[q4 * 4 + 3]) * scale;
                            *reinterpret_cast<float4 *>(dkrow + 32 * c + 4 * q4) = f;
                        }
                    }
                }
            }
        }
        if (!ok && !*abort_flag) raise_error_b(err, abort_flag);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// dQhat
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreadsBwd, 1)
k_bwd_dq_tc(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
            const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
            const float *__restrict__ lse, const float *__restrict__ dlt,
            float *__restrict__ dqhat, int S, int H, int G, int n_qt, unsigned int *err) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ BwdBarriers bars;
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sQ = smem;
    uint8_t *sDO = smem + C::kOwnTile;
    uint8_t *sStage = smem + 2 * C::kOwnTile;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = gridDim.x / n_qt;
    const int i = n_qt - 1 - (int)(blockIdx.x / BH);   // query tile, longest first
    const int bh = blockIdx.x % BH;
    const int b = bh / H, h = bh - b * H, g = h / (H / G);
    const int n_k64 = (S + kStream - 1) / kStream;
    const int T = min(2 * i + 2, n_k64);               // key tiles at or before the rows
    volatile int *abort_flag = &bars.abort_flag;

    if (threadIdx.x == 0) init_bwd_barriers(bars, 1);
    if (warp == 5) {
        tmem_alloc(&bars.tmem_base, 512);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&map_q);
            tma_prefetch_desc(&map_do);
            tma_prefetch_desc(&map_k);
            tma_prefetch_desc(&map_v);
            mbar_expect_tx(&bars.own_full, 2 * C::kOwnTile);
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_3d(sQ + c * 16384, &map_q, &bars.own_full, c * 64, i * kOwn, bh);
                tma_load_4d(sDO + c * 16384, &map_do, &bars.own_full, c * 64, h, i * kOwn, b);
            }
            int issued = 0;
            for (int t = 0; t < T; ++t) {
                const int st = t % kStages;
                if (t >= kStages &&
                    !mbar_wait(&bars.st_empty[st], ((t / kStages) - 1) & 1, abort_flag)) {
                    if (!*abort_flag) raise_error_b(err, abort_flag);
                    break;
                }
                uint8_t *base = sStage + st * C::kStageBytes;
                mbar_expect_tx(&bars.st_full[st], 2 * C::kStreamTile);
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_3d(base + c * 8192, &map_k, &bars.st_full[st], c * 64, t * kStream,
                                b * G + g);
                    tma_load_4d(base + C::kStreamTile + c * 8192, &map_v, &bars.st_full[st],
                                c * 64, g, t * kStream, b);
                }
                issued = t + 1;
            }
            mbar_wait(&bars.own_full, 0, nullptr);
            for (int t = max(0, issued - kStages); t < issued; ++t)
                mbar_wait(&bars.st_full[t % kStages], (t / kStages) & 1, nullptr);
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16_f32(kOwn, kStream, 0, 0);
            const uint32_t idesc_acc = idesc_bf16_f32(kOwn, D, 0, 1);
            const uint32_t aQ = smem_u32(sQ), aDO = smem_u32(sDO);
            bool ok = mbar_wait(&bars.own_full, 0, abort_flag);
            for (int t = 0; ok && t <= T; ++t) {
                if (t < T) {
                    const int st = t % kStages, buf = t & 1;
                    if (!(ok = mbar_wait(&bars.st_full[st], (t / kStages) & 1, abort_flag))) break;
                    if (t >= 2 && !(ok = mbar_wait(&bars.s_free[buf], ((t >> 1) - 1) & 1, abort_flag)))
                        break;
                    tc_fence_after();
                    const uint32_t aK = smem_u32(sStage + st * C::kStageBytes);
                    const uint32_t aV = aK + C::kStreamTile;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)      // S = Qhat Khat^T
                        mma_ss(tmem + 128 * buf, kmajor_desc(aQ, kk, 16384),
                               kmajor_desc(aK, kk, 8192), idesc_s, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)      // dP = dO V^T
                        mma_ss(tmem + 128 * buf + 64, kmajor_desc(aDO, kk, 16384),
                               kmajor_desc(aV, kk, 8192), idesc_s, kk > 0);
                    mma_commit(&bars.s_full[buf]);
                }
                if (t >= 1) {
                    const int tp = t - 1, bp = tp & 1, stp = tp % kStages;
                    if (!(ok = mbar_wait(&bars.p_full[bp], (tp >> 1) & 1, abort_flag))) break;
                    tc_fence_after();
                    const uint32_t aK = smem_u32(sStage + stp * C::kStageBytes);
#pragma unroll
                    for (int kk = 0; kk < kStream / 16; ++kk)   // dQhat += dS Khat
                        mma_ts(tmem + 256, tmem + 128 * bp + kk * 8, mnmajor_desc(aK, kk, 8192),
                               idesc_acc, (tp > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&bars.s_free[bp]);
                    mma_commit(&bars.st_empty[stp]);
                }
            }
            if (ok) mma_commit(&bars.acc_done);
            else if (!*abort_flag) raise_error_b(err, abort_flag);
            mma_commit(&bars.drain);
            mbar_wait(&bars.drain, 0, nullptr);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int r = warp * 32 + lane;                // owned query row = TMEM lane
        const int tq = i * kOwn + r;                   // query position
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const float sl2 = kLog2e * rsqrtf((float)D);
        const float lse2 = tq < S ? lse[(size_t)bh * S + tq] * kLog2e : 0.f;
        const float dl = tq < S ? dlt[(size_t)bh * S + tq] : 0.f;
        bool ok = true;
        for (int t = 0; t < T; ++t) {
            const int buf = t & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full[buf], (t >> 1) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            const int k0 = t * kStream;
            const uint32_t tS = tmem + 128 * buf + lane_off;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t s[32], dp[32], dd[16];
                tmem_ld32_sync(tS + 32 * c, s);
                tmem_ld32_sync(tS + 64 + 32 * c, dp);
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float dsv[2];
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        const int kpos = k0 + 32 * c + e + x;
                        const float p = (kpos <= tq)
                                            ? fast_exp2(__uint_as_float(s[e + x]) * sl2 - lse2)
                                            : 0.f;
                        dsv[x] = p * (__uint_as_float(dp[e + x]) - dl);
                    }
                    dd[e >> 1] = pack_bf16x2(dsv[0], dsv[1]);
                }
                tmem_st16_sync(tS + 16 * c, dd);
            }
            tc_fence_before();
            mbar_arrive(&bars.p_full[buf]);
        }
        if (ok) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars.acc_done, 0, abort_flag));
            if (ok) {
                tc_fence_after();
                const float scale = rsqrtf((float)D);
                float *dst = dqhat + ((size_t)bh * S + tq) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t a[32];
                    tmem_ld32_sync(tmem + 256 + lane_off + 32 * c, a);
                    if (tq < S) {
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4) {
                            float4 f;
                            f.x = __uint_as_float(a[q4 * 4 + 0]) * scale;
                            f.y = __uint_as_float(a[q4 * 4 + 1]) * scale;
                            f.z = __uint_as_float(a[q4 * 4 + 2]) * scale;
                            f.w = __uint_as_float(a[q4 * 4 + 3]) * scale;
                            *reinterpret_cast<float4 *>(dst + 32 * c + 4 * q4) = f;
                        }
                    }
                }
            }
        }
        if (!ok && !*abort_flag) raise_error_b(err, abort_flag);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
struct BwdMaps {
    CUtensorMap q, k, v, dout;
};

// Qhat [B*H, S, D] / Khat [B*G, S, D] as 3-D maps; V [B, S, G, D] and
// dO [B, S, H, D] as 4-D maps (D, heads, S, B); boxes of 64 columns x rows.
cudaError_t make_maps(const Problem &p, const void *qhat, const void *khat, const void *v,
                      const void *dout, int q_rows, int k_rows, BwdMaps &m) {
    const uint64_t esz = 2, D = (uint64_t)p.D;
    cudaError_t e;
    {
        const uint64_t dims[3] = {D, (uint64_t)p.S, (uint64_t)p.B * p.H};
        const uint64_t strides[2] = {D * esz, (uint64_t)p.S * D * esz};
        const uint32_t box[3] = {64, (uint32_t)q_rows, 1};
        if ((e = encode_tmap_bf16(&m.q, qhat, 3, dims, strides, box)) != cudaSuccess) return e;
    }
    {
        const uint64_t dims[3] = {D, (uint64_t)p.S, (uint64_t)p.B * p.G};
        const uint64_t strides[2] = {D * esz, (uint64_t)p.S * D * esz};
        const uint32_t box[3] = {64, (uint32_t)k_rows, 1};
        if ((e = encode_tmap_bf16(&m.k, khat, 3, dims, strides, box)) != cudaSuccess) return e;
    }
    {
        const uint64_t dims[4] = {D, (uint64_t)p.G, (uint64_t)p.S, (uint64_t)p.B};
        const uint64_t strides[3] = {D * esz, (uint64_t)p.G * D * esz, (uint64_t)p.S * p.G * D * esz};
        const uint32_t box[4] = {64, 1, (uint32_t)k_rows, 1};
        if ((e = encode_tmap_bf16(&m.v, v, 4, dims, strides, box)) != cudaSuccess) return e;
    }
    {
        const uint64_t dims[4] = {D, (uint64_t)p.H, (uint64_t)p.S, (uint64_t)p.B};
        const uint64_t strides[3] = {D * esz, (uint64_t)p.H * D * esz, (uint64_t)p.S * p.H * D * esz};
        const uint32_t box[4] = {64, 1, (uint32_t)q_rows, 1};
        if ((e = encode_tmap_bf16(&m.dout, dout, 4, dims, strides, box)) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int D>
cudaError_t launch_dkdv_d(const Problem &p, const void *qhat, const void *khat, const void *v,
                          const void *dout, const float *lse, const float *dlt, float *dkhat,
                          void *dv, unsigned int *err, cudaStream_t st) {
    using C = BwdCfg<D>;
    BwdMaps m;
    cudaError_t e = make_maps(p, qhat, khat, v, dout, kStream, kOwn, m);
    if (e != cudaSuccess) return e;
    const int n_kvt = (p.S + kOwn - 1) / kOwn;
    const long blocks = (long)p.B * p.G * n_kvt;
    if ((e = cudaFuncSetAttribute(k_bwd_dkdv_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  C::kSmemBytes)) != cudaSuccess)
        return e;
    k_bwd_dkdv_tc<D><<<(unsigned)blocks, kThreadsBwd, C::kSmemBytes, st>>>(
        m.k, m.v, m.q, m.dout, lse, dlt, dkhat, (bf16 *)dv, p.S, p.H, p.G, n_kvt, err);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_dq_d(const Problem &p, const void *qhat, const void *khat, const void *v,
                        const void *dout, const float *lse, const float *dlt, float *dqhat,
                        unsigned int *err, cudaStream_t st) {
    using C = BwdCfg<D>;
    BwdMaps m;
    cudaError_t e = make_maps(p, qhat, khat, v, dout, kOwn, kStream, m);
    if (e != cudaSuccess) return e;
    const int n_qt = (p.S + kOwn - 1) / kOwn;
    const long blocks = (long)p.B * p.H * n_qt;
    if ((e = cudaFuncSetAttribute(k_bwd_dq_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  C::kSmemBytes)) != cudaSuccess)
        return e;
    k_bwd_dq_tc<D><<<(unsigned)blocks, kThreadsBwd, C::kSmemBytes, st>>>(
        m.q, m.dout, m.k, m.v, lse, dlt, dqhat, p.S, p.H, p.G, n_qt, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv_tc(const Problem &p, const void *qhat, const void *khat,
                               const void *v, const void *dout, const float *lse,
                               const float *dlt, float *dkhat, void *dv, unsigned int *err,
                               cudaStream_t st) {
    if (p.D == 128) return launch_dkdv_d<128>(p, qhat, khat, v, dout, lse, dlt, dkhat, dv, err, st);
    if (p.D == 64) return launch_dkdv_d<64>(p, qhat, khat, v, dout, lse, dlt, dkhat, dv, err, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dq_tc(const Problem &p, const void *qhat, const void *khat, const void *v,
                             const void *dout, const float *lse, const float *dlt, float *dqhat,
                             unsigned int *err, cudaStream_t st) {
    if (p.D == 128) return launch_dq_d<128>(p, qhat, khat, v, dout, lse, dlt, dqhat, err, st);
    if (p.D == 64) return launch_dq_d<64>(p, qhat, khat, v, dout, lse, dlt, dqhat, err, st);
    return cudaErrorInvalidValue;
}

}  // namespace xt
