// xt_fwd_tc.cu -- bf16 causal GQA flash forward on sm_103a tensor cores.
//
// Operation (web pages): xtrain "Phase T5: Tiny Transformer", multi-head
// pipeline (per head: scores = q k^T / sqrt(hd) + causal mask, softmax,
// P V); Mint project report 5.3.1 (max-subtracted softmax, a_t = sum_j
// p_tj v_j); xtrain "Phase T15: GQA" (query head h reads kv head
// h / group); xtrain "Phase T12: bf16 mixed precision" (bf16 operands, fp32
// accumulation and softmax). Keys j > t are skipped; the pages' additive
// -1e9 mask makes their probabilities exactly 0 in fp32 anyway.
//
// A work item is two consecutive 128-row query tiles (2p, 2p+1) of one
// (batch, head); a persistent grid of one CTA per SM walks the items (longest
// first), ping-ponging the item's two tiles so that the tensor core works on
// one while the softmax warps work on the other:
//   warps 0-3  softmax + epilogue of query tile 0 (thread = one query row)
//   warps 4-7  softmax + epilogue of query tile 1
//   warp  8    TMA producer: each item's Q tiles, then its K and V tiles into
//              two rings (a K tile is released after its last S MMA, an
//              iteration before its V tile)
//   warp  9    TMEM allocator and MMA issuer (the whole warp runs the issue
//              loop; one elected lane issues each MMA)
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [384,384+D).
// S_i = Q_i K^T is an SS MMA (both operands K-major, 128B swizzle); the
// softmax warps overwrite the first 64 columns of S_i with P_i as packed
// bf16, and O_i += P_i V is a TS MMA (A = P from TMEM, B = V MN-major).
// Online softmax in the log2 domain with lazy rescaling: the running max
// used for exp2 is only raised when a row's max grows by more than 8, so O
// is rescaled in TMEM rarely; the final 1/l and lse use the same max.
//
// Every barrier wait is bounded (xt_tc.cuh); on a timeout the CTA raises the
// library's error word, drains its own copies and MMAs, frees TMEM and exits.
#include <algorithm>

#include "xt_common.cuh"
#include "xt_internal.h"
#include "xt_tc.cuh"

namespace xt {

namespace {

using namespace tc;

constexpr int kBM = 128;         // query rows per tile
constexpr int kBN = 128;         // key rows per tile
constexpr int kThreadsFwd = 320;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D> struct FwdCfg {
    using A = Atoms<D>;
    static constexpr int kChunks = A::kPerRow;              // swizzle atoms (TMA boxes) per row
    static constexpr int kBox = A::box_bytes(128);          // one box of a 128-row tile
    static constexpr int kTileBytes = kChunks * kBox;       // one 128-row tile
    // separate K and V rings: a K tile is released once the last S MMA that reads
    // it has run (an iteration before its V tile), so each ring refills on its own
    static constexpr int kKStages = (D == 128) ? 2 : 5;
    static constexpr int kVStages = (D == 128) ? 3 : 5;
    static constexpr int kSmemBytes = (2 + kKStages + kVStages) * kTileBytes + 1024;
};
constexpr int kMaxRing = 8;

struct FwdBarriers {
    uint64_t q_full, q_empty;
    uint64_t k_full[kMaxRing], k_empty[kMaxRing], v_full[kMaxRing], v_empty[kMaxRing];
    uint64_t s_full[2], p_full[2], o_done[2];
    uint64_t drain;
    uint64_t stall;   // never arrived on (xt_test_inject_stall)
    uint32_t tmem_base;
    int abort_flag;
};

// Work item w: query tiles 2 pair and 2 pair + 1 of head h of unit `unit`.
// Items run longest first (pair descending); consecutive items are
// consecutive heads of one unit, so CTAs working at the same time share K/V
// tiles in L2. n_kv[i]: key tiles of query tile i (0 past a short sample).
struct FwdItem {
    int pair, h, g;
    SeqSpan sp;
    int n_kv[2];
};

__device__ __forceinline__ FwdItem fwd_item(int w, int BH, int n_pairs, int H, int G,
                                            const SeqRows &sr) {
    FwdItem it;
    it.pair = n_pairs - 1 - w / BH;
    const int bh = w - (w / BH) * BH;
    const int unit = bh / H;
    it.h = bh - unit * H;
    it.g = it.h / (H / G);
    it.sp = seq_span(sr, unit);
    const int n_qtiles = (it.sp.len + kBM - 1) / kBM;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int qt = 2 * it.pair + i;
        it.n_kv[i] = qt < n_qtiles ? qt + 1 : 0;
    }
    return it;
}

__device__ __forceinline__ void raise_error(unsigned int *err, volatile int *abort_flag) {
    atomicOr(err, ERR_TIMEOUT);
    *abort_flag = 1;
}

// Epilogue of one query row: O / l from TMEM (this warp's lanes, columns
// [tO, tO + D)) -> bf16 row `dst`; lse = (m + log2 l) ln 2. A separate
// function, so that the softmax loop keeps its registers.
template <int D>
__device__ __noinline__ void write_out_row(uint32_t tO, float l, float m_used, bool row_ok,
                                           bf16 *dst, float *lse_row) {
    const float inv_l = 1.0f / l;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32_sync(tO + c * 32, o);
        if (row_ok) {
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(o[q8 * 8 + 0]) * inv_l, __uint_as_float(o[q8 * 8 + 1]) * inv_l);
                v.y = pack_bf16x2(__uint_as_float(o[q8 * 8 + 2]) * inv_l, __uint_as_float(o[q8 * 8 + 3]) * inv_l);
                v.z = pack_bf16x2(__uint_as_float(o[q8 * 8 + 4]) * inv_l, __uint_as_float(o[q8 * 8 + 5]) * inv_l);
                v.w = pack_bf16x2(__uint_as_float(o[q8 * 8 + 6]) * inv_l, __uint_as_float(o[q8 * 8 + 7]) * inv_l);
                *reinterpret_cast<uint4 *>(dst + c * 32 + q8 * 8) = v;
            }
        }
    }
    if (row_ok) *lse_row = (m_used + __log2f(l)) * kLn2;
}

template <int D>
__global__ void __launch_bounds__(kThreadsFwd, 1)
k_fwd_tc(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
         const __grid_constant__ CUtensorMap map_v, bf16 *__restrict__ out,
         float *__restrict__ lse, const SeqRows sr, int H, int G, int BH, int n_pairs,
         int n_items, unsigned int *err, int stall) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ FwdBarriers bars;
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sQ = smem;                                   // 2 tiles
    uint8_t *sK = smem + 2 * C::kTileBytes;               // kKStages tiles
    uint8_t *sV = sK + C::kKStages * C::kTileBytes;       // kVStages tiles

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &bars.abort_flag;

    if (threadIdx.x == 0) {
        bars.abort_flag = 0;
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.q_empty, 1);
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(&bars.k_full[s], 1);
            mbar_init(&bars.k_empty[s], 1);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(&bars.v_full[s], 1);
            mbar_init(&bars.v_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.p_full[i], 128);
            mbar_init(&bars.o_done[i], 1);
        }
        mbar_init(&bars.drain, 1);
        mbar_init(&bars.stall, 1);
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc(&bars.tmem_base, 512);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    pdl_enter();
    const uint32_t tmem = bars.tmem_base;

    // Every role walks the same items (snake_item: rounds of gridDim.x items,
    // walked forwards and backwards in turn) and
    // skips the same empty ones; barrier phases are counted across items.
    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&map_q);
            tma_prefetch_desc(&map_k);
            tma_prefetch_desc(&map_v);
            int q_issued = 0, k_issued = 0, v_issued = 0;
            bool ok = true;
            for (int rnd = 0, w = snake_item(0); ok && w < n_items; w = snake_item(++rnd)) {
                const FwdItem it = fwd_item(w, BH, n_pairs, H, G, sr);
                if (it.n_kv[0] == 0) continue;   // a packed sample shorter than this pair's rows
                const int n_iter = max(it.n_kv[0], it.n_kv[1]);
                const int qplane = it.sp.plane * H + it.h, kplane = it.sp.plane * G + it.g;
                // the Q tiles are reloaded once the previous item's S MMAs have read them
                if (q_issued > 0 &&
                    !(ok = mbar_wait(&bars.q_empty, (q_issued - 1) & 1, abort_flag)))
                    break;
                const int nq = (it.n_kv[1] > 0) ? 2 : 1;
                mbar_expect_tx(&bars.q_full, nq * C::kTileBytes);
                for (int i = 0; i < nq; ++i)
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(sQ + i * C::kTileBytes + c * C::kBox, &map_q, &bars.q_full,
                                    c * C::A::kCols, it.sp.start + (2 * it.pair + i) * kBM, qplane);
                ++q_issued;
                for (int j = 0; j < n_iter; ++j) {
                    const int x = v_issued;   // == k_issued here
                    const int ks = x % C::kKStages, vs = x % C::kVStages;
                    if (x >= C::kKStages &&
                        !(ok = mbar_wait(&bars.k_empty[ks], ((x / C::kKStages) - 1) & 1, abort_flag)))
                        break;
                    mbar_expect_tx(&bars.k_full[ks], C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(sK + ks * C::kTileBytes + c * C::kBox, &map_k, &bars.k_full[ks],
                                    c * C::A::kCols, it.sp.start + j * kBN, kplane);
                    ++k_issued;
                    if (x >= C::kVStages &&
                        !(ok = mbar_wait(&bars.v_empty[vs], ((x / C::kVStages) - 1) & 1, abort_flag)))
                        break;
                    mbar_expect_tx(&bars.v_full[vs], C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_4d(sV + vs * C::kTileBytes + c * C::kBox, &map_v, &bars.v_full[vs],
                                    c * C::A::kCols, it.g, it.sp.start + j * kBN, it.sp.plane);
                    ++v_issued;
                }
            }
            if (!ok && !*abort_flag) raise_error(err, abort_flag);
            // Drain: every copy this CTA issued must land before it exits (at most the
            // last Q load, the last kKStages K tiles and the last kVStages V tiles can
            // still be in flight).
            if (q_issued > 0) mbar_wait(&bars.q_full, (q_issued - 1) & 1, nullptr);
            for (int x = max(0, k_issued - C::kKStages); x < k_issued; ++x)
                mbar_wait(&bars.k_full[x % C::kKStages], (x / C::kKStages) & 1, nullptr);
            for (int x = max(0, v_issued - C::kVStages); x < v_issued; ++x)
                mbar_wait(&bars.v_full[x % C::kVStages], (x / C::kVStages) & 1, nullptr);
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        // Issue order per key tile j: PV_{j,0}, S_{j+1,0}, PV_{j,1}, S_{j+1,1}, so the
        // next S of query tile 0 queues right behind its PV while tile 1's softmax runs.
        // The MMA warp waits for data (TMA) and for P (softmax), never for its own
        // MMAs: the tensor pipe executes one thread's MMAs in issue order. The first
        // PV of an item overwrites O_i: the softmax threads of tile i read the
        // previous item's O_i (epilogue) before they signal that item's first P_i.
        {
            // the whole warp runs this loop; one elected lane issues each MMA / commit
            const uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0, 0);
            const uint32_t idesc_o = idesc_bf16_f32(kBM, D, 0, 1);
            const uint32_t tS[2] = {tmem, tmem + 128};
            const uint32_t tO[2] = {tmem + 256, tmem + 384};
            // Descriptors are built once; per MMA only a compile-time offset (>> 4, the
            // start-address field) is added, which keeps the single issuing thread fast.
            using A = typename C::A;
            const uint64_t dQ0 = smem_desc(smem_u32(sQ), 16, A::kSBO, A::kMode);
            const uint64_t dK0 = smem_desc(smem_u32(sK), 16, A::kSBO, A::kMode);
            const uint64_t dV0 = smem_desc(smem_u32(sV), C::kBox, A::kSBO, A::kMode);
            constexpr uint64_t kTileStep = (uint64_t)C::kTileBytes >> 4;
            auto issue_s = [&](int i, int ks) {
                const uint64_t dQ = dQ0 + (uint64_t)i * kTileStep;
                const uint64_t dK = dK0 + (uint64_t)ks * kTileStep;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)A::kstep(kk, kBM) >> 4;
                    mma_ss_w(tS[i], dQ + off, dK + off, idesc_s, kk > 0);
                }
                mma_commit_w(&bars.s_full[i]);
            };
            bool ok = !stall ||
                      __all_sync(0xffffffffu, mbar_wait_for(&bars.stall, 0, abort_flag, kStallLimitNs));
            int items = 0, kv_used = 0, p_cnt[2] = {0, 0};
            for (int rnd = 0, w = snake_item(0); ok && w < n_items; w = snake_item(++rnd)) {
                const FwdItem it = fwd_item(w, BH, n_pairs, H, G, sr);
                if (it.n_kv[0] == 0) continue;
                const int n_iter = max(it.n_kv[0], it.n_kv[1]);
                const int ks0 = kv_used % C::kKStages;
                ok = mbar_wait_w(&bars.q_full, items & 1, abort_flag) &&
                     mbar_wait_w(&bars.k_full[ks0], (kv_used / C::kKStages) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                for (int i = 0; i < 2; ++i)
                    if (it.n_kv[i] > 0) issue_s(i, ks0);
                mma_commit_w(&bars.k_empty[ks0]);   // K tile 0 of the item is read by then
                for (int j = 0; ok && j < n_iter; ++j) {
                    const int x = kv_used + j;
                    const int vs = x % C::kVStages, ks1 = (x + 1) % C::kKStages;
                    const uint64_t dV = dV0 + (uint64_t)vs * kTileStep;
                    if (!(ok = mbar_wait_w(&bars.v_full[vs], (x / C::kVStages) & 1, abort_flag))) break;
                    bool k_next = false;
                    for (int i = 0; i < 2 && ok; ++i) {
                        if (j >= it.n_kv[i]) continue;
                        if (!(ok = mbar_wait_w(&bars.p_full[i], p_cnt[i] & 1, abort_flag))) break;
                        ++p_cnt[i];
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk)
                            mma_ts_w(tO[i], tS[i] + kk * 8, dV + (uint64_t)(A::mnstep(kk) >> 4),
                                   idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                        mma_commit_w(&bars.o_done[i]);
                        if (j + 1 < it.n_kv[i]) {
                            if (!k_next) {
                                if (!(ok = mbar_wait_w(&bars.k_full[ks1], ((x + 1) / C::kKStages) & 1,
                                                     abort_flag)))
                                    break;
                                k_next = true;
                            }
                            // No wait for PV_{j,i} to finish reading P_i: tcgen05.mma
                            // operations issued by one thread execute in issue order.
                            issue_s(i, ks1);
                        }
                    }
                    if (!ok) break;
                    mma_commit_w(&bars.v_empty[vs]);                // V tile j is read
                    if (k_next) mma_commit_w(&bars.k_empty[ks1]);   // and K tile j + 1
                }
                if (!ok) break;
                mma_commit_w(&bars.q_empty);   // every S MMA of this item has read sQ
                kv_used += n_iter;
                ++items;
            }
            if (!ok && lane == 0 && !*abort_flag) raise_error(err, abort_flag);
            // Drain: all MMAs issued by this warp complete before TMEM is freed.
            mma_commit_w(&bars.drain);
            mbar_wait_w(&bars.drain, 0, nullptr);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int i = warp >> 2;                 // query tile of this warpgroup
        const int quarter = warp & 3;            // TMEM lanes [32*quarter, 32*quarter+32)
        const int r = quarter * 32 + lane;       // row within the tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + i * 128 + lane_off;
        const uint32_t tO = tmem + 256 + i * 128 + lane_off;
        const float sl2 = kLog2e * rsqrtf((float)D);
        bool ok = true;
        int s_cnt = 0;   // S_i tiles (and PV_i MMAs) of the previous items
        for (int rnd = 0, w = snake_item(0); ok && w < n_items; w = snake_item(++rnd)) {
            const FwdItem it = fwd_item(w, BH, n_pairs, H, G, sr);
            const int n = it.n_kv[i];
            if (n == 0) continue;                // no query tile i in this item
            const int t = (2 * it.pair + i) * kBM + r;   // query position inside the unit
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < n; ++j) {
                ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full[i], (s_cnt + j) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                uint32_t sr[128];
                tmem_ld128_sync(tS, sr);
                if (j == n - 1) {
                    // diagonal tile: key column c is visible to row r iff c <= r
#pragma unroll
                    for (int e = 0; e < 128; ++e)
                        if (e > r) sr[e] = __float_as_uint(-INFINITY);
                }
                float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
                for (int e = 0; e < 128; e += 4) {
                    m0 = fmax3(m0, __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
                    m1 = fmax3(m1, __uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3]));
                }
                const float mx = fmaxf(m0, m1) * sl2;
                const float m_new = fmaxf(m_used, mx);
                const bool need = m_new - m_used > kRescaleThreshold;   // true on the first tile
                float alpha = 1.f;
                if (need) {
                    alpha = fast_exp2(m_used - m_new);
                    m_used = m_new;
                }
                // O rescale in TMEM (warp-uniform: tcgen05.ld/st are warp-collective)
                if (j > 0 && __any_sync(0xffffffffu, need)) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&bars.o_done[i], (s_cnt + j - 1) & 1,
                                                           abort_flag));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32_sync(tO + c * 32, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32_sync(tO + c * 32, o);
                    }
                }
                // element pairs through the packed fp32 pipe (f32x2 FMA / add)
                const float2 nm2 = make_float2(-m_used, -m_used), sl2v = make_float2(sl2, sl2);
                float2 rs01 = make_float2(0.f, 0.f), rs23 = make_float2(0.f, 0.f);
                uint32_t pk[64];
#pragma unroll
                for (int e = 0; e < 128; e += 4) {
                    const float2 a01 = ffma2(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
                                             sl2v, nm2);
                    const float2 a23 = ffma2(make_float2(__uint_as_float(sr[e + 2]),
                                                         __uint_as_float(sr[e + 3])), sl2v, nm2);
                    const float2 p01 = make_float2(fast_exp2(a01.x), fast_exp2(a01.y));
                    const float2 p23 = make_float2(fast_exp2(a23.x), fast_exp2(a23.y));
                    rs01 = fadd2(rs01, p01);
                    rs23 = fadd2(rs23, p23);
                    pk[e >> 1] = pack_bf16x2(p01.x, p01.y);
                    pk[(e >> 1) + 1] = pack_bf16x2(p23.x, p23.y);
                }
                const float rowsum = (rs01.x + rs01.y) + (rs23.x + rs23.y);
                tmem_st64_sync(tS, pk);
                tc_fence_before();
                mbar_arrive(&bars.p_full[i]);
                l = l * alpha + rowsum;
            }
            if (!ok) break;
            // epilogue: O / l -> bf16 rows of out [B, S, H, D]; lse = (m + log2 l) ln 2
            ok = __all_sync(0xffffffffu, mbar_wait(&bars.o_done[i], (s_cnt + n - 1) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            const size_t row = (size_t)it.sp.plane * sr.S + it.sp.start + t;
            write_out_row<D>(tO, l, m_used, t < it.sp.len, out + (row * H + it.h) * D,
                             lse + ((size_t)it.sp.plane * H + it.h) * sr.S + it.sp.start + t);
            s_cnt += n;
        }
        if (!ok && !*abort_flag) raise_error(err, abort_flag);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
cudaError_t launch_fwd_tc_d(const Problem &p, const void *qhat, const void *khat, const void *v,
                            void *out, float *lse, unsigned int *err, cudaStream_t st) {
    using C = FwdCfg<D>;
    CUtensorMap mq, mk, mv;
    const uint64_t esz = 2;
    {
        const uint64_t dims[3] = {(uint64_t)D, (uint64_t)p.S, (uint64_t)p.B * p.H};
        const uint64_t strides[2] = {D * esz, (uint64_t)p.S * D * esz};
        const uint32_t box[3] = {(uint32_t)C::A::kCols, kBM, 1};
        cudaError_t e = encode_tmap_bf16(&mq, qhat, 3, dims, strides, box, C::A::kSwizzleBytes);
        if (e != cudaSuccess) return e;
    }
    {
        const uint64_t dims[3] = {(uint64_t)D, (uint64_t)p.S, (uint64_t)p.B * p.G};
        const uint64_t strides[2] = {D * esz, (uint64_t)p.S * D * esz};
        const uint32_t box[3] = {(uint32_t)C::A::kCols, kBN, 1};
        cudaError_t e = encode_tmap_bf16(&mk, khat, 3, dims, strides, box, C::A::kSwizzleBytes);
        if (e != cudaSuccess) return e;
    }
    {
        const uint64_t dims[4] = {(uint64_t)D, (uint64_t)p.G, (uint64_t)p.S, (uint64_t)p.B};
        const uint64_t strides[3] = {D * esz, (uint64_t)p.G * D * esz, (uint64_t)p.S * p.G * D * esz};
        const uint32_t box[4] = {(uint32_t)C::A::kCols, 1, kBN, 1};
        cudaError_t e = encode_tmap_bf16(&mv, v, 4, dims, strides, box, C::A::kSwizzleBytes);
        if (e != cudaSuccess) return e;
    }
    const int n_qtiles = (p.max_len + kBM - 1) / kBM;
    const int n_pairs = (n_qtiles + 1) / 2;
    const long BH = (long)p.units * p.H;
    const long n_items = BH * n_pairs;
    if (n_items >= (1L << 31)) return cudaErrorInvalidValue;
    // persistent grid: one CTA per SM walks the items (one CTA fits an SM: 512 TMEM columns)
    const long blocks = std::min<long>(n_items, sm_count());
    cudaError_t e = cudaFuncSetAttribute(k_fwd_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_dependent(k_fwd_tc<D>, dim3((unsigned)blocks), dim3(kThreadsFwd), C::kSmemBytes,
                            st, mq, mk, mv, (bf16 *)out, lse, SeqRows{p.cu, p.S, p.max_len}, p.H,
                            p.G, (int)BH, n_pairs, (int)n_items, err,
                            (int)((test_stall_mask() & STALL_FWD_TC) != 0));
}

}  // namespace

cudaError_t launch_fwd_tc(const Problem &p, const void *qhat, const void *khat, const void *v,
                          void *out, float *lse, unsigned int *err, cudaStream_t st) {
    if (p.D == 128) return launch_fwd_tc_d<128>(p, qhat, khat, v, out, lse, err, st);
    if (p.D == 64) return launch_fwd_tc_d<64>(p, qhat, khat, v, out, lse, err, st);
    if (p.D == 32) return launch_fwd_tc_d<32>(p, qhat, khat, v, out, lse, err, st);
    return cudaErrorInvalidValue;
}

}  // namespace xt
