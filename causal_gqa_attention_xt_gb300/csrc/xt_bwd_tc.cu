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
//    the group's query heads r = 0..group-1 in order, each over the 128-row
//    query tiles at or after its keys, accumulating dV += P^T dO and
//    dKhat += dS^T Qhat in TMEM: the group sum happens inside the CTA.
//    k_bwd_dkdv_tc_p is its persistent form for short items at D <= 64.
//  * k_bwd_dq_tc: a persistent CTA walks (batch, head, 128 query rows) items;
//    for each it walks the 128-row key tiles at or before the rows,
//    accumulating dQhat += dS Khat; its epilogue finishes dq (RoPE backward,
//    then RMSNorm backward: Mint project report 5.4.4 and 5.5.2) and writes the
//    item's dgamma_q partial, so dQhat never leaves TMEM.
// Both recompute S from the saved Qhat, Khat and lse.
//
// TMEM: S (or S^T) in columns [0,128), dP (or dP^T) in [128,256), the
// accumulators from 256. Four softmax warpgroups split the streamed tile's 128
// columns (warpgroup w takes [32w, 32w+32)) and form P and dS; the
// accumulating MMAs (TS form, A from TMEM) read them packed as bf16 k-step by
// k-step; the causal-mask select runs only on tiles that cross the diagonal or
// the end of the sequence.
//
// dK/dV pipeline: S^T and dP^T are issued per half of the streamed tile
// (queries [64h, 64h+64), N = 64), each half with its own "S ready" and "P
// ready" mbarriers, warpgroups 2h and 2h+1 being that half's, which write
// packed P^T/dS^T over the first 16 of the columns they read. Once half h's
// P/dS are in TMEM, the MMA warp issues that half's 4 k-steps of dV and dKhat
// and then S^T/dP^T of the same half of the next tile: the tensor core works on
// one half while the other half's softmax runs. tcgen05.mma operations issued
// by one thread execute in issue order, so the next tile's S/dP cannot
// overwrite P/dS before they are read. The softmax threads hold their columns
// as 16-lane TMEM fragments, so each needs the (lse, Dlt) of 8 columns only,
// loaded from the half stage as soon as it lands.
//
// dQ pipeline: S = Qhat Khat^T is TS-form (the owned Qhat rows are a
// TMEM-resident A operand, TMA'd into the owned-row slot and copied into TMEM
// by tcgen05.cp from the MMA warp, after which the slot takes the dO rows),
// dP = dO V^T SS-form (the owned dO rows in shared memory); packed dS has its
// own 64 columns. As soon as every softmax thread holds S(t) in registers,
// S(t+1) is issued, and dP(t+1) once they hold dP(t), so both run during the
// softmax of t; dQ(t) follows once dS(t) is in TMEM. K and V tiles come
// through separate rings (a V tile is released after its dP MMA, a K tile
// after its dQ MMA); the next item's Qhat copy, first S and first dP run during
// the current item's epilogue, whose staged dq tile the producer stores by TMA
// when it reloads the slot. The kernel also computes Dlt = rowsum(dO o O) of
// its rows and writes it for the dK/dV kernel, which is launched after it.
//
// An mbarrier poll right after tcgen05.commit stalls the issuing thread until
// earlier MMAs drain, so the TMA-arrival check for the next tile is done by the
// softmax warps before they signal the current one.
//
// Warps: 0-15 the four softmax warpgroups (thread = owned row = TMEM lane of
// its warp's quarter); 16 TMA producer; 17 TMEM allocator + MMA issuer.
#include <type_traits>

#include <algorithm>

#include "xt_common.cuh"
#include "xt_internal.h"
#include "xt_tc.cuh"

namespace xt {

namespace {

using namespace tc;

constexpr int kTile = 128;         // owned rows (MMA M) and streamed rows (MMA N of S/dP)
constexpr int kSoftmaxWGs = 4;     // softmax warpgroups; WG w takes columns [32w, 32w+32)
constexpr int kWgCols = kTile / kSoftmaxWGs;
constexpr int kWarpTma = 4 * kSoftmaxWGs, kWarpMma = kWarpTma + 1;
constexpr int kThreadsBwd = 32 * (kWarpMma + 1);
constexpr int kMaxStages = 8;

template <int D> struct BwdCfg {
    using A = Atoms<D>;
    static constexpr int kChunks = A::kPerRow;            // swizzle atoms (TMA boxes) per row
    static constexpr int kBox = A::box_bytes(kTile);      // one box of 128 rows
    static constexpr int kHalfBox = A::box_bytes(kTile / 2);
    static constexpr int kTileBytes = kChunks * kBox;     // 128 rows x D bf16
    static constexpr int kHalfBytes = kChunks * kHalfBox; // 64 rows x D bf16
    // dQ kernel: a ring of K tiles and a ring of V tiles (a V tile is released
    // after its dP MMA, a K tile only after its dQ MMA), plus the owned dO rows;
    // the dq epilogue's inputs go into freed slots after the last tile: the owned
    // q rows into the V ring, their RoPE (cos, sin) rows (two 64-row halves of
    // D/32 boxes of 16 pairs) into two K slots
    static constexpr int kKStages = (D == 128) ? 3 : 4;
    static constexpr int kVStages = (D == 128) ? 2 : 3;
    static_assert(kKStages >= 3, "the cos/sin rows take two K slots besides the last K tile");
    static constexpr int kSmemB = (kKStages + kVStages + 1) * kTileBytes + 1024;
    // dK/dV kernel: a ring of half tiles, each the Qhat and dO rows of one half
    // of a streamed query tile plus their 2 x 64 row statistics, so that a half
    // is reloaded as soon as its own MMAs are done
    static constexpr int kHStages = (D == 128) ? 4 : 8;
    static constexpr int kHStageBytes = 2 * kHalfBytes + 1024;
    static constexpr int kSmemA = 2 * kTileBytes + kHStages * kHStageBytes + 1024;
    // the dk epilogue takes three half stages after the last streamed half: the
    // k rows (a whole tile) and two 64-row halves of their (cos, sin) rows
    static_assert(kTileBytes <= kHStageBytes && (D / 32) * 64 * 128 <= kHStageBytes &&
                  kHStages >= 4, "dk epilogue inputs must fit the half stages");
};

// One piece of the dk epilogue's (cos, sin) rows: 64 rows x 16 pairs (128 bytes).
constexpr int kCsPieceBytes = 64 * 128;

struct BwdBarriers {
    uint64_t own_full;
    uint64_t st_full[kMaxStages], st_empty[kMaxStages];
    uint64_t v_full[kMaxStages], v_empty[kMaxStages];   // dQ kernel: the V ring
    uint64_t s_full[2], p_full[2];   // per half of the streamed tile (columns [64h, 64h+64))
    uint64_t acc_done;
    uint64_t drain;
    uint64_t x_full;                 // dQ kernel: the owned rows of dO are in shared memory
    uint64_t dp_full, dp_taken;      // dQ kernel: dP of a tile is in TMEM / in every softmax thread
    uint64_t do_free;                // dQ kernel: the item's dP MMAs and its Dlt have read the dO rows
    uint64_t q_read;                 // dQ kernel: the Qhat rows are copied from the dO slot into TMEM
    uint64_t stall;                  // never arrived on (xt_test_inject_stall)
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ void raise_error_b(unsigned int *err, volatile int *abort_flag) {
    atomicOr(err, ERR_TIMEOUT);
    *abort_flag = 1;
}

// split_p: one p_full barrier per half of the streamed tile (the dK/dV kernel);
// otherwise p_full[0] collects every softmax thread.
__device__ __forceinline__ void init_bwd_barriers(BwdBarriers &bars, uint32_t own_count,
                                                  uint32_t st_full_count, int stages,
                                                  bool split_p) {
    bars.abort_flag = 0;
    mbar_init(&bars.own_full, own_count);
    for (int s = 0; s < stages; ++s) {
        mbar_init(&bars.st_full[s], st_full_count);
        mbar_init(&bars.st_empty[s], 1);
        mbar_init(&bars.v_full[s], 1);
        mbar_init(&bars.v_empty[s], 1);
    }
    for (int h = 0; h < 2; ++h) {
        mbar_init(&bars.s_full[h], 1);
        mbar_init(&bars.p_full[h], split_p ? 32 * 4 * kSoftmaxWGs / 2    // the half's two warpgroups
                                           : 32 * 4 * kSoftmaxWGs);      // every softmax thread
    }
    mbar_init(&bars.acc_done, 1);
    mbar_init(&bars.drain, 1);
    mbar_init(&bars.x_full, 1);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.dp_taken, 32 * 4 * kSoftmaxWGs);
    mbar_init(&bars.do_free, 2);   // the last dP MMA's commit + the softmax threads after Dlt
    mbar_init(&bars.q_read, 1);
    mbar_init(&bars.stall, 1);
    fence_barrier_init();
}

// TMEM column of the packed-bf16 A operand (P or dS) for k-step kk of 16 rows:
// warpgroup w wrote rows [32w, 32w+32) packed two per column at columns
// [32w, 32w+16) (relative to the S or dP region).
__device__ __forceinline__ uint32_t packed_col(int kk) {
    return (uint32_t)((kk >> 1) * kWgCols + (kk & 1) * 8);
}

// Operand descriptor offsets (tc::Atoms: 128- or 64-byte swizzle rows, 8-row
// groups): a K-major operand advances 16 elements by +32 B inside an atom
// column, atom columns a box apart (128 rows, or 64 for a half tile); an
// MN-major B operand advances 16 rows by 16 atom rows, its N atoms a box apart
// (in the descriptor).
template <int D> constexpr uint64_t kmajor_off(int kk) { return (uint64_t)Atoms<D>::kstep(kk, kTile) >> 4; }
template <int D> constexpr uint64_t kmajor_off_half(int kk) { return (uint64_t)Atoms<D>::kstep(kk, kTile / 2) >> 4; }
template <int D> constexpr uint64_t mnmajor_off(int kk) { return (uint64_t)Atoms<D>::mnstep(kk) >> 4; }

// ---------------------------------------------------------------------------
// dKhat, dV
// ---------------------------------------------------------------------------
// Work split. Key tile j of a (unit, kv head) has group * (n_q - j) (head,
// query tile) iterations; when that is more than `chunk` (chunk > 0), the
// iterations are cut into chunks of `chunk`, one CTA each, whose fp32 dKhat/dV
// partials go to `part` and are summed in chunk order by k_dkdv_reduce (so the
// group sum stays in a fixed order). Work items of a (unit, kv head) are
// numbered key tile by key tile, chunks in order: nw of them.
__host__ __device__ inline int dkdv_chunks(int iters, int chunk) {
    return (chunk > 0 && iters > chunk) ? (iters + chunk - 1) / chunk : 1;
}

// Scratch of the row epilogue (finish_rows): per-warpgroup parts of each row's
// norm dot product, per-(warpgroup, row quarter) column sums of the dgamma
// terms, and the rows' rstd and gamma.
struct EpiScratch {
    float dot[kSoftmaxWGs][kTile];
    float g[kSoftmaxWGs][4][32];
    float rstd[kTile];               // rstd_q of the owned rows (0 past the end)
    float gamma[kTile];              // gamma_q (D <= kTile)
};

// The 512 softmax threads (warps 0-15) only.
__device__ __forceinline__ void softmax_bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * 4 * kSoftmaxWGs) : "memory");
}

// Named barrier 1 for the 512 softmax threads with an OR over their flags: every
// thread gets the same answer (the persistent dQ kernel's softmax threads
// decide together whether to stop, so that no named barrier is left waiting).
__device__ __forceinline__ bool softmax_bar_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n"
        " bar.red.or.pred p, 1, %2, q;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r) : "r"((uint32_t)v), "n"(32 * 4 * kSoftmaxWGs) : "memory");
    return r != 0;
}

// Work item w of the dQ kernel: query tile i of (unit, head) bh, longest first
// (i descending, heads and units fastest). T: key tiles at or before the rows
// (0 for a packed sample shorter than this tile).
struct DqItem {
    int i, bh, h, g, T;
    SeqSpan sp;
};

__device__ __forceinline__ DqItem dq_item(int w, int BH, int n_qt, int H, int G,
                                          const SeqRows &sr) {
    DqItem it;
    it.i = n_qt - 1 - w / BH;
    it.bh = w - (w / BH) * BH;
    const int unit = it.bh / H;
    it.h = it.bh - unit * H;
    it.g = it.h / (H / G);
    it.sp = seq_span(sr, unit);
    it.T = it.i * kTile < it.sp.len ? it.i + 1 : 0;
    return it;
}

// Element e of bf16 values packed two per word (the lower index in the low half).
template <int N>
__device__ __forceinline__ float bf16_lo_or_hi(const uint32_t (&w)[N], int e) {
    const uint32_t v = w[e >> 1];
    return __uint_as_float((e & 1) ? (v & 0xffff0000u) : (v << 16));
}

// Transposing butterfly: every lane holds V values v[c] (c = column, V = 8, 16
// or 32); after log2 V exchange steps lane l holds the sum over its group of V
// lanes of column l % V (each step a lane keeps half of its columns, sends the
// other half to the partner lane and adds the partner's copy of the kept half),
// and the 32 / V groups are then added by xor shuffles: every lane l ends with
// the sum over the warp of column l % V. Fixed association.
template <int V>
__device__ __forceinline__ float transpose_sum(float (&v)[V], int lane) {
#pragma unroll
    for (int n = V / 2; n >= 1; n >>= 1) {
        const bool up = (lane & n) != 0;
#pragma unroll
        for (int e = 0; e < n; ++e) {
            const float send = up ? v[e] : v[e + n];
            const float keep = up ? v[e + n] : v[e];
            v[e] = keep + __shfl_xor_sync(0xffffffffu, send, n);
        }
    }
    float s = v[0];
#pragma unroll
    for (int m = V; m < 32; m <<= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
    return s;
}

// N consecutive TMEM columns (N = 4, 8 or 16) from each of two addresses, then
// one wait (32x32b shape: thread i of the warp reads lane base + i).
template <int N>
__device__ __forceinline__ void tmem_ld_pair_n(uint32_t ta, uint32_t (&a)[N], uint32_t tb,
                                               uint32_t (&b)[N]) {
    if constexpr (N == 16) {
        tmem_ld16_pair_sync(ta, a, tb, b);
    } else if constexpr (N == 8) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%16];\n"
            "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%17];\n"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]),
              "=r"(a[7]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]),
              "=r"(b[6]), "=r"(b[7])
            : "r"(ta), "r"(tb)
            : "memory");
    } else {
        static_assert(N == 4, "4, 8 or 16 columns");
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%8];\n"
            "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%4, %5, %6, %7}, [%9];\n"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]),
              "=r"(b[3])
            : "r"(ta), "r"(tb)
            : "memory");
    }
}

// The epilogue that turns the gradient of 128 normed-and-rotated rows into the
// gradient of the raw rows (Mint project report 5.4.4: RoPE backward, the
// rotation by the negative angle; 5.5.2: RMSNorm backward with the shared
// gamma) and the CTA's dgamma partial, for the 512 softmax threads (thread =
// row r = TMEM lane). Inputs: the accumulator in TMEM columns [0, D) at `tacc`
// (this warp's lanes; the gradient times sqrt(D)), the raw rows in shared
// memory as D / kCols TMA boxes of 128 rows (tc::Atoms<D> layout), this
// thread's row of the (cos, sin) pieces at `cs_row` (piece c holds pairs
// [16 c, 16 c + 16): a 128-byte row of a 128-byte-swizzled fp32 box at
// cs_row + c * kCsPieceBytes, unswizzled start), and rstd and gamma in escr
// (written before the call by other threads: the first named barrier orders
// them). Warpgroup wg takes the P = D/8 pairs [P wg, P wg + P) (columns P wg..
// and D/2 + P wg..) of its row; the row's dot product is summed over the four
// warpgroups in order. The dgamma terms are summed over the warp's rows by a
// transposing butterfly, then over the four row quarters in order, into
// part[0, D). Every softmax thread must call this (it holds three named
// barriers); with ok false it only writes a zero partial.
template <int D>
__device__ __forceinline__ void finish_rows(bool ok, int wg, int quarter, int lane,
                                            uint32_t tacc, const uint8_t *sX,
                                            const uint8_t *cs_row, bool row_ok,
                                            EpiScratch &escr, bf16 *dst_row, float *part,
                                            uint8_t *stage) {
    using A = Atoms<D>;
    constexpr int kHalf = D / 2;
    constexpr int kP = D / 8;             // pairs per warpgroup (all four take part)
    constexpr int kXW = kP / 2;           // 32-bit words of x (and of dq) per row half
    const int i0 = wg * kP;
    const int r = quarter * 32 + lane;
    // the swizzled place of column `col` of this thread's row in a tile
    auto xoff = [&](int col) -> uint32_t {
        return swizzled<A::kRowBytes>((uint32_t)((col / A::kCols) * A::box_bytes(kTile) +
                                                 r * A::kRowBytes + (col % A::kCols) * 2));
    };
    softmax_bar_sync();   // the stashed gamma and rstd are visible from here on
    uint32_t xw[2 * kXW]; // the row's x: kXW words of the low pairs' columns, then kXW of the high
    float dy[2 * kP];     // dy[e] (e < kP): column i0 + e; dy[kP + e]: column D/2 + i0 + e
#pragma unroll
    for (int e = 0; e < 2 * kP; ++e) dy[e] = 0.f;
#pragma unroll
    for (int e = 0; e < 2 * kXW; ++e) xw[e] = 0u;
    if (ok) {
        tc_fence_after();
        // x: kP columns of each half, in 16-byte chunks of 8 (8 bytes when kP = 4)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int cb = hh * kHalf + i0;
            if constexpr (kP >= 8) {
#pragma unroll
                for (int c8 = 0; c8 < kP / 8; ++c8) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(sX + xoff(cb + 8 * c8));
                    xw[hh * kXW + 4 * c8] = v.x; xw[hh * kXW + 4 * c8 + 1] = v.y;
                    xw[hh * kXW + 4 * c8 + 2] = v.z; xw[hh * kXW + 4 * c8 + 3] = v.w;
                }
            } else {
                const uint2 v = *reinterpret_cast<const uint2 *>(sX + xoff(cb));
                xw[hh * kXW] = v.x; xw[hh * kXW + 1] = v.y;
            }
        }
        uint32_t a[kP], b[kP];
        tmem_ld_pair_n<kP>(tacc + i0, a, tacc + kHalf + i0, b);
        const float scale = rsqrtf((float)D);
        // this warpgroup's pairs lie in piece i0 / 16 (kP divides 16), from pair i0 % 16
        const uint8_t *cs_p = cs_row + (i0 >> 4) * kCsPieceBytes;
        const int j0 = kP == 16 ? 0 : (i0 & 15);
        float dotp = 0.f;
#pragma unroll
        for (int e = 0; e < kP; e += 2) {
            // (cos, sin) of pairs i0 + e, i0 + e + 1: 16-byte chunk (j0 + e) / 2 of the
            // swizzled row
            const float4 c2 = *reinterpret_cast<const float4 *>(
                cs_p + ((((j0 + e) >> 1) ^ (r & 7)) << 4));
            const float cv[2] = {c2.x, c2.z}, sv[2] = {c2.y, c2.w};
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                const float gl = __uint_as_float(a[e + x]) * scale;
                const float gh = __uint_as_float(b[e + x]) * scale;
                // rotation by the negative angle
                const float dyl = gl * cv[x] + gh * sv[x];
                const float dyh = gh * cv[x] - gl * sv[x];
                dy[e + x] = dyl;
                dy[kP + e + x] = dyh;
                dotp = fmaf(escr.gamma[i0 + e + x] * dyl, bf16_lo_or_hi(xw, e + x), dotp);
                dotp = fmaf(escr.gamma[kHalf + i0 + e + x] * dyh,
                            bf16_lo_or_hi(xw, 2 * kXW + e + x), dotp);
            }
        }
        escr.dot[wg][r] = dotp;
    }
    softmax_bar_sync();
    if (ok) {
        const float dot = ((escr.dot[0][r] + escr.dot[1][r]) + escr.dot[2][r]) + escr.dot[3][r];
        const float rr = escr.rstd[r];
        const float corr = dot * rr * rr * rr * (1.0f / (float)D);
        uint32_t ow[2 * kXW];
#pragma unroll
        for (int e = 0; e < kP; e += 2) {
            float ol[2], oh[2];
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                const float xl = bf16_lo_or_hi(xw, e + x);
                const float xh = bf16_lo_or_hi(xw, 2 * kXW + e + x);
                ol[x] = escr.gamma[i0 + e + x] * dy[e + x] * rr - xl * corr;
                oh[x] = escr.gamma[kHalf + i0 + e + x] * dy[kP + e + x] * rr - xh * corr;
                // the dgamma terms replace dy
                dy[e + x] = dy[e + x] * xl * rr;
                dy[kP + e + x] = dy[kP + e + x] * xh * rr;
            }
            ow[e / 2] = pack_bf16x2(ol[0], ol[1]);
            ow[kXW + e / 2] = pack_bf16x2(oh[0], oh[1]);
        }
        if (stage != nullptr) {
            // in place of the x pieces this thread read (the caller stores the tile by TMA)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int cb = hh * kHalf + i0;
                if constexpr (kP >= 8) {
#pragma unroll
                    for (int c8 = 0; c8 < kP / 8; ++c8)
                        *reinterpret_cast<uint4 *>(stage + xoff(cb + 8 * c8)) =
                            make_uint4(ow[hh * kXW + 4 * c8], ow[hh * kXW + 4 * c8 + 1],
                                       ow[hh * kXW + 4 * c8 + 2], ow[hh * kXW + 4 * c8 + 3]);
                } else {
                    *reinterpret_cast<uint2 *>(stage + xoff(cb)) =
                        make_uint2(ow[hh * kXW], ow[hh * kXW + 1]);
                }
            }
            fence_proxy_async_smem();
        } else if (row_ok) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                bf16 *dst = dst_row + hh * kHalf + i0;
                if constexpr (kP >= 8) {
#pragma unroll
                    for (int c8 = 0; c8 < kP / 8; ++c8)
                        reinterpret_cast<uint4 *>(dst)[c8] =
                            make_uint4(ow[hh * kXW + 4 * c8], ow[hh * kXW + 4 * c8 + 1],
                                       ow[hh * kXW + 4 * c8 + 2], ow[hh * kXW + 4 * c8 + 3]);
                } else {
                    *reinterpret_cast<uint2 *>(dst) = make_uint2(ow[hh * kXW], ow[hh * kXW + 1]);
                }
            }
        }
        // column sums over the warp's 32 rows: lane l ends with column l % 2P of dy
        const float g = transpose_sum<2 * kP>(dy, lane);
        if (lane < 2 * kP) escr.g[wg][quarter][lane] = g;
    }
    softmax_bar_sync();
    if (threadIdx.x < D) {
        // column d of the partial: the four row quarters of its warpgroup, in order
        const int d = threadIdx.x;
        const int pd = d < kHalf ? d : d - kHalf;
        const int w = pd / kP;
        const int l = (d < kHalf ? 0 : kP) + pd % kP;
        float sum = 0.f;
        if (ok) {
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) sum += escr.g[w][qq][l];
        }
        part[d] = sum;
    }
}

// finish_rows as a separate function: the dQ kernel calls it this way, which
// keeps its main loop free of register spills (its live state there is at
// the 96-register limit of 576-thread blocks).
template <int D>
__device__ __noinline__ void finish_rows_call(bool ok, int wg, int quarter, int lane,
                                              uint32_t tacc, const uint8_t *sX,
                                              const uint8_t *cs_row, bool row_ok,
                                              EpiScratch &escr, bf16 *dst_row, float *part,
                                              uint8_t *stage) {
    finish_rows<D>(ok, wg, quarter, lane, tacc, sX, cs_row, row_ok, escr, dst_row, part, stage);
}

// The dK/dV kernel's accumulator stores (a separate function, so that its
// softmax loop keeps its registers): dV (bf16) and, unless the kernel
// finishes dk itself, dKhat (fp32, scaled by 1/sqrt(D)) of this thread's key
// row, or both as fp32 chunk partials when prow is set. 32-column chunks: dV
// chunks 0..D/32-1, then dKhat; warpgroup w writes chunks w, w + 4, ...
template <int D, bool kSplit>
__device__ __noinline__ void store_dkdv_acc(int wg, uint32_t tacc, bool row_ok, bf16 *dvrow,
                                            float *dkrow, float *prow) {
    constexpr bool kFuse = !kSplit;
    const float scale = rsqrtf((float)D);
#pragma unroll
    for (int cc = wg; cc < (kFuse ? 1 : 2) * (D / 32); cc += kSoftmaxWGs) {
        const bool isv = cc < D / 32;
        const int c = isv ? cc : cc - D / 32;
        uint32_t a[32];
        tmem_ld32_sync(tacc + (isv ? 256 : 384) + 32 * c, a);
        if (row_ok && prow != nullptr) {
            const float sc = isv ? 1.f : scale;
            float *dst = prow + (isv ? 0 : (size_t)kTile * D) + 32 * c;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
                *reinterpret_cast<float4 *>(dst + 4 * q4) =
                    make_float4(__uint_as_float(a[q4 * 4 + 0]) * sc,
                                __uint_as_float(a[q4 * 4 + 1]) * sc,
                                __uint_as_float(a[q4 * 4 + 2]) * sc,
                                __uint_as_float(a[q4 * 4 + 3]) * sc);
        } else if (row_ok) {
            if (isv) {
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) {
                    uint4 v4;
                    v4.x = pack_bf16x2(__uint_as_float(a[q8 * 8 + 0]), __uint_as_float(a[q8 * 8 + 1]));
                    v4.y = pack_bf16x2(__uint_as_float(a[q8 * 8 + 2]), __uint_as_float(a[q8 * 8 + 3]));
                    v4.z = pack_bf16x2(__uint_as_float(a[q8 * 8 + 4]), __uint_as_float(a[q8 * 8 + 5]));
                    v4.w = pack_bf16x2(__uint_as_float(a[q8 * 8 + 6]), __uint_as_float(a[q8 * 8 + 7]));
                    *reinterpret_cast<uint4 *>(dvrow + 32 * c + 8 * q8) = v4;
                }
            } else {
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

// finish_rows for the dK/dV kernel: its own out-of-line copy (sharing one
// with the dQ kernel changes the dQ kernel's register allocation).
template <int D>
__device__ __noinline__ void finish_rows_dk(bool ok, int wg, int quarter, int lane,
                                            uint32_t tacc, const uint8_t *sX,
                                            const uint8_t *cs_row, bool row_ok,
                                            EpiScratch &escr, bf16 *dst_row, float *part) {
    finish_rows<D>(ok, wg, quarter, lane, tacc, sX, cs_row, row_ok, escr, dst_row, part, nullptr);
}

// kSplit: the chunked work split is on (a separate instantiation keeps the
// unsplit kernel free of its index arithmetic). The unsplit kernel finishes dk
// itself (finish_rows on dKhat; one dgamma_k partial per CTA at part_k); the
// split one writes fp32 dKhat (or chunk partials) for the reduce and the k-row
// epilogue.
template <int D, bool kSplit>
__global__ void __launch_bounds__(kThreadsBwd, 1)
k_bwd_dkdv_tc(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
              const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
              const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_cs,
              const float *__restrict__ lse, const float *__restrict__ dlt,
              float *__restrict__ dkhat, bf16 *__restrict__ dv, float *__restrict__ part,
              const float *__restrict__ gamma_k, const float *__restrict__ rstd_k,
              bf16 *__restrict__ dk, float *__restrict__ part_k, const SeqRows sr, int H, int G,
              int n_kvt, int chunk, int nw, unsigned int *err, int stall) {
    using C = BwdCfg<D>;
    constexpr int HS = C::kHStages;
    constexpr bool kFuse = !kSplit;
    extern __shared__ uint8_t smem_raw[];
    __shared__ BwdBarriers bars;
    __shared__ EpiScratch escr;
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sK = smem;
    uint8_t *sV = smem + C::kTileBytes;
    uint8_t *sStage = smem + 2 * C::kTileBytes;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BG = gridDim.x / nw;
    const int witem = (int)(blockIdx.x / BG);      // work item, longest first
    const int bg = blockIdx.x % BG;
    const int unit = bg / G, g = bg - unit * G, group = H / G;
    int j = witem, cidx = 0, nc = 1;               // key tile, chunk of it, its chunk count
    if constexpr (kSplit) {
        j = 0;
        cidx = witem;
        for (;;) {
            nc = dkdv_chunks(group * (n_kvt - j), chunk);
            if (cidx < nc || j + 1 >= n_kvt) break;
            cidx -= nc;
            ++j;
        }
    }
    const SeqSpan sp = seq_span(sr, unit);
    const int S = sp.len;                           // rows of this unit
    const int n_q = (S + kTile - 1) / kTile;
    float *pk = kFuse ? part_k + ((size_t)bg * nw + witem) * D : nullptr;   // dgamma_k partial
    if (j >= n_q || cidx >= nc) {                   // a packed sample shorter than this tile
        if constexpr (kFuse)
            for (int d = threadIdx.x; d < D; d += blockDim.x) pk[d] = 0.f;
        return;
    }
    const int nU = n_q - j;                         // query tiles at/after the keys, per head
    const int t0 = kSplit && nc > 1 ? cidx * chunk : 0;   // this CTA's iterations [t0, t0 + T)
    const int T = kSplit && nc > 1 ? min(chunk, group * nU - t0) : group * nU;
    volatile int *abort_flag = &bars.abort_flag;

    if (threadIdx.x == 0) init_bwd_barriers(bars, 1, 2, HS, true);
    if (warp == kWarpMma) {
        tmem_alloc(&bars.tmem_base, 512);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    pdl_enter();
    const uint32_t tmem = bars.tmem_base;

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&map_k);
            tma_prefetch_desc(&map_v);
            tma_prefetch_desc(&map_q);
            tma_prefetch_desc(&map_do);
            mbar_expect_tx(&bars.own_full, 2 * C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_3d(sK + c * C::kBox, &map_k, &bars.own_full, c * C::A::kCols,
                            sp.start + j * kTile, sp.plane * G + g);
                tma_load_4d(sV + c * C::kBox, &map_v, &bars.own_full, c * C::A::kCols, g,
                            sp.start + j * kTile, sp.plane);
            }
        }
        // half tile x = 2 t + hf: rows [64 hf, 64 hf + 64) of streamed tile t
        int issued = 0;
        for (int x = 0; x < 2 * T; ++x) {
            const int hs = x % HS, t = t0 + (x >> 1), hf = x & 1;
            bool ok = true;
            if (x >= HS && lane == 0)
                ok = mbar_wait(&bars.st_empty[hs], ((x / HS) - 1) & 1, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0 && !*abort_flag) raise_error_b(err, abort_flag);
                break;
            }
            const int r = t / nU, u = j + (t - r * nU);
            const int h = g * group + r;
            const int q0 = u * kTile + 64 * hf;
            uint8_t *base = sStage + hs * C::kHStageBytes;
            if (lane == 0) {
                mbar_expect_tx(&bars.st_full[hs], 2 * C::kHalfBytes);
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_3d(base + c * C::kHalfBox, &map_q, &bars.st_full[hs],
                                c * C::A::kCols, sp.start + q0, sp.plane * H + h);
                    tma_load_4d(base + C::kHalfBytes + c * C::kHalfBox, &map_do,
                                &bars.st_full[hs], c * C::A::kCols, h, sp.start + q0, sp.plane);
                }
            }
            // the half's row statistics (lse at [0,64), Dlt at [64,128)) by 4-byte
            // asynchronous copies that the stage's barrier waits for, so the producer
            // never stalls on a global load; rows past the end read as 0
            float *sl = reinterpret_cast<float *>(base + 2 * C::kHalfBytes);
            const size_t row0 = ((size_t)sp.plane * H + h) * sr.S + sp.start;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                // column kq of the half: lse at 4 (kq / 2) + kq % 2, Dlt two words on
                // (one 16-byte word per column pair, the softmax's load unit)
                const int kq = lane + 32 * e, q = q0 + kq;
                const int o = 4 * (kq >> 1) + (kq & 1);
                if (q < S) {
                    cp_async4(sl + o, lse + row0 + q);
                    cp_async4(sl + o + 2, dlt + row0 + q);
                } else {
                    sl[o] = 0.f;
                    sl[o + 2] = 0.f;
                }
            }
            // each lane's copies become one pending arrival of the stage barrier
            // (registered before lane 0's arrival below, hence the __syncwarp)
            cp_async_mbar_arrive(&bars.st_full[hs]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.st_full[hs]);
            issued = x + 1;
        }
        if constexpr (kFuse) {
            // the dk epilogue's inputs, in the next three half stages as they free up:
            // the owned k rows (one 128-row tile), then their (cos, sin) rows in two
            // 64-row halves (D/32 boxes of 64 rows x 16 pairs each)
            for (int e = 0; issued == 2 * T + e && e < 3; ++e) {
                const int x = 2 * T + e, hs = x % HS;
                bool ok = true;
                if (x >= HS && lane == 0)
                    ok = mbar_wait(&bars.st_empty[hs], ((x / HS) - 1) & 1, abort_flag);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    if (lane == 0 && !*abort_flag) raise_error_b(err, abort_flag);
                    break;
                }
                uint8_t *base = sStage + hs * C::kHStageBytes;
                if (lane == 0) {
                    if (e == 0) {
                        mbar_expect_tx(&bars.st_full[hs], C::kTileBytes);
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_4d(base + c * C::kBox, &map_x, &bars.st_full[hs],
                                        c * C::A::kCols, g, sp.start + j * kTile, sp.plane);
                    } else {
                        mbar_expect_tx(&bars.st_full[hs], (D / 32) * kCsPieceBytes);
                        for (int c = 0; c < D / 32; ++c)
                            tma_load_2d(base + c * kCsPieceBytes, &map_cs, &bars.st_full[hs],
                                        32 * c, sp.start + j * kTile + 64 * (e - 1));
                    }
                    mbar_arrive(&bars.st_full[hs]);
                }
                issued = x + 1;
            }
        }
        if (lane == 0) {
            // drain: every copy issued by this CTA lands before it exits
            mbar_wait(&bars.own_full, 0, nullptr);
            for (int x = max(0, issued - HS); x < issued; ++x)
                mbar_wait(&bars.st_full[x % HS], (x / HS) & 1, nullptr);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        {
            // the whole warp runs this loop; one elected lane issues each MMA / commit
            const uint32_t idesc_s = idesc_bf16_f32(kTile, kTile / 2, 0, 0);
            const uint32_t idesc_acc = idesc_bf16_f32(kTile, D, 0, 1);
            using A = typename C::A;
            const uint64_t dK = smem_desc(smem_u32(sK), 16, A::kSBO, A::kMode);
            const uint64_t dV = smem_desc(smem_u32(sV), 16, A::kSBO, A::kMode);
            const uint64_t dQk0 = smem_desc(smem_u32(sStage), 16, A::kSBO, A::kMode);
            const uint64_t dDOk0 = smem_desc(smem_u32(sStage + C::kHalfBytes), 16, A::kSBO, A::kMode);
            const uint64_t dQm0 = smem_desc(smem_u32(sStage), C::kHalfBox, A::kSBO, A::kMode);
            const uint64_t dDOm0 = smem_desc(smem_u32(sStage + C::kHalfBytes), C::kHalfBox, A::kSBO,
                                             A::kMode);
            constexpr uint64_t kStep = (uint64_t)C::kHStageBytes >> 4;
            // S^T = Khat Qhat^T and dP^T = V dO^T for the queries [64h, 64h+64) of
            // tile t, from half stage (2t + h) % HS
            auto issue_sp = [&](int t, int h) {
                const uint64_t so = (uint64_t)((2 * t + h) % HS) * kStep;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss_w(tmem + 64 * h, dK + kmajor_off<D>(kk), dQk0 + so + kmajor_off_half<D>(kk),
                           idesc_s, kk > 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss_w(tmem + 128 + 64 * h, dV + kmajor_off<D>(kk),
                           dDOk0 + so + kmajor_off_half<D>(kk), idesc_s, kk > 0);
                mma_commit_w(&bars.s_full[h]);
            };
            bool ok = !stall ||
                      __all_sync(0xffffffffu, mbar_wait_for(&bars.stall, 0, abort_flag, kStallLimitNs));
            ok = ok && mbar_wait_w(&bars.own_full, 0, abort_flag) &&
                 mbar_wait_w(&bars.st_full[0], 0, abort_flag) &&
                 mbar_wait_w(&bars.st_full[1], 0, abort_flag);   // both halves of tile 0
            if (ok) {
                tc_fence_after();
                issue_sp(0, 0);
                issue_sp(0, 1);
            }
            // Per half h: once its P/dS are in TMEM, accumulate its 4 k-steps of
            // dV += P^T dO and dKhat += dS^T Qhat, then start S/dP of the same half
            // of the next tile (in-order execution keeps them behind those reads).
            for (int t = 0; ok && t < T; ++t) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int hs = (2 * t + h) % HS;
                    const uint64_t so = (uint64_t)hs * kStep;
                    if (!(ok = mbar_wait_w(&bars.p_full[h], t & 1, abort_flag))) break;
                    tc_fence_after();
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {   // dV += P^T dO
                        const int kk = 4 * h + k4;
                        mma_ts_w(tmem + 256, tmem + packed_col(kk), dDOm0 + so + mnmajor_off<D>(k4),
                               idesc_acc, (t > 0 || kk > 0) ? 1u : 0u);
                    }
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {   // dKhat += dS^T Qhat
                        const int kk = 4 * h + k4;
                        mma_ts_w(tmem + 384, tmem + 128 + packed_col(kk), dQm0 + so + mnmajor_off<D>(k4),
                               idesc_acc, (t > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit_w(&bars.st_empty[hs]);       // this half stage may be reloaded
                    if (t + 1 < T) issue_sp(t + 1, h);   // operands checked by the softmax warps
                }
            }
            if (ok) mma_commit_w(&bars.acc_done);
            else if (lane == 0 && !*abort_flag) raise_error_b(err, abort_flag);
            mma_commit_w(&bars.drain);
            mbar_wait_w(&bars.drain, 0, nullptr);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int wg = warp >> 2, quarter = warp & 3;
        const int r = quarter * 32 + lane;              // owned key row = TMEM lane
        const int kp = j * kTile + r;                   // key position
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float sl2 = kLog2e * rsqrtf((float)D);
        if (kFuse && wg == kSoftmaxWGs - 1) {
            // for the dk epilogue (read after its first named barrier)
            escr.rstd[r] = kp < S ? rstd_k[((size_t)sp.plane * sr.S + sp.start + kp) * G + g] : 0.f;
            if (r < D) escr.gamma[r] = gamma_k[r];
        }
        bool ok = true;
        const int hf = wg >> 1;                         // this warpgroup's half of the tile
        for (int t = 0; t < T; ++t) {
            const int x = 2 * t + hf, hs = x % HS;
            // the half stage first: its row statistics are loaded into registers while
            // S^T/dP^T are still being computed (their shared-memory loads would
            // otherwise queue behind the tensor core's operand reads)
            ok = __all_sync(0xffffffffu, mbar_wait(&bars.st_full[hs], (x / HS) & 1, abort_flag));
            if (!ok) break;
            float4 st4[4];
            {
                // (lse, lse, Dlt, Dlt) of the column pairs 8 k + 2 (lane % 4) of this
                // warpgroup's 32 columns
                const float4 *sl4 = reinterpret_cast<const float4 *>(
                    sStage + hs * C::kHStageBytes + 2 * C::kHalfBytes);
#pragma unroll
                for (int k = 0; k < 4; ++k) st4[k] = sl4[16 * (wg & 1) + 4 * k + (lane & 3)];
            }
            ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full[hf], t & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            const int u = j + ((t0 + t) % nU);
            const int c0 = wg * kWgCols;                // this warpgroup's columns
            const int q0 = u * kTile + c0;
            const uint32_t tS = tmem + lane_off + c0;         // S^T columns
            const uint32_t tP = tmem + lane_off + 128 + c0;   // dP^T columns
            // no masking when every query of these columns is at/after every owned key and < S
            const bool interior = (q0 >= j * kTile + kTile - 1) && (q0 + kWgCols <= S);
            // 16-lane TMEM shapes (xt_tc.cuh): this thread holds rows
            // 16 L + lane/4 + 8 jh of its warp's 32 and the column pairs 8 k + 2 (lane % 4)
            // of the warpgroup's 32, so it needs the statistics of 8 columns only (st4).
            uint32_t pp[kWgCols / 2], dd[kWgCols / 2];
            {
                uint32_t sv[32], dpv[32];
                tmem_ld16x256b_x4_rows32_pair_sync(tS, sv, tP, dpv);
                const int cp = 2 * (lane & 3);
                // masked columns (the diagonal tile, the ragged end) take the select;
                // interior tiles (all but about one in n_q) run without it
                auto body = [&](auto masked) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 nl = fmul2(make_float2(st4[k].x, st4[k].y),
                                                make_float2(-kLog2e, -kLog2e));
                        const float2 ndl = make_float2(-st4[k].z, -st4[k].w);
#pragma unroll
                        for (int L = 0; L < 2; ++L) {
#pragma unroll
                            for (int jh = 0; jh < 2; ++jh) {
                                // column pairs through the packed fp32 pipe (f32x2 FMA / add / mul)
                                const int e = 16 * L + 4 * k + 2 * jh;
                                const float2 a = ffma2(make_float2(__uint_as_float(sv[e]),
                                                                   __uint_as_float(sv[e + 1])),
                                                       make_float2(sl2, sl2), nl);
                                float2 p = make_float2(fast_exp2(a.x), fast_exp2(a.y));
                                if constexpr (decltype(masked)::value) {
                                    const int q = q0 + 8 * k + cp;
                                    const int kr = j * kTile + quarter * 32 + 16 * L + (lane >> 2) + 8 * jh;
                                    if (!(q >= kr && q < S)) p.x = 0.f;
                                    if (!(q + 1 >= kr && q + 1 < S)) p.y = 0.f;
                                }
                                const float2 ds = fmul2(p, fadd2(make_float2(__uint_as_float(dpv[e]),
                                                                             __uint_as_float(dpv[e + 1])),
                                                                 ndl));
                                pp[8 * L + 2 * k + jh] = pack_bf16x2(p.x, p.y);
                                dd[8 * L + 2 * k + jh] = pack_bf16x2(ds.x, ds.y);
                            }
                        }
                    }
                };
                if (interior) body(std::false_type{});
                else body(std::true_type{});
            }
            if (t + 1 < T) {   // operands of this half of tile t+1, issued right behind its dV/dK
                ok = __all_sync(0xffffffffu, mbar_wait(&bars.st_full[(x + 2) % HS],
                                                       ((x + 2) / HS) & 1, abort_flag));
                if (!ok) break;
            }
            tmem_st16x128b_x4_rows32_pair_sync(tS, pp, tP, dd);
            tc_fence_before();
            mbar_arrive(&bars.p_full[wg >> 1]);
        }
        if (ok) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars.acc_done, 0, abort_flag));
            if (ok) {
                tc_fence_after();
                store_dkdv_acc<D, kSplit>(
                    wg, tmem + lane_off, kp < S,
                    dv + (((size_t)sp.plane * sr.S + sp.start + kp) * G + g) * D,
                    dkhat + (((size_t)sp.plane * G + g) * sr.S + sp.start + kp) * D,
                    kSplit && nc > 1
                        ? part + ((size_t)bg * nw + witem) * 2 * kTile * D + (size_t)r * D
                        : nullptr);
            }
        }
        if constexpr (kFuse) {
            // dk and the CTA's dgamma_k partial from dKhat in TMEM, with the k rows
            // and their (cos, sin) rows that the producer loaded after the last half
            const int x0 = 2 * T;
            if (ok) ok = __all_sync(0xffffffffu,
                                    mbar_wait(&bars.st_full[x0 % HS], (x0 / HS) & 1, abort_flag) &&
                                    mbar_wait(&bars.st_full[(x0 + 1) % HS], ((x0 + 1) / HS) & 1,
                                              abort_flag) &&
                                    mbar_wait(&bars.st_full[(x0 + 2) % HS], ((x0 + 2) / HS) & 1,
                                              abort_flag));
            const uint8_t *sX = sStage + (x0 % HS) * C::kHStageBytes;
            const uint8_t *cs_row = sStage + ((x0 + 1 + (r >> 6)) % HS) * C::kHStageBytes +
                                    (r & 63) * 128;
            finish_rows_dk<D>(ok, wg, quarter, lane, tmem + 384 + lane_off, sX, cs_row, kp < S,
                              escr, dk + (((size_t)sp.plane * sr.S + sp.start + kp) * G + g) * D,
                              pk);
        }
        if (!ok && !*abort_flag) raise_error_b(err, abort_flag);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Work item w of the dK/dV kernel: 128 key rows (key tile j) of (unit, kv head)
// bg, or with the chunked split one chunk cidx of that tile's iterations; items
// run longest first (key tile ascending, units and kv heads fastest). T: the
// item's (head, query tile) iterations starting at t0 (0: nothing to do, a
// packed sample shorter than the tile). witem: the item's index within its bg.
struct DkdvItem {
    int witem, bg, g, j, T, t0, nU;
    bool split;   // a chunk of a split tile (its partials go to the chunk reduce)
    SeqSpan sp;
};

template <bool kSplit>
__device__ __forceinline__ DkdvItem dkdv_item(int w, int BG, int H, int G, int n_kvt, int chunk,
                                              const SeqRows &sr) {
    DkdvItem it;
    it.witem = w / BG;
    it.bg = w - it.witem * BG;
    const int unit = it.bg / G, group = H / G;
    it.g = it.bg - unit * G;
    int j = it.witem, cidx = 0, nc = 1;
    if constexpr (kSplit) {
        j = 0;
        cidx = it.witem;
        for (;;) {
            nc = dkdv_chunks(group * (n_kvt - j), chunk);
            if (cidx < nc || j + 1 >= n_kvt) break;
            cidx -= nc;
            ++j;
        }
    }
    it.j = j;
    it.sp = seq_span(sr, unit);
    const int n_q = (it.sp.len + kTile - 1) / kTile;
    it.split = kSplit && nc > 1;
    if (j >= n_q || cidx >= nc) {
        it.T = 0; it.t0 = 0; it.nU = 0;
        return it;
    }
    it.nU = n_q - j;                                // query tiles at/after the keys, per head
    it.t0 = it.split ? cidx * chunk : 0;            // this item's iterations [t0, t0 + T)
    it.T = it.split ? min(chunk, group * it.nU - it.t0) : group * it.nU;
    return it;
}

// The persistent form of k_bwd_dkdv_tc (used at D <= 64, where items are short
// and a CTA's set-up, pipeline fill and epilogue are a large share of each): a
// grid of one CTA per SM walks the items in snake order (snake_item), barrier
// phases and half-stage uses counted across items, the next item's own K/V
// tiles loaded once the last S^T/dP^T MMA of the current one has read the old
// ones. Same arguments as k_bwd_dkdv_tc plus the item count.
template <int D, bool kSplit>
__global__ void __launch_bounds__(kThreadsBwd, 1)
k_bwd_dkdv_tc_p(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
              const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
              const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_cs,
              const float *__restrict__ lse, const float *__restrict__ dlt,
              float *__restrict__ dkhat, bf16 *__restrict__ dv, float *__restrict__ part,
              const float *__restrict__ gamma_k, const float *__restrict__ rstd_k,
              bf16 *__restrict__ dk, float *__restrict__ part_k, const SeqRows sr, int H, int G,
              int n_kvt, int chunk, int nw, int BG, int n_items, unsigned int *err, int stall) {
    using C = BwdCfg<D>;
    constexpr int HS = C::kHStages;
    constexpr bool kFuse = !kSplit;
    constexpr int kEpiStages = kFuse ? 3 : 0;       // k rows + two (cos, sin) halves per item
    extern __shared__ uint8_t smem_raw[];
    __shared__ BwdBarriers bars;
    __shared__ EpiScratch escr;
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sK = smem;
    uint8_t *sV = smem + C::kTileBytes;
    uint8_t *sStage = smem + 2 * C::kTileBytes;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = H / G;
    volatile int *abort_flag = &bars.abort_flag;

    if (threadIdx.x == 0) init_bwd_barriers(bars, 1, 2, HS, true);
    if (warp == kWarpMma) {
        tmem_alloc(&bars.tmem_base, 512);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    pdl_enter();
    const uint32_t tmem = bars.tmem_base;

    // Every role walks the same items (snake_item) and skips
    // the same empty ones. Half stages are used in one sequence across items: an
    // item's 2T streamed half tiles (x = 2 t + hf: rows [64 hf, 64 hf + 64) of
    // streamed tile t), then (kFuse) its three epilogue-input stages, which the
    // softmax threads release after the epilogue. Barrier phases count items
    // (own_full, acc_done) or streamed tiles (s_full, p_full) across items.
    if (warp == kWarpTma) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&map_k);
            tma_prefetch_desc(&map_v);
            tma_prefetch_desc(&map_q);
            tma_prefetch_desc(&map_do);
        }
        int items = 0, issued = 0;   // items whose own tiles were loaded; half stages used
        bool ok = true;
        for (int rnd = 0, w = snake_item(0); ok && w < n_items; w = snake_item(++rnd)) {
            const DkdvItem it = dkdv_item<kSplit>(w, BG, H, G, n_kvt, chunk, sr);
            if (it.T == 0) continue;
            const SeqSpan sp = it.sp;
            const int S = sp.len, T = it.T, g = it.g, j = it.j;
            // the item's own K and V tiles, once the previous item's S^T/dP^T MMAs
            // have read the old ones
            if (lane == 0 && items > 0)
                ok = mbar_wait(&bars.acc_done, (items - 1) & 1, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane == 0) {
                mbar_expect_tx(&bars.own_full, 2 * C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_3d(sK + c * C::kBox, &map_k, &bars.own_full, c * C::A::kCols,
                                sp.start + j * kTile, sp.plane * G + g);
                    tma_load_4d(sV + c * C::kBox, &map_v, &bars.own_full, c * C::A::kCols, g,
                                sp.start + j * kTile, sp.plane);
                }
            }
            ++items;
            for (int x = 0; x < 2 * T + kEpiStages; ++x) {
                const int xs = issued, hs = xs % HS;
                if (lane == 0 && xs >= HS)
                    ok = mbar_wait(&bars.st_empty[hs], ((xs / HS) - 1) & 1, abort_flag);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                uint8_t *base = sStage + hs * C::kHStageBytes;
                if (x >= 2 * T) {
                    // the dk epilogue's inputs: the owned k rows (one 128-row tile),
                    // then their (cos, sin) rows in two 64-row halves (D/32 boxes of 64
                    // rows x 16 pairs each)
                    const int e = x - 2 * T;
                    if (lane == 0) {
                        if (e == 0) {
                            mbar_expect_tx(&bars.st_full[hs], C::kTileBytes);
                            for (int c = 0; c < C::kChunks; ++c)
                                tma_load_4d(base + c * C::kBox, &map_x, &bars.st_full[hs],
                                            c * C::A::kCols, g, sp.start + j * kTile, sp.plane);
                        } else {
                            mbar_expect_tx(&bars.st_full[hs], (D / 32) * kCsPieceBytes);
                            for (int c = 0; c < D / 32; ++c)
                                tma_load_2d(base + c * kCsPieceBytes, &map_cs, &bars.st_full[hs],
                                            32 * c, sp.start + j * kTile + 64 * (e - 1));
                        }
                        mbar_arrive(&bars.st_full[hs]);
                    }
                    ++issued;
                    continue;
                }
                const int t = it.t0 + (x >> 1), hf = x & 1;
                const int rr = t / it.nU, u = j + (t - rr * it.nU);
                const int h = g * group + rr;
                const int q0 = u * kTile + 64 * hf;
                if (lane == 0) {
                    mbar_expect_tx(&bars.st_full[hs], 2 * C::kHalfBytes);
                    for (int c = 0; c < C::kChunks; ++c) {
                        tma_load_3d(base + c * C::kHalfBox, &map_q, &bars.st_full[hs],
                                    c * C::A::kCols, sp.start + q0, sp.plane * H + h);
                        tma_load_4d(base + C::kHalfBytes + c * C::kHalfBox, &map_do,
                                    &bars.st_full[hs], c * C::A::kCols, h, sp.start + q0, sp.plane);
                    }
                }
                // the half's row statistics by 4-byte asynchronous copies that the stage's
                // barrier waits for (so the producer never stalls on a global load):
                // column kq at 4 (kq / 2) + kq % 2 (lse) and two words on (Dlt), one
                // 16-byte word per column pair; rows past the end read as 0
                float *sl = reinterpret_cast<float *>(base + 2 * C::kHalfBytes);
                const size_t row0 = ((size_t)sp.plane * H + h) * sr.S + sp.start;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int kq = lane + 32 * e, q = q0 + kq;
                    const int o = 4 * (kq >> 1) + (kq & 1);
                    if (q < S) {
                        cp_async4(sl + o, lse + row0 + q);
                        cp_async4(sl + o + 2, dlt + row0 + q);
                    } else {
                        sl[o] = 0.f;
                        sl[o + 2] = 0.f;
                    }
                }
                // each lane's copies become one pending arrival of the stage barrier
                // (registered before lane 0's arrival below, hence the __syncwarp)
                cp_async_mbar_arrive(&bars.st_full[hs]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.st_full[hs]);
                ++issued;
            }
        }
        if (!ok && lane == 0 && !*abort_flag) raise_error_b(err, abort_flag);
        if (lane == 0) {
            // drain: every copy issued by this CTA lands before it exits
            if (items > 0) mbar_wait(&bars.own_full, (items - 1) & 1, nullptr);
            for (int x = max(0, issued - HS); x < issued; ++x)
                mbar_wait(&bars.st_full[x % HS], (x / HS) & 1, nullptr);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        {
            // the whole warp runs this loop; one elected lane issues each MMA / commit
            const uint32_t idesc_s = idesc_bf16_f32(kTile, kTile / 2, 0, 0);
            const uint32_t idesc_acc = idesc_bf16_f32(kTile, D, 0, 1);
            using A = typename C::A;
            const uint64_t dK = smem_desc(smem_u32(sK), 16, A::kSBO, A::kMode);
            const uint64_t dV = smem_desc(smem_u32(sV), 16, A::kSBO, A::kMode);
            const uint64_t dQk0 = smem_desc(smem_u32(sStage), 16, A::kSBO, A::kMode);
            const uint64_t dDOk0 = smem_desc(smem_u32(sStage + C::kHalfBytes), 16, A::kSBO, A::kMode);
            const uint64_t dQm0 = smem_desc(smem_u32(sStage), C::kHalfBox, A::kSBO, A::kMode);
            const uint64_t dDOm0 = smem_desc(smem_u32(sStage + C::kHalfBytes), C::kHalfBox, A::kSBO,
                                             A::kMode);
            constexpr uint64_t kStep = (uint64_t)C::kHStageBytes >> 4;
            // S^T = Khat Qhat^T and dP^T = V dO^T for the queries [64h, 64h+64) of a
            // streamed tile, from half stage xs (its use index) % HS
            auto issue_sp = [&](int xs, int h) {
                const uint64_t so = (uint64_t)(xs % HS) * kStep;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss_w(tmem + 64 * h, dK + kmajor_off<D>(kk), dQk0 + so + kmajor_off_half<D>(kk),
                             idesc_s, kk > 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss_w(tmem + 128 + 64 * h, dV + kmajor_off<D>(kk),
                             dDOk0 + so + kmajor_off_half<D>(kk), idesc_s, kk > 0);
                mma_commit_w(&bars.s_full[h]);
            };
            bool ok = !stall ||
                      __all_sync(0xffffffffu, mbar_wait_for(&bars.stall, 0, abort_flag, kStallLimitNs));
            int items = 0, xb = 0, tg = 0;   // items, half stages and streamed tiles before this item
            for (int rnd = 0, w = snake_item(0); ok && w < n_items; w = snake_item(++rnd)) {
                const DkdvItem it = dkdv_item<kSplit>(w, BG, H, G, n_kvt, chunk, sr);
                if (it.T == 0) continue;
                const int T = it.T;
                ok = mbar_wait_w(&bars.own_full, items & 1, abort_flag) &&
                     mbar_wait_w(&bars.st_full[xb % HS], (xb / HS) & 1, abort_flag) &&
                     mbar_wait_w(&bars.st_full[(xb + 1) % HS], ((xb + 1) / HS) & 1,
                                 abort_flag);   // both halves of tile 0
                if (!ok) break;
                tc_fence_after();
                issue_sp(xb, 0);
                issue_sp(xb + 1, 1);
                // Per half h: once its P/dS are in TMEM, accumulate its 4 k-steps of
                // dV += P^T dO and dKhat += dS^T Qhat, then start S/dP of the same half
                // of the next tile (in-order execution keeps them behind those reads).
                // The first accumulating MMA of an item overwrites the accumulators: the
                // softmax threads read the previous item's out (epilogue) before they
                // signal this item's first P.
                for (int t = 0; ok && t < T; ++t) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int xs = xb + 2 * t + h;
                        const uint64_t so = (uint64_t)(xs % HS) * kStep;
                        if (!(ok = mbar_wait_w(&bars.p_full[h], (tg + t) & 1, abort_flag))) break;
                        tc_fence_after();
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) {   // dV += P^T dO
                            const int kk = 4 * h + k4;
                            mma_ts_w(tmem + 256, tmem + packed_col(kk), dDOm0 + so + mnmajor_off<D>(k4),
                                     idesc_acc, (t > 0 || kk > 0) ? 1u : 0u);
                        }
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) {   // dKhat += dS^T Qhat
                            const int kk = 4 * h + k4;
                            mma_ts_w(tmem + 384, tmem + 128 + packed_col(kk), dQm0 + so + mnmajor_off<D>(k4),
                                     idesc_acc, (t > 0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit_w(&bars.st_empty[xs % HS]);   // this half stage may be reloaded
                        if (t + 1 < T) issue_sp(xs + 2, h);      // operands checked by the softmax warps
                    }
                }
                if (!ok) break;
                mma_commit_w(&bars.acc_done);   // also frees the own K/V tiles
                xb += 2 * T + kEpiStages;
                tg += T;
                ++items;
            }
            if (!ok && lane == 0 && !*abort_flag) raise_error_b(err, abort_flag);
            mma_commit_w(&bars.drain);
            mbar_wait_w(&bars.drain, 0, nullptr);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int wg = warp >> 2, quarter = warp & 3;
        const int r = quarter * 32 + lane;              // owned key row = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float sl2 = kLog2e * rsqrtf((float)D);
        const int hf = wg >> 1;                         // this warpgroup's half of the tile
        int items = 0, xb = 0, tg = 0;
        for (int rnd = 0, w = snake_item(0); w < n_items; w = snake_item(++rnd)) {
            const DkdvItem it = dkdv_item<kSplit>(w, BG, H, G, n_kvt, chunk, sr);
            float *pk = kFuse ? part_k + ((size_t)it.bg * nw + it.witem) * D : nullptr;   // dgamma_k partial
            if (it.T == 0) {                            // a packed sample shorter than this tile
                if constexpr (kFuse)
                    if (threadIdx.x < D) pk[threadIdx.x] = 0.f;
                continue;
            }
            const SeqSpan sp = it.sp;
            const int S = sp.len, T = it.T, g = it.g, j = it.j;
            const int kp = j * kTile + r;               // key position
            if (kFuse && wg == kSoftmaxWGs - 1) {
                // for the dk epilogue (read after its first named barrier; the previous
                // item's epilogue finished reading these before the stop barrier below)
                escr.rstd[r] = kp < S ? rstd_k[((size_t)sp.plane * sr.S + sp.start + kp) * G + g] : 0.f;
                if (r < D) escr.gamma[r] = gamma_k[r];
            }
            bool ok = true;
            for (int t = 0; t < T; ++t) {
                const int x = xb + 2 * t + hf, hs = x % HS;
                // the half stage first: its row statistics are loaded into registers while
                // S^T/dP^T are still being computed (their shared-memory loads would
                // otherwise queue behind the tensor core's operand reads)
                ok = __all_sync(0xffffffffu, mbar_wait(&bars.st_full[hs], (x / HS) & 1, abort_flag));
                if (!ok) break;
                float4 st4[4];
                {
                    // (lse, lse, Dlt, Dlt) of the column pairs 8 k + 2 (lane % 4) of this
                    // warpgroup's 32 columns
                    const float4 *sl4 = reinterpret_cast<const float4 *>(
                        sStage + hs * C::kHStageBytes + 2 * C::kHalfBytes);
#pragma unroll
                    for (int k = 0; k < 4; ++k) st4[k] = sl4[16 * (wg & 1) + 4 * k + (lane & 3)];
                }
                ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full[hf], (tg + t) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                const int u = j + ((it.t0 + t) % it.nU);
                const int c0 = wg * kWgCols;                // this warpgroup's columns
                const int q0 = u * kTile + c0;
                const uint32_t tS = tmem + lane_off + c0;         // S^T columns
                const uint32_t tP = tmem + lane_off + 128 + c0;   // dP^T columns
                // no masking when every query of these columns is at/after every owned key and < S
                const bool interior = (q0 >= j * kTile + kTile - 1) && (q0 + kWgCols <= S);
                // 16-lane TMEM shapes (xt_tc.cuh): this thread holds rows
                // 16 L + lane/4 + 8 jh of its warp's 32 and the column pairs 8 k + 2 (lane % 4)
                // of the warpgroup's 32, so it needs the statistics of 8 columns only (st4).
                uint32_t pp[kWgCols / 2], dd[kWgCols / 2];
                {
                    uint32_t sv[32], dpv[32];
                    tmem_ld16x256b_x4_rows32_pair_sync(tS, sv, tP, dpv);
                    const int cp = 2 * (lane & 3);
                    // masked columns (the diagonal tile, the ragged end) take the select;
                    // interior tiles (all but about one in n_q) run without it
                    auto body = [&](auto masked) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float2 nl = fmul2(make_float2(st4[k].x, st4[k].y),
                                                    make_float2(-kLog2e, -kLog2e));
                            const float2 ndl = make_float2(-st4[k].z, -st4[k].w);
#pragma unroll
                            for (int L = 0; L < 2; ++L) {
#pragma unroll
                                for (int jh = 0; jh < 2; ++jh) {
                                    // column pairs through the packed fp32 pipe (f32x2 FMA / add / mul)
                                    const int e = 16 * L + 4 * k + 2 * jh;
                                    const float2 a = ffma2(make_float2(__uint_as_float(sv[e]),
                                                                       __uint_as_float(sv[e + 1])),
                                                           make_float2(sl2, sl2), nl);
                                    float2 p = make_float2(fast_exp2(a.x), fast_exp2(a.y));
                                    if constexpr (decltype(masked)::value) {
                                        const int q = q0 + 8 * k + cp;
                                        const int kr = j * kTile + quarter * 32 + 16 * L + (lane >> 2) + 8 * jh;
                                        if (!(q >= kr && q < S)) p.x = 0.f;
                                        if (!(q + 1 >= kr && q + 1 < S)) p.y = 0.f;
                                    }
                                    const float2 ds = fmul2(p, fadd2(make_float2(__uint_as_float(dpv[e]),
                                                                                 __uint_as_float(dpv[e + 1])),
                                                                     ndl));
                                    pp[8 * L + 2 * k + jh] = pack_bf16x2(p.x, p.y);
                                    dd[8 * L + 2 * k + jh] = pack_bf16x2(ds.x, ds.y);
                                }
                            }
                        }
                    };
                    if (interior) body(std::false_type{});
                    else body(std::true_type{});
                }
                if (t + 1 < T) {   // operands of this half of tile t+1, issued right behind its dV/dK
                    ok = __all_sync(0xffffffffu, mbar_wait(&bars.st_full[(x + 2) % HS],
                                                           ((x + 2) / HS) & 1, abort_flag));
                    if (!ok) break;
                }
                tmem_st16x128b_x4_rows32_pair_sync(tS, pp, tP, dd);
                tc_fence_before();
                mbar_arrive(&bars.p_full[hf]);
            }
            if (ok) {
                ok = __all_sync(0xffffffffu, mbar_wait(&bars.acc_done, items & 1, abort_flag));
                if (ok) {
                    tc_fence_after();
                    store_dkdv_acc<D, kSplit>(
                        wg, tmem + lane_off, kp < S,
                        dv + (((size_t)sp.plane * sr.S + sp.start + kp) * G + g) * D,
                        dkhat + (((size_t)sp.plane * G + g) * sr.S + sp.start + kp) * D,
                        it.split ? part + ((size_t)it.bg * nw + it.witem) * 2 * kTile * D + (size_t)r * D
                                 : nullptr);
                }
            }
            if (!ok && !*abort_flag) raise_error_b(err, abort_flag);
            if constexpr (kFuse) {
                // dk and the item's dgamma_k partial from dKhat in TMEM, with the k rows
                // and their (cos, sin) rows that the producer loaded after the last half
                const int x0 = xb + 2 * T;
                if (ok) ok = __all_sync(0xffffffffu,
                                        mbar_wait(&bars.st_full[x0 % HS], (x0 / HS) & 1, abort_flag) &&
                                        mbar_wait(&bars.st_full[(x0 + 1) % HS], ((x0 + 1) / HS) & 1,
                                                  abort_flag) &&
                                        mbar_wait(&bars.st_full[(x0 + 2) % HS], ((x0 + 2) / HS) & 1,
                                                  abort_flag));
                if (!ok && !*abort_flag) raise_error_b(err, abort_flag);
                const uint8_t *sX = sStage + (x0 % HS) * C::kHStageBytes;
                const uint8_t *cs_row = sStage + ((x0 + 1 + (r >> 6)) % HS) * C::kHStageBytes +
                                        (r & 63) * 128;
                finish_rows_dk<D>(ok, wg, quarter, lane, tmem + 384 + lane_off, sX, cs_row, kp < S,
                                  escr, dk + (((size_t)sp.plane * sr.S + sp.start + kp) * G + g) * D,
                                  pk);
                // every softmax thread is done with the epilogue inputs (finish_rows ends
                // on a named barrier): their half stages may be refilled
                if (threadIdx.x == 0) {
                    mbar_arrive(&bars.st_empty[x0 % HS]);
                    mbar_arrive(&bars.st_empty[(x0 + 1) % HS]);
                    mbar_arrive(&bars.st_empty[(x0 + 2) % HS]);
                }
            }
            // stop together (a failed wait here, or one raised by another warp); the
            // barrier also keeps the next item's P signals (and so its first
            // accumulating MMAs) behind every thread's reads of the accumulators
            if (softmax_bar_any(!ok || *abort_flag)) break;
            xb += 2 * T + kEpiStages;
            tg += T;
            ++items;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}


// Sums the chunk partials of the split key tiles in chunk order: block =
// (split key tile j, unit x kv head), threads over the tile's rows x D.
__global__ void __launch_bounds__(256)
k_dkdv_reduce(const float *__restrict__ part, float *__restrict__ dkhat, bf16 *__restrict__ dv,
              const SeqRows sr, int H, int G, int D, int n_kvt, int chunk, int nw) {
    pdl_enter();
    const int j = blockIdx.x, bg = blockIdx.y;
    const int unit = bg / G, g = bg - unit * G, group = H / G;
    int w0 = 0;
    for (int i = 0; i < j; ++i) w0 += dkdv_chunks(group * (n_kvt - i), chunk);
    const int nc = dkdv_chunks(group * (n_kvt - j), chunk);
    if (nc <= 1) return;
    const SeqSpan sp = seq_span(sr, unit);
    const size_t stride = (size_t)2 * kTile * D;   // one chunk's [dV | dKhat]
    const float *base = part + ((size_t)bg * nw + w0) * stride;
    for (int e = threadIdx.x; e < kTile * D; e += blockDim.x) {
        const int r = e / D, d = e - r * D;
        const int kp = j * kTile + r;
        if (kp >= sp.len) break;
        float sv = 0.f, sk = 0.f;
        for (int c = 0; c < nc; ++c) {
            sv += base[c * stride + e];
            sk += base[c * stride + (size_t)kTile * D + e];
        }
        dv[(((size_t)sp.plane * sr.S + sp.start + kp) * G + g) * D + d] = __float2bfloat16_rn(sv);
        dkhat[(((size_t)sp.plane * G + g) * sr.S + sp.start + kp) * D + d] = sk;
    }
}

// ---------------------------------------------------------------------------
// dQhat and the dq epilogue
// ---------------------------------------------------------------------------
// L2 prefetch of [p, p + bytes), widened to 16-byte boundaries.
__device__ __forceinline__ void l2_prefetch_span(const void *p, size_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p) & ~(uintptr_t)15;
    const uintptr_t e = (reinterpret_cast<uintptr_t>(p) + bytes + 15) & ~(uintptr_t)15;
    l2_prefetch_bulk(reinterpret_cast<const void *>(a), (uint32_t)(e - a));
}

template <int D>
__global__ void __launch_bounds__(kThreadsBwd, 1)
k_bwd_dq_tc(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
            const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_cs,
            const __grid_constant__ CUtensorMap map_do, const __grid_constant__ CUtensorMap map_o,
            const __grid_constant__ CUtensorMap map_dq, const __grid_constant__ CUtensorMap map_qh,
            const bf16 *__restrict__ out, const float *__restrict__ lse, float *__restrict__ dlt,
            const float *__restrict__ gamma_q, const float *__restrict__ rstd_q,
            bf16 *__restrict__ dq, float *__restrict__ part_q, const SeqRows sr, int H, int G,
            int BH, int n_qt, int n_items, unsigned int *err, int stall) {
    using C = BwdCfg<D>;
    constexpr int KS = C::kKStages, VS = C::kVStages;
    // TMEM: S [0,128), dP [128,256), dQhat accumulator [256, 256+D), the resident
    // Qhat A operand at 384 (D/2 packed columns) and packed dS at 448 (64 columns:
    // k-step kk of 16 keys at [448 + 8 kk, +8)), so that dS of one key tile and
    // S/dP of the next live side by side
    constexpr uint32_t kTQ = 384, kTDS = 448;
    extern __shared__ uint8_t smem_raw[];
    __shared__ BwdBarriers bars;
    __shared__ EpiScratch escr;
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sK = smem;                                // KS K tiles
    uint8_t *sV = sK + KS * C::kTileBytes;             // VS V tiles
    // the owned rows: first Qhat (copied into TMEM as the S MMA's A), then dO (the
    // dP MMA's A, and Dlt's)
    uint8_t *sDO = sV + VS * C::kTileBytes;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &bars.abort_flag;
    // s_full[0] / dp_full: S / dP of a key tile are in TMEM; p_full[1] / dp_taken:
    // every softmax thread holds them in registers (the columns may be
    // overwritten); p_full[0]: packed dS is in TMEM; s_full[1]: dQ has read dS
    // (its columns may be overwritten). Their phases count key tiles across items.
    uint64_t *ds_ready = &bars.p_full[0];
    uint64_t *s_taken = &bars.p_full[1];
    uint64_t *ds_free = &bars.s_full[1];

    if (threadIdx.x == 0) init_bwd_barriers(bars, 1, 1, KS > VS ? KS : VS, false);
    if (warp == kWarpMma) {
        tmem_alloc(&bars.tmem_base, 512);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    pdl_enter();
    const uint32_t tmem = bars.tmem_base;

    // Every role walks the same items (snake_item: rounds of gridDim.x items,
    // walked forwards and backwards in turn) and skips
    // the same empty ones. Ring uses per item: K ring, its T key tiles and then
    // the two (cos, sin) halves of its rows; V ring, its T value tiles and then its
    // q rows (the epilogue's inputs, released by the softmax threads after it; the
    // epilogue writes the dq rows over them, and the producer stores that tile by
    // TMA before it reloads the slot, so the softmax threads never wait for it).
    // The owned-row slot takes the item's Qhat rows (own_full), which the MMA warp
    // copies into TMEM once the previous item's last S MMA has run (q_read), then
    // its dO rows (x_full), held until its dP MMAs and Dlt are done (do_free): the
    // next item's Qhat copy, first S and first dP run during the current item's
    // epilogue.
    if (warp == kWarpTma) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&map_k);
            tma_prefetch_desc(&map_v);
            tma_prefetch_desc(&map_x);
            tma_prefetch_desc(&map_cs);
            tma_prefetch_desc(&map_do);
            tma_prefetch_desc(&map_o);
            tma_prefetch_desc(&map_dq);
            int items = 0, x_issued = 0, k_issued = 0, v_issued = 0;
            // a V slot holding an item's staged dq rows, to be stored by TMA once the
            // softmax threads release the slot: (head, first row, plane), or h < 0
            int pend_h[VS], pend_row[VS], pend_plane[VS];
#pragma unroll
            for (int v = 0; v < VS; ++v) pend_h[v] = -1;
            auto store_dq = [&](int vs) {
                for (int c = 0; c < C::kChunks; ++c)
                    tma_store_4d(&map_dq, sV + vs * C::kTileBytes + c * C::kBox, c * C::A::kCols,
                                 pend_h[vs], pend_row[vs], pend_plane[vs]);
                bulk_commit();
                pend_h[vs] = -1;
            };
            bool ok = true;
            for (int rnd = 0, w = snake_item(0); ok && w < n_items; w = snake_item(++rnd)) {
                const DqItem it = dq_item(w, BH, n_qt, H, G, sr);
                if (it.T == 0) continue;
                const int T = it.T, row0 = it.sp.start + it.i * kTile;
                {
                    // L2 prefetch of what the softmax threads read with plain loads when
                    // the item starts (after the previous item's epilogue): the O rows,
                    // the rows' lse and the rstd_q block of the rows (all heads)
                    const int rows = min(kTile, it.sp.len - it.i * kTile);
                    for (int c = 0; c < C::kChunks; ++c)
                        l2_prefetch_4d(&map_o, c * C::A::kCols, it.h, row0, it.sp.plane);
                    l2_prefetch_span(lse + ((size_t)it.sp.plane * H + it.h) * sr.S + row0,
                                     (size_t)rows * 4);
                    l2_prefetch_span(rstd_q + ((size_t)it.sp.plane * sr.S + row0) * H,
                                     (size_t)rows * H * 4);
                }
                // the item's Qhat rows, once the previous item's dP MMAs and Dlt have read
                // its dO rows
                if (items > 0 && !(ok = mbar_wait(&bars.do_free, (items - 1) & 1, abort_flag)))
                    break;
                mbar_expect_tx(&bars.own_full, C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sDO + c * C::kBox, &map_qh, &bars.own_full, c * C::A::kCols, row0,
                                it.sp.plane * H + it.h);
                ++items;
                for (int u = 0; ok && u < T + 2; ++u) {
                    const int ks = k_issued % KS;
                    if (k_issued >= KS &&
                        !(ok = mbar_wait(&bars.st_empty[ks], ((k_issued / KS) - 1) & 1, abort_flag)))
                        break;
                    uint8_t *kb = sK + ks * C::kTileBytes;
                    if (u < T) {
                        mbar_expect_tx(&bars.st_full[ks], C::kTileBytes);
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_3d(kb + c * C::kBox, &map_k, &bars.st_full[ks],
                                        c * C::A::kCols, it.sp.start + u * kTile,
                                        it.sp.plane * G + it.g);
                    } else {
                        // (cos, sin) rows [64 e, 64 e + 64) of the owned rows: D/32 pieces
                        mbar_expect_tx(&bars.st_full[ks], (D / 32) * kCsPieceBytes);
                        for (int c = 0; c < D / 32; ++c)
                            tma_load_2d(kb + c * kCsPieceBytes, &map_cs, &bars.st_full[ks],
                                        32 * c, row0 + 64 * (u - T));
                    }
                    ++k_issued;
                    if (u > T) continue;
                    const int vs = v_issued % VS;
                    if (v_issued >= VS &&
                        !(ok = mbar_wait(&bars.v_empty[vs], ((v_issued / VS) - 1) & 1, abort_flag)))
                        break;
                    if (pend_h[vs] >= 0) {
                        // the dq rows an earlier epilogue staged here: stored before the
                        // slot is reloaded
                        store_dq(vs);
                        bulk_wait_read0();
                    }
                    uint8_t *vb = sV + vs * C::kTileBytes;
                    mbar_expect_tx(&bars.v_full[vs], C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c) {
                        if (u < T)
                            tma_load_4d(vb + c * C::kBox, &map_v, &bars.v_full[vs],
                                        c * C::A::kCols, it.g, it.sp.start + u * kTile,
                                        it.sp.plane);
                        else
                            tma_load_4d(vb + c * C::kBox, &map_x, &bars.v_full[vs],
                                        c * C::A::kCols, it.h, row0, it.sp.plane);
                    }
                    // the epilogue stages dq over the q rows unless the tile reaches past
                    // a packed sample (those rows are stored one by one)
                    if (u == T && (sr.cu == nullptr || it.i * kTile + kTile <= it.sp.len)) {
                        pend_h[vs] = it.h;
                        pend_row[vs] = row0;
                        pend_plane[vs] = it.sp.plane;
                    }
                    ++v_issued;
                    if (u == 0) {
                        // the item's dO rows, once its Qhat rows are in TMEM (behind its
                        // first K and V tiles, whose slots free up earlier)
                        if (!(ok = mbar_wait(&bars.q_read, (items - 1) & 1, abort_flag))) break;
                        mbar_expect_tx(&bars.x_full, C::kTileBytes);
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_4d(sDO + c * C::kBox, &map_do, &bars.x_full, c * C::A::kCols,
                                        it.h, row0, it.sp.plane);
                        ++x_issued;
                    }
                }
            }
            // the last items' staged dq rows, in ring order, once their epilogues are done
            for (int x = max(0, v_issued - VS); ok && x < v_issued; ++x) {
                const int vs = x % VS;
                if (pend_h[vs] < 0) continue;
                if ((ok = mbar_wait(&bars.v_empty[vs], (x / VS) & 1, abort_flag))) store_dq(vs);
            }
            if (!ok && !*abort_flag) raise_error_b(err, abort_flag);
            bulk_wait0();   // every dq store has completed
            // drain: every copy issued by this CTA lands before it exits (at most the
            // last Qhat and dO loads, the last KS K-ring and the last VS V-ring loads
            // in flight)
            if (items > 0) mbar_wait(&bars.own_full, (items - 1) & 1, nullptr);
            if (x_issued > 0) mbar_wait(&bars.x_full, (x_issued - 1) & 1, nullptr);
            for (int x = max(0, k_issued - KS); x < k_issued; ++x)
                mbar_wait(&bars.st_full[x % KS], (x / KS) & 1, nullptr);
            for (int x = max(0, v_issued - VS); x < v_issued; ++x)
                mbar_wait(&bars.v_full[x % VS], (x / VS) & 1, nullptr);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        {
            // the whole warp runs this loop; one elected lane issues each MMA / commit
            const uint32_t idesc_s = idesc_bf16_f32(kTile, kTile, 0, 0);
            const uint32_t idesc_acc = idesc_bf16_f32(kTile, D, 0, 1);
            using A = typename C::A;
            const uint64_t dKk0 = smem_desc(smem_u32(sK), 16, A::kSBO, A::kMode);
            const uint64_t dVk0 = smem_desc(smem_u32(sV), 16, A::kSBO, A::kMode);
            const uint64_t dKm0 = smem_desc(smem_u32(sK), C::kBox, A::kSBO, A::kMode);
            const uint64_t dDO = smem_desc(smem_u32(sDO), 16, A::kSBO, A::kMode);
            constexpr uint64_t kStep = (uint64_t)C::kTileBytes >> 4;
            // S = Qhat Khat^T (A in TMEM) and dP = dO V^T (both operands in shared
            // memory), full 128-key tiles (N = 128 runs at the full MMA rate); kx / vx
            // are the tiles' K-ring / V-ring use indices
            auto issue_s = [&](int kx) {
                const uint64_t ko = (uint64_t)(kx % KS) * kStep;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ts_w(tmem, tmem + kTQ + kk * 8, dKk0 + ko + kmajor_off<D>(kk), idesc_s, kk > 0);
                mma_commit_w(&bars.s_full[0]);         // S of the tile is in TMEM
            };
            auto issue_dp = [&](int vx) {
                const uint64_t vo = (uint64_t)(vx % VS) * kStep;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss_w(tmem + 128, dDO + kmajor_off<D>(kk), dVk0 + vo + kmajor_off<D>(kk),
                             idesc_s, kk > 0);
                mma_commit_w(&bars.dp_full);           // dP of the tile is in TMEM
                mma_commit_w(&bars.v_empty[vx % VS]);  // its V tile is read
            };
            bool ok = !stall ||
                      __all_sync(0xffffffffu, mbar_wait_for(&bars.stall, 0, abort_flag, kStallLimitNs));
            int items = 0, kt = 0, vt = 0, tg = 0;   // ring uses and key tiles before this item
            for (int rnd = 0, w = snake_item(0); ok && w < n_items; w = snake_item(++rnd)) {
                const DqItem it = dq_item(w, BH, n_qt, H, G, sr);
                if (it.T == 0) continue;
                const int T = it.T;
                // the item's Qhat rows from the owned-row slot into TMEM. The previous
                // item's last S MMA, which read the old ones, has completed: its dS
                // was signalled (after the softmax threads had waited for that S)
                // before the previous dQ MMA was issued. The copy's commit releases the
                // slot for the dO rows and orders the copy before the S MMAs.
                if (!(ok = mbar_wait_w(&bars.own_full, items & 1, abort_flag))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    tmem_cp128x256b_w(tmem + kTQ + kk * 8, dDO + kmajor_off<D>(kk));
                mma_commit_w(&bars.q_read);
                ok = mbar_wait_w(&bars.q_read, items & 1, abort_flag) &&
                     mbar_wait_w(&bars.st_full[kt % KS], (kt / KS) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                issue_s(kt);
                // the first dP once the dO rows and the first V tile have landed
                ok = mbar_wait_w(&bars.x_full, items & 1, abort_flag) &&
                     mbar_wait_w(&bars.v_full[vt % VS], (vt / VS) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                issue_dp(vt);
                if (T == 1) mma_commit_w(&bars.do_free);
                // Per tile t: once every softmax thread holds S(t) in registers, S(t+1)
                // is issued, and once they hold dP(t), dP(t+1) (both run during the
                // softmax of t, and the dP loads overlap S(t+1)); once dS(t) is packed
                // in its own columns, dQ(t). The softmax of t+1 writes dS(t+1) only
                // after dQ(t) has read dS(t) (ds_free).
                for (int t = 0; ok && t < T; ++t) {
                    const int x = tg + t;
                    if (t + 1 < T) {
                        if (!(ok = mbar_wait_w(s_taken, x & 1, abort_flag) &&
                                   mbar_wait_w(&bars.st_full[(kt + t + 1) % KS],
                                               ((kt + t + 1) / KS) & 1, abort_flag)))
                            break;
                        tc_fence_after();
                        issue_s(kt + t + 1);
                        if (!(ok = mbar_wait_w(&bars.dp_taken, x & 1, abort_flag) &&
                                   mbar_wait_w(&bars.v_full[(vt + t + 1) % VS],
                                               ((vt + t + 1) / VS) & 1, abort_flag)))
                            break;
                        tc_fence_after();
                        issue_dp(vt + t + 1);
                        if (t + 2 == T) mma_commit_w(&bars.do_free);   // the item's last dP
                    }
                    if (!(ok = mbar_wait_w(ds_ready, x & 1, abort_flag))) break;
                    tc_fence_after();
                    const uint64_t ko = (uint64_t)((kt + t) % KS) * kStep;
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)   // dQhat += dS Khat
                        mma_ts_w(tmem + 256, tmem + kTDS + kk * 8, dKm0 + ko + mnmajor_off<D>(kk),
                                 idesc_acc, (t > 0 || kk > 0) ? 1u : 0u);
                    mma_commit_w(&bars.st_empty[(kt + t) % KS]);   // K tile t is read
                    mma_commit_w(ds_free);
                }
                if (!ok) break;
                mma_commit_w(&bars.acc_done);
                kt += T + 2;
                vt += T + 1;
                tg += T;
                ++items;
            }
            if (!ok && lane == 0 && !*abort_flag) raise_error_b(err, abort_flag);
            mma_commit_w(&bars.drain);
            mbar_wait_w(&bars.drain, 0, nullptr);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int wg = warp >> 2, quarter = warp & 3;
        const int r = quarter * 32 + lane;             // owned query row = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float sl2 = kLog2e * rsqrtf((float)D);
        int items = 0, kt = 0, vt = 0, tg = 0;
        for (int rnd = 0, w = snake_item(0); w < n_items; w = snake_item(++rnd)) {
            const DqItem it = dq_item(w, BH, n_qt, H, G, sr);
            float *part = part_q + ((size_t)it.bh * n_qt + it.i) * D;   // the item's dgamma_q partial
            if (it.T == 0) {                       // a packed sample shorter than this tile
                if (threadIdx.x < D) part[threadIdx.x] = 0.f;
                continue;
            }
            const int T = it.T, S = it.sp.len, h = it.h;
            const int tq = it.i * kTile + r;           // query position
            const size_t qrow0 = ((size_t)it.sp.plane * H + h) * sr.S + it.sp.start;
            const size_t xrow = ((size_t)it.sp.plane * sr.S + it.sp.start + tq) * H + h;   // [.., S, H, ..]
            // Rows past the sample's end hold whatever the Qhat tile's TMA load brought
            // (zeros past the tensor, the next sample's rows in a packed batch): an
            // infinite lse gives them P = 0 exactly, so dS = 0 and their dQhat rows
            // stay finite (they are never stored, and their dgamma terms are zero).
            const float lse2 = tq < S ? lse[qrow0 + tq] * kLog2e : INFINITY;
            // rstd_q of the row for the dq epilogue (stashed below, read after the
            // epilogue's first named barrier)
            const float rstd_v = (wg == kSoftmaxWGs - 1 && tq < S) ? rstd_q[xrow] : 0.f;
            // Dlt = rowsum(dO o O) of the owned rows (the softmax backward's row term;
            // the dK/dV kernel, launched after this one, reads it). Row-contiguous
            // mapping: warp w takes rows [8w, 8w + 8) with D/8 lanes per row, a lane one
            // 16-byte chunk (8 columns), so each load instruction reads whole O rows.
            // O comes from global memory (loaded before the wait for the dO tile, so the
            // two latencies overlap), dO from the TMA'd tile; the lanes of a row are
            // summed by a fixed butterfly and the sum reaches the row's owner through
            // shared memory.
            constexpr int kLpr = D / 8;              // lanes per row
            constexpr int kRpi = 32 / kLpr;          // rows per load instruction
            constexpr int kNi = 8 / kRpi;            // load instructions per warp
            const int dch = lane % kLpr;
            uint4 orow[kNi];
#pragma unroll
            for (int k = 0; k < kNi; ++k) {
                const int q = it.i * kTile + 8 * warp + k * kRpi + lane / kLpr;
                orow[k] = q < S ? *reinterpret_cast<const uint4 *>(
                                      out + (((size_t)it.sp.plane * sr.S + it.sp.start + q) * H + h) * D +
                                      8 * dch)
                                : make_uint4(0, 0, 0, 0);
            }
            bool ok = __all_sync(0xffffffffu, mbar_wait(&bars.x_full, items & 1, abort_flag));
            {
                using A = Atoms<D>;
                const int col = 8 * dch;
#pragma unroll
                for (int k = 0; k < kNi; ++k) {
                    const int rr = 8 * warp + k * kRpi + lane / kLpr;
                    float part0 = 0.f, part1 = 0.f;
                    if (ok) {
                        const uint32_t off = (uint32_t)((col / A::kCols) * A::box_bytes(kTile) +
                                                        rr * A::kRowBytes + (col % A::kCols) * 2);
                        const uint4 gv = *reinterpret_cast<const uint4 *>(sDO + swizzled<A::kRowBytes>(off));
                        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
                        const uint32_t ow[4] = {orow[k].x, orow[k].y, orow[k].z, orow[k].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            part0 = fmaf(__uint_as_float(gw[e] << 16), __uint_as_float(ow[e] << 16), part0);
                            part1 = fmaf(__uint_as_float(gw[e] & 0xffff0000u),
                                         __uint_as_float(ow[e] & 0xffff0000u), part1);
                        }
                    }
                    float sum = part0 + part1;
#pragma unroll
                    for (int o = kLpr / 2; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                    if (dch == 0) escr.dot[0][rr] = sum;
                }
            }
            softmax_bar_sync();   // every softmax thread reaches this (no wait above is unbounded)
            if (threadIdx.x == 0) mbar_arrive(&bars.do_free);   // no softmax thread reads sDO any more
            if (wg == kSoftmaxWGs - 1) {
                // for the dq epilogue (the previous item's epilogue finished reading these
                // before the stop barrier below)
                escr.rstd[r] = rstd_v;
                if (r < D) escr.gamma[r] = gamma_q[r];
            }
            const float dl = escr.dot[0][r];
            if (ok && wg == 0 && tq < S) dlt[qrow0 + tq] = dl;
            for (int t = 0; ok && t < T; ++t) {
                const int x = tg + t;                   // key tiles before this one
                ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full[0], x & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                const int c0 = wg * kWgCols;
                const int k0 = t * kTile + c0;
                const uint32_t tS = tmem + lane_off + c0;
                const uint32_t tP = tmem + lane_off + 128 + c0;
                // no masking when every key of these columns is at/before every owned query
                const bool interior = (k0 + kWgCols - 1 <= it.i * kTile);
                uint32_t dd[kWgCols / 2];
                {
                    uint32_t sv[32], dpv[32];
                    tmem_ld32_sync(tS, sv);
                    tc_fence_before();
                    mbar_arrive(s_taken);                   // S of the next tile may be issued
                    if (!__all_sync(0xffffffffu, mbar_wait(&bars.dp_full, x & 1, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    tmem_ld32_sync(tP, dpv);
                    tc_fence_before();
                    mbar_arrive(&bars.dp_taken);            // dP of the next tile may be issued
                    // only tiles that reach past the owned rows' diagonal take the select
                    // element pairs through the packed fp32 pipe (f32x2 FMA / add / mul)
                    auto body = [&](auto masked) {
                        const float2 sl2v = make_float2(sl2, sl2), nl = make_float2(-lse2, -lse2);
                        const float2 ndl = make_float2(-dl, -dl);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 a = ffma2(make_float2(__uint_as_float(sv[e]),
                                                               __uint_as_float(sv[e + 1])), sl2v, nl);
                            float2 p = make_float2(fast_exp2(a.x), fast_exp2(a.y));
                            if constexpr (decltype(masked)::value) {
                                if (k0 + e > tq) p.x = 0.f;
                                if (k0 + e + 1 > tq) p.y = 0.f;
                            }
                            const float2 ds = fmul2(p, fadd2(make_float2(__uint_as_float(dpv[e]),
                                                                         __uint_as_float(dpv[e + 1])),
                                                             ndl));
                            dd[e >> 1] = pack_bf16x2(ds.x, ds.y);
                        }
                    };
                    if (interior) body(std::false_type{});
                    else body(std::true_type{});
                }
                if (x > 0) {   // the previous dQ MMA has read the dS columns
                    ok = __all_sync(0xffffffffu, mbar_wait(ds_free, (x - 1) & 1, abort_flag));
                    if (!ok) break;
                    tc_fence_after();
                }
                tmem_st16_sync(tmem + lane_off + kTDS + 16 * wg, dd);   // packed dS, k-steps 2 wg, 2 wg + 1
                tc_fence_before();
                mbar_arrive(ds_ready);
            }
            // ---- epilogue: dq and the item's dgamma_q partial from dQhat in TMEM; the
            // producer loaded the q rows into the V slot after the item's last V tile
            // and their (cos, sin) rows into the two K slots after its last K tile (row
            // half r/64; piece wg = pairs [16 wg, 16 wg + 16))
            const int xq = vt + T, xc = kt + T;         // their ring use indices
            if (ok) ok = __all_sync(0xffffffffu,
                                    mbar_wait(&bars.acc_done, items & 1, abort_flag) &&
                                    mbar_wait(&bars.v_full[xq % VS], (xq / VS) & 1, abort_flag) &&
                                    mbar_wait(&bars.st_full[xc % KS], (xc / KS) & 1, abort_flag) &&
                                    mbar_wait(&bars.st_full[(xc + 1) % KS], ((xc + 1) / KS) & 1,
                                              abort_flag));
            if (!ok && !*abort_flag) raise_error_b(err, abort_flag);
            const uint8_t *sX = sV + (xq % VS) * C::kTileBytes;
            const uint8_t *cs_row = sK + ((xc + (r >> 6)) % KS) * C::kTileBytes + (r & 63) * 128;
            // dq rows: written over the q rows in shared memory and stored by one TMA
            // store, unless the tile reaches past a packed sample (its last rows would
            // land on the next sample's; those tiles store row by row)
            const bool tma_out = sr.cu == nullptr || it.i * kTile + kTile <= S;
            finish_rows_call<D>(ok, wg, quarter, lane, tmem + 256 + lane_off, sX, cs_row, tq < S, escr,
                                dq + xrow * D, part,
                                tma_out ? const_cast<uint8_t *>(sX) : nullptr);
            // every softmax thread is done with the item (finish_rows ends on a named
            // barrier, after each thread's fence for its staged dq rows): its epilogue
            // inputs' ring slots may be refilled (the producer first stores the staged
            // dq tile)
            if (threadIdx.x == 0) {
                mbar_arrive(&bars.v_empty[xq % VS]);
                mbar_arrive(&bars.st_empty[xc % KS]);
                mbar_arrive(&bars.st_empty[(xc + 1) % KS]);
            }
            // stop together: a failed wait here, or one raised by another warp
            if (softmax_bar_any(!ok || *abort_flag)) break;
            kt += T + 2;
            vt += T + 1;
            tg += T;
            ++items;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
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
// dO [B, S, H, D] as 4-D maps (D, heads, S, B); boxes of one swizzle atom's
// columns (tc::Atoms) x 128 rows (K, V: whole tiles) or x 64 rows (Qhat, dO:
// the dK/dV kernel's half tiles).
template <int DD>
cudaError_t make_maps(const Problem &p, const void *qhat, const void *khat, const void *v,
                      const void *dout, BwdMaps &m) {
    using A = Atoms<DD>;
    const uint64_t esz = 2, D = (uint64_t)p.D;
    const uint32_t bc = (uint32_t)A::kCols;
    const int sw = A::kSwizzleBytes;
    cudaError_t e;
    {
        const uint64_t dims[3] = {D, (uint64_t)p.S, (uint64_t)p.B * p.H};
        const uint64_t strides[2] = {D * esz, (uint64_t)p.S * D * esz};
        const uint32_t box[3] = {bc, (uint32_t)kTile / 2, 1};
        if ((e = encode_tmap_bf16(&m.q, qhat, 3, dims, strides, box, sw)) != cudaSuccess) return e;
    }
    {
        const uint64_t dims[3] = {D, (uint64_t)p.S, (uint64_t)p.B * p.G};
        const uint64_t strides[2] = {D * esz, (uint64_t)p.S * D * esz};
        const uint32_t box[3] = {bc, (uint32_t)kTile, 1};
        if ((e = encode_tmap_bf16(&m.k, khat, 3, dims, strides, box, sw)) != cudaSuccess) return e;
    }
    {
        const uint64_t dims[4] = {D, (uint64_t)p.G, (uint64_t)p.S, (uint64_t)p.B};
        const uint64_t strides[3] = {D * esz, (uint64_t)p.G * D * esz, (uint64_t)p.S * p.G * D * esz};
        const uint32_t box[4] = {bc, 1, (uint32_t)kTile, 1};
        if ((e = encode_tmap_bf16(&m.v, v, 4, dims, strides, box, sw)) != cudaSuccess) return e;
    }
    {
        const uint64_t dims[4] = {D, (uint64_t)p.H, (uint64_t)p.S, (uint64_t)p.B};
        const uint64_t strides[3] = {D * esz, (uint64_t)p.H * D * esz, (uint64_t)p.S * p.H * D * esz};
        const uint32_t box[4] = {bc, 1, (uint32_t)kTile / 2, 1};
        if ((e = encode_tmap_bf16(&m.dout, dout, 4, dims, strides, box, sw)) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Chunk size of the dK/dV work split (0: no split). When the longest key
// tile's iterations exceed half of an SM's share of the whole work (few kv
// heads with long sequences and large groups, e.g. MQA: the makespan is then
// set by single CTAs), key tiles are cut into chunks of a quarter of that
// share; otherwise nothing is split (its partials and reduce would only cost).
// Plain batches only (a packed batch's sample lengths are on the device).
struct DkdvPlan {
    int n_kvt, chunk, nw, n_split;   // key tiles, chunk, work items per (unit, kv head), split tiles
    size_t part_bytes;
};

DkdvPlan dkdv_plan(const Problem &p) {
    DkdvPlan pl = {};
    pl.n_kvt = (p.max_len + kTile - 1) / kTile;
    const int group = p.H / p.G;
    const long bgs = (long)p.units * p.G;
    if (p.cu == nullptr) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms < 1)
            sms = 148;
        long total = 0;
        for (int j = 0; j < pl.n_kvt; ++j) total += (long)group * (pl.n_kvt - j);
        total *= bgs;
        const long share = total / sms;
        const long target = (total + 4L * sms - 1) / (4L * sms);
        if (2L * group * pl.n_kvt > share && target < (1L << 30))
            pl.chunk = (int)std::max<long>(8, target);
    }
    pl.nw = 0;
    for (int j = 0; j < pl.n_kvt; ++j) {
        const int nc = dkdv_chunks(group * (pl.n_kvt - j), pl.chunk);
        pl.nw += nc;
        if (nc > 1) pl.n_split = j + 1;
    }
    pl.part_bytes = pl.n_split > 0
        ? (size_t)bgs * pl.nw * 2 * kTile * p.D * sizeof(float) : 0;
    return pl;
}

// The row epilogue's inputs: x (q or k) [B, S, heads, D] as a 4-D map with
// 128-row boxes of one swizzle atom's columns, and the fp32 RoPE table
// [S, D/2] (cos, sin) pairs as a 2-D map of D floats per row, boxes of 32
// floats (16 pairs) x cs_rows rows with the 128-byte swizzle.
template <int DD>
cudaError_t make_epi_maps(const Problem &p, const RowEpilogue &ep, int heads, int cs_rows,
                          CUtensorMap &mx, CUtensorMap &mcs) {
    using A = Atoms<DD>;
    const uint64_t esz = 2, D = (uint64_t)p.D, NH = (uint64_t)heads;
    cudaError_t e;
    {
        const uint64_t dims[4] = {D, NH, (uint64_t)p.S, (uint64_t)p.B};
        const uint64_t strides[3] = {D * esz, NH * D * esz, (uint64_t)p.S * NH * D * esz};
        const uint32_t box[4] = {(uint32_t)A::kCols, 1, (uint32_t)kTile, 1};
        if ((e = encode_tmap_bf16(&mx, ep.x, 4, dims, strides, box, A::kSwizzleBytes)) !=
            cudaSuccess)
            return e;
    }
    {
        const uint64_t dims[2] = {D, (uint64_t)p.S};
        const uint64_t strides[1] = {D * sizeof(float)};
        const uint32_t box[2] = {32, (uint32_t)cs_rows};
        if ((e = encode_tmap_f32(&mcs, ep.tab, 2, dims, strides, box, 128)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

template <int D>
cudaError_t launch_dkdv_d(const Problem &p, const BwdMaps &m, const float *lse, const float *dlt,
                          float *dkhat, void *dv, float *part, const RowEpilogue &ek,
                          unsigned int *err, cudaStream_t st) {
    using C = BwdCfg<D>;
    const DkdvPlan pl = dkdv_plan(p);
    const long blocks = (long)p.units * p.G * pl.nw;
    const bool split = pl.n_split > 0;
    CUtensorMap mx, mcs;
    cudaError_t e = split ? cudaSuccess : make_epi_maps<D>(p, ek, p.G, 64, mx, mcs);
    if (e != cudaSuccess) return e;
    if (split) mx = mcs = m.k;   // unused by the split kernel
    // persistent when every item is short (at most kPersistTiles streamed tiles: the
    // longest item, key tile 0, streams group x n_q) and there are several per SM,
    // where a CTA's set-up, fill and epilogue would dominate; longer items keep one
    // CTA each (the persistent form's extra loop state spills at the 96-register limit)
    if constexpr (D <= 64) {
        constexpr int kPersistTiles = 8;
        const int n_q = (p.max_len + kTile - 1) / kTile;
        if (!split && (p.H / p.G) * n_q <= kPersistTiles && blocks >= 2L * sm_count()) {
            const long BG = (long)p.units * p.G;
            const long n_items = blocks;
            const long grid = std::min<long>(n_items, sm_count());
            auto pk = k_bwd_dkdv_tc_p<D, false>;
            e = cudaFuncSetAttribute(pk, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemA);
            if (e != cudaSuccess) return e;
            return launch_dependent(pk, dim3((unsigned)grid), dim3(kThreadsBwd), C::kSmemA, st,
                                    m.k, m.v, m.q, m.dout, mx, mcs, lse, dlt, dkhat, (bf16 *)dv,
                                    part, ek.gamma, ek.rstd, (bf16 *)ek.out, ek.part,
                                    SeqRows{p.cu, p.S, p.max_len}, p.H, p.G, pl.n_kvt, pl.chunk,
                                    pl.nw, (int)BG, (int)n_items, err,
                                    (int)((test_stall_mask() & STALL_DKDV_TC) != 0));
        }
    }
    auto kern = split ? k_bwd_dkdv_tc<D, true> : k_bwd_dkdv_tc<D, false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemA);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, dim3((unsigned)blocks), dim3(kThreadsBwd), C::kSmemA, st, m.k,
                            m.v, m.q, m.dout, mx, mcs, lse, dlt, dkhat, (bf16 *)dv, part, ek.gamma,
                            ek.rstd, (bf16 *)ek.out, ek.part, SeqRows{p.cu, p.S, p.max_len}, p.H,
                            p.G, pl.n_kvt, pl.chunk, pl.nw, err,
                            (int)((test_stall_mask() & STALL_DKDV_TC) != 0));
}

template <int D>
cudaError_t launch_dq_d(const Problem &p, const BwdMaps &m, const void *qhat, const void *dout,
                        const void *out, const float *lse, float *dlt, const RowEpilogue &ep,
                        unsigned int *err, cudaStream_t st) {
    using C = BwdCfg<D>;
    const int n_qt = (p.max_len + kTile - 1) / kTile;
    const long BH = (long)p.units * p.H;
    const long n_items = BH * n_qt;
    if (n_items >= (1L << 31)) return cudaErrorInvalidValue;
    // persistent grid: one CTA per SM walks the items (one CTA fits an SM: 512 TMEM columns)
    const long blocks = std::min<long>(n_items, sm_count());
    CUtensorMap mx, mcs, mdo;
    cudaError_t e = make_epi_maps<D>(p, ep, p.H, 64, mx, mcs);
    if (e != cudaSuccess) return e;
    // dO [B, S, H, D] with 128-row boxes (the owned rows, the dP MMA's A operand)
    RowEpilogue eo = ep;
    eo.x = dout;
    CUtensorMap unused;
    e = make_epi_maps<D>(p, eo, p.H, kTile, mdo, unused);
    if (e != cudaSuccess) return e;
    // the forward output O (L2 prefetch of the rows Dlt reads) and dq (TMA store of the rows)
    CUtensorMap mo, mdq;
    eo.x = out;
    if ((e = make_epi_maps<D>(p, eo, p.H, kTile, mo, unused)) != cudaSuccess) return e;
    eo.x = ep.out;
    if ((e = make_epi_maps<D>(p, eo, p.H, kTile, mdq, unused)) != cudaSuccess) return e;
    // Qhat [B, H, S, D] with 128-row boxes (the owned rows, copied into TMEM)
    CUtensorMap mqh;
    {
        using A = Atoms<D>;
        const uint64_t dims[3] = {D, (uint64_t)p.S, (uint64_t)p.B * p.H};
        const uint64_t strides[2] = {D * 2, (uint64_t)p.S * D * 2};
        const uint32_t box[3] = {(uint32_t)A::kCols, (uint32_t)kTile, 1};
        if ((e = encode_tmap_bf16(&mqh, qhat, 3, dims, strides, box, A::kSwizzleBytes)) !=
            cudaSuccess)
            return e;
    }
    e = cudaFuncSetAttribute(k_bwd_dq_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemB);
    if (e != cudaSuccess) return e;
    return launch_dependent(k_bwd_dq_tc<D>, dim3((unsigned)blocks), dim3(kThreadsBwd), C::kSmemB,
                            st, m.k, m.v, mx, mcs, mdo, mo, mdq, mqh, (const bf16 *)out, lse, dlt,
                            ep.gamma, ep.rstd, (bf16 *)ep.out, ep.part,
                            SeqRows{p.cu, p.S, p.max_len}, p.H, p.G, (int)BH, n_qt, (int)n_items,
                            err, (int)((test_stall_mask() & STALL_DQ_TC) != 0));
}

template <int D>
cudaError_t run_dkdv(const Problem &p, const void *qhat, const void *khat, const void *v,
                     const void *dout, const float *lse, const float *dlt, float *dkhat, void *dv,
                     float *part, const RowEpilogue &ek, unsigned int *err, cudaStream_t st) {
    BwdMaps m;
    cudaError_t e = make_maps<D>(p, qhat, khat, v, dout, m);
    if (e != cudaSuccess) return e;
    return launch_dkdv_d<D>(p, m, lse, dlt, dkhat, dv, part, ek, err, st);
}

template <int D>
cudaError_t run_dq(const Problem &p, const void *qhat, const void *khat, const void *v,
                   const void *dout, const void *out, const float *lse, float *dlt,
                   const RowEpilogue &ep, unsigned int *err, cudaStream_t st) {
    BwdMaps m;
    cudaError_t e = make_maps<D>(p, qhat, khat, v, dout, m);
    if (e != cudaSuccess) return e;
    return launch_dq_d<D>(p, m, qhat, dout, out, lse, dlt, ep, err, st);
}

}  // namespace

size_t dkdv_part_bytes(const Problem &p) { return dkdv_plan(p).part_bytes; }

size_t dk_part_count(const Problem &p) { return (size_t)p.units * p.G * dkdv_plan(p).nw; }

cudaError_t launch_bwd_dkdv_tc(const Problem &p, const void *qhat, const void *khat,
                               const void *v, const void *dout, const float *lse,
                               const float *dlt, float *dkhat, void *dv, float *part,
                               const RowEpilogue &ek, unsigned int *err, cudaStream_t st) {
    if (p.D == 128)
        return run_dkdv<128>(p, qhat, khat, v, dout, lse, dlt, dkhat, dv, part, ek, err, st);
    if (p.D == 64)
        return run_dkdv<64>(p, qhat, khat, v, dout, lse, dlt, dkhat, dv, part, ek, err, st);
    if (p.D == 32)
        return run_dkdv<32>(p, qhat, khat, v, dout, lse, dlt, dkhat, dv, part, ek, err, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_dkdv_reduce(const Problem &p, const float *part, float *dkhat, void *dv,
                               cudaStream_t st) {
    const DkdvPlan pl = dkdv_plan(p);
    if (pl.n_split == 0) return cudaSuccess;
    dim3 grid((unsigned)pl.n_split, (unsigned)((long)p.units * p.G));
    return launch_dependent(k_dkdv_reduce, grid, dim3(256), 0, st, part, dkhat, (bf16 *)dv,
                            SeqRows{p.cu, p.S, p.max_len}, p.H, p.G, p.D, pl.n_kvt, pl.chunk,
                            pl.nw);
}

size_t dq_part_count(const Problem &p) {
    return (size_t)p.units * p.H * ((p.max_len + kTile - 1) / kTile);
}

cudaError_t launch_bwd_dq_tc(const Problem &p, const void *qhat, const void *khat, const void *v,
                             const void *dout, const void *out, const float *lse, float *dlt,
                             const RowEpilogue &ep, unsigned int *err, cudaStream_t st) {
    if (p.D == 128) return run_dq<128>(p, qhat, khat, v, dout, out, lse, dlt, ep, err, st);
    if (p.D == 64) return run_dq<64>(p, qhat, khat, v, dout, out, lse, dlt, ep, err, st);
    if (p.D == 32) return run_dq<32>(p, qhat, khat, v, dout, out, lse, dlt, ep, err, st);
    return cudaErrorInvalidValue;
}

}  // namespace xt
