// xt_common.cuh -- small device helpers shared by the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace xt {

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// 16-byte vector of T: 4 floats or 8 bf16.
template <typename T> struct Vec16 {
    static constexpr int N = 16 / sizeof(T);
    uint4 raw;
};

template <typename T>
__device__ __forceinline__ void load16(const T *p, float *dst) {
    uint4 r = *reinterpret_cast<const uint4 *>(p);
    if constexpr (sizeof(T) == 4) {
        dst[0] = __uint_as_float(r.x); dst[1] = __uint_as_float(r.y);
        dst[2] = __uint_as_float(r.z); dst[3] = __uint_as_float(r.w);
    } else {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            dst[2 * i] = __uint_as_float(w[i] << 16);
            dst[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
}

template <typename T>
__device__ __forceinline__ void store16(T *p, const float *src) {
    uint4 r;
    if constexpr (sizeof(T) == 4) {
        r.x = __float_as_uint(src[0]); r.y = __float_as_uint(src[1]);
        r.z = __float_as_uint(src[2]); r.w = __float_as_uint(src[3]);
    } else {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(src[2 * i], src[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        r.x = w[0]; r.y = w[1]; r.z = w[2]; r.w = w[3];
    }
    *reinterpret_cast<uint4 *>(p) = r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Sum over an aligned group of `width` lanes (width a power of two <= 32).
__device__ __forceinline__ float group_sum(float v, int width) {
    for (int o = width >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Work item of a persistent CTA in round k: rounds walk the CTAs forwards and
// backwards in turn ("snake"), so that with items sorted longest first every
// CTA gets a long and a short item of each pair of rounds (a plain stride gives
// CTA 0 the longest item of every round: 5-14% slower at the bench shapes).
__device__ __forceinline__ int snake_item(int k) {
    const int c = (k & 1) ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
    return k * (int)gridDim.x + c;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Rows of the attention kernels. A unit is either a batch element b (plane b
// of the [B, ..., S, ...] tensors, rows 0..S-1) or, for a packed batch (cu set;
// Mint report 8.2: samples flattened into one [total] row dimension), a sample
// u on rows cu[u]..cu[u+1]-1 of plane 0 of tensors whose row count S is the
// total. Causal masking inside the unit is then the block-causal mask: a
// unit's tiles never start before its first row, and rows past its end are
// only visible to query rows past its end, which are not stored.
struct SeqRows {
    const int *cu;   // [units + 1] row offsets (device), or nullptr
    int S;           // rows per plane
    int max_len;     // longest unit: S, or the packed batch's longest sample
};
struct SeqSpan {
    int plane, start, len;
};
// Offsets out of order or out of range are clamped into [0, S] (with a
// length of at most max_len), so every access stays inside the tensors; the
// library's offset check reports them.
__device__ __forceinline__ SeqSpan seq_span(const SeqRows &sr, int u) {
    if (sr.cu == nullptr) return SeqSpan{u, 0, sr.S};
    const int s0 = min(max(sr.cu[u], 0), sr.S);
    const int s1 = min(max(sr.cu[u + 1], s0), min(sr.S, s0 + sr.max_len));
    return SeqSpan{0, s0, s1 - s0};
}

// Programmatic dependent launch (kernels launched with launch_dependent): lets
// the next kernel on the stream be scheduled (its CTAs take SMs as they free up
// and run their set-up), then waits until the earlier grids on the stream have
// completed and their writes are visible. Every thread calls it before its
// first global-memory access; in a kernel launched the ordinary way it returns
// at once.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace xt
