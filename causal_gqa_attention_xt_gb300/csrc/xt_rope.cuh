// xt_rope.cuh -- the RoPE angle of the kernels: cos and sin of
// pos * theta^(-2i/D) (xtrain "Phase T9: Export to xserv", architecture-diff
// table: rotate_half RoPE with freq = theta^(-2i/hd) and pos = token row; Mint
// project report 5.4.1-5.4.2).
//
// The inverse frequency f_i = theta^(-2i/D) is formed on the host in double
// and split into fp32 hi + lo (hi + lo is that double to ~48 bits). For
// positions below 2^21 the product pos * f_i is formed in fp32 with the
// rounding error of pos * hi recovered exactly by an fma, then reduced by 2*pi
// with Cody and Waite's three-constant scheme; beyond 2^21 product and
// reduction are done in double. The reduced angle (|r| <= pi + small, within a
// few fp32 ulps) goes to the fp32 sincosf.
#pragma once

#include <cuda_runtime.h>
#include <math.h>

namespace xt {

constexpr int kRopeMaxHalf = 64;             // D / 2 for D <= 128
constexpr int kRopeFp32Limit = 1 << 21;      // positions with the fp32 angle path

// 2*pi = kRopeC1 + kRopeC2 + kRopeC3 (Cody-Waite): kRopeC1 has 5 significant
// bits, so k * kRopeC1 is exact for |k| < 2^19; the other two carry the rest.
constexpr double kRopeTwoPi = 6.283185307179586476925;
constexpr float kRopeC1 = 6.25f;
constexpr float kRopeC2 = (float)(kRopeTwoPi - 6.25);
constexpr float kRopeC3 = (float)((kRopeTwoPi - 6.25) - (double)kRopeC2);
constexpr float kRopeInvTwoPi = (float)(1.0 / kRopeTwoPi);

struct RopeConsts {
    float fhi[kRopeMaxHalf], flo[kRopeMaxHalf];
    double fd[kRopeMaxHalf];
};

inline RopeConsts make_rope_consts(double theta, int D) {
    RopeConsts f = {};
    for (int i = 0; i < D / 2 && i < kRopeMaxHalf; ++i) {
        const double v = pow(theta, -2.0 * (double)i / (double)D);
        f.fd[i] = v;
        f.fhi[i] = (float)v;
        f.flo[i] = (float)(v - (double)f.fhi[i]);
    }
    return f;
}

// The frequencies of the last (theta, D) this host thread asked for: calls
// with the same model shape skip the D/2 pow() evaluations, which otherwise
// delay the first launch of each call.
inline const RopeConsts &rope_consts(double theta, int D) {
    thread_local double c_theta = -1.0;
    thread_local int c_D = -1;
    thread_local RopeConsts c;
    if (theta != c_theta || D != c_D) {
        c = make_rope_consts(theta, D);
        c_theta = theta;
        c_D = D;
    }
    return c;
}

// (cos, sin) of s * f for f = hi + lo (fd the same frequency in double).
__device__ __forceinline__ float2 rope_cos_sin(int s, float hi, float lo, double fd) {
    float red;
    if (s < kRopeFp32Limit) {
        const float fs = (float)s;   // exact
        const float p = __fmul_rn(fs, hi);
        const float tail = fmaf(fs, lo, fmaf(fs, hi, -p));   // s * f - p
        const float k = rintf(p * kRopeInvTwoPi);
        float r = fmaf(-k, kRopeC1, p);   // exact
        r = fmaf(-k, kRopeC2, r);
        red = __fadd_rn(r, fmaf(-k, kRopeC3, tail));
    } else {
        const double ang = (double)s * fd;
        red = (float)fma(-rint(ang * (1.0 / kRopeTwoPi)), kRopeTwoPi, ang);
    }
    float sv, cv;
    sincosf(red, &sv, &cv);
    return make_float2(cv, sv);
}

}  // namespace xt
