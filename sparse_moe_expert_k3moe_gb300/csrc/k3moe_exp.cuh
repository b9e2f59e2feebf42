// k3moe_exp.cuh -- exp(x) rounded to the nearest float, from fp32 arithmetic alone.
//
// The router's score is sc = 1/(1+expf(-logit)) in float (kimi-k3-in-c README, Part II,
// section 9, the k3_router listing), and the float rounding of the exponential decides
// near-equal scores.  The fp64 pipe that a double exponential would use is very slow on
// this GPU (about 10 us for one warp-wide call), so the value is built from float
// operations with the error-free transformations of double-float arithmetic
// (Dekker, Knuth; products split exactly with fma):
//   1. x = k ln2 + r, k = rint(x / ln2), |r| <= ~0.35: ln2 is held as three floats (the
//      first with 16 significant bits, so k * ln2_hi is exact for |k| <= 255), and r as an
//      unevaluated pair (rh, rl) good to ~2^-60 absolute;
//   2. exp(r) = sum_{i <= 11} r^i / i!: the terms from r^7 on are below 2^-23 of the sum
//      and are added in float, the rest by a Horner scheme in pairs (1/i! as float pairs);
//      the truncation error is below 2^-42 relative;
//   3. the pair is rounded to float once and scaled by 2^k (exact in the normal range).
// The result is the correctly rounded float except when exp(x) lies within ~2^-40
// (relative) of a rounding tie.  Below x = -103 it returns 0 and above the float range
// +inf (exp(x) there is below the smallest subnormal, or above the largest float).
#pragma once

#include <cmath>
#include <cstdint>
#include <cstring>

namespace k3moe {

#ifdef __CUDA_ARCH__
#define K3_ADD(a, b) __fadd_rn((a), (b))
#define K3_SUB(a, b) __fsub_rn((a), (b))
#define K3_MUL(a, b) __fmul_rn((a), (b))
#define K3_FMA(a, b, c) __fmaf_rn((a), (b), (c))
#else
#define K3_ADD(a, b) ((a) + (b))
#define K3_SUB(a, b) ((a) - (b))
#define K3_MUL(a, b) ((a) * (b))
#define K3_FMA(a, b, c) fmaf((a), (b), (c))
#endif

__host__ __device__ __forceinline__ float bits_to_float(uint32_t u)
{
#ifdef __CUDA_ARCH__
    return __uint_as_float(u);
#else
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
#endif
}

struct DF {
    float h, l;
};

// a + b = s + e exactly.
__host__ __device__ __forceinline__ DF df_two_sum(float a, float b)
{
    const float s = K3_ADD(a, b);
    const float bb = K3_SUB(s, a);
    const float e = K3_ADD(K3_SUB(a, K3_SUB(s, bb)), K3_SUB(b, bb));
    return DF{s, e};
}
// a + b = s + e exactly, given |a| >= |b|.
__host__ __device__ __forceinline__ DF df_fast_two_sum(float a, float b)
{
    const float s = K3_ADD(a, b);
    return DF{s, K3_SUB(b, K3_SUB(s, a))};
}
__host__ __device__ __forceinline__ DF df_mul(DF a, DF b)
{
    const float p = K3_MUL(a.h, b.h);
    float e = K3_FMA(a.h, b.h, -p);
    e = K3_FMA(a.h, b.l, e);
    e = K3_FMA(a.l, b.h, e);
    return df_fast_two_sum(p, e);
}
__host__ __device__ __forceinline__ DF df_add(DF a, DF b)
{
    DF s = df_two_sum(a.h, b.h);
    s.l = K3_ADD(s.l, K3_ADD(a.l, b.l));
    return df_fast_two_sum(s.h, s.l);
}

__host__ __device__ __forceinline__ float exp_rn(float x)
{
    if (x != x) return x;
    if (x > 88.8f) return bits_to_float(0x7F800000u);
    if (x < -103.0f) return 0.0f;
    const float k = rintf(K3_MUL(x, 0x1.715476p+0f));
    // r = x - k ln2 = (x - k ln2_hi) - k ln2_lo - k ln2_lo2; the first difference is exact
    const float ln2_hi = 0x1.62e4p-1f, ln2_lo = 0x1.7f7d1cp-20f, ln2_lo2 = 0x1.ef357ap-45f;
    const float rh0 = K3_SUB(x, K3_MUL(k, ln2_hi));
    const float p2 = K3_MUL(k, ln2_lo);
    const float e2 = K3_FMA(k, ln2_lo, -p2);
    DF r = df_two_sum(rh0, -p2);
    r.l = K3_SUB(K3_SUB(r.l, e2), K3_MUL(k, ln2_lo2));
    r = df_fast_two_sum(r.h, r.l);
    // the float tail: sum_{i=7..11} r^(i-7) / i!
    float t = 0x1.ae6456p-26f;                          // 1/11!
    t = K3_FMA(t, r.h, 0x1.27e4fcp-22f);                // 1/10!
    t = K3_FMA(t, r.h, 0x1.71de3ap-19f);                // 1/9!
    t = K3_FMA(t, r.h, 0x1.a01a02p-16f);                // 1/8!
    t = K3_FMA(t, r.h, 0x1.a01a02p-13f);                // 1/7!
    // pairs: y = y r + 1/i! for i = 6 .. 0
    const DF c[7] = {{1.0f, 0.0f},
                     {1.0f, 0.0f},
                     {0.5f, 0.0f},
                     {0x1.555556p-3f, -0x1.555556p-28f},
                     {0x1.555556p-5f, -0x1.555556p-30f},
                     {0x1.111112p-7f, -0x1.ddddde0p-32f},
                     {0x1.6c16c2p-10f, -0x1.27d27ep-35f}};
    DF y{t, 0.0f};
#pragma unroll
    for (int i = 6; i >= 0; i--) y = df_add(df_mul(y, r), c[i]);
    const float m = K3_ADD(y.h, y.l);
    // 2^k in two exact factors (|k| <= 150)
    const int ki = (int)k, k1 = ki / 2, k2 = ki - k1;
    const float s1 = bits_to_float((uint32_t)(k1 + 127) << 23);
    const float s2 = bits_to_float((uint32_t)(k2 + 127) << 23);
    return K3_MUL(K3_MUL(m, s1), s2);
}

}  // namespace k3moe
