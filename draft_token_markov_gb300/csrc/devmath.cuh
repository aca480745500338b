// devmath.cuh -- the device's own scalar arithmetic for Markov draft sampling.
//
// Every operation is an explicitly rounded IEEE fp32 intrinsic (__fadd_rn,
// __fmul_rn, __fmaf_rn, __fdiv_rn): no contraction and no fast-math, so each
// function is a fixed sequence of correctly rounded steps whose result does
// not depend on the compiler.  The algorithms:
//   log  -- x = 2^k m, m in [sqrt(1/2), sqrt(2)); s = (m-1)/((m-1)+2);
//           ln m = 2s + 2s R(s^2) with R the odd atanh series through s^12/13
//           (Abramowitz & Stegun 4.1.27); ln x = k ln2_hi + (k ln2_lo + ln m),
//           the two-part ln 2 of fdlibm's single-precision log.
//   exp  -- k = rint(x log2 e), Cody & Waite reduction with the same ln 2
//           split, degree-7 Taylor polynomial, scale by 2^k; x < -87 gives 0.
//   tanh -- |u| < 1/2: Taylor series through u^15; otherwise
//           1 - 2 / (exp(2|u|) + 1); odd.
//   BF16 -- round to nearest, ties to even.
//   splitmix64 -- Steele, Lea & Flood (OOPSLA 2014): golden gamma, then the
//           mix64 finalizer.
// The noise is u = ((h >> 41) + 1/2) 2^-23, gumbel = -log(-log u), with
// h = sm(sm(sm(sm(seed) ^ row) ^ step) ^ v): a counter hash of (seed, row,
// position, vocab id), which the sharded_markov page's _shard_noise_kernel
// docstring requires to depend on seeds and positions only.
#pragma once
#include <cstdint>

namespace dtm {

__device__ __forceinline__ float dm_log_core(float x, int kadj = 0) {
    // x positive, finite and normal; kadj is added to the binary exponent.
    uint32_t t = __float_as_uint(x) + 0x004afb0du;  // 0x3f800000 - 0x3f3504f3
    int k = (int)(t >> 23) - 127 + kadj;
    float m = __uint_as_float((t & 0x007fffffu) + 0x3f3504f3u);
    float f = __fsub_rn(m, 1.0f);
    float s = __fdiv_rn(f, __fadd_rn(f, 2.0f));
    float z = __fmul_rn(s, s);
    float p = 0x1.3b13b2p-4f;
    p = __fmaf_rn(p, z, 0x1.745d18p-4f);
    p = __fmaf_rn(p, z, 0x1.c71c72p-4f);
    p = __fmaf_rn(p, z, 0x1.24924ap-3f);
    p = __fmaf_rn(p, z, 0x1.99999ap-3f);
    p = __fmaf_rn(p, z, 0x1.555556p-2f);
    float R = __fmul_rn(p, z);
    float hs = __fadd_rn(s, s);
    float lnm = __fmaf_rn(hs, R, hs);
    float kf = __int2float_rn(k);
    float lo = __fmaf_rn(kf, 0x1.2fefa2p-17f, lnm);
    return __fmaf_rn(kf, 0x1.62e300p-1f, lo);
}

__device__ __forceinline__ float dm_log(float x) {
    uint32_t ix = __float_as_uint(x);
    if (x != x) return x;
    if ((ix & 0x7fffffffu) == 0u) return __uint_as_float(0xff800000u);
    if (ix & 0x80000000u) return __uint_as_float(0x7fc00000u);
    if (ix == 0x7f800000u) return x;
    if (ix < 0x00800000u) return dm_log_core(__fmul_rn(x, 0x1p23f), -23);  // subnormal
    return dm_log_core(x);
}

__device__ __forceinline__ float dm_exp(float x) {
    if (x != x) return x;
    if (x > 0x1.62e42ep+6f) return __uint_as_float(0x7f800000u);
    if (x < -87.0f) return 0.0f;
    float kf = rintf(__fmul_rn(x, 0x1.715476p+0f));
    float r = __fmaf_rn(-kf, 0x1.62e300p-1f, x);
    r = __fmaf_rn(-kf, 0x1.2fefa2p-17f, r);
    float p = 0x1.a01a02p-13f;
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
    p = __fmaf_rn(p, r, 0x1.111112p-7f);
    p = __fmaf_rn(p, r, 0x1.555556p-5f);
    p = __fmaf_rn(p, r, 0x1.555556p-3f);
    p = __fmaf_rn(p, r, 0x1.000000p-1f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    int k = __float2int_rn(kf);
    if (k > 127) {
        p = __fmul_rn(p, 2.0f);
        k -= 1;
    }
    return __fmul_rn(p, __uint_as_float((uint32_t)(k + 127) << 23));
}

// The inverse-CDF integer weight floor(exp(d) 2^40) of d = fp32(x / T) - M
// for d <= 0 (M the row's maximum of fp32(x / T), finite): dm_exp's steps
// with the 2^40 folded into its final power-of-two scale, and zero below
// d = -28.  Both are exact rewrites: for -28 <= d <= 0, k = rint(d log2 e)
// lies in [-41, 0], so p 2^k and p 2^(k + 40) are normal and the two
// power-of-two products exact; below -28 the exp is under e^-28 (1 + 2^-20)
// < 2^-40, whose scaled floor is 0 (as it is for d = -inf).  The select
// keeps lanes of a warp from diverging.  The integer steps stay on the
// FMA and integer pipes: rint of the rounded product by adding and
// subtracting 1.5 2^23 (for |y| < 2^22 that sum's unit in the last place is
// 1, so it rounds y to the nearest integer, ties to even, and its low bits
// are that integer), and the floor of w = m 2^(e - 23) (m the 24-bit
// significand) by shifting m.
__device__ __forceinline__ uint64_t dm_cdf_weight(float d) {
    const float y = __fmul_rn(d, 0x1.715476p+0f);
    const float t = __fadd_rn(y, 0x1.8p23f);
    const float kf = __fsub_rn(t, 0x1.8p23f);
    float r = __fmaf_rn(-kf, 0x1.62e300p-1f, d);
    r = __fmaf_rn(-kf, 0x1.2fefa2p-17f, r);
    float p = 0x1.a01a02p-13f;
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
    p = __fmaf_rn(p, r, 0x1.111112p-7f);
    p = __fmaf_rn(p, r, 0x1.555556p-5f);
    p = __fmaf_rn(p, r, 0x1.555556p-3f);
    p = __fmaf_rn(p, r, 0x1.000000p-1f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int k = (int)(__float_as_uint(t) - 0x4B400000u);
    const uint32_t wb = __float_as_uint(__fmul_rn(p, __uint_as_float((uint32_t)(k + 167) << 23)));
    // w >= 1/2 here: its biased exponent e >= 126, w = m 2^(e - 150)
    const int sh = (int)(wb >> 23) - 150;
    const uint32_t m = (wb & 0x007fffffu) | 0x00800000u;
    const uint64_t q = sh >= 0 ? (uint64_t)m << (sh & 63) : (uint64_t)(m >> (-sh < 31 ? -sh : 31));
    return d >= -28.0f ? q : 0ull;
}

// fp32(x / T).  For T a positive normal power of two, 1 / T is exact and
// the product x (1 / T) is the same real number as x / T, rounded once: the
// multiply is the division's exact rewrite (kPow2 selects it; rT = 1 / T).
__device__ __forceinline__ bool dm_pow2_temperature(float T) {
    const uint32_t b = __float_as_uint(T);
    return (b & 0x007fffffu) == 0u && (b >> 23) - 1u < 0xfeu;
}
template <bool kPow2>
__device__ __forceinline__ float dm_div_T(float x, float T, float rT) {
    return kPow2 ? __fmul_rn(x, rT) : __fdiv_rn(x, T);
}

__device__ __forceinline__ float dm_tanh(float u) {
    float a = fabsf(u);
    if (a < 0.5f) {
        float z = __fmul_rn(u, u);
        float p = -0x1.7da364p-10f;
        p = __fmaf_rn(p, z, 0x1.d6d3d0p-9f);
        p = __fmaf_rn(p, z, -0x1.226e36p-7f);
        p = __fmaf_rn(p, z, 0x1.664f48p-6f);
        p = __fmaf_rn(p, z, -0x1.ba1ba2p-5f);
        p = __fmaf_rn(p, z, 0x1.111112p-3f);
        p = __fmaf_rn(p, z, -0x1.555556p-2f);
        return __fmaf_rn(u, __fmul_rn(p, z), u);
    }
    float e = dm_exp(__fadd_rn(a, a));
    float t = __fsub_rn(1.0f, __fdiv_rn(2.0f, __fadd_rn(e, 1.0f)));
    return copysignf(t, u);
}

// fp32 -> BF16 bits, round to nearest even; NaN -> quiet NaN.
__device__ __forceinline__ uint32_t dm_bf16_bits(float f) {
    uint32_t x = __float_as_uint(f);
    if ((x & 0x7fffffffu) > 0x7f800000u) return 0x7fc0u;
    x += 0x7fffu + ((x >> 16) & 1u);
    return x >> 16;
}

__device__ __forceinline__ float dm_bf16_f32(uint32_t h) { return __uint_as_float(h << 16); }

__device__ __forceinline__ uint64_t dm_splitmix64(uint64_t x) {
    uint64_t z = x + 0x9e3779b97f4a7c15ull;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t dm_row_step_hash(uint64_t seed, uint32_t row, uint32_t step) {
    return dm_splitmix64(dm_splitmix64(dm_splitmix64(seed) ^ (uint64_t)row) ^ (uint64_t)step);
}

__device__ __forceinline__ uint64_t dm_cdf_hash(uint64_t row_step) {
    return dm_splitmix64(row_step ^ 0x8000000000000000ull);
}

// gumbel = -log(-log u), u = ((h >> 41) + 1/2) 2^-23 (exact, in [2^-24, 1)).
__device__ __forceinline__ float dm_gumbel_from_hash(uint64_t h) {
    uint32_t m = (uint32_t)(h >> 41);
    // 1 + m 2^-23 minus (1 - 2^-24) is exactly (m + 1/2) 2^-23
    float u = __fsub_rn(__uint_as_float(0x3f800000u | m), 0x1.fffffep-1f);
    float w = -dm_log_core(u);            // u in [2^-24, 1): normal, positive
    return -dm_log_core(w);               // w in (0, 17): normal, positive
}

__device__ __forceinline__ float dm_gumbel(uint64_t row_step, uint32_t v) {
    return dm_gumbel_from_hash(dm_splitmix64(row_step ^ (uint64_t)v));
}

}  // namespace dtm
