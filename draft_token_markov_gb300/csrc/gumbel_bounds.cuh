// gumbel_bounds.cuh -- cheap bounds on the Gumbel noise and on Gumbel keys,
// used to prune the exact key computation in the persistent chain.
//
// The Gumbel-max token of a position is the lowest id of the largest key
// fp32(l / T) + gumbel(u), u drawn by the counter hash (sharded_markov page,
// module docstring: Gumbel-max over the cached logits; _shard_noise_kernel:
// noise from seeds and positions).  Only ids whose key can reach the largest
// key need the exact (own-log) noise.  One byte per (position, id, row)
// stores q = ceil((g_up + 4) 12) for an upper bound g_up on the noise, from
// which an upper and a lower bound on the exact noise follow; a key's
// bounds add the logit term with a relative margin.  Every bound is checked
// on the device over all 2^23 values u can take.
#pragma once
#include <cstdint>

#include "devmath.cuh"

namespace dtm {

// One byte per (position, id, row) holding an upper bound on the Gumbel
// value: q = ceil((bound + 4) * 12).  Every value the hash can give lies in
// (-2.8, 16.7), so q fits a byte; q / 12 - 4 >= bound >= the exact value.
__device__ __forceinline__ uint32_t quantize_upper(float g_up) {
    const float t = ceilf(__fmul_rn(__fadd_rn(g_up, 4.0f), 12.0f));
    return t < 0.0f ? 0u : (t > 255.0f ? 255u : (uint32_t)t);
}
__device__ __forceinline__ float dequantize_upper(uint32_t q) {
    return __fmaf_rn((float)q, 1.0f / 12.0f, -4.0f) + 0.001f;
}
// A lower bound on the Gumbel value from the same byte: the fast estimate
// lies within 2e-4 of the exact value and q - 1 < (estimate + 0.01 + 4) 12,
// so the value exceeds (q - 1) / 12 - 4 - 0.0103.
__device__ __forceinline__ float dequantize_lower(uint32_t q) {
    return __fmaf_rn((float)q, 1.0f / 12.0f, -4.0f - 1.0f / 12.0f - 0.02f);
}

// An upper bound on gumbel = -log(-log u) for the u of hash h.  w = -ln u
// from the hardware log2 (absolute error <= 2^-22 on [1/2, 2), 2 ulp
// elsewhere) while u <= 0.999, where w >= 1e-3 keeps its relative error
// below 2e-4; above, the series d + d^2/2 + d^3/3 of -ln(1 - d), d = 1 - u
// (exact) <= 1e-3.  Then -ln w adds at most ~3e-6, so the estimate is within
// 2e-4 of the exact value and the 0.01 margin makes it a bound.
__device__ __forceinline__ float gumbel_upper(uint64_t h) {
    const uint32_t m = (uint32_t)(h >> 41);
    const float u = __fsub_rn(__uint_as_float(0x3f800000u | m), 0x1.fffffep-1f);
    const float d = __fsub_rn(1.0f, u);
    const float ws = d * (1.0f + d * (0.5f + d * (1.0f / 3.0f)));
    const float wl = -__log2f(u) * 0.6931472f;
    const float w = u > 0.999f ? ws : wl;
    return -__log2f(w) * 0.6931472f + 0.01f;
}

// A lower bound on the Gumbel key of an id from its cached logit lf, 1 / T
// (rounded) and its noise byte: lf * invT is within two roundings of
// fp32(lf / T), far inside the 1e-5 relative margin, and the noise byte's
// lower end is below the exact noise; rounding the sum is monotone.  NaN
// when lf * invT is +inf (no bound: it never raises a threshold).
__device__ __forceinline__ float key_lower(float lf, float invT, uint32_t qb) {
    const float xa = lf * invT;
    return __fadd_rn(__fmaf_rn(fabsf(xa), -1e-5f, xa), dequantize_lower(qb));
}

// An upper bound on the Gumbel key of an id, as key_lower with the margin
// the other way.  NaN when lf * invT is -inf (treated as "may win").
__device__ __forceinline__ float key_upper(float lf, float invT, uint32_t qb) {
    const float xa = lf * invT;
    return __fadd_rn(__fmaf_rn(fabsf(xa), 1e-5f, xa), dequantize_upper(qb));
}

// The exact Gumbel key fp32(l / T) + gumbel of one id, given its hash.
__device__ __forceinline__ float exact_key(float l, float T, uint64_t h) {
    const float x = (T == 1.0f) ? l : __fdiv_rn(l, T);
    return __fadd_rn(x, dm_gumbel_from_hash(h));
}

}  // namespace dtm
