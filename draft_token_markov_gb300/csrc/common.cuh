// common.cuh -- device helpers shared by the Markov sampling kernels.
#pragma once
#include <cstdint>

#include "devmath.cuh"
#include "internal.h"

namespace dtm {

// ------------------------------------------------------------------ PTX

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add_u32(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_cg_u64(const uint64_t *p) {
    return (uint64_t)__ldcg((const unsigned long long *)p);
}

// Record the first device error: status word = code, plus where it
// happened.  Never traps.
__device__ __forceinline__ void set_status(uint32_t *status, uint32_t code, uint32_t where) {
    if (atomicCAS(status, 0u, code) == 0u) atomicExch(status + 1, where);
}

// --------------------------------------------------------------- keys

// Order-preserving map of a key to uint32: NaN (any payload) maps above
// +inf so that the lowest NaN id wins the maximum; -0 maps to +0.
__device__ __forceinline__ uint32_t ordered_key(float k) {
    uint32_t b = __float_as_uint(k);
    b = (b == 0x80000000u) ? 0u : b;                           // -0 == +0
    const uint32_t o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((b & 0x7fffffffu) > 0x7f800000u) ? 0xffffffffu : o;   // NaN above all
}

__device__ __forceinline__ float key_from_ordered(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// (ordered key, id) packed so that the u64 maximum is the largest key and,
// among equal keys, the lowest id (the torch.argmax order).
__device__ __forceinline__ uint64_t pack_key(float k, uint32_t v) {
    return ((uint64_t)ordered_key(k) << 32) | (uint64_t)(0xffffffffu - v);
}

__device__ __forceinline__ uint32_t packed_id(uint64_t p) {
    return 0xffffffffu - (uint32_t)(p & 0xffffffffu);
}

__device__ __forceinline__ uint32_t packed_ordered(uint64_t p) { return (uint32_t)(p >> 32); }

// ---------------------------------------------------------- epilogue

// The cached logit of one element, as an fp32 value, from its base logit
// and its fp32 bias sum: bias = bf16(sum); s = f32(base) + f32(bias) in
// fp32, rounded to BF16 for a BF16 cache; with a transform y = s * mult,
// then cap * tanh(y * inv_cap) when capped, rounded to BF16 for a BF16
// cache.  (sharded_markov page, "Per call" diagram: cache_round(base +
// bf16(head . embed)), its chain compiled for BF16 or fp32 base logits and
// caches; muse_spark markov page, fused_markov_params: the output-logit
// transform in the epilogue, multiplier and cap rounded to fp32.  For an
// fp32 cache the transform's fp32 steps are a reading: the pages give the
// transform for BF16 caches only.)
__device__ __forceinline__ float logit_value(float base, float bias_sum, const Transform &tf,
                                             bool cache_f32) {
    float s = __fadd_rn(base, dm_bf16_f32(dm_bf16_bits(bias_sum)));
    if (!cache_f32) s = dm_bf16_f32(dm_bf16_bits(s));
    if (!tf.has_transform) return s;
    float y = __fmul_rn(s, tf.mult);
    if (tf.has_cap) y = __fmul_rn(tf.cap, dm_tanh(__fmul_rn(y, tf.inv_cap)));
    return cache_f32 ? y : dm_bf16_f32(dm_bf16_bits(y));
}

// Base logit (row, position i, id v) as fp32, from a BF16 or an fp32 base.
__device__ __forceinline__ float base_value(const SampleArgs &a, int row, int i, int v) {
    const int64_t o = row * a.base_s0 + (int64_t)i * a.base_s1 + v;
    return a.base_f ? a.base_f[o] : dm_bf16_f32(a.base[o]);
}

// Cache element (row, i, v) as fp32 (a BF16 cache's values are exact in fp32).
__device__ __forceinline__ float cache_value(const SampleArgs &a, int row, int i, int v) {
    const int64_t o = row * a.cache_s0 + (int64_t)i * a.cache_s1 + v;
    return a.cache_f ? a.cache_f[o] : dm_bf16_f32(a.cache[o]);
}

// Store a logit from logit_value into the cache (for a BF16 cache the value
// is a BF16 value: its top 16 bits).
__device__ __forceinline__ void cache_put(const SampleArgs &a, int row, int i, int v, float l) {
    const int64_t o = row * a.cache_s0 + (int64_t)i * a.cache_s1 + v;
    if (a.cache_f)
        a.cache_f[o] = l;
    else
        a.cache[o] = (uint16_t)(__float_as_uint(l) >> 16);
}

// Two fp32 values rounded to BF16 (nearest, ties to even) in one
// instruction: lo in bits 0-15, hi in bits 16-31.  A NaN becomes a NaN
// (the hardware's canonical one, not necessarily 0x7FC0).
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Whether a temperature samples (T > 0); 0, negatives and NaN are greedy.
__device__ __forceinline__ bool samples(float T) { return T > 0.0f; }

// ----------------------------------------------------- grid barrier

// A bounded grid-wide barrier for a co-resident (cooperative) grid.  The
// counter only grows: barrier number `epoch` (1-based) of a launch completes
// when the counter reaches base + epoch * gridDim.x.  Gives up after
// timeout_ns (device status MARKOV_ETIMEOUT) or as soon as another CTA has
// recorded an error; returns false then, and the caller must return.
__device__ __forceinline__ bool grid_barrier(uint32_t *count, uint32_t target, uint32_t *status,
                                             uint64_t timeout_ns, uint32_t where,
                                             uint32_t *smem_flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        red_release_add_u32(count, 1u);
        uint32_t ok = 1u;
        uint64_t t0 = globaltimer_ns();
        uint32_t spins = 0;
        while ((int32_t)(ld_acquire_u32(count) - target) < 0) {
            if ((++spins & 63u) == 0u) {
                if (ld_acquire_u32(status) != 0u) { ok = 0u; break; }
                if (globaltimer_ns() - t0 > timeout_ns || spins > (1u << 30)) {
                    set_status(status, 4u /* MARKOV_ETIMEOUT */, where);
                    ok = 0u;
                    break;
                }
            }
        }
        __threadfence();
        *smem_flag = ok;
    }
    __syncthreads();
    return *smem_flag != 0u;
}

}  // namespace dtm
