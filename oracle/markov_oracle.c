/*
 * markov_oracle.c -- plain CPU oracle for DSpark sequential Markov sampling
 * of draft tokens.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * Sources (the three documentation pages the method is taken from):
 *   [sharded]  "vllm.models.deepseek_v41.nvidia.specialized_decode.sampling.
 *               sharded_markov" -- module docstring, _shard_noise_kernel,
 *               DSparkShardedMarkovSampler.sample / fork_noise.
 *   [fused]    "vllm.models.deepseek_v41.nvidia.ops.fused_markov" -- module
 *               docstring, FusedMarkovSampler.
 *   [muse]     "vllm.models.muse_spark.nvidia.specialized_decode.runtime.
 *               markov" -- module docstring, FusedMarkovParams,
 *               fused_markov_params, MarkovSampler.sample.
 *
 * What is computed, for every request row b whose request-state index is
 * >= 0 (padding rows, index < 0, are inert: nothing is written) and every
 * draft position i = 0 .. N-1, with p = the anchor token at i = 0 and the
 * previous position's token afterwards ([sharded] module docstring, "Per
 * call" diagram; [muse] MarkovSampler.sample, markov_embeds[i+1]):
 *
 *   bias[v]  = bf16( sum_k f32(head[v,k]) * f32(embed[p,k]) )   fp32, k order
 *   s[v]     = bf16( f32(base[b,i,v]) + f32(bias[v]) )          ("cache_round")
 *   l[v]     = bf16( transform(f32(s[v])) )                     ([muse] epilogue)
 *              transform(y) = y * mult, then cap * tanh(y * inv_cap) if capped
 *   cache[b,i,v] = l[v]
 *   token    = Gumbel-max of l/T + gumbel, or inverse CDF of softmax(l/T),
 *              or argmax at T = 0, NaN rule first ([muse] docstring,
 *              [fused] docstring)
 *
 * The noise is the counter-based splitmix64 hash of (seed, row, step, vocab
 * id) mapped to u in (0,1) and gumbel = -log(-log u); the pages leave their
 * own hash undefined, so this composition is a stated reading.
 *
 * All floating point is fp32 with IEEE round-to-nearest, compiled with
 * -ffp-contract=off; every fused multiply-add is an explicit fmaf.  log, exp
 * and tanh are this file's own, written from the textbook methods named at
 * each function, so that results do not depend on the host's libm.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_GUMBEL 0
#define ORC_INVCDF 1

/* ------------------------------------------------------------------ bits */

static inline uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static inline float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* fp32 -> bf16, IEEE round to nearest, ties to even.  NaN becomes the quiet
 * NaN 0x7FC0.  ([sharded] docstring: logits are rounded to BF16.) */
uint16_t orc_bf16_rne(float f)
{
    uint32_t x = f2u(f);
    if ((x & 0x7fffffffu) > 0x7f800000u) return (uint16_t)0x7fc0u;
    uint32_t lsb = (x >> 16) & 1u;
    x += 0x7fffu + lsb;
    return (uint16_t)(x >> 16);
}

float orc_bf16_to_f32(uint16_t h) { return u2f((uint32_t)h << 16); }

/* ------------------------------------------------------------ own math */

/* Natural log.  Reduce x = 2^k * m with m in [sqrt(1/2), sqrt(2)); with
 * f = m - 1 (exact) and s = f / (f + 2), ln m = 2 atanh(s) = 2s + 2s R(s^2),
 * R(z) = z/3 + z^2/5 + ... + z^6/13 (the odd atanh series, Abramowitz &
 * Stegun 4.1.27); ln x = k ln2_hi + (k ln2_lo + ln m) with the Cody & Waite
 * two-part ln 2 of fdlibm's single-precision log. */
float orc_log(float x)
{
    uint32_t ix = f2u(x);
    if (x != x) return x;
    if (ix == 0u || ix == 0x80000000u) return -INFINITY;
    if (ix & 0x80000000u) return NAN;
    if (ix == 0x7f800000u) return x;
    int ksub = 0;
    if (ix < 0x00800000u) {            /* subnormal: scale into the normals */
        x = x * 0x1p23f;
        ix = f2u(x);
        ksub = -23;
    }
    uint32_t t = ix + (0x3f800000u - 0x3f3504f3u);
    int k = (int)(t >> 23) - 127 + ksub;
    float m = u2f((t & 0x007fffffu) + 0x3f3504f3u);
    float f = m - 1.0f;
    float s = f / (f + 2.0f);
    float z = s * s;
    float p = 0x1.3b13b2p-4f;          /* 1/13 */
    p = fmaf(p, z, 0x1.745d18p-4f);    /* 1/11 */
    p = fmaf(p, z, 0x1.c71c72p-4f);    /* 1/9  */
    p = fmaf(p, z, 0x1.24924ap-3f);    /* 1/7  */
    p = fmaf(p, z, 0x1.99999ap-3f);    /* 1/5  */
    p = fmaf(p, z, 0x1.555556p-2f);    /* 1/3  */
    float R = p * z;
    float hs = s + s;
    float lnm = fmaf(hs, R, hs);
    float kf = (float)k;
    float lo = fmaf(kf, 0x1.2fefa2p-17f, lnm);   /* ln2_lo */
    return fmaf(kf, 0x1.62e300p-1f, lo);         /* ln2_hi */
}

/* Exponential.  k = rint(x log2 e); r = x - k ln2_hi - k ln2_lo (Cody &
 * Waite 1980); e^r by its degree-7 Taylor polynomial in Horner form; the
 * result is scaled by 2^k.  Results below e^-87 are flushed to zero (no
 * caller uses them: they are far below every weight that matters). */
float orc_exp(float x)
{
    if (x != x) return x;
    if (x > 0x1.62e42ep+6f) return INFINITY;
    if (x < -87.0f) return 0.0f;
    float kf = rintf(x * 0x1.715476p+0f);
    float r = fmaf(-kf, 0x1.62e300p-1f, x);
    r = fmaf(-kf, 0x1.2fefa2p-17f, r);
    float p = 0x1.a01a02p-13f;         /* 1/7! */
    p = fmaf(p, r, 0x1.6c16c2p-10f);   /* 1/6! */
    p = fmaf(p, r, 0x1.111112p-7f);    /* 1/5! */
    p = fmaf(p, r, 0x1.555556p-5f);    /* 1/4! */
    p = fmaf(p, r, 0x1.555556p-3f);    /* 1/3! */
    p = fmaf(p, r, 0x1.000000p-1f);    /* 1/2! */
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    int k = (int)kf;
    if (k > 127) {
        p = p * 2.0f;
        k -= 1;
    }
    return p * u2f((uint32_t)(k + 127) << 23);
}

/* Hyperbolic tangent.  |u| < 1/2: the Taylor series of tanh through u^15
 * (coefficients from the Bernoulli numbers: 1, -1/3, 2/15, -17/315, 62/2835,
 * -1382/155925, 21844/6081075, -929569/638512875); otherwise
 * 1 - 2 / (e^{2|u|} + 1) with this file's exp.  Odd in u. */
float orc_tanh(float u)
{
    float a = fabsf(u);
    float t;
    if (a < 0.5f) {
        float z = u * u;
        float p = -0x1.7da364p-10f;
        p = fmaf(p, z, 0x1.d6d3d0p-9f);
        p = fmaf(p, z, -0x1.226e36p-7f);
        p = fmaf(p, z, 0x1.664f48p-6f);
        p = fmaf(p, z, -0x1.ba1ba2p-5f);
        p = fmaf(p, z, 0x1.111112p-3f);
        p = fmaf(p, z, -0x1.555556p-2f);
        return fmaf(u, p * z, u);
    }
    float e = orc_exp(a + a);
    t = 1.0f - 2.0f / (e + 1.0f);
    return copysignf(t, u);
}

/* --------------------------------------------------------------- noise */

/* splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014): add the golden gamma, then the mix64 finalizer
 * (xor-shift 30, multiply, xor-shift 27, multiply, xor-shift 31). */
uint64_t orc_splitmix64(uint64_t x)
{
    uint64_t z = x + 0x9e3779b97f4a7c15ull;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

/* Hash of one (row, step): sm(sm(sm(seed) ^ row) ^ step).  The noise
 * depends on the seed and the position only, never on the chain ([sharded]
 * fork_noise docstring). */
uint64_t orc_row_step_hash(uint64_t seed, uint32_t row, uint32_t step)
{
    return orc_splitmix64(orc_splitmix64(orc_splitmix64(seed) ^ (uint64_t)row) ^
                          (uint64_t)step);
}

/* u = ((h >> 41) + 1/2) 2^-23 in [2^-24, 1 - 2^-24], exactly. */
float orc_uniform(uint64_t h)
{
    uint32_t m = (uint32_t)(h >> 41);
    return ((float)m + 0.5f) * 0x1p-23f;
}

/* Gumbel noise of vocab id v at (seed, row, step): -log(-log u). */
float orc_gumbel(uint64_t seed, uint32_t row, uint32_t step, uint32_t v)
{
    uint64_t h = orc_splitmix64(orc_row_step_hash(seed, row, step) ^ (uint64_t)v);
    float u = orc_uniform(h);
    return -orc_log(-orc_log(u));
}

/* The inverse-CDF target hash of (row, step): salted with the top bit,
 * which no vocab id can set. */
uint64_t orc_cdf_hash(uint64_t seed, uint32_t row, uint32_t step)
{
    return orc_splitmix64(orc_row_step_hash(seed, row, step) ^ 0x8000000000000000ull);
}

/* ----------------------------------------------------- one position's math */

/* bias = bf16(sum_k f32(head[v,k]) * f32(e[k])), fp32, sequential in k.
 * The BF16 x BF16 product is exact in fp32, so the only rounding is the
 * running sum's. */
uint16_t orc_bias(const uint16_t *head_row, const uint16_t *e, int r)
{
    float acc = 0.0f;
    for (int k = 0; k < r; ++k)
        acc = acc + orc_bf16_to_f32(head_row[k]) * orc_bf16_to_f32(e[k]);
    return orc_bf16_rne(acc);
}

/* The cached logit from the base logit and the bias, both BF16 bits:
 * s = bf16(f32(base) + f32(bias)), then, when the draft has an output
 * transform, l = bf16(cap * tanh((f32(s) * mult) * inv_cap)) (capped) or
 * bf16(f32(s) * mult).  inv_cap = fp32(1) / fp32(cap) ([muse]
 * FusedMarkovParams, fused_markov_params).  Without a transform l = s. */
uint16_t orc_logit(uint16_t base, uint16_t bias, int has_transform, float mult,
                   int has_cap, float cap, float inv_cap)
{
    uint16_t s = orc_bf16_rne(orc_bf16_to_f32(base) + orc_bf16_to_f32(bias));
    if (!has_transform) return s;
    float y = orc_bf16_to_f32(s) * mult;
    if (has_cap) y = cap * orc_tanh(y * inv_cap);
    return orc_bf16_rne(y);
}

/* The cached logit for either cache dtype, as an fp32 value.  The sharded
 * page's chain takes BF16 or fp32 base logits and caches ([sharded]
 * DSparkShardedMarkovSampler set-up, _kernel: base and cache dtypes) and
 * rounds to the cache's dtype ("cache_round" in the module docstring):
 *   s = f32(base) + f32(bias)            fp32 sum
 *   BF16 cache: s = bf16(s), then the transform and bf16 as orc_logit;
 *   fp32 cache: no BF16 rounding; the transform (a reading: the same fp32
 *               steps, as the pages give the transform only for BF16
 *               caches) and l = its fp32 result.
 * With a BF16 base and a BF16 cache this is orc_logit's value. */
float orc_logit_typed(float base, uint16_t bias, int cache_f32, int has_transform, float mult,
                      int has_cap, float cap, float inv_cap)
{
    float s = base + orc_bf16_to_f32(bias);
    if (!cache_f32) s = orc_bf16_to_f32(orc_bf16_rne(s));
    if (!has_transform) return s;
    float y = s * mult;
    if (has_cap) y = cap * orc_tanh(y * inv_cap);
    return cache_f32 ? y : orc_bf16_to_f32(orc_bf16_rne(y));
}

/* Gumbel key of one cached logit: fp32(l / T) + gumbel (T > 0). */
float orc_gumbel_key(uint16_t l, float T, uint64_t seed, uint32_t row, uint32_t step,
                     uint32_t v)
{
    return orc_bf16_to_f32(l) / T + orc_gumbel(seed, row, step, v);
}

/* Whether the row samples greedily: T = 0, and, as a reading, any T that is
 * not > 0 (negative or NaN). */
static int greedy_temperature(float T) { return !(T > 0.0f); }

/* The key of id v at one position: l at T = 0 (greedy), fp32(l / T) in
 * inverse-CDF mode, fp32(l / T) + gumbel in Gumbel mode. */
static float position_key(const float *l, int v, float T, int mode, uint64_t seed,
                          uint32_t row, uint32_t step)
{
    if (greedy_temperature(T)) return l[v];
    if (mode == ORC_INVCDF) return l[v] / T;
    return l[v] / T + orc_gumbel(seed, row, step, (uint32_t)v);
}

/* Select the token of one position from its cached logits l[0..V-1] (fp32
 * values; a BF16 cache's values are exact in fp32).
 *   NaN rule: the lowest id whose key (the noised logit) is NaN ([muse]
 *   docstring); applied in every mode, a reading.
 *   T = 0: the lowest id of max l (the torch.argmax order).
 *   Gumbel: the lowest id of max (fp32(l/T) + gumbel).
 *   Inverse CDF: x = fp32(l/T), M = max x; M = +inf picks the lowest +inf
 *   id, an all -inf row picks id 0; otherwise the weights
 *   q = floor(exp(fp32(x - M)) 2^40) are summed exactly as integers and the
 *   token is the smallest j whose prefix sum exceeds mulhi64(H, S).
 * Returns the token; *k1 / *k2 receive the winning and runner-up keys (NaN
 * when the NaN rule decided). */
int64_t orc_select_f(const float *l, int V, float T, int mode, uint64_t seed, uint32_t row,
                     uint32_t step, float *k1, float *k2)
{
    float best = -INFINITY, second = -INFINITY;
    int64_t arg = -1;
    for (int v = 0; v < V; ++v) {
        float key = position_key(l, v, T, mode, seed, row, step);
        if (key != key) {
            if (k1) *k1 = NAN;
            if (k2) *k2 = NAN;
            return v;
        }
        if (arg < 0 || key > best) {
            if (arg >= 0) second = best;
            best = key;
            arg = v;
        } else if (key > second) {
            second = key;
        }
    }
    if (k1) *k1 = best;
    if (k2) *k2 = second;
    if (greedy_temperature(T) || mode == ORC_GUMBEL) return arg;
    /* inverse CDF; best is M */
    float M = best;
    if (M == INFINITY) return arg;             /* the lowest +inf id */
    if (M == -INFINITY) return 0;              /* every weight is zero */
    uint64_t S = 0;
    for (int v = 0; v < V; ++v) {
        float w = orc_exp(l[v] / T - M);
        S += (uint64_t)(w * 0x1p40f);          /* exact scale, then truncation */
    }
    uint64_t H = orc_cdf_hash(seed, row, step);
    uint64_t t = (uint64_t)(((unsigned __int128)H * (unsigned __int128)S) >> 64);
    uint64_t prefix = 0;
    for (int v = 0; v < V; ++v) {
        float w = orc_exp(l[v] / T - M);
        prefix += (uint64_t)(w * 0x1p40f);
        if (prefix > t) return v;
    }
    return V - 1;                              /* unreachable: prefix(V-1) = S > t */
}

/* orc_select_f on a BF16 cache row (raw bits). */
int64_t orc_select(const uint16_t *l, int V, float T, int mode, uint64_t seed,
                   uint32_t row, uint32_t step, float *k1, float *k2)
{
    float *lf = (float *)malloc((size_t)(V > 0 ? V : 1) * sizeof(float));
    if (!lf) return -1;
    for (int v = 0; v < V; ++v) lf[v] = orc_bf16_to_f32(l[v]);
    int64_t tok = orc_select_f(lf, V, T, mode, seed, row, step, k1, k2);
    free(lf);
    return tok;
}

/* -------------------------------------------------------------- the chain */

/* Run the chain for `rows` request rows.  base[b, i, v] is at
 * base[b*base_s0 + i*base_s1 + v], BF16 bits (base_f32 == 0) or fp32; the
 * cache likewise with cache_s0 / cache_s1 and cache_f32; head and embed are
 * BF16 bits; tokens at tokens[b*tok_s0 + i].  start_step / start_prev (both
 * NULL, or both [rows]) restart row b at position start_step[b] with
 * previous token start_prev[b], leaving earlier positions untouched: the
 * acceptance check uses this to continue a row from a token the GPU drew.
 * has_cap == 0 means no soft cap; has_transform == 0 means l = s.  Returns
 * 0, or -1 on a bad argument (an anchor or previous token out of range). */
int orc_chain_typed(int V, int r, int N, int rows, const void *base, int base_f32,
                    int64_t base_s0, int64_t base_s1, const uint16_t *head, const uint16_t *embed,
                    const int32_t *anchor, const float *temperature, const int64_t *seeds,
                    const int64_t *row_state_idx, int mode, int has_transform, float mult,
                    int has_cap, float cap, int64_t *tokens, int64_t tok_s0, void *cache,
                    int cache_f32, int64_t cache_s0, int64_t cache_s1, const int32_t *start_step,
                    const int64_t *start_prev, int nthreads)
{
    float inv_cap = has_cap ? 1.0f / cap : 1.0f;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    float *lrow = (float *)malloc((size_t)(V > 0 ? V : 1) * sizeof(float));
    if (!lrow) return -1;
    for (int b = 0; b < rows; ++b) {
        if (row_state_idx[b] < 0) continue;           /* padding rows are inert */
        int i0 = start_step ? start_step[b] : 0;
        int64_t p = start_prev ? start_prev[b] : (int64_t)anchor[b];
        if (p < 0 || p >= V) { free(lrow); return -1; }
        for (int i = i0; i < N; ++i) {
            const uint16_t *e = embed + (size_t)p * (size_t)r;
            const int64_t bo = b * base_s0 + i * base_s1, co = b * cache_s0 + i * cache_s1;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
            for (int v = 0; v < V; ++v) {
                uint16_t bv = orc_bias(head + (size_t)v * (size_t)r, e, r);
                float bf = base_f32 ? ((const float *)base)[bo + v]
                                    : orc_bf16_to_f32(((const uint16_t *)base)[bo + v]);
                float l = orc_logit_typed(bf, bv, cache_f32, has_transform, mult, has_cap, cap,
                                          inv_cap);
                lrow[v] = l;
                if (cache_f32) ((float *)cache)[co + v] = l;
                else ((uint16_t *)cache)[co + v] = orc_bf16_rne(l);
            }
            int64_t tok = orc_select_f(lrow, V, temperature[b], mode, (uint64_t)seeds[b],
                                       (uint32_t)b, (uint32_t)i, NULL, NULL);
            tokens[b * tok_s0 + i] = tok;
            p = tok;
        }
    }
    free(lrow);
    return 0;
}

/* orc_chain_typed with a BF16 base and a BF16 cache (raw bits). */
int orc_chain(int V, int r, int N, int rows, const uint16_t *base, int64_t base_s0,
              int64_t base_s1, const uint16_t *head, const uint16_t *embed,
              const int32_t *anchor, const float *temperature, const int64_t *seeds,
              const int64_t *row_state_idx, int mode, int has_transform, float mult,
              int has_cap, float cap, int64_t *tokens, int64_t tok_s0, uint16_t *cache,
              int64_t cache_s0, int64_t cache_s1, const int32_t *start_step,
              const int64_t *start_prev, int nthreads)
{
    return orc_chain_typed(V, r, N, rows, base, 0, base_s0, base_s1, head, embed, anchor,
                           temperature, seeds, row_state_idx, mode, has_transform, mult, has_cap,
                           cap, tokens, tok_s0, cache, 0, cache_s0, cache_s1, start_step,
                           start_prev, nthreads);
}

/* ------------------------------------------------------- array helpers */
/* Element-wise wrappers so tests can evaluate the pieces over arrays. */

void orc_bf16_rne_n(const float *x, uint16_t *y, int64_t n)
{
    for (int64_t j = 0; j < n; ++j) y[j] = orc_bf16_rne(x[j]);
}
void orc_log_n(const float *x, float *y, int64_t n)
{
    for (int64_t j = 0; j < n; ++j) y[j] = orc_log(x[j]);
}
void orc_exp_n(const float *x, float *y, int64_t n)
{
    for (int64_t j = 0; j < n; ++j) y[j] = orc_exp(x[j]);
}
void orc_tanh_n(const float *x, float *y, int64_t n)
{
    for (int64_t j = 0; j < n; ++j) y[j] = orc_tanh(x[j]);
}
void orc_splitmix64_n(const uint64_t *x, uint64_t *y, int64_t n)
{
    for (int64_t j = 0; j < n; ++j) y[j] = orc_splitmix64(x[j]);
}
/* Gumbel noise of ids v0 .. v0+n-1 at one (seed, row, step). */
void orc_gumbel_n(uint64_t seed, uint32_t row, uint32_t step, uint32_t v0, float *y,
                  int64_t n)
{
    for (int64_t j = 0; j < n; ++j) y[j] = orc_gumbel(seed, row, step, v0 + (uint32_t)j);
}
/* bias of every id for one previous token p (BF16 bits out). */
void orc_bias_all(const uint16_t *head, const uint16_t *embed, int V, int r, int64_t p,
                  uint16_t *out)
{
    const uint16_t *e = embed + (size_t)p * (size_t)r;
    for (int v = 0; v < V; ++v) out[v] = orc_bias(head + (size_t)v * (size_t)r, e, r);
}
