// batch_tc.cu -- the per-position logits kernel for batches above the chain
// limit, on the 5th-generation tensor cores (fused_markov page,
// FusedMarkovSampler: per draft position a bias contraction, a logits
// epilogue over (row, vocab block) and a per-row select step; sharded_markov
// page, module docstring: batches above the chain's rows take this loop;
// muse_spark markov page, MarkovSampler: per-step kernels launched with
// programmatic dependent launch).
//
// One CTA per SM and row group of 64 rows; a CTA owns a contiguous run of
// 128-id vocab tiles and takes them in pairs (X, Y).  The head's K chunks
// [128 ids x 64 K] stream from L2 (the head stays there across positions)
// into a ring of shared-memory stages by TMA.  The rows are the MMA's M side
// and the ids its N side, so that a thread of the epilogue owns one row and
// a run of consecutive ids (16-byte loads and stores of base logits and
// cache): the previous tokens' embeddings E [64 rows x K] sit in Tensor
// Memory twice, as the A operands [E; 0] (rows in lanes 0-63) and [0; E]
// (lanes 64-127); one thread issues M = 128, N = 128, K = 16 MMAs of tile X
// through [E; 0] and of tile Y through [0; E] into one accumulator, which
// then holds the 64 rows' biases of X in lanes 0-63 and of Y in lanes
// 64-127 (each MMA adds exact zeros to the other half).  Two accumulators
// alternate, so the tensor core works on pair p + 1 while the epilogue reads
// pair p.
//
// Warp roles (18 warps, 576 threads):
//   0      allocates TMEM; lane 0 streams the head chunks (TMA) ahead of the
//          MMAs
//   1      lane 0 issues the MMAs (accumulator p % 2 for pair p)
//   2-17   the epilogue: warp w reads TMEM lane quarter q = w % 4 (rows
//          32 (q % 2) .. of tile X for q < 2, of tile Y for q >= 2) and
//          columns 32 cg .. 32 cg + 31, cg = (w - 2) / 4 (ids of the tile),
//          so each thread owns one row and 32 consecutive ids: bias
//          rounding, base add, transform, cache store, and the row's best
//          key with its lowest id; at the start it writes its row's
//          embedding slice into the A operands
// After the tiles the block's best per row goes into the row's winner word
// (u64 atomic maximum).  In Gumbel mode the last block of the row group
// writes every row's token; in inverse-CDF mode the inverse-CDF kernel that
// follows (batch.cu) writes the tokens the maxima decide and samples the
// others.
#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace dtm {

namespace {

constexpr int kBtThreads = 576;
constexpr int kBtGroup = 64;                   // rows per row group = MMA N
constexpr int kBtStages = 12;                  // head K-chunk stages of 16 KB
constexpr uint32_t kBtChunk = 128 * 128;       // 128 ids x 64 BF16
constexpr uint32_t kBtIdesc = tc::idesc_bf16(128, 128);
constexpr uint32_t kBtTmemCols = 512;          // A [E; 0], A [0; E], two accumulators
constexpr uint32_t kBtA0 = 0, kBtA1 = 128, kBtD = 256;   // TMEM columns

struct BtCtl {
    uint64_t full[kBtStages];     // stage s holds a landed chunk
    uint64_t empty[kBtStages];    // stage s read by its MMAs
    uint64_t accf[2];             // accumulator b holds a finished tile
    uint64_t accr[2];             // accumulator b read out by the 16 epilogue warps
    uint64_t fin;                 // every MMA complete (exit)
    unsigned long long best[kBtGroup];
    float T[kBtGroup];
    int live[kBtGroup];
    int resc[kBtGroup];
    uint32_t issued[kBtStages];   // producer: loads issued per stage
    unsigned int vmin;
    int flag;
    uint32_t tmem_base;
    uint32_t abort;
};

__device__ __forceinline__ void bt_pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void bt_pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void bt_fail(BtCtl &c, const SampleArgs &a, uint32_t where) {
    set_status(a.status, 4u /* MARKOV_ETIMEOUT */, where);
    c.abort = 1u;
}

__device__ __forceinline__ bool bt_aborted(const BtCtl &c) {
    return *(volatile const uint32_t *)&c.abort != 0u;
}

// Whether this block is the last of `total` blocks to pass `counter`.  Every
// block calls it once, after its results are written; the fences order each
// block's writes before its increment and the last block's reads after it.
__device__ bool bt_last_block(uint32_t *counter, uint32_t total, int *s_flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        *s_flag = atomicAdd(counter, 1u) == total - 1u;
    }
    __syncthreads();
    const bool last = *s_flag != 0;
    if (last) __threadfence();
    return last;
}

// ordered_key in fewer instructions: -0 is first made +0 (x + 0 rounds it
// so), then negative keys flip all bits and others the sign bit; any NaN
// maps above all.
__device__ __forceinline__ uint32_t bt_ordered(float k) {
    const uint32_t b = __float_as_uint(__fadd_rn(k, 0.0f));
    const uint32_t o = b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u);
    return (b & 0x7fffffffu) > 0x7f800000u ? 0xffffffffu : o;
}

// One 32-byte global store (the address 32-byte aligned).
__device__ __forceinline__ void st_v8(void *p, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                      uint32_t a4, uint32_t a5, uint32_t a6, uint32_t a7) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a0), "r"(a1),
                 "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
                 : "memory");
}

// The output-logit transforms (out of line: only transformed heads take them).
__device__ __noinline__ float bt_transform_f32(float s, const Transform tf) {
    float y = __fmul_rn(s, tf.mult);
    if (tf.has_cap) y = __fmul_rn(tf.cap, dm_tanh(__fmul_rn(y, tf.inv_cap)));
    return y;
}
__device__ __noinline__ uint32_t bt_transform_bf16x2(uint32_t lp, const Transform tf) {
    float y0 = __fmul_rn(__uint_as_float(lp << 16), tf.mult);
    float y1 = __fmul_rn(__uint_as_float(lp & 0xffff0000u), tf.mult);
    if (tf.has_cap) {
        y0 = __fmul_rn(tf.cap, dm_tanh(__fmul_rn(y0, tf.inv_cap)));
        y1 = __fmul_rn(tf.cap, dm_tanh(__fmul_rn(y1, tf.inv_cap)));
    }
    return bf16x2_rn(y0, y1);
}

}  // namespace

template <int RANK, bool kBaseF32>
__global__ void __launch_bounds__(kBtThreads, 1)
batch_tc_logits_kernel(const SampleArgs a, const __grid_constant__ CUtensorMap tmap, int i) {
    constexpr int cpt = RANK / 64;                    // K chunks per tile
    extern __shared__ uint8_t bt_raw[];
    __shared__ BtCtl c;
    uint8_t *st_s = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(bt_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t st_sa = tc::smem_u32(st_s);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = gridDim.x, cta = blockIdx.x;
    const int row0 = blockIdx.y * kBtGroup;
    const int V = a.V;
    const int T_total = (V + 127) / 128;
    const int t0 = (int)((int64_t)cta * T_total / G);
    const int t1 = (int)((int64_t)(cta + 1) * T_total / G);
    const int nt = t1 - t0;
    const int np = (nt + 1) / 2;                      // tile pairs
    const int nch = nt * cpt;
    const uint64_t timeout = a.timeout_ns;
    bt_pdl_trigger();

    // ---- input-side set-up (may overlap the kernel before this one)
    if (tid == 0) {
        for (int s = 0; s < kBtStages; ++s) {
            tc::mbar_init(tc::smem_u32(&c.full[s]), 1);
            tc::mbar_init(tc::smem_u32(&c.empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(tc::smem_u32(&c.accf[b]), 1);
            tc::mbar_init(tc::smem_u32(&c.accr[b]), 16);
        }
        tc::mbar_init(tc::smem_u32(&c.fin), 1);
        tc::mbar_init_fence();
        c.abort = 0u;
        c.vmin = 0xffffffffu;
    }
    if (warp == 0) tc::tmem_alloc(tc::smem_u32(&c.tmem_base), kBtTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = c.tmem_base;
    int produced = 0;
    if (warp == 0 && lane == 0) {
        // the first stages' head chunks (the head is an input: never written)
        for (int s = 0; s < kBtStages; ++s) c.issued[s] = 0u;
        for (; produced < nch && produced < kBtStages; ++produced) {
            const uint32_t bar = tc::smem_u32(&c.full[produced]);
            tc::mbar_expect_tx(bar, kBtChunk);
            tc::tma_load_2d(st_sa + produced * kBtChunk, &tmap, (produced % cpt) * 64,
                            (t0 + produced / cpt) * 128, bar);
            ++c.issued[produced];
        }
    }
    // epilogue threads: row (32 (q % 2) + lane) of the group, tile X (q < 2)
    // or Y (q >= 2) of each pair, ids 32 cg .. 32 cg + 31 of the tile
    const int q = warp & 3, cg = (warp - 2) >> 2;
    const int rr = 32 * (q & 1) + lane, b = row0 + rr;
    const int hy = q >> 1;
    bt_pdl_wait();

    if (tid < kBtGroup) {
        const int b = row0 + tid;
        c.best[tid] = 0ull;
        c.T[tid] = b < a.rows ? a.temperature[b] : 0.0f;
        c.live[tid] = b < a.rows && a.row_state_idx[b] >= 0;
    }
    if (warp >= 2) {
        // ---- the A operands: this thread's lane holds row rr of [E; 0]
        // (q < 2) or of [0; E] (q >= 2), columns 32 cg .. 32 cg + 31 (K
        // elements 64 cg .. 64 cg + 63, two per column, low half first);
        // the lane of the other operand is zero
        uint32_t e[32];
        bool ok = false;
        if (b < a.rows && a.row_state_idx[b] >= 0) {
            const int64_t p = i == 0 ? (int64_t)a.anchor[b] : a.tokens[b * a.tok_s0 + i - 1];
            if (p >= 0 && p < V) {
                ok = true;
                const uint4 *src = reinterpret_cast<const uint4 *>(a.embed + p * RANK + 64 * cg);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint4 x = (64 * cg + 8 * u < RANK) ? __ldg(src + u) : make_uint4(0u, 0u, 0u, 0u);
                    e[4 * u] = x.x;
                    e[4 * u + 1] = x.y;
                    e[4 * u + 2] = x.z;
                    e[4 * u + 3] = x.w;
                }
            } else if (cg == 0) {
                set_status(a.status, 1u /* MARKOV_EINVAL */, 0x300u + (uint32_t)i);
            }
        }
        if (!ok) {
#pragma unroll
            for (int u = 0; u < 32; ++u) e[u] = 0u;
        }
        uint32_t z[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) z[u] = 0u;
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        const uint32_t mine = hy ? kBtA1 : kBtA0, other = hy ? kBtA0 : kBtA1;
        // (columns past RANK / 2 are never read by the MMAs)
        uint32_t e0[16], e1[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            e0[u] = e[u];
            e1[u] = e[16 + u];
        }
        __syncwarp();
        tc::st_32x32b_x16(tmem + lanes + mine + 32 * cg, e0);
        tc::st_32x32b_x16(tmem + lanes + mine + 32 * cg + 16, e1);
        tc::st_32x32b_x16(tmem + lanes + other + 32 * cg, z);
        tc::st_32x32b_x16(tmem + lanes + other + 32 * cg + 16, z);
        tc::wait_st();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    if (warp == 0) {
        // ---- producer: the remaining chunks, each into the stage its MMAs freed
        if (lane == 0) {
            for (int j = produced; j < nch; ++j) {
                if (bt_aborted(c)) break;
                const int s = j % kBtStages;
                if (!tc::mbar_wait_for(tc::smem_u32(&c.empty[s]), (uint32_t)((j / kBtStages) - 1) & 1u, timeout)) {
                    bt_fail(c, a, 0x310u);
                    break;
                }
                const uint32_t bar = tc::smem_u32(&c.full[s]);
                tc::mbar_expect_tx(bar, kBtChunk);
                tc::tma_load_2d(st_sa + s * kBtChunk, &tmap, (j % cpt) * 64, (t0 + j / cpt) * 128, bar);
                ++c.issued[s];
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issuer: pair p into accumulator p % 2 once the epilogue
        // has read that accumulator's previous pair; tile X through [E; 0],
        // tile Y through [0; E]
        if (lane == 0) {
            for (int p = 0; p < np; ++p) {
                if (bt_aborted(c)) break;
                const int ab = p & 1, use = p >> 1;
                if (use > 0 &&
                    !tc::mbar_wait_for(tc::smem_u32(&c.accr[ab]), (uint32_t)(use - 1) & 1u, timeout)) {
                    bt_fail(c, a, 0x320u);
                    break;
                }
                tc::fence_after_sync();
                const uint32_t d = tmem + kBtD + (uint32_t)(ab * 128);
                bool ok = true;
                const int ntile = 2 * p + 1 < nt ? 2 : 1;
                for (int h = 0; h < ntile && ok; ++h) {
                    const int k = 2 * p + h;
                    const uint32_t aop = tmem + (h == 0 ? kBtA0 : kBtA1);
#pragma unroll
                    for (int kc = 0; kc < cpt; ++kc) {
                        const int j = k * cpt + kc, s = j % kBtStages;
                        if (!tc::mbar_wait_for(tc::smem_u32(&c.full[s]), (uint32_t)(j / kBtStages) & 1u, timeout)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
                        const uint64_t bd = tc::sw128_desc(st_sa + s * kBtChunk);
                        const uint32_t at = aop + 32u * (uint32_t)kc;
                        tc::mma_tmemA(d, at, bd, kBtIdesc, (h == 0 && kc == 0) ? 0u : 1u);
                        tc::mma_tmemA(d, at + 8u, bd + 2u, kBtIdesc, 1u);
                        tc::mma_tmemA(d, at + 16u, bd + 4u, kBtIdesc, 1u);
                        tc::mma_tmemA(d, at + 24u, bd + 6u, kBtIdesc, 1u);
                        tc::commit(tc::smem_u32(&c.empty[s]));
                    }
                }
                if (!ok) {
                    bt_fail(c, a, 0x330u);
                    break;
                }
                tc::commit(tc::smem_u32(&c.accf[ab]));
            }
        }
        __syncwarp();
    } else if (warp >= 2) {
        // ---- epilogue: one row and 32 consecutive ids per thread and pair,
        // in two halves of 16 ids
        const bool live = c.live[rr] != 0;
        const float T = c.T[rr];
        const bool gum = live && a.mode == 0 && samples(T);
        const bool cache_f32 = a.cache_f != nullptr;
        const int64_t brow = b * a.base_s0 + (int64_t)i * a.base_s1;
        const int64_t crow = b * a.cache_s0 + (int64_t)i * a.cache_s1;
        const float *nrow = a.noise + (int64_t)(b * a.N + i) * a.noise_s0;
        // 16-byte base loads need 16-byte aligned rows
        constexpr int kEpV = kBaseF32 ? 4 : 8;       // elements per 16 bytes
        const bool vec = ((reinterpret_cast<uintptr_t>(kBaseF32 ? (const void *)a.base_f : (const void *)a.base) &
                           15u) == 0u) &&
                         (a.base_s0 % kEpV) == 0 && (a.base_s1 % kEpV) == 0;
        // the row's best key so far and its id (kNone: no key yet)
        constexpr uint32_t kNone = 0xffffffffu;
        float bf = 0.0f;
        uint32_t bid = kNone;
        // 32-byte cache stores need 32-byte aligned rows
        const bool st32 = ((reinterpret_cast<uintptr_t>(cache_f32 ? (void *)a.cache_f : (void *)a.cache) & 31u) == 0u) &&
                          ((a.cache_s0 * (cache_f32 ? 4 : 2)) % 32) == 0 && ((a.cache_s1 * (cache_f32 ? 4 : 2)) % 32) == 0;
        constexpr int kNB = kBaseF32 ? 32 : 16;      // base words of 32 ids
        // the base logits of this thread's 32 ids of pair p (zeros outside)
        auto load_base = [&](int p, uint32_t (&w)[kNB]) {
            const int k = 2 * p + hy;
            const int v0 = (t0 + k) * 128 + 32 * cg;
            const bool on = live && p < np && k < nt && v0 < V;
            if (kBaseF32) {
                const float *src = a.base_f + brow + v0;
#pragma unroll
                for (int u = 0; u < 32; u += 4) {
                    uint4 x = make_uint4(0u, 0u, 0u, 0u);
                    if (on && vec && v0 + u < V) {
                        x = __ldg(reinterpret_cast<const uint4 *>(src + u));
                    } else if (on && !vec) {
                        x.x = v0 + u < V ? __float_as_uint(__ldg(src + u)) : 0u;
                        x.y = v0 + u + 1 < V ? __float_as_uint(__ldg(src + u + 1)) : 0u;
                        x.z = v0 + u + 2 < V ? __float_as_uint(__ldg(src + u + 2)) : 0u;
                        x.w = v0 + u + 3 < V ? __float_as_uint(__ldg(src + u + 3)) : 0u;
                    }
                    w[u] = x.x;
                    w[u + 1] = x.y;
                    w[u + 2] = x.z;
                    w[u + 3] = x.w;
                }
            } else {
                const uint16_t *src = a.base + brow + v0;
#pragma unroll
                for (int u = 0; u < 16; u += 4) {
                    uint4 x = make_uint4(0u, 0u, 0u, 0u);
                    if (on && vec && v0 + 2 * u < V) {
                        x = __ldg(reinterpret_cast<const uint4 *>(src + 2 * u));
                    } else if (on && !vec) {
                        uint32_t y[4];
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            const int v = v0 + 2 * (u + e2);
                            const uint32_t lo = v < V ? (uint32_t)__ldg(src + 2 * (u + e2)) : 0u;
                            const uint32_t hi = v + 1 < V ? (uint32_t)__ldg(src + 2 * (u + e2) + 1) : 0u;
                            y[e2] = lo | (hi << 16);
                        }
                        x = make_uint4(y[0], y[1], y[2], y[3]);
                    }
                    w[u] = x.x;
                    w[u + 1] = x.y;
                    w[u + 2] = x.z;
                    w[u + 3] = x.w;
                }
            }
        };
        uint32_t nb[kNB];
        if (!kBaseF32) load_base(0, nb);   // BF16 base: one pair ahead
        for (int p = 0; p < np; ++p) {
            uint32_t cb[kNB];
            if (kBaseF32) {
                load_base(p, cb);
            } else {
#pragma unroll
                for (int u = 0; u < kNB; ++u) cb[u] = nb[u];
                load_base(p + 1, nb);
            }
            const int ab = p & 1;
            bool ok = true;
            if (lane == 0)
                ok = tc::mbar_wait_for(tc::smem_u32(&c.accf[ab]), (uint32_t)(p >> 1) & 1u, timeout);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) bt_fail(c, a, 0x340u);
                break;
            }
            tc::fence_after_sync();
            const int k = 2 * p + hy;
            const int v0 = (t0 + k) * 128 + 32 * cg;
            const bool on = live && k < nt && v0 < V;
            const uint32_t dcol = tmem + ((uint32_t)(q * 32) << 16) + kBtD + (uint32_t)(ab * 128 + 32 * cg);
#pragma unroll
            for (int h16 = 0; h16 < 2; ++h16) {
                uint32_t acc[16];
                __syncwarp();   // (the lanes' rows differ in liveness)
                tc::ld_32x32b_x16(dcol + 16u * (uint32_t)h16, acc);
                tc::wait_ld();
                if (h16 == 1) {
                    // the accumulator is read out: the MMAs of pair p + 2 may start
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(tc::smem_u32(&c.accr[ab]));
                }
                const int vh = v0 + 16 * h16;
                if (!on || vh >= V) continue;
                // 8 id pairs: bias = bf16(sum); l = f32(base) + f32(bias),
                // rounded to the cache's type and transformed
                uint32_t lp[8];
                float lf[16];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t bb = bf16x2_rn(__uint_as_float(acc[2 * j]), __uint_as_float(acc[2 * j + 1]));
                    const float b0 = kBaseF32 ? __uint_as_float(cb[16 * h16 + 2 * j])
                                              : __uint_as_float(cb[(8 * h16 + j) % kNB] << 16);
                    const float b1 = kBaseF32 ? __uint_as_float(cb[16 * h16 + 2 * j + 1])
                                              : __uint_as_float(cb[(8 * h16 + j) % kNB] & 0xffff0000u);
                    float l0 = __fadd_rn(b0, __uint_as_float(bb << 16));
                    float l1 = __fadd_rn(b1, __uint_as_float(bb & 0xffff0000u));
                    if (cache_f32) {
                        if (a.tf.has_transform) {
                            l0 = bt_transform_f32(l0, a.tf);
                            l1 = bt_transform_f32(l1, a.tf);
                        }
                    } else {
                        uint32_t w = bf16x2_rn(l0, l1);
                        if (a.tf.has_transform) w = bt_transform_bf16x2(w, a.tf);
                        lp[j] = w;
                        l0 = __uint_as_float(w << 16);
                        l1 = __uint_as_float(w & 0xffff0000u);
                    }
                    lf[2 * j] = l0;
                    lf[2 * j + 1] = l1;
                }
                // the cache: one 32-byte store per 16 BF16 ids where the
                // cache rows are 32-byte aligned, else 16-byte stores (the
                // rows are 16-byte aligned); the vocabulary is a multiple of
                // 16, so a half is whole
                if (cache_f32) {
                    float *dst = a.cache_f + crow + vh;
                    if (st32) {
#pragma unroll
                        for (int u = 0; u < 2; ++u)
                            st_v8(dst + 8 * u, __float_as_uint(lf[8 * u]), __float_as_uint(lf[8 * u + 1]),
                                  __float_as_uint(lf[8 * u + 2]), __float_as_uint(lf[8 * u + 3]),
                                  __float_as_uint(lf[8 * u + 4]), __float_as_uint(lf[8 * u + 5]),
                                  __float_as_uint(lf[8 * u + 6]), __float_as_uint(lf[8 * u + 7]));
                    } else {
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            *reinterpret_cast<float4 *>(dst + 4 * u) =
                                make_float4(lf[4 * u], lf[4 * u + 1], lf[4 * u + 2], lf[4 * u + 3]);
                    }
                } else {
                    uint16_t *dst = a.cache + crow + vh;
                    if (st32) {
                        st_v8(dst, lp[0], lp[1], lp[2], lp[3], lp[4], lp[5], lp[6], lp[7]);
                    } else {
#pragma unroll
                        for (int u = 0; u < 2; ++u)
                            *reinterpret_cast<uint4 *>(dst + 8 * u) =
                                make_uint4(lp[4 * u], lp[4 * u + 1], lp[4 * u + 2], lp[4 * u + 3]);
                    }
                }
                // keys: the logit, or for a sampling Gumbel row fp32(l / T)
                // + the call's noise
                float key[16];
                if (gum) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float4 x = __ldg(reinterpret_cast<const float4 *>(nrow + vh) + u);
                        key[4 * u] = __fadd_rn(__fdiv_rn(lf[4 * u], T), x.x);
                        key[4 * u + 1] = __fadd_rn(__fdiv_rn(lf[4 * u + 1], T), x.y);
                        key[4 * u + 2] = __fadd_rn(__fdiv_rn(lf[4 * u + 2], T), x.z);
                        key[4 * u + 3] = __fadd_rn(__fdiv_rn(lf[4 * u + 3], T), x.w);
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < 16; ++u) key[u] = lf[u];
                }
                // the half's best: a tree of strict comparisons, the
                // lower-id side winning ties (16 keys in id order), and a
                // NaN / infinity test (x 0 is NaN for both)
                float tv[8];
                uint32_t ti[8];
                float poison = 0.0f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const bool r = key[2 * j + 1] > key[2 * j];
                    tv[j] = r ? key[2 * j + 1] : key[2 * j];
                    ti[j] = r ? 2u * j + 1u : 2u * j;
                    poison = __fmaf_rn(key[2 * j], 0.0f, poison);
                    poison = __fmaf_rn(key[2 * j + 1], 0.0f, poison);
                }
#pragma unroll
                for (int w = 4; w >= 1; w >>= 1) {
#pragma unroll
                    for (int j = 0; j < w; ++j) {
                        const bool r = tv[2 * j + 1] > tv[2 * j];
                        tv[j] = r ? tv[2 * j + 1] : tv[2 * j];
                        ti[j] = r ? ti[2 * j + 1] : ti[2 * j];
                    }
                }
                if (poison == 0.0f) {
                    // halves come in increasing id order: a strict
                    // comparison keeps the earlier of equal keys
                    const bool better = bid == kNone || tv[0] > bf;
                    bf = better ? tv[0] : bf;
                    bid = better ? (uint32_t)vh + ti[0] : bid;
                } else {
                    // a NaN or an infinity in the half: the exact ordered
                    // keys (a NaN above all, the lowest NaN id first)
                    uint32_t ob = bid == kNone ? 0u : bt_ordered(bf);
#pragma unroll
                    for (int e2 = 0; e2 < 16; ++e2) {
                        const uint32_t o = bt_ordered(key[e2]);
                        const bool better = o > ob;
                        ob = better ? o : ob;
                        bf = better ? key[e2] : bf;
                        bid = better ? (uint32_t)(vh + e2) : bid;
                    }
                }
            }
        }
        // the thread's best into the block's (4 threads share a row)
        if (live && bid != kNone)
            atomicMax(&c.best[rr],
                      ((unsigned long long)bt_ordered(bf) << 32) | (unsigned long long)(0xffffffffu - bid));
    }

    // ---- every async operation completes before TMEM is released
    if (warp == 1 && lane == 0) {
        tc::commit(tc::smem_u32(&c.fin));
        tc::mbar_wait_for(tc::smem_u32(&c.fin), 0u, 1000000000ull);
    }
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < kBtStages; ++s) {
            if (c.issued[s] == 0u) continue;
            tc::mbar_wait_for(tc::smem_u32(&c.full[s]), (c.issued[s] - 1u) & 1u, 1000000000ull);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, kBtTmemCols);

    // ---- the block's best per row into the row's winner word; inverse-CDF
    // rows that sample: the block's key is fl(max l / T), which is
    // max fl(l / T) since rounding is monotone; only the id of a +inf key
    // needs the exact keys (their lowest id), so such rows rescan
    bool resc = false;
    if (tid < kBtGroup) {
        const uint64_t bw = c.best[tid];
        const float T = c.T[tid];
        if (a.mode == 1 && bw != 0ull && samples(T)) {
            const uint32_t o = packed_ordered(bw);
            if (o != 0xffffffffu) {
                const float kq = __fdiv_rn(key_from_ordered(o), T);
                if (kq == __uint_as_float(0x7f800000u))
                    resc = true;
                else
                    c.best[tid] = pack_key(kq, packed_id(bw));
            }
        }
        c.resc[tid] = resc;
    }
    const int v_begin = t0 * 128, v_end = t1 * 128 < V ? t1 * 128 : V;
    if (__syncthreads_or(resc)) {
        // rare: the lowest id of this block whose key fl(l / T) is +inf
        for (int rr = 0; rr < kBtGroup; ++rr) {
            if (!c.resc[rr]) continue;
            const float T = c.T[rr];
            for (int v = v_begin + tid; v < v_end; v += kBtThreads) {
                if (__fdiv_rn(cache_value(a, row0 + rr, i, v), T) == __uint_as_float(0x7f800000u)) {
                    atomicMin(&c.vmin, (unsigned int)v);
                    break;
                }
            }
            __syncthreads();
            if (tid == 0) {
                c.best[rr] = pack_key(__uint_as_float(0x7f800000u), c.vmin);
                c.vmin = 0xffffffffu;
            }
            __syncthreads();
        }
    }
    unsigned long long *wins = reinterpret_cast<unsigned long long *>(a.bwin + (size_t)i * kMaxRows);
    if (tid < kBtGroup && c.best[tid]) atomicMax(wins + row0 + tid, c.best[tid]);
    // inverse CDF: the inverse-CDF kernel that follows (it waits for this
    // grid) writes the tokens the maxima decide, so no block here waits for
    // the others (no fence, no done counter)
    if (a.mode == 1) return;
    uint32_t *cnt = a.bcnt + (size_t)i * kBatchCntPerStep + blockIdx.y;
    if (!bt_last_block(cnt, (uint32_t)G, &c.flag)) return;

    // last block of the row group: every block's maximum is in
    if (tid == 0) *cnt = 0u;
    const int bq = row0 + tid;
    if (tid < kBtGroup && c.live[tid]) {
        unsigned long long *ws = wins + bq;
        const uint64_t win = __ldcg(ws);
        const float T = c.T[tid];
        const uint32_t o = packed_ordered(win);
        const float M = key_from_ordered(o);
        const bool decided = a.mode == 0 || !samples(T) || o == 0xffffffffu ||
                             M == __uint_as_float(0x7f800000u) || M == __uint_as_float(0xff800000u);
        if (decided) {
            int64_t tok = (int64_t)packed_id(win);
            if (a.mode == 1 && samples(T) && o != 0xffffffffu && M == __uint_as_float(0xff800000u)) tok = 0;
            if (win == 0ull) {
                set_status(a.status, 6u /* MARKOV_EDEVICE */, 0x350u + (uint32_t)i);
                tok = 0;
            }
            a.tokens[bq * a.tok_s0 + i] = tok;
            *ws = 0ull;
        }
    }
}

size_t batch_tc_smem(int) { return (size_t)kBtStages * kBtChunk + 1024; }

static const void *bt_kernel(int r, bool base_f32) {
    switch (r) {
        case 64: return base_f32 ? (const void *)batch_tc_logits_kernel<64, true>
                                 : (const void *)batch_tc_logits_kernel<64, false>;
        case 128: return base_f32 ? (const void *)batch_tc_logits_kernel<128, true>
                                  : (const void *)batch_tc_logits_kernel<128, false>;
        case 256: return base_f32 ? (const void *)batch_tc_logits_kernel<256, true>
                                  : (const void *)batch_tc_logits_kernel<256, false>;
        default: return nullptr;
    }
}

cudaError_t batch_tc_prepare() {
    for (int r : {64, 128, 256})
        for (int f = 0; f < 2; ++f) {
            cudaError_t e = cudaFuncSetAttribute(bt_kernel(r, f != 0), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)batch_tc_smem(r));
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

// One logits launch of position i: grid (CTAs per row group, row groups of
// 64); pdl: as a programmatic dependent of the launch before it.
cudaError_t launch_batch_tc_logits(const SampleArgs &a, const CUtensorMap &tmap, int i, int ctas,
                                   cudaStream_t stream, bool pdl) {
    const void *fn = bt_kernel(a.r, a.base_f != nullptr);
    if (!fn) return cudaErrorInvalidValue;
    const int groups = (a.rows + kBtGroup - 1) / kBtGroup;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas, groups);
    cfg.blockDim = dim3(kBtThreads);
    cfg.dynamicSmemBytes = batch_tc_smem(a.r);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    void *args[] = {(void *)&a, (void *)&tmap, (void *)&i};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace dtm
