// batch.cu -- the per-position path for batches above the chain limit
// (fused_markov page, FusedMarkovSampler: per draft position a bias
// contraction plus a logits kernel over (row, vocab block) and a per-row
// select step; sharded_markov page, module docstring: batches above
// max_rows take this loop; muse_spark markov page, MarkovSampler: the
// per-step kernels are launched with programmatic dependent launch).
//
// Per position i, in launch order on one stream:
//   logits  grid (blocks, row groups of 16 rows up to 16 rows, else 32),
//           or the tcgen05 logits kernel (batch_tc.cu) when the plan has
//           the head's tensor map:
//           bias tiles [16 ids x group rows] by mma.m16n8k16 with the
//           previous tokens' embeddings staged in shared memory, the
//           epilogue (BF16 rounding, base add, transform,
//           cache store) and each block's best (key, id) per row, merged
//           into the row's winner word by one u64 atomicMax per block.  The
//           last block of a row group to finish (a done counter) writes the
//           token of every row the winner decides: all rows in Gumbel mode,
//           greedy rows and rows with a NaN, +inf or all -inf maximum in
//           inverse-CDF mode;
//   cdf     (inverse CDF only) grid (vocab blocks of kCdfIds ids, rows):
//           the integer weights floor(exp(x - M) 2^40) summed per 256-id
//           unit; the last block of a row scans the row's unit sums for
//           mulhi64(H, S), then one warp the target unit's weights, and
//           writes the token.
// The next position's logits kernel reads token i from draft_tokens.  Every
// block that takes the last-block step resets the counter and the winner
// word it consumed, so each call leaves them zero for the next.
//
// Every launch after the first of a call is a programmatic dependent launch:
// it may start while the kernel before it still runs, does only input-side
// work (block ranges, L2 prefetch of its head and base-logit rows) until
// griddepcontrol.wait, and every block of every kernel passes that wait
// before it reads or writes anything the path writes, and before it exits.
// A grid therefore completes only after the grid before it has, and a
// kernel's wait covers the whole chain of launches before it.
#include <type_traits>

#include "common.cuh"
#include "tc.cuh"

namespace dtm {

namespace {

constexpr int kBW = kBatchThreads / 32;    // warps per block
constexpr int kBPad = 32;

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Programmatic dependent launch: pdl_wait() returns once the kernel before
// this one on the stream has completed and its writes are visible (at once
// for an ordinary launch); pdl_trigger() lets the next kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// L2 eviction policies: the head is read at every position and should stay
// in L2 across them; base logits are read once and cache entries written
// once per call.
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// Loads of data no kernel of the call writes (the head, the base logits),
// bypassing L1, with an L2 cache policy.
__device__ __forceinline__ uint4 ld_nc_v4(const void *ptr, uint64_t pol) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(ptr), "l"(pol));
    return v;
}
__device__ __forceinline__ uint32_t ld_nc_u32(const void *ptr, uint64_t pol) {
    uint32_t v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;"
        : "=r"(v)
        : "l"(ptr), "l"(pol));
    return v;
}
__device__ __forceinline__ float2 ld_nc_f2(const void *ptr, uint64_t pol) {
    float2 v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.f32 {%0, %1}, [%2], %3;"
        : "=f"(v.x), "=f"(v.y)
        : "l"(ptr), "l"(pol));
    return v;
}
__device__ __forceinline__ void st_u32(void *ptr, uint32_t v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.u32 [%0], %1, %2;" ::"l"(ptr), "r"(v), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void st_f2(void *ptr, float2 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(ptr), "f"(v.x),
                 "f"(v.y), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ int64_t prev_token(const SampleArgs &a, int b, int i) {
    return i == 0 ? (int64_t)a.anchor[b] : a.tokens[b * a.tok_s0 + i - 1];
}

__device__ __forceinline__ bool row_live(const SampleArgs &a, int b) {
    return b < a.rows && a.row_state_idx[b] >= 0;
}

// The block's vocab range: contiguous 16-id tiles, split evenly.
__device__ __forceinline__ void block_range(int V, int nblk, int blk, int &v0, int &v1) {
    int nt = V / kTile;
    v0 = (int)((int64_t)blk * nt / nblk) * kTile;
    v1 = (int)((int64_t)(blk + 1) * nt / nblk) * kTile;
}

__device__ __forceinline__ unsigned long long *win_slot(const SampleArgs &a, int i, int b) {
    return reinterpret_cast<unsigned long long *>(a.bwin + (size_t)i * kMaxRows + b);
}
__device__ __forceinline__ uint32_t *group_counter(const SampleArgs &a, int i, int grp) {
    return a.bcnt + (size_t)i * kBatchCntPerStep + grp;
}
__device__ __forceinline__ uint32_t *row_counter(const SampleArgs &a, int i, int b) {
    return a.bcnt + (size_t)i * kBatchCntPerStep + kMaxRows / 16 + b;
}

// Whether this block is the last of `total` blocks to pass `counter`.  Every
// block calls it once, after its results are written; the fences order each
// block's writes before its increment and the last block's reads after it.
__device__ bool last_block(uint32_t *counter, uint32_t total, int *s_flag) {
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

// Whether an inverse-CDF row with this winner needs the weight sums: its
// maximum is finite (a NaN or +inf maximum decides the token directly; an
// all -inf row takes id 0).
__device__ __forceinline__ bool needs_sums(uint64_t win) {
    uint32_t o = packed_ordered(win);
    float M = key_from_ordered(o);
    return o != 0xffffffffu && M != __uint_as_float(0x7f800000u) &&
           M != __uint_as_float(0xff800000u);
}

// ordered_key in fewer instructions: -0 is first made +0 (x + 0 rounds it
// so), then negative keys flip all bits and others the sign bit; any NaN
// maps above all.
__device__ __forceinline__ uint32_t ordered_canonical(float k) {
    const uint32_t b = __float_as_uint(__fadd_rn(k, 0.0f));
    const uint32_t o = b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u);
    return (b & 0x7fffffffu) > 0x7f800000u ? 0xffffffffu : o;
}

// The token of a row that its winner decides without weight sums.
__device__ __forceinline__ int64_t direct_token(const SampleArgs &a, uint64_t win, float T) {
    int64_t tok = (int64_t)packed_id(win);
    if (a.mode == 1 && samples(T)) {
        const uint32_t o = packed_ordered(win);
        if (o != 0xffffffffu && key_from_ordered(o) == __uint_as_float(0xff800000u)) tok = 0;
    }
    return tok;
}

// The output-logit transform of one fp32 cached logit, and of two packed
// BF16 cached logits (out of line: only transformed heads take them).
__device__ __noinline__ float transform_one_f32(float s, const Transform tf) {
    float y = __fmul_rn(s, tf.mult);
    if (tf.has_cap) y = __fmul_rn(tf.cap, dm_tanh(__fmul_rn(y, tf.inv_cap)));
    return y;
}

__device__ __noinline__ uint32_t transform_two_bf16(uint32_t lp, const Transform tf) {
    float y0 = __fmul_rn(__uint_as_float(lp << 16), tf.mult);
    float y1 = __fmul_rn(__uint_as_float(lp & 0xffff0000u), tf.mult);
    if (tf.has_cap) {
        y0 = __fmul_rn(tf.cap, dm_tanh(__fmul_rn(y0, tf.inv_cap)));
        y1 = __fmul_rn(tf.cap, dm_tanh(__fmul_rn(y1, tf.inv_cap)));
    }
    return bf16x2_rn(y0, y1);
}

// Integer inverse-CDF weight floor(exp(x / T - M) 2^40) of cached logit x
// (kPow2: T a power of two, rT = 1 / T).
template <bool kPow2>
__device__ __forceinline__ uint64_t cdf_weight_of(float x, float T, float rT, float M) {
    return dm_cdf_weight(__fsub_rn(dm_div_T<kPow2>(x, T, rT), M));
}

// The weight sum of 8 cached logits.
template <bool kPow2>
__device__ __forceinline__ uint64_t cdf_weight8(const float (&x)[8], float T, float rT, float M) {
    uint64_t s = 0ull;
#pragma unroll
    for (int e = 0; e < 8; ++e) s += cdf_weight_of<kPow2>(x[e], T, rT, M);
    return s;
}

}  // namespace

// The logits kernel of position i, for row groups of 16 MT rows.  MMA
// roles: M = 16 rows (the previous tokens' embeddings, staged in shared
// memory), N = 8 vocab ids (head rows, read from global), K = rank, so that
// each thread's accumulators hold pairs of consecutive ids of one row: base
// logits are read and cache entries written two ids at a time.  Rows of a thread: row0 + 16 m + 8 h + g for
// M-tile m < MT and half h < 2 (bit 2 m + h of `live`).  The head fragments
// of a tile are fetched kDepth k-chunks ahead of their MMAs: the whole tile
// at once for 16-row groups (few accumulators leave the registers for it),
// two chunks for 32-row groups.
template <int RANK, bool kBaseF32, int MT>
__global__ void __launch_bounds__(kBatchThreads, 2)
batch_logits_kernel(const SampleArgs a, int i) {
    constexpr int kGroupRows = 16 * MT;
    constexpr int kMT = MT;
    constexpr int kChunks = RANK / 32;
    constexpr int kDepth = MT == 1 ? kChunks : 2;
    extern __shared__ __align__(16) uint16_t e_smem[];      // [kGroupRows][RANK + kBPad]
    __shared__ unsigned long long s_best[kGroupRows];
    __shared__ float s_T[kGroupRows];
    __shared__ int s_resc[kGroupRows];
    __shared__ unsigned int s_vmin;
    __shared__ int s_flag;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int blk = blockIdx.x, nblk = gridDim.x;
    const int row0 = blockIdx.y * kGroupRows;
    const int V = a.V;
    int v_begin, v_end;
    block_range(V, nblk, blk, v_begin, v_end);
    pdl_trigger();
    {
        // input side only: this block's head rows (kept in L2 across
        // positions) and its base-logit rows of position i into L2
        const char *hp = reinterpret_cast<const char *>(a.head + (int64_t)v_begin * RANK);
        const int hlines = (v_end - v_begin) * RANK * 2 / 128;
        for (int l = tid; l < hlines; l += kBatchThreads)
            asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(hp + (int64_t)l * 128));
        constexpr int esz = kBaseF32 ? 4 : 2;
        const char *bp = kBaseF32 ? reinterpret_cast<const char *>(a.base_f)
                                  : reinterpret_cast<const char *>(a.base);
        const int lines = ((v_end - v_begin) * esz + 127) / 128 + 1;
        for (int idx = tid; idx < kGroupRows * lines; idx += kBatchThreads) {
            const int b = idx / lines, l = idx - b * lines;
            if (!row_live(a, row0 + b)) continue;
            const int64_t o0 = (row0 + b) * a.base_s0 + (int64_t)i * a.base_s1 + v_begin;
            const char *q = bp + o0 * esz + (int64_t)l * 128;
            if (q < bp + (o0 + (v_end - v_begin)) * esz)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(q));
        }
    }
    pdl_wait();

    for (int idx = tid; idx < kGroupRows * (RANK / 8); idx += kBatchThreads) {
        int b = idx / (RANK / 8), c = idx % (RANK / 8);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row_live(a, row0 + b)) {
            int64_t p = prev_token(a, row0 + b, i);
            if (p >= 0 && p < V) v = *reinterpret_cast<const uint4 *>(a.embed + p * RANK + 8 * c);
        }
        *reinterpret_cast<uint4 *>(e_smem + b * (RANK + kBPad) + 8 * c) = v;
    }
    if (tid < kGroupRows) {
        s_best[tid] = 0ull;
        s_T[tid] = row0 + tid < a.rows ? a.temperature[row0 + tid] : 0.0f;
    }
    if (tid == 0) s_vmin = 0xffffffffu;
    uint32_t live = 0u;
#pragma unroll
    for (int q = 0; q < 2 * kMT; ++q)
        if (row_live(a, row0 + 16 * (q >> 1) + 8 * (q & 1) + g)) live |= 1u << q;
    __syncthreads();

    // per row of this thread: the best ordered key so far and its id (ids
    // are visited in increasing order, so a strict comparison keeps the
    // lowest id of equal keys); ordered key 0 is below every real key
    uint32_t bo[kMT][2], bi[kMT][2];
#pragma unroll
    for (int m = 0; m < kMT; ++m) bo[m][0] = bo[m][1] = bi[m][0] = bi[m][1] = 0u;
    const int nm = min(kMT, (a.rows - row0 + 15) / 16);
    const uint64_t keep = policy_evict_last(), once = policy_evict_first();
    const bool cache_f32 = a.cache_f != nullptr;
    // paired base loads need the pair's alignment
    const bool vec = ((reinterpret_cast<uintptr_t>(kBaseF32 ? (const void *)a.base_f
                                                             : (const void *)a.base) &
                       (kBaseF32 ? 7u : 3u)) == 0u) &&
                     ((a.base_s0 | a.base_s1) & 1) == 0;
    // the key of a row is its logit except for Gumbel rows that sample
    // (inverse-CDF rows divide their maximum by T once, at the end)
    uint32_t divides = 0u;
    if (a.mode == 0) {
#pragma unroll
        for (int q = 0; q < 2 * kMT; ++q)
            if (samples(s_T[16 * (q >> 1) + 8 * (q & 1) + g])) divides |= 1u << q;
    }

    for (int v0 = v_begin + warp * kTile; v0 < v_end; v0 += kBW * kTile) {
        // this tile's base logits first: their latency overlaps the MMAs
        using BaseT = typename std::conditional<kBaseF32, float2, uint32_t>::type;
        BaseT bv[kMT][2][2];
#pragma unroll
        for (int m = 0; m < kMT; ++m)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int n = 0; n < 2; ++n) {
                    const int q = 2 * m + h;
                    const int64_t o = (row0 + 16 * m + 8 * h + g) * a.base_s0 +
                                      (int64_t)i * a.base_s1 + v0 + 8 * n + 2 * t;
                    if constexpr (kBaseF32) {
                        bv[m][h][n] = make_float2(0.0f, 0.0f);
                        if (m < nm && ((live >> q) & 1u))
                            bv[m][h][n] = vec ? ld_nc_f2(a.base_f + o, once)
                                              : make_float2(__ldg(a.base_f + o),
                                                            __ldg(a.base_f + o + 1));
                    } else {
                        bv[m][h][n] = 0u;
                        if (m < nm && ((live >> q) & 1u))
                            bv[m][h][n] = vec ? ld_nc_u32(a.base + o, once)
                                              : ((uint32_t)__ldg(a.base + o) |
                                                 ((uint32_t)__ldg(a.base + o + 1) << 16));
                    }
                }

        float acc[kMT][2][4];
#pragma unroll
        for (int m = 0; m < kMT; ++m)
#pragma unroll
            for (int n = 0; n < 2; ++n) acc[m][n][0] = acc[m][n][1] = acc[m][n][2] = acc[m][n][3] = 0.0f;
        const uint16_t *h0 = a.head + (int64_t)(v0 + g) * RANK + 8 * t;
        const uint16_t *h1 = h0 + 8 * RANK;
        // head fragments kDepth k-chunks ahead of the MMAs that use them
        uint4 hx[kDepth], hy[kDepth];
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
            hx[d] = ld_nc_v4(h0 + 32 * d, keep);
            hy[d] = ld_nc_v4(h1 + 32 * d, keep);
        }
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
            const uint4 x = hx[j % kDepth], y = hy[j % kDepth];
            if (j + kDepth < kChunks) {
                hx[j % kDepth] = ld_nc_v4(h0 + 32 * (j + kDepth), keep);
                hy[j % kDepth] = ld_nc_v4(h1 + 32 * (j + kDepth), keep);
            }
#pragma unroll
            for (int m = 0; m < kMT; ++m) {
                if (m >= nm) break;
                const uint16_t *er = e_smem + (16 * m + g) * (RANK + kBPad) + 8 * t + 32 * j;
                const uint4 ea = *reinterpret_cast<const uint4 *>(er);
                const uint4 eb = *reinterpret_cast<const uint4 *>(er + 8 * (RANK + kBPad));
                mma16816(acc[m][0], ea.x, eb.x, ea.y, eb.y, x.x, x.y);
                mma16816(acc[m][1], ea.x, eb.x, ea.y, eb.y, y.x, y.y);
                mma16816(acc[m][0], ea.z, eb.z, ea.w, eb.w, x.z, x.w);
                mma16816(acc[m][1], ea.z, eb.z, ea.w, eb.w, y.z, y.w);
            }
        }
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
            if (m >= nm) break;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int q = 2 * m + h;
                if (!((live >> q) & 1u)) continue;
                const int rr = 16 * m + 8 * h + g;
                const int row = row0 + rr;
#pragma unroll
                for (int n = 0; n < 2; ++n) {
                    const int v = v0 + 8 * n + 2 * t;
                    // bias = bf16(sum); s = f32(base) + f32(bias)
                    const uint32_t bb = bf16x2_rn(acc[m][n][2 * h], acc[m][n][2 * h + 1]);
                    float b0, b1;
                    if constexpr (kBaseF32) {
                        b0 = bv[m][h][n].x;
                        b1 = bv[m][h][n].y;
                    } else {
                        b0 = __uint_as_float(bv[m][h][n] << 16);
                        b1 = __uint_as_float(bv[m][h][n] & 0xffff0000u);
                    }
                    float l0 = __fadd_rn(b0, __uint_as_float(bb << 16));
                    float l1 = __fadd_rn(b1, __uint_as_float(bb & 0xffff0000u));
                    const int64_t co = row * a.cache_s0 + (int64_t)i * a.cache_s1 + v;
                    if (cache_f32) {
                        if (a.tf.has_transform) {
                            l0 = transform_one_f32(l0, a.tf);
                            l1 = transform_one_f32(l1, a.tf);
                        }
                        st_f2(a.cache_f + co, make_float2(l0, l1), once);
                    } else {
                        uint32_t lp = bf16x2_rn(l0, l1);
                        if (a.tf.has_transform) lp = transform_two_bf16(lp, a.tf);
                        st_u32(a.cache + co, lp, once);
                        l0 = __uint_as_float(lp << 16);
                        l1 = __uint_as_float(lp & 0xffff0000u);
                    }
                    float k0 = l0, k1 = l1;
                    if ((divides >> q) & 1u) {
                        const float T = s_T[rr];
                        const float2 gn = *reinterpret_cast<const float2 *>(
                            a.noise + (int64_t)(row * a.N + i) * a.noise_s0 + v);
                        k0 = __fadd_rn(__fdiv_rn(l0, T), gn.x);
                        k1 = __fadd_rn(__fdiv_rn(l1, T), gn.y);
                    }
                    const uint32_t o0 = ordered_canonical(k0), o1 = ordered_canonical(k1);
                    if (o0 > bo[m][h]) {
                        bo[m][h] = o0;
                        bi[m][h] = (uint32_t)v;
                    }
                    if (o1 > bo[m][h]) {
                        bo[m][h] = o1;
                        bi[m][h] = (uint32_t)v + 1u;
                    }
                }
            }
        }
    }
#pragma unroll
    for (int m = 0; m < kMT; ++m) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint64_t v = bo[m][h] ? ((uint64_t)bo[m][h] << 32) | (uint64_t)(0xffffffffu - bi[m][h])
                                  : 0ull;
#pragma unroll
            for (int o = 1; o < 4; o <<= 1) {
                uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
                v = w > v ? w : v;
            }
            if (t == 0 && v) atomicMax(&s_best[16 * m + 8 * h + g], (unsigned long long)v);
        }
    }
    __syncthreads();
    // inverse-CDF rows that sample: the block's key is fl(max l / T), which
    // is max fl(l / T) since rounding is monotone; only the id of a +inf
    // key needs the exact keys (their lowest id), so such rows rescan
    bool resc = false;
    if (tid < kGroupRows) {
        const uint64_t bw = s_best[tid];
        const float T = s_T[tid];
        if (a.mode == 1 && bw != 0ull && samples(T)) {
            const uint32_t o = packed_ordered(bw);
            if (o != 0xffffffffu) {
                const float k = __fdiv_rn(key_from_ordered(o), T);
                if (k == __uint_as_float(0x7f800000u))
                    resc = true;
                else
                    s_best[tid] = pack_key(k, packed_id(bw));
            }
        }
        s_resc[tid] = resc;
    }
    if (__syncthreads_or(resc)) {
        // rare: the lowest id of this block whose key fl(l / T) is +inf
        for (int rr = 0; rr < kGroupRows; ++rr) {
            if (!s_resc[rr]) continue;
            const float T = s_T[rr];
            for (int v = v_begin + tid; v < v_end; v += kBatchThreads) {
                if (__fdiv_rn(cache_value(a, row0 + rr, i, v), T) == __uint_as_float(0x7f800000u)) {
                    atomicMin(&s_vmin, (unsigned int)v);
                    break;
                }
            }
            __syncthreads();
            if (tid == 0) {
                s_best[rr] = pack_key(__uint_as_float(0x7f800000u), s_vmin);
                s_vmin = 0xffffffffu;
            }
            __syncthreads();
        }
    }
    // the block's best per row into the row's winner word
    if (tid < kGroupRows && s_best[tid]) atomicMax(win_slot(a, i, row0 + tid), s_best[tid]);
    if (!last_block(group_counter(a, i, blockIdx.y), (uint32_t)nblk, &s_flag)) return;

    // last block of the row group: every block's maximum is in
    if (tid == 0) *group_counter(a, i, blockIdx.y) = 0u;
    const int b = row0 + tid;
    if (tid < kGroupRows && row_live(a, b)) {
        unsigned long long *ws = win_slot(a, i, b);
        const uint64_t win = __ldcg(ws);
        const float T = s_T[tid];
        if (a.mode == 0 || !samples(T) || !needs_sums(win)) {
            a.tokens[b * a.tok_s0 + i] = direct_token(a, win, T);
            *ws = 0ull;
        }
    }
}

// Eight consecutive cached logits as fp32, read once more (the cache's last
// read of the position: evict-first in L2).
__device__ __forceinline__ void cache8_last(const SampleArgs &a, int b, int i, int v, uint64_t pol,
                                            float (&x)[8]) {
    const int64_t o = b * a.cache_s0 + (int64_t)i * a.cache_s1 + v;
    if (a.cache_f) {
        const uint4 p = tc::ld_nc_v4_hint(a.cache_f + o, pol);
        const uint4 q = tc::ld_nc_v4_hint(a.cache_f + o + 4, pol);
        x[0] = __uint_as_float(p.x); x[1] = __uint_as_float(p.y);
        x[2] = __uint_as_float(p.z); x[3] = __uint_as_float(p.w);
        x[4] = __uint_as_float(q.x); x[5] = __uint_as_float(q.y);
        x[6] = __uint_as_float(q.z); x[7] = __uint_as_float(q.w);
    } else {
        const uint4 p = tc::ld_nc_v4_hint(a.cache + o, pol);
        const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = __uint_as_float(w[k] << 16);
            x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    }
}

// The inverse-CDF step of position i for the rows the logits kernel left
// open: grid (blocks of kCdfIds ids, rows).  A block's warp takes 256
// consecutive ids per round (8 per lane), so each (round, warp) is one
// 256-id unit of the vocabulary; its weight sum goes to the row's unit
// array (a.sums + b nu, in id order).  The last block of the row scans the
// unit sums for the target mulhi64(H, S), then one warp re-reads the target
// unit's 256 ids and scans their weights for the token.
__global__ void __launch_bounds__(kBatchThreads, 4)
batch_cdf_kernel(const SampleArgs a, int i, int nb2, int nu) {
    __shared__ unsigned long long s_w[kBW];
    __shared__ unsigned long long s_pre, s_target;
    __shared__ int s_unit, s_flag;
    const int b = blockIdx.y, c = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_trigger();
    pdl_wait();
    // the row's state, temperature and winner word in one round trip (b < rows)
    unsigned long long *ws = win_slot(a, i, b);
    const int64_t idx = a.row_state_idx[b];
    const float T = a.temperature[b];
    const uint64_t win = __ldcg(ws);
    // padding, or a row whose token the logits kernel's last block wrote
    if (idx < 0 || win == 0ull) return;
    if (!samples(T) || !needs_sums(win)) {
        // decided by its maximum (greedy, a NaN, +inf, all -inf): the row's
        // first block writes the token (the tcgen05 logits kernel leaves it)
        if (c == 0 && tid == 0) {
            a.tokens[b * a.tok_s0 + i] = direct_token(a, win, T);
            *ws = 0ull;
        }
        return;
    }
    const float M = key_from_ordered(packed_ordered(win));
    const bool p2 = dm_pow2_temperature(T);
    const float rT = p2 ? __frcp_rn(T) : 0.0f;
    const uint64_t pol = tc::policy_evict_first();
    uint64_t *units = a.sums + (int64_t)b * nu;

    // every round's 8 logits are loaded before any weight
    const int v0 = c * kCdfIds;
    float x[kCdfRounds][8];
    bool ok[kCdfRounds];
#pragma unroll
    for (int r = 0; r < kCdfRounds; ++r) {
        const int vv = v0 + r * (8 * kBatchThreads) + tid * 8;
        ok[r] = vv < a.V;
        if (ok[r]) cache8_last(a, b, i, vv, pol, x[r]);
    }
#pragma unroll
    for (int r = 0; r < kCdfRounds; ++r) {
        uint64_t part = 0ull;
        if (ok[r]) part = p2 ? cdf_weight8<true>(x[r], T, rT, M) : cdf_weight8<false>(x[r], T, rT, M);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        const int u = (c * kCdfRounds + r) * kBW + warp;
        if (lane == 0 && u < nu) units[u] = part;
    }
    if (!last_block(row_counter(a, i, b), (uint32_t)nb2, &s_flag)) return;

    // last block of the row: the unit whose prefix range holds the target;
    // thread t takes units 4t .. 4t + 3 (nu <= 4 kBatchThreads)
    if (tid == 0) {
        *row_counter(a, i, b) = 0u;
        s_unit = -1;
    }
    uint64_t w4[4];
    uint64_t mine = 0ull;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int u = 4 * tid + k;
        w4[k] = u < nu ? __ldcg(reinterpret_cast<const unsigned long long *>(units) + u) : 0ull;
        mine += w4[k];
    }
    uint64_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    uint64_t wpre = 0ull, S = 0ull;
#pragma unroll
    for (int w = 0; w < kBW; ++w) {
        wpre += w < warp ? s_w[w] : 0ull;
        S += s_w[w];
    }
    const uint64_t target =
        __umul64hi(dm_cdf_hash(dm_row_step_hash((uint64_t)a.seeds[b], (uint32_t)b, (uint32_t)i)), S);
    uint64_t pre = wpre + incl - mine;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (w4[k] && pre <= target && target < pre + w4[k]) {
            s_unit = 4 * tid + k;
            s_pre = pre;
            s_target = target;
        }
        pre += w4[k];
    }
    __syncthreads();
    const int u = s_unit;
    if (warp != 0) return;
    int64_t tok = -1;
    if (u >= 0) {
        // the target unit: lane l takes ids 256 u + 8 l .. + 7, in order
        const uint64_t tgt = s_target;
        const int v = u * 256 + lane * 8;
        float y[8];
        uint64_t wl = 0ull;
        if (v < a.V) {
            cache8_last(a, b, i, v, pol, y);
            wl = p2 ? cdf_weight8<true>(y, T, rT, M) : cdf_weight8<false>(y, T, rT, M);
        }
        uint64_t inc = wl;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t z = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += z;
        }
        uint64_t run = s_pre + inc - wl;
        int hit = -1;
        if (wl && run <= tgt && tgt < run + wl) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                run += p2 ? cdf_weight_of<true>(y[e], T, rT, M) : cdf_weight_of<false>(y[e], T, rT, M);
                if (hit < 0 && run > tgt) hit = e;
            }
        }
        const unsigned m = __ballot_sync(0xffffffffu, hit >= 0);
        if (m) {
            const int src = __ffs(m) - 1;
            const int h = __shfl_sync(0xffffffffu, hit, src);
            tok = (int64_t)u * 256 + src * 8 + h;
        }
    }
    if (lane == 0) {
        if (tok < 0) {
            set_status(a.status, 6u /* MARKOV_EDEVICE */, 0x200u + i);
            tok = 0;
        }
        a.tokens[b * a.tok_s0 + i] = tok;
        *ws = 0ull;
    }
}

int batch_blocks(int V) {
    // about two blocks per SM on a 152-SM part; at least one tile per warp
    int nt = V / kTile;
    int nblk = 304;
    if (nblk > nt / kBW) nblk = nt / kBW > 0 ? nt / kBW : 1;
    return nblk;
}

// One launch of the path; pdl: as a programmatic dependent of the launch
// before it on the stream.
template <typename... Params, typename... Args>
static cudaError_t launch_one(void (*kernel)(Params...), dim3 grid, size_t smem,
                              cudaStream_t stream, bool pdl, Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kBatchThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int MT>
static void (*logits_kernel(int r, bool base_f32))(const SampleArgs, int) {
    switch (r) {
        case 64: return base_f32 ? batch_logits_kernel<64, true, MT> : batch_logits_kernel<64, false, MT>;
        case 128:
            return base_f32 ? batch_logits_kernel<128, true, MT> : batch_logits_kernel<128, false, MT>;
        case 256:
            return base_f32 ? batch_logits_kernel<256, true, MT> : batch_logits_kernel<256, false, MT>;
        default: return nullptr;
    }
}

cudaError_t launch_batch(const SampleArgs &a, cudaStream_t stream, int *launches, const CUtensorMap *tmap,
                         int sms) {
    // the launch variant by row count: 16-row groups (whole-tile head
    // prefetch) up to 16 rows, 32-row groups above
    const int mt = a.rows <= 16 ? 1 : 2;
    const int group_rows = 16 * mt;
    const int groups = (a.rows + group_rows - 1) / group_rows;
    // one wave: the plan's vocab blocks shared out over the row groups
    const int nblk = a.grid / groups > 0 ? a.grid / groups : 1;
    const int nb2 = (a.V + kCdfIds - 1) / kCdfIds;
    const int nu = (a.V + 255) / 256;            // 256-id weight units per row
    const size_t smem = (size_t)group_rows * (a.r + kBPad) * sizeof(uint16_t);
    *launches = 0;
    if (nb2 > 64 || a.rows > kMaxRows || a.N > kMaxSteps) return cudaErrorInvalidValue;
    void (*logits)(const SampleArgs, int) =
        mt == 1 ? logits_kernel<1>(a.r, a.base_f != nullptr) : logits_kernel<2>(a.r, a.base_f != nullptr);
    if (!logits) return cudaErrorInvalidValue;
    // the tcgen05 logits kernel: row groups of 64, one CTA per SM shared out
    // over the groups, each CTA a contiguous run of 128-id tiles
    const int tgroups = (a.rows + 63) / 64;
    const int tiles = (a.V + 127) / 128;
    int tctas = sms > 0 ? sms / tgroups : 1;
    if (tctas < 1) tctas = 1;
    if (tctas > tiles) tctas = tiles;
    int n = 0;
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < a.N && e == cudaSuccess; ++i) {
        // the first launch of a call waits for the stream as usual
        if (tmap)
            e = launch_batch_tc_logits(a, *tmap, i, tctas, stream, i > 0);
        else
            e = launch_one(logits, dim3(nblk, groups), smem, stream, i > 0, a, i);
        ++n;
        if (e == cudaSuccess && a.mode == 1) {
            e = launch_one(batch_cdf_kernel, dim3(nb2, a.rows), 0, stream, true, a, i, nb2, nu);
            ++n;
        }
    }
    *launches = n;
    return e;
}

}  // namespace dtm
