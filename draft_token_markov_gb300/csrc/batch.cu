// batch.cu -- the per-position path for batches above the chain limit
// (fused_markov page, FusedMarkovSampler: per draft position a bias
// contraction plus a logits kernel over (row, vocab block) and a per-row
// select kernel; sharded_markov page, module docstring: batches above
// max_rows take this loop).
//
// Per position i, in launch order on one stream:
//   logits  grid (blocks, row groups of 64): bias tiles [16 ids x 64 rows] by
//           mma.m16n8k16 with the previous tokens' embeddings staged in
//           shared memory, the epilogue (BF16 rounding, base add, transform,
//           cache store) and each block's best (key, id) per row;
//   cdfsum  (inverse CDF only) grid (blocks, rows): the block's integer
//           weight sum floor(exp(x - M) 2^40) once M is reduced;
//   pick    grid (rows): reduce the blocks' partials; in inverse-CDF mode find
//           the block whose prefix holds mulhi64(H, S) and scan it.
// The next position's logits kernel reads token i from draft_tokens.
#include "common.cuh"

namespace dtm {

namespace {

constexpr int kBW = kBatchThreads / 32;    // warps per block
constexpr int kGroupRows = 64;             // rows per row group (8 MMA n-tiles)
constexpr int kNT = kGroupRows / 8;
constexpr int kBPad = 32;

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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

}  // namespace

template <int RANK>
__global__ void __launch_bounds__(kBatchThreads)
batch_logits_kernel(const SampleArgs a, int i) {
    extern __shared__ __align__(16) uint16_t e_smem[];      // [64][RANK + kBPad]
    __shared__ unsigned long long s_best[kGroupRows];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int blk = blockIdx.x, nblk = gridDim.x;
    const int row0 = blockIdx.y * kGroupRows;
    const int V = a.V;
    int v_begin, v_end;
    block_range(V, nblk, blk, v_begin, v_end);

    for (int idx = tid; idx < kGroupRows * (RANK / 8); idx += kBatchThreads) {
        int b = idx / (RANK / 8), c = idx % (RANK / 8);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row_live(a, row0 + b)) {
            int64_t p = prev_token(a, row0 + b, i);
            if (p >= 0 && p < V) v = *reinterpret_cast<const uint4 *>(a.embed + p * RANK + 8 * c);
        }
        *reinterpret_cast<uint4 *>(e_smem + b * (RANK + kBPad) + 8 * c) = v;
    }
    if (tid < kGroupRows) s_best[tid] = 0ull;
    __syncthreads();

    // rows handled by this thread: row0 + 8 nt + 2t + {0, 1}
    uint64_t best[kNT][2];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) best[nt][0] = best[nt][1] = 0ull;
    const int ngroups = min(kNT, (a.rows - row0 + 7) / 8);

    for (int v0 = v_begin + warp * kTile; v0 < v_end; v0 += kBW * kTile) {
        float acc[kNT][4];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
        const uint16_t *ha = a.head + (int64_t)(v0 + g) * RANK + 8 * t;
        const uint16_t *hb = ha + 8 * RANK;
#pragma unroll 2
        for (int j = 0; j < RANK / 32; ++j) {
            uint4 x = *reinterpret_cast<const uint4 *>(ha + 32 * j);
            uint4 y = *reinterpret_cast<const uint4 *>(hb + 32 * j);
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
                if (nt >= ngroups) break;
                uint4 e = *reinterpret_cast<const uint4 *>(e_smem + (nt * 8 + g) * (RANK + kBPad) +
                                                           8 * t + 32 * j);
                mma16816(acc[nt], x.x, y.x, x.y, y.y, e.x, e.y);
                mma16816(acc[nt], x.z, y.z, x.w, y.w, e.z, e.w);
            }
        }
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
            if (nt >= ngroups) break;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = row0 + nt * 8 + 2 * t + (e & 1);
                if (!row_live(a, row)) continue;
                const int v = v0 + g + ((e & 2) ? 8 : 0);
                const float l = logit_value(base_value(a, row, i, v), acc[nt][e], a.tf,
                                            a.cache_f != nullptr);
                cache_put(a, row, i, v, l);
                const float T = a.temperature[row];
                float key = l;
                if (samples(T)) {
                    key = __fdiv_rn(key, T);
                    if (a.mode == 0)
                        key = __fadd_rn(key, a.noise[(int64_t)(row * a.N + i) * a.noise_s0 + v]);
                }
                const uint64_t pk = pack_key(key, (uint32_t)v);
                best[nt][e & 1] = pk > best[nt][e & 1] ? pk : best[nt][e & 1];
            }
        }
    }
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint64_t v = best[nt][h];
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
                v = w > v ? w : v;
            }
            if (g == 0 && v) atomicMax(&s_best[nt * 8 + 2 * t + h], (unsigned long long)v);
        }
    }
    __syncthreads();
    if (tid < kGroupRows && row0 + tid < a.rows)
        a.keys[(int64_t)(row0 + tid) * nblk + blk] = s_best[tid];
}

// Reduce the blocks' partial maxima of one row (the packed key).
__device__ uint64_t reduce_partials(const SampleArgs &a, int b, int nblk, uint64_t *s_red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint64_t m = 0ull;
    for (int c = tid; c < nblk; c += blockDim.x) {
        uint64_t k = a.keys[(int64_t)b * nblk + c];
        m = k > m ? k : m;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        uint64_t w = __shfl_xor_sync(0xffffffffu, m, o);
        m = w > m ? w : m;
    }
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    uint64_t r = 0ull;
    for (int w = 0; w < (int)(blockDim.x / 32); ++w) r = s_red[w] > r ? s_red[w] : r;
    __syncthreads();
    return r;
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

__global__ void __launch_bounds__(kBatchThreads)
batch_cdfsum_kernel(const SampleArgs a, int i, int nblk) {
    __shared__ uint64_t s_red[kBatchThreads / 32];
    __shared__ unsigned long long s_sum;
    const int b = blockIdx.y, blk = blockIdx.x;
    if (!row_live(a, b) || !samples(a.temperature[b])) return;
    const uint64_t win = reduce_partials(a, b, nblk, s_red);
    if (!needs_sums(win)) return;
    const float M = key_from_ordered(packed_ordered(win));
    const float T = a.temperature[b];
    int v0, v1;
    block_range(a.V, nblk, blk, v0, v1);
    if (threadIdx.x == 0) s_sum = 0ull;
    __syncthreads();
    uint64_t part = 0ull;
    for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
        float x = __fdiv_rn(cache_value(a, b, i, v), T);
        part += (uint64_t)__float2ull_rz(__fmul_rn(dm_exp(__fsub_rn(x, M)), 0x1p40f));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if ((threadIdx.x & 31) == 0) atomicAdd(&s_sum, (unsigned long long)part);
    __syncthreads();
    if (threadIdx.x == 0) a.sums[(int64_t)b * nblk + blk] = s_sum;
}

__global__ void __launch_bounds__(kBatchThreads)
batch_pick_kernel(const SampleArgs a, int i, int nblk) {
    __shared__ uint64_t s_red[kBatchThreads / 32];
    __shared__ uint64_t s_scan[kBatchThreads / 32];
    __shared__ uint64_t s_blkpre;
    __shared__ int s_blk;
    __shared__ int64_t s_tok;
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (!row_live(a, b)) return;
    const uint64_t win = reduce_partials(a, b, nblk, s_red);
    const float T = a.temperature[b];
    int64_t tok = (int64_t)packed_id(win);
    if (a.mode == 1 && samples(T)) {
        uint32_t o = packed_ordered(win);
        if (o != 0xffffffffu && key_from_ordered(o) == __uint_as_float(0xff800000u)) tok = 0;
        if (needs_sums(win)) {
            const float M = key_from_ordered(o);
            const uint64_t *sums = a.sums + (int64_t)b * nblk;
            // total and the block holding the target (serial over blocks: few hundred)
            if (tid == 0) {
                uint64_t S = 0ull;
                for (int c = 0; c < nblk; ++c) S += sums[c];
                const uint64_t H = dm_cdf_hash(dm_row_step_hash((uint64_t)a.seeds[b], (uint32_t)b,
                                                                (uint32_t)i));
                const uint64_t target = __umul64hi(H, S);
                uint64_t pre = 0ull;
                int c = 0;
                for (; c < nblk; ++c) {
                    if (target < pre + sums[c]) break;
                    pre += sums[c];
                }
                s_blk = c < nblk ? c : nblk - 1;
                s_blkpre = pre;
                s_red[0] = target;
                s_tok = -1;
            }
            __syncthreads();
            const uint64_t target = s_red[0];
            int v0, v1;
            block_range(a.V, nblk, s_blk, v0, v1);
            const int len = v1 - v0;
            const int chunk = (len + kBatchThreads - 1) / kBatchThreads;
            const int c0 = v0 + tid * chunk, c1 = min(c0 + chunk, v1);
            uint64_t mine = 0ull;
            for (int v = c0; v < c1; ++v) {
                float x = __fdiv_rn(cache_value(a, b, i, v), T);
                mine += (uint64_t)__float2ull_rz(__fmul_rn(dm_exp(__fsub_rn(x, M)), 0x1p40f));
            }
            uint64_t incl = mine;
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) {
                uint64_t y = __shfl_up_sync(0xffffffffu, incl, o2);
                if (lane >= o2) incl += y;
            }
            if (lane == 31) s_scan[warp] = incl;
            __syncthreads();
            uint64_t wpre = 0ull;
            for (int w = 0; w < warp; ++w) wpre += s_scan[w];
            uint64_t run = s_blkpre + wpre + incl - mine;
            if (run <= target && target < run + mine) {
                for (int v = c0; v < c1; ++v) {
                    float x = __fdiv_rn(cache_value(a, b, i, v), T);
                    run += (uint64_t)__float2ull_rz(__fmul_rn(dm_exp(__fsub_rn(x, M)), 0x1p40f));
                    if (run > target) {
                        s_tok = v;
                        break;
                    }
                }
            }
            __syncthreads();
            tok = s_tok;
            if (tok < 0) {
                if (tid == 0) set_status(a.status, 6u /* MARKOV_EDEVICE */, 0x200u + i);
                tok = 0;
            }
        }
    }
    if (tid == 0) a.tokens[b * a.tok_s0 + i] = tok;
}

int batch_blocks(int V) {
    // about two blocks per SM on a 152-SM part; at least one tile per warp
    int nt = V / kTile;
    int nblk = 304;
    if (nblk > nt / kBW) nblk = nt / kBW > 0 ? nt / kBW : 1;
    return nblk;
}

cudaError_t launch_batch(const SampleArgs &a, cudaStream_t stream, int *launches) {
    const int nblk = a.grid;
    const int groups = (a.rows + kGroupRows - 1) / kGroupRows;
    const size_t smem = (size_t)kGroupRows * (a.r + kBPad) * sizeof(uint16_t);
    int n = 0;
    for (int i = 0; i < a.N; ++i) {
        dim3 grid(nblk, groups);
        switch (a.r) {
            case 64: batch_logits_kernel<64><<<grid, kBatchThreads, smem, stream>>>(a, i); break;
            case 128: batch_logits_kernel<128><<<grid, kBatchThreads, smem, stream>>>(a, i); break;
            case 256: batch_logits_kernel<256><<<grid, kBatchThreads, smem, stream>>>(a, i); break;
            default: return cudaErrorInvalidValue;
        }
        ++n;
        if (a.mode == 1) {
            batch_cdfsum_kernel<<<dim3(nblk, a.rows), kBatchThreads, 0, stream>>>(a, i, nblk);
            ++n;
        }
        batch_pick_kernel<<<a.rows, kBatchThreads, 0, stream>>>(a, i, nblk);
        ++n;
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    *launches = n;
    return cudaSuccess;
}

}  // namespace dtm
