// chain.cu -- the persistent Markov chain kernel: all N draft positions of up
// to 8 request rows in one cooperative launch.
//
// Design (sharded_markov page, module docstring: one cooperative kernel runs
// the whole chain; up to 8 request rows are the columns of the tensor-core
// MMA; each shard agrees on the position's winner through one 64-bit
// (score, index) key): here the shards are the CTAs of one GPU.  CTA c owns a
// contiguous range of 16-id vocab tiles.  Per position i:
//   1. every CTA stages markov_embed[p_b] of the live rows in shared memory;
//   2. each warp computes bias tiles [16 ids x 8 rows] with
//      mma.m16n8k16 (BF16 in, fp32 accumulate), head rows read from L2/HBM
//      with 16-byte loads, and runs the epilogue in registers: BF16 rounding,
//      base add, transform, cache store and the row's key;
//   3. the CTA's best (key, id) per row goes to a slot; one bounded grid
//      barrier; every CTA reduces the slots of all CTAs and so knows the
//      winner, which is token i and the next position's previous token.
// In inverse-CDF mode two more barriers follow: once the row maximum M is
// known, every CTA sums its integer weights floor(exp(x - M) 2^40); once the
// sums are known, the one CTA whose prefix range holds the target
// mulhi64(H, S) scans its slice for the token.
#include "common.cuh"
#include "mma_tile.cuh"

namespace dtm {

namespace {

constexpr int kWarps = kChainThreads / 32;

// Per-row state of one launch, in shared memory.
struct RowState {
    int live[kChainRows];
    int sampling[kChainRows];      // T > 0
    float T[kChainRows];
    uint64_t seed[kChainRows];
    int64_t prev[kChainRows];
};

}  // namespace

template <int RANK>
__global__ void __launch_bounds__(kChainThreads, 1) chain_kernel(const SampleArgs a) {
    __shared__ __align__(16) uint16_t e_smem[kChainRows * (RANK + kEPad)];
    __shared__ RowState rs;
    __shared__ unsigned long long s_best[kChainRows];
    __shared__ unsigned long long s_sum[kChainRows];
    __shared__ uint64_t s_win[kChainRows];
    __shared__ uint32_t s_flag;
    __shared__ uint32_t s_base;
    __shared__ uint64_t s_scan[kChainThreads / 32];
    __shared__ uint64_t s_tot, s_pre;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int G = gridDim.x, cta = blockIdx.x;
    const int R = a.rows, N = a.N, V = a.V;
    const int ntiles = V / kTile;
    const int tile_begin = (int)((int64_t)cta * ntiles / G);
    const int tile_end = (int)((int64_t)(cta + 1) * ntiles / G);
    const int v_begin = tile_begin * kTile, v_end = tile_end * kTile;
    const int Gp = (G + kKeyPad - 1) / kKeyPad * kKeyPad;

    if (tid < kChainRows) {
        int b = tid;
        bool live = b < R && a.row_state_idx[b] >= 0;
        rs.live[b] = live;
        float T = live ? a.temperature[b] : 0.0f;
        rs.T[b] = T;
        rs.sampling[b] = live && samples(T);
        rs.seed[b] = live ? (uint64_t)a.seeds[b] : 0ull;
        int64_t p = live ? (int64_t)a.anchor[b] : 0;
        if (p < 0 || p >= V) {         // an anchor outside the vocabulary
            set_status(a.status, 1u /* MARKOV_EINVAL */, 0x100u + b);
            p = 0;
        }
        rs.prev[b] = p;
    }
    if (tid == 0) s_base = *(volatile uint32_t *)a.bar_base;
    __syncthreads();
    const uint32_t base = s_base;
    uint32_t epoch = 0;

    for (int i = 0; i < N; ++i) {
        // 1. stage the previous tokens' embeddings (zeros for absent rows)
        for (int idx = tid; idx < kChainRows * (RANK / 8); idx += kChainThreads) {
            int b = idx / (RANK / 8), c = idx % (RANK / 8);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (rs.live[b])
                v = *reinterpret_cast<const uint4 *>(a.embed + rs.prev[b] * RANK + 8 * c);
            *reinterpret_cast<uint4 *>(e_smem + b * (RANK + kEPad) + 8 * c) = v;
        }
        if (tid < kChainRows) s_best[tid] = 0ull;
        __syncthreads();

        // 2. bias tiles, epilogue, per-row best key
        uint64_t best0 = 0ull, best1 = 0ull;      // rows 2t, 2t+1
        const int r0 = 2 * t, r1 = 2 * t + 1;
        const bool l0 = rs.live[r0], l1 = rs.live[r1];
        const float T0 = rs.T[r0], T1 = rs.T[r1];
        const bool s0 = rs.sampling[r0], s1 = rs.sampling[r1];
        for (int tile = tile_begin + warp; tile < tile_end; tile += kWarps) {
            const int v0 = tile * kTile;
            float acc[4];
            bias_tile<RANK>(a.head, v0, e_smem, g, t, acc);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = (e & 1) ? r1 : r0;
                const bool live = (e & 1) ? l1 : l0;
                if (!live) continue;
                const int v = v0 + g + ((e & 2) ? 8 : 0);
                const float lf = logit_value(base_value(a, row, i, v), acc[e], a.tf, a.cache_f != nullptr);
                cache_put(a, row, i, v, lf);
                const bool smp = (e & 1) ? s1 : s0;
                float key = lf;
                if (smp) {
                    key = __fdiv_rn(lf, (e & 1) ? T1 : T0);
                    if (a.mode == 0)
                        key = __fadd_rn(key, a.noise[(int64_t)(row * N + i) * a.noise_s0 + v]);
                }
                const uint64_t pk = pack_key(key, (uint32_t)v);
                if (e & 1) best1 = pk > best1 ? pk : best1;
                else best0 = pk > best0 ? pk : best0;
            }
        }
        // reduce over the 8 lanes that share t (lane bits 2..4)
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            uint64_t w0 = __shfl_xor_sync(0xffffffffu, best0, o);
            uint64_t w1 = __shfl_xor_sync(0xffffffffu, best1, o);
            best0 = w0 > best0 ? w0 : best0;
            best1 = w1 > best1 ? w1 : best1;
        }
        if (g == 0) {
            if (l0) atomicMax(&s_best[r0], (unsigned long long)best0);
            if (l1) atomicMax(&s_best[r1], (unsigned long long)best1);
        }
        __syncthreads();

        // 3. publish, barrier, reduce over all CTAs
        uint64_t *slots = a.keys + (int64_t)(i * 2 + 0) * kChainRows * Gp;
        if (tid < kChainRows && rs.live[tid]) slots[tid * Gp + cta] = s_best[tid];
        if (!grid_barrier(a.bar_count, base + (++epoch) * (uint32_t)G, a.status, a.timeout_ns,
                          (uint32_t)(i * 4 + 1), &s_flag))
            return;
        if (warp < kChainRows && rs.live[warp]) {
            uint64_t m = 0ull;
            for (int c = lane; c < G; c += 32) {
                uint64_t k = ld_cg_u64(slots + warp * Gp + c);
                m = k > m ? k : m;
            }
            m = warp_max_u64_shfl(m);
            if (lane == 0) s_win[warp] = m;
        }
        __syncthreads();

        // 4. inverse CDF: rows whose maximum is finite need the weight sums
        bool cdf_any = false;
        if (a.mode == 1) {
            for (int b = 0; b < R && b < kChainRows; ++b) {
                if (!rs.sampling[b]) continue;
                uint32_t o = packed_ordered(s_win[b]);
                float M = key_from_ordered(o);
                if (o != 0xffffffffu && M != __uint_as_float(0x7f800000u) &&
                    M != __uint_as_float(0xff800000u))
                    cdf_any = true;
            }
        }
        if (cdf_any) {
            if (tid < kChainRows) s_sum[tid] = 0ull;
            __syncthreads();
            for (int b = 0; b < R && b < kChainRows; ++b) {
                if (!rs.sampling[b]) continue;
                uint32_t o = packed_ordered(s_win[b]);
                const float M = key_from_ordered(o);
                if (o == 0xffffffffu || M == __uint_as_float(0x7f800000u) ||
                    M == __uint_as_float(0xff800000u))
                    continue;
                uint64_t part = 0ull;
                for (int v = v_begin + tid; v < v_end; v += kChainThreads) {
                    float x = __fdiv_rn(cache_value(a, b, i, v), rs.T[b]);
                    part += dm_cdf_weight(__fsub_rn(x, M));
                }
#pragma unroll
                for (int o2 = 16; o2 > 0; o2 >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o2);
                if (lane == 0) atomicAdd(&s_sum[b], (unsigned long long)part);
            }
            __syncthreads();
            uint64_t *sums = a.sums + (int64_t)i * kChainRows * Gp;
            uint64_t *tok_slot = a.keys + (int64_t)(i * 2 + 1) * kChainRows * Gp;
            if (tid < kChainRows && rs.sampling[tid]) {
                sums[tid * Gp + cta] = s_sum[tid];
                if (cta == 0) tok_slot[tid] = (uint64_t)V;   // no token yet
            }
            if (!grid_barrier(a.bar_count, base + (++epoch) * (uint32_t)G, a.status,
                              a.timeout_ns, (uint32_t)(i * 4 + 2), &s_flag))
                return;
            for (int b = 0; b < R && b < kChainRows; ++b) {
                if (!rs.sampling[b]) continue;
                uint32_t o = packed_ordered(s_win[b]);
                const float M = key_from_ordered(o);
                if (o == 0xffffffffu || M == __uint_as_float(0x7f800000u) ||
                    M == __uint_as_float(0xff800000u))
                    continue;
                // total S and this CTA's prefix, from every CTA's sum
                if (warp == 0) {
                    uint64_t tot = 0ull, pre = 0ull;
                    for (int c = lane; c < G; c += 32) {
                        uint64_t s = ld_cg_u64(sums + b * Gp + c);
                        tot += s;
                        if (c < cta) pre += s;
                    }
#pragma unroll
                    for (int o2 = 16; o2 > 0; o2 >>= 1) {
                        tot += __shfl_xor_sync(0xffffffffu, tot, o2);
                        pre += __shfl_xor_sync(0xffffffffu, pre, o2);
                    }
                    if (lane == 0) { s_tot = tot; s_pre = pre; }
                }
                __syncthreads();
                const uint64_t S = s_tot, P = s_pre, Sc = s_sum[b];
                const uint64_t H = dm_cdf_hash(dm_row_step_hash(rs.seed[b], (uint32_t)b, (uint32_t)i));
                const uint64_t target = __umul64hi(H, S);
                if (P <= target && target < P + Sc) {
                    // this CTA holds the token: each thread takes a contiguous
                    // chunk of the slice, chunk sums are scanned across the CTA
                    const int len = v_end - v_begin;
                    const int chunk = (len + kChainThreads - 1) / kChainThreads;
                    const int c0 = v_begin + tid * chunk;
                    const int c1 = min(c0 + chunk, v_end);
                    uint64_t mine = 0ull;
                    for (int v = c0; v < c1; ++v) {
                        float x = __fdiv_rn(cache_value(a, b, i, v), rs.T[b]);
                        mine += dm_cdf_weight(__fsub_rn(x, M));
                    }
                    // exclusive scan of `mine` over the CTA, in thread order
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
                    uint64_t run = P + wpre + incl - mine;
                    if (run <= target && target < run + mine) {
                        for (int v = c0; v < c1; ++v) {
                            float x = __fdiv_rn(cache_value(a, b, i, v), rs.T[b]);
                            run += dm_cdf_weight(__fsub_rn(x, M));
                            if (run > target) {
                                tok_slot[b] = (uint64_t)v;
                                break;
                            }
                        }
                    }
                }
                __syncthreads();
            }
            if (!grid_barrier(a.bar_count, base + (++epoch) * (uint32_t)G, a.status,
                              a.timeout_ns, (uint32_t)(i * 4 + 3), &s_flag))
                return;
            if (tid < kChainRows && rs.sampling[tid]) {
                uint32_t o = packed_ordered(s_win[tid]);
                const float M = key_from_ordered(o);
                if (!(o == 0xffffffffu || M == __uint_as_float(0x7f800000u) ||
                      M == __uint_as_float(0xff800000u))) {
                    uint64_t v = ld_cg_u64(tok_slot + tid);
                    if (v >= (uint64_t)V) {           // no CTA found the target
                        set_status(a.status, 6u /* MARKOV_EDEVICE */, (uint32_t)(i * 4 + 3));
                        v = 0ull;
                    }
                    s_win[tid] = (s_win[tid] & 0xffffffff00000000ull) | (0xffffffffull - v);
                }
            }
            __syncthreads();
        }

        // 5. the token: all -inf inverse-CDF rows take id 0
        if (tid < kChainRows && rs.live[tid]) {
            const int b = tid;
            uint32_t id = packed_id(s_win[b]);
            if (a.mode == 1 && rs.sampling[b]) {
                uint32_t o = packed_ordered(s_win[b]);
                if (o != 0xffffffffu && key_from_ordered(o) == __uint_as_float(0xff800000u)) id = 0u;
            }
            rs.prev[b] = (int64_t)id;
            if (cta == 0) a.tokens[b * a.tok_s0 + i] = (int64_t)id;
        }
        __syncthreads();
    }
    if (cta == 0 && tid == 0) *(volatile uint32_t *)a.bar_base = base + epoch * (uint32_t)G;
}

cudaError_t chain_occupancy(int *blocks_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, chain_kernel<256>,
                                                         kChainThreads, 0);
}

cudaError_t launch_chain(const SampleArgs &a, cudaStream_t stream) {
    void *args[] = {(void *)&a};
    const void *fn = nullptr;
    switch (a.r) {
        case 64: fn = (const void *)chain_kernel<64>; break;
        case 128: fn = (const void *)chain_kernel<128>; break;
        case 256: fn = (const void *)chain_kernel<256>; break;
        default: return cudaErrorInvalidValue;
    }
    return cudaLaunchCooperativeKernel(fn, dim3(a.grid), dim3(kChainThreads), args, 0, stream);
}

}  // namespace dtm
