// sharded.cu -- the vocabulary-sharded chain of the sharded_markov page, its
// ranks emulated as groups of CTAs of one cooperative launch on one GPU.
//
// The page's design (module docstring and "Per call" diagram): rank k of
// `world` owns head rows [k V / world, (k + 1) V / world).  Per draft
// position every rank computes its shard's logits, writes them into its own
// cache and into every peer's staging buffer, takes its shard's best key
// (fp32(l / T) + gumbel, or l at T = 0; lowest id among equal keys, a NaN
// above all) and exchanges one 64-bit key per (rank, row, position) through
// a mailbox in every peer's memory; the best key of the world is the
// position's token on every rank.  After the last position each rank copies
// its peers' columns from its staging buffer into its cache, so every rank
// ends with the full-vocabulary cache.  The page samples Gumbel-max (and
// argmax at T = 0); so does this kernel.
//
// Emulation: CTA c belongs to rank c / Gr and takes a contiguous run of
// 16-id tiles of that rank's shard (the bias tile of the simple chain:
// mma.sync m16n8k16, head rows read with 16-byte loads).  Everything a rank
// owns lives in its own allocations: head shard (the caller's), noise shard,
// staging buffer, mailbox, CTA slots, outputs.  A rank writes into a peer's
// memory only what the page sends through its peer mappings: the staging
// copy of its logits and its mailbox key.  Inside a rank the CTAs agree
// through tagged slots in the rank's memory, read by the rank's first CTA;
// across ranks through the mailboxes.  Keys carry the call's epoch in their
// low 14 bits, so no slot is cleared between calls; every wait is
// bounded.  With one GPU per rank the same protocol runs on peer-mapped
// memory with system-scope release and acquire; here the ranks share one
// GPU, so GPU scope orders them.
#include <cmath>
#include <cstring>

#include "../../include/markov.h"
#include "common.cuh"
#include "internal.h"
#include "mma_tile.cuh"

namespace dtm {

namespace {

constexpr int kMaxWorld = 8;
constexpr int kShThreads = kChainThreads;
constexpr int kShWarps = kShThreads / 32;
constexpr int kShPer = 5;              // slots a lane reads per poll round (Gr <= 160)

struct ShardedArgs {
    const uint16_t *base;              // [rows, N, V] full-vocabulary base logits
    int64_t base_s0, base_s1;
    const uint16_t *embed;             // [V, r], on every rank
    const int32_t *anchor;
    const float *temperature;
    const int64_t *seeds;
    const int64_t *row_state_idx;
    int rows, N, V, Vs, world, Gr, Grp;
    Transform tf;
    int64_t tok_s0, cache_s0, cache_s1, noise_s0, stg_s0;
    const uint16_t *head[kMaxWorld];   // rank k's head rows [Vs, r]
    const float *noise[kMaxWorld];     // rank k's noise [rows * N, noise_s0], its shard's ids
    uint16_t *cache[kMaxWorld];        // rank k's [rows, N, V] cache (output)
    uint16_t *staging[kMaxWorld];      // rank k's [rows, N, V] copy of its peers' logits
    int64_t *tokens[kMaxWorld];        // rank k's [rows, N] tokens (output)
    uint64_t *mailbox[kMaxWorld];      // rank k's [N][8][kMaxWorld] keys of every rank
    uint64_t *slots[kMaxWorld];        // rank k's [N][8][Grp] keys of its CTAs
    uint32_t *status;                  // [2] sticky status, where
    uint32_t *call_counter;
    uint64_t timeout_ns;
};

// packed key: ordered key (32) | 0x3FFFF - id (18) | epoch tag (14)
__device__ __forceinline__ uint64_t sh_pack(float key, uint32_t v, uint32_t tag) {
    return ((uint64_t)ordered_key(key) << 32) | ((uint64_t)(0x3FFFFu - v) << 14) | (uint64_t)tag;
}
__device__ __forceinline__ uint32_t sh_id(uint64_t p) {
    return 0x3FFFFu - (uint32_t)((p >> 14) & 0x3FFFFu);
}

__device__ __forceinline__ void st_release_u64(uint64_t *p, uint64_t v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// One warp waits until the n tagged words at p all carry `tag`, then
// returns their maximum (acquire: what their writers released is visible).
// False after the bounded wait (or when another CTA recorded an error).
__device__ bool poll_tagged(const uint64_t *p, int n, uint32_t tag, uint64_t timeout_ns,
                            uint32_t *status, uint64_t &out) {
    const int lane = threadIdx.x & 31;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t spin = 0;; ++spin) {
        uint64_t k[kShPer];
#pragma unroll
        for (int u = 0; u < kShPer; ++u)
            k[u] = lane + 32 * u < n ? ld_relaxed_u64(p + lane + 32 * u) : (uint64_t)tag;
        bool fresh = true;
        uint64_t m = 0ull;
#pragma unroll
        for (int u = 0; u < kShPer; ++u) {
            fresh = fresh && (uint32_t)(k[u] & 0x3FFFu) == tag;
            m = k[u] > m ? k[u] : m;
        }
        if (__all_sync(0xffffffffu, fresh)) {
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            out = warp_max_u64_shfl(m);
            return true;
        }
        if ((spin & 15u) == 15u) {
            const bool bad = globaltimer_ns() - t0 > timeout_ns || ld_acquire_u32(status) != 0u;
            if (__any_sync(0xffffffffu, bad)) return false;
        }
    }
}

}  // namespace

template <int RANK>
__global__ void __launch_bounds__(kShThreads, 1) sharded_chain_kernel(const ShardedArgs a) {
    __shared__ __align__(16) uint16_t e_smem[kChainRows * (RANK + kEPad)];
    __shared__ int s_live[kChainRows], s_samp[kChainRows];
    __shared__ float s_T[kChainRows];
    __shared__ int64_t s_prev[kChainRows];
    __shared__ unsigned long long s_best[kChainRows];
    __shared__ uint64_t s_win[kChainRows];
    __shared__ uint32_t s_call;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int rank = blockIdx.x / a.Gr, lc = blockIdx.x % a.Gr;
    const int N = a.N, V = a.V;
    const int ntiles = a.Vs / kTile;
    const int tile_begin = (int)((int64_t)lc * ntiles / a.Gr);
    const int tile_end = (int)((int64_t)(lc + 1) * ntiles / a.Gr);
    const int voff = rank * a.Vs;       // global id of the shard's column 0
    const uint16_t *head = a.head[rank];
    const float *noise = a.noise[rank];
    uint16_t *cache = a.cache[rank];

    if (tid < kChainRows) {
        const int b = tid;
        const bool live = b < a.rows && a.row_state_idx[b] >= 0;
        s_live[b] = live;
        const float T = live ? a.temperature[b] : 0.0f;
        s_T[b] = T;
        s_samp[b] = live && samples(T);
        int64_t p = live ? (int64_t)a.anchor[b] : 0;
        if (p < 0 || p >= V) {
            set_status(a.status, 1u /* MARKOV_EINVAL */, 0xE100u + b);
            p = 0;
        }
        s_prev[b] = p;
    }
    if (tid == 0) s_call = *(volatile const uint32_t *)a.call_counter;
    __syncthreads();
    // a status left by an earlier call, or an anchor outside the vocabulary
    // (every CTA checks the same anchors): this call writes nothing (the
    // host's status read clears the status, and the slots with it)
    if (__syncthreads_or(tid == 0 && ld_acquire_u32(a.status) != 0u)) return;

    for (int i = 0; i < N; ++i) {
        // in [1, 16383]: zeroed slots are never taken for fresh ones
        const uint32_t tag = (s_call * (uint32_t)kMaxSteps + (uint32_t)i) % 16383u + 1u;
        // 1. the previous tokens' embeddings (zeros for absent rows)
        for (int idx = tid; idx < kChainRows * (RANK / 8); idx += kShThreads) {
            const int b = idx / (RANK / 8), c = idx % (RANK / 8);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (s_live[b]) v = *reinterpret_cast<const uint4 *>(a.embed + s_prev[b] * RANK + 8 * c);
            *reinterpret_cast<uint4 *>(e_smem + b * (RANK + kEPad) + 8 * c) = v;
        }
        if (tid < kChainRows) s_best[tid] = 0ull;
        __syncthreads();

        // 2. the CTA's tiles: logits into this rank's cache and every peer's
        //    staging buffer, the rows' best keys
        uint64_t best0 = 0ull, best1 = 0ull;      // rows 2t, 2t+1
        const int r0 = 2 * t, r1 = 2 * t + 1;
        const bool l0 = s_live[r0], l1 = s_live[r1];
        const float T0 = s_T[r0], T1 = s_T[r1];
        const bool s0 = s_samp[r0], s1 = s_samp[r1];
        for (int tile = tile_begin + warp; tile < tile_end; tile += kShWarps) {
            const int vl0 = tile * kTile;
            float acc[4];
            bias_tile<RANK>(head, vl0, e_smem, g, t, acc);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = (e & 1) ? r1 : r0;
                const bool live = (e & 1) ? l1 : l0;
                if (!live) continue;
                const int vl = vl0 + g + ((e & 2) ? 8 : 0);
                const int v = voff + vl;
                const float base = dm_bf16_f32(a.base[row * a.base_s0 + (int64_t)i * a.base_s1 + v]);
                const float lf = logit_value(base, acc[e], a.tf, false);
                const uint16_t lb = (uint16_t)(__float_as_uint(lf) >> 16);
                cache[row * a.cache_s0 + (int64_t)i * a.cache_s1 + v] = lb;
                for (int q = 0; q < a.world; ++q)
                    if (q != rank) a.staging[q][row * a.stg_s0 + (int64_t)i * V + v] = lb;
                const bool smp = (e & 1) ? s1 : s0;
                float key = lf;
                if (smp)
                    key = __fadd_rn(__fdiv_rn(lf, (e & 1) ? T1 : T0),
                                    noise[(int64_t)(row * N + i) * a.noise_s0 + vl]);
                const uint64_t pk = sh_pack(key, (uint32_t)v, tag);
                if (e & 1) best1 = pk > best1 ? pk : best1;
                else best0 = pk > best0 ? pk : best0;
            }
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            const uint64_t w0 = __shfl_xor_sync(0xffffffffu, best0, o);
            const uint64_t w1 = __shfl_xor_sync(0xffffffffu, best1, o);
            best0 = w0 > best0 ? w0 : best0;
            best1 = w1 > best1 ? w1 : best1;
        }
        if (g == 0) {
            if (l0 && best0) atomicMax(&s_best[r0], (unsigned long long)best0);
            if (l1 && best1) atomicMax(&s_best[r1], (unsigned long long)best1);
        }
        __syncthreads();

        // 3. the CTA's key into the rank's slots (released after its cache
        //    and staging writes, which the __syncthreads ordered before it);
        //    a CTA without tiles reports the lowest key of the epoch
        if (tid < kChainRows && s_live[tid]) {
            const uint64_t k = s_best[tid] ? (uint64_t)s_best[tid] : (uint64_t)tag;
            st_release_u64(a.slots[rank] + ((int64_t)i * kChainRows + tid) * a.Grp + lc, k);
        }
        // 4. the rank's first CTA: the rank's key per row into every rank's mailbox
        bool ok = true;
        if (lc == 0 && warp < kChainRows && s_live[warp]) {
            uint64_t m = 0ull;
            ok = poll_tagged(a.slots[rank] + ((int64_t)i * kChainRows + warp) * a.Grp, a.Gr, tag,
                             a.timeout_ns, a.status, m);
            if (ok && lane < a.world)
                st_release_u64(a.mailbox[lane] + ((int64_t)i * kChainRows + warp) * kMaxWorld + rank, m);
        }
        // 5. every CTA: the world's best key per row
        if (ok && warp < kChainRows && s_live[warp]) {
            uint64_t m = 0ull;
            ok = poll_tagged(a.mailbox[rank] + ((int64_t)i * kChainRows + warp) * kMaxWorld, a.world,
                             tag, a.timeout_ns, a.status, m);
            if (ok && lane == 0) s_win[warp] = m;
        }
        if (!ok && lane == 0) set_status(a.status, 4u /* MARKOV_ETIMEOUT */, 0xE200u + (uint32_t)i);
        if (__syncthreads_or(!ok)) return;

        // 6. the token
        if (tid < kChainRows && s_live[tid]) {
            uint32_t id = sh_id(s_win[tid]);
            if (id >= (uint32_t)V) {
                set_status(a.status, 6u /* MARKOV_EDEVICE */, 0xE300u + (uint32_t)i);
                id = 0u;
            }
            s_prev[tid] = (int64_t)id;
            if (lc == 0) a.tokens[rank][tid * a.tok_s0 + i] = (int64_t)id;
        }
        __syncthreads();
    }

    // tail: the peers' columns from this rank's staging buffer into its
    // cache (every peer's staging writes were released before its key of
    // the last position, which this CTA acquired), 8 ids per 16-byte copy
    const int per_row = (a.world - 1) * (a.Vs / 8);     // 16-byte pieces of peers' columns
    const int64_t total = (int64_t)kChainRows * N * per_row;
    for (int64_t w = (int64_t)lc * kShThreads + tid; w < total; w += (int64_t)a.Gr * kShThreads) {
        const int piece = (int)(w % per_row);
        const int ri = (int)(w / per_row);
        const int b = ri / N, i = ri % N;
        if (!s_live[b]) continue;
        int col = piece * 8;                            // among the peers' columns
        const int q = col / a.Vs;
        const int v = (q >= rank ? q + 1 : q) * a.Vs + (col - q * a.Vs);
        const uint4 x =
            *reinterpret_cast<const uint4 *>(a.staging[rank] + b * a.stg_s0 + (int64_t)i * V + v);
        *reinterpret_cast<uint4 *>(cache + b * a.cache_s0 + (int64_t)i * a.cache_s1 + v) = x;
    }
    if (blockIdx.x == 0 && tid == 0 && ld_acquire_u32(a.status) == 0u)
        *(volatile uint32_t *)a.call_counter = s_call + 1u;
}

namespace {

const void *sharded_kernel_for(int r) {
    switch (r) {
        case 64: return (const void *)sharded_chain_kernel<64>;
        case 128: return (const void *)sharded_chain_kernel<128>;
        case 256: return (const void *)sharded_chain_kernel<256>;
        default: return nullptr;
    }
}

}  // namespace
}  // namespace dtm

// ------------------------------------------------------------------ C ABI

struct markov_shard_plan {
    int dev = 0;
    markov_desc d{};
    int world = 1, Vs = 0, Gr = 0, Grp = 0;
    uint64_t timeout_ns = 0;
    float *noise[dtm::kMaxWorld] = {};
    uint16_t *staging[dtm::kMaxWorld] = {};
    uint64_t *mailbox[dtm::kMaxWorld] = {};
    uint64_t *slots[dtm::kMaxWorld] = {};
    uint32_t *ctrl = nullptr;          // [0] status, [1] where, [2] call counter
};

namespace {

void shard_free(markov_shard_plan *p) {
    for (int k = 0; k < dtm::kMaxWorld; ++k) {
        if (p->noise[k]) cudaFree(p->noise[k]);
        if (p->staging[k]) cudaFree(p->staging[k]);
        if (p->mailbox[k]) cudaFree(p->mailbox[k]);
        if (p->slots[k]) cudaFree(p->slots[k]);
    }
    if (p->ctrl) cudaFree(p->ctrl);
    delete p;
}

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0u; }

}  // namespace

extern "C" markov_status markov_shard_plan_create(const markov_desc *desc, int32_t world,
                                                  markov_shard_plan **out) {
    if (!out) return MARKOV_EINVAL;
    *out = nullptr;
    if (!desc) return MARKOV_EINVAL;
    const markov_desc d = *desc;
    if (world != 1 && world != 2 && world != 4 && world != 8) return MARKOV_EINVAL;
    if (d.vocab <= 0 || d.vocab > dtm::kMaxVocab || d.vocab % (16 * world) != 0) return MARKOV_EINVAL;
    if (d.rank != 64 && d.rank != 128 && d.rank != 256) return MARKOV_EINVAL;
    if (d.num_steps < 1 || d.num_steps > dtm::kMaxSteps) return MARKOV_EINVAL;
    if (d.max_rows < 1 || d.max_rows > dtm::kChainRows) return MARKOV_EINVAL;
    if (d.timeout_ms < 0) return MARKOV_EINVAL;
    if (cudaSetDevice(d.device) != cudaSuccess) {
        cudaGetLastError();
        return MARKOV_EDEVICE;
    }
    markov_shard_plan *p = new markov_shard_plan();
    p->dev = d.device;
    p->d = d;
    p->world = world;
    p->Vs = d.vocab / world;
    p->timeout_ns = (uint64_t)(d.timeout_ms > 0 ? d.timeout_ms : 100) * 1000000ull;
    int sms = 0, occ = 0;
    const void *fn = dtm::sharded_kernel_for(d.rank);
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d.device) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, dtm::kShThreads, 0) != cudaSuccess ||
        occ < 1) {
        cudaGetLastError();
        shard_free(p);
        return MARKOV_ECUDA;
    }
    // every rank gets the same CTA count, each CTA at least one 16-id tile
    int gr = sms * occ / world;
    if (gr > 160) gr = 160;
    if (gr > p->Vs / 16) gr = p->Vs / 16;
    if (gr < 1) {
        shard_free(p);
        return MARKOV_ENOTRESIDENT;
    }
    p->Gr = gr;
    p->Grp = (gr + dtm::kKeyPad - 1) / dtm::kKeyPad * dtm::kKeyPad;
    const size_t R = (size_t)d.max_rows, N = (size_t)d.num_steps;
    // each rank's buffers in allocations of their own, as on separate GPUs
    for (int k = 0; k < world; ++k) {
        if (cudaMalloc(&p->noise[k], R * N * p->Vs * sizeof(float)) != cudaSuccess ||
            cudaMalloc(&p->staging[k], R * N * d.vocab * sizeof(uint16_t)) != cudaSuccess ||
            cudaMalloc(&p->mailbox[k], N * dtm::kChainRows * dtm::kMaxWorld * sizeof(uint64_t)) !=
                cudaSuccess ||
            cudaMalloc(&p->slots[k], N * dtm::kChainRows * p->Grp * sizeof(uint64_t)) != cudaSuccess ||
            cudaMemset(p->mailbox[k], 0, N * dtm::kChainRows * dtm::kMaxWorld * sizeof(uint64_t)) !=
                cudaSuccess ||
            cudaMemset(p->slots[k], 0, N * dtm::kChainRows * p->Grp * sizeof(uint64_t)) != cudaSuccess) {
            cudaGetLastError();
            shard_free(p);
            return MARKOV_ECUDA;
        }
    }
    if (cudaMalloc(&p->ctrl, 4 * sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(p->ctrl, 0, 4 * sizeof(uint32_t)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        shard_free(p);
        return MARKOV_ECUDA;
    }
    *out = p;
    return MARKOV_OK;
}

extern "C" void markov_shard_plan_destroy(markov_shard_plan *p) {
    if (!p) return;
    cudaSetDevice(p->dev);
    cudaDeviceSynchronize();
    shard_free(p);
}

extern "C" int32_t markov_shard_plan_ctas(const markov_shard_plan *p) {
    return p ? p->world * p->Gr : -1;
}

extern "C" markov_status markov_shard_plan_status(markov_shard_plan *p) {
    if (!p) return MARKOV_EINVAL;
    if (cudaSetDevice(p->dev) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return MARKOV_ECUDA;
    }
    uint32_t st[2] = {0u, 0u};
    if (cudaMemcpy(st, p->ctrl, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) return MARKOV_ECUDA;
    if (st[0] != 0u) {
        // a call that stopped part way may have left keys with the epoch the
        // next call takes (the call counter only moves after a clean call)
        const size_t N = (size_t)p->d.num_steps;
        for (int k = 0; k < p->world; ++k)
            if (cudaMemset(p->mailbox[k], 0, N * dtm::kChainRows * dtm::kMaxWorld * sizeof(uint64_t)) !=
                    cudaSuccess ||
                cudaMemset(p->slots[k], 0, N * dtm::kChainRows * p->Grp * sizeof(uint64_t)) != cudaSuccess)
                return MARKOV_ECUDA;
        if (cudaMemset(p->ctrl, 0, 2 * sizeof(uint32_t)) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess)
            return MARKOV_ECUDA;
    }
    return (markov_status)st[0];
}

extern "C" markov_status markov_chain_sample_sharded(
    markov_shard_plan *p, const uint16_t *base_logits, int64_t base_s0, int64_t base_s1,
    const uint16_t *const *head_shards, const uint16_t *embed, const int32_t *anchor_tokens,
    const float *temperature, const int64_t *seeds, const int64_t *row_state_idx, int32_t rows,
    float output_multiplier, float soft_cap, int64_t *const *draft_tokens, int64_t tok_s0,
    uint16_t *const *logit_caches, int64_t cache_s0, int64_t cache_s1, void *stream) {
    if (!p) return MARKOV_EINVAL;
    const int N = p->d.num_steps, V = p->d.vocab, W = p->world;
    if (rows < 1 || rows > p->d.max_rows) return MARKOV_EINVAL;
    if (!base_logits || !head_shards || !embed || !anchor_tokens || !temperature || !seeds ||
        !row_state_idx || !draft_tokens || !logit_caches)
        return MARKOV_EINVAL;
    if (base_s1 < V || base_s0 < (int64_t)N * base_s1) return MARKOV_EINVAL;
    if (tok_s0 < N || cache_s1 < V || cache_s0 < (int64_t)N * cache_s1) return MARKOV_EINVAL;
    if (cache_s0 % 8 != 0 || cache_s1 % 8 != 0 || !al16(embed)) return MARKOV_EINVAL;
    if (!std::isfinite(output_multiplier) || std::isnan(soft_cap)) return MARKOV_EINVAL;
    for (int k = 0; k < W; ++k)
        if (!head_shards[k] || !al16(head_shards[k]) || !draft_tokens[k] || !logit_caches[k] ||
            !al16(logit_caches[k]))
            return MARKOV_EINVAL;
    if (cudaSetDevice(p->dev) != cudaSuccess) {
        cudaGetLastError();
        return MARKOV_EDEVICE;
    }
    cudaStream_t s = (cudaStream_t)stream;
    dtm::ShardedArgs a;
    std::memset(&a, 0, sizeof(a));
    a.base = base_logits;
    a.base_s0 = base_s0;
    a.base_s1 = base_s1;
    a.embed = embed;
    a.anchor = anchor_tokens;
    a.temperature = temperature;
    a.seeds = seeds;
    a.row_state_idx = row_state_idx;
    a.rows = rows;
    a.N = N;
    a.V = V;
    a.Vs = p->Vs;
    a.world = W;
    a.Gr = p->Gr;
    a.Grp = p->Grp;
    // the output-logit transform as the other entry points take it
    a.tf.mult = output_multiplier;
    a.tf.has_cap = soft_cap > 0.0f;
    a.tf.cap = a.tf.has_cap ? soft_cap : 1.0f;
    a.tf.inv_cap = a.tf.has_cap ? 1.0f / a.tf.cap : 1.0f;   // fp32(1) / fp32(cap)
    a.tf.has_transform = output_multiplier != 1.0f || a.tf.has_cap;
    a.tok_s0 = tok_s0;
    a.cache_s0 = cache_s0;
    a.cache_s1 = cache_s1;
    a.noise_s0 = p->Vs;
    a.stg_s0 = (int64_t)N * V;
    for (int k = 0; k < W; ++k) {
        a.head[k] = head_shards[k];
        a.noise[k] = p->noise[k];
        a.cache[k] = logit_caches[k];
        a.staging[k] = p->staging[k];
        a.tokens[k] = draft_tokens[k];
        a.mailbox[k] = p->mailbox[k];
        a.slots[k] = p->slots[k];
    }
    a.status = p->ctrl;
    a.call_counter = p->ctrl + 2;
    a.timeout_ns = p->timeout_ns;
    // each rank's noise: its shard's ids (sharded_markov page, fork_noise)
    for (int k = 0; k < W; ++k)
        if (dtm::launch_noise(seeds, temperature, row_state_idx, rows, N, p->Vs, p->noise[k], p->Vs, 1, s,
                              k * p->Vs) != cudaSuccess)
            return MARKOV_ECUDA;
    const void *fn = dtm::sharded_kernel_for(p->d.rank);
    void *args[] = {(void *)&a};
    if (cudaLaunchCooperativeKernel(fn, dim3(W * p->Gr), dim3(dtm::kShThreads), args, 0, s) !=
        cudaSuccess) {
        cudaGetLastError();
        return MARKOV_ECUDA;
    }
    return MARKOV_OK;
}
