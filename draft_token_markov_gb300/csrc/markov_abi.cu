// markov_abi.cu -- host side of the C ABI declared in include/markov.h:
// plan creation (all scratch allocated once), argument validation (the
// conditions the sharded_markov page's unsupported_reason and sample()
// assert), path dispatch (the persistent chain up to 8 rows, the
// per-position kernels above), the optional side-stream noise fork, and the
// sticky device status.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>

#include "../../include/markov.h"
#include "internal.h"

using namespace dtm;

struct markov_plan {
    markov_desc d;
    int sm_count = 0;
    int chain_occ = 0;            // chain CTAs per SM
    int chain_grid = 0;
    int batch_grid = 0;
    float *noise = nullptr;       // [max_rows * N, V]
    int64_t noise_s0 = 0;
    uint64_t *keys = nullptr;
    uint64_t *sums = nullptr;
    uint32_t *ctrl = nullptr;     // [0] barrier count, [1] barrier base, [2..3] status,
                                  // [4] call counter of the tcgen05 chain
    size_t keys_n = 0;
    // the tcgen05 chain: exchange slots and words, and the head's TMA descriptor
    bool tc_ok = false;
    bool batch_tc_ok = false;     // the per-position logits on the tcgen05 kernel
    int tc_grid = 0;
    uint64_t *tc_sums = nullptr;
    uint64_t *tok_slots = nullptr;
    uint64_t *win_max = nullptr;
    uint32_t *win_cnt = nullptr;
    // the per-position path's winner words and done counters; every call
    // leaves them zero, except one whose launches failed part way
    uint64_t *bwin = nullptr;
    uint32_t *bcnt = nullptr;
    bool batch_dirty = false;
    size_t tc_slots_n = 0;
    CUtensorMap tmap;
    const void *tmap_head = nullptr;
    cudaStream_t side = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_noise = nullptr;
    int noise_state = 0;          // 0 none, 1 forked, 2 forked and joined
    int forked_rows = 0;
    markov_path path = MARKOV_PATH_AUTO;
    int last_launches = 0;
    int last_path = 0;
};

namespace {

// Makes the plan's device current for the duration of a call and restores
// the caller's device afterwards.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0u; }

bool valid_rank(int r) { return r == 64 || r == 128 || r == 256; }

void free_plan(markov_plan *p) {
    if (!p) return;
    if (p->noise) cudaFree(p->noise);
    if (p->keys) cudaFree(p->keys);
    if (p->sums) cudaFree(p->sums);
    if (p->ctrl) cudaFree(p->ctrl);
    if (p->tc_sums) cudaFree(p->tc_sums);
    if (p->bwin) cudaFree(p->bwin);
    if (p->bcnt) cudaFree(p->bcnt);
    if (p->tok_slots) cudaFree(p->tok_slots);
    if (p->win_max) cudaFree(p->win_max);
    if (p->win_cnt) cudaFree(p->win_cnt);
    if (p->ev_fork) cudaEventDestroy(p->ev_fork);
    if (p->ev_noise) cudaEventDestroy(p->ev_noise);
    if (p->side) cudaStreamDestroy(p->side);
    delete p;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The head [V, r] BF16 as 2-D tiles of 128 rows x 64 elements, 128-byte
// swizzle (the K-major MMA operand layout); rows past V read as zero.
bool encode_head_map(CUtensorMap *m, const void *head, int V, int r) {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !f)
            return false;
        fn = (EncodeTiledFn)f;
    }
    cuuint64_t dims[2] = {(cuuint64_t)r, (cuuint64_t)V};
    cuuint64_t strides[1] = {(cuuint64_t)r * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(head), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

Transform make_transform(float mult, float cap) {
    Transform tf{};
    tf.mult = mult;
    tf.has_cap = cap > 0.0f;
    tf.cap = tf.has_cap ? cap : 1.0f;
    tf.inv_cap = tf.has_cap ? 1.0f / tf.cap : 1.0f;   // fp32(1) / fp32(cap)
    tf.has_transform = (mult != 1.0f) || tf.has_cap;
    return tf;
}

}  // namespace

extern "C" {

const char *markov_status_string(markov_status s) {
    switch (s) {
        case MARKOV_OK: return "ok";
        case MARKOV_EINVAL: return "invalid argument";
        case MARKOV_EUNSUPPORTED: return "unsupported configuration";
        case MARKOV_ECUDA: return "CUDA runtime error";
        case MARKOV_ETIMEOUT: return "an in-kernel bounded wait timed out";
        case MARKOV_ENOTRESIDENT: return "persistent grid cannot be co-resident";
        case MARKOV_EDEVICE: return "device error or unusable device";
    }
    return "unknown status";
}

markov_status markov_plan_create(const markov_desc *desc, markov_plan **out) {
    if (!out) return MARKOV_EINVAL;
    *out = nullptr;
    if (!desc) return MARKOV_EINVAL;
    const markov_desc d = *desc;
    if (d.vocab <= 0 || d.vocab % kTile != 0 || d.vocab > kMaxVocab) return MARKOV_EINVAL;
    if (!valid_rank(d.rank)) return MARKOV_EINVAL;
    if (d.num_steps < 1 || d.num_steps > kMaxSteps) return MARKOV_EINVAL;
    if (d.max_rows < 1 || d.max_rows > kMaxRows) return MARKOV_EINVAL;
    if (d.timeout_ms < 0) return MARKOV_EINVAL;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || d.device < 0 || d.device >= ndev)
        return MARKOV_EDEVICE;
    DeviceGuard guard(d.device);
    if (!guard.ok) return MARKOV_EDEVICE;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, d.device) != cudaSuccess) return MARKOV_EDEVICE;
    if (prop.major < 10) return MARKOV_EUNSUPPORTED;    // the kernels are built for sm_103a
    if (!prop.cooperativeLaunch) return MARKOV_EUNSUPPORTED;

    markov_plan *p = new (std::nothrow) markov_plan();
    if (!p) return MARKOV_ECUDA;
    p->d = d;
    if (p->d.timeout_ms == 0) p->d.timeout_ms = 100;
    p->sm_count = prop.multiProcessorCount;
    if (chain_occupancy(&p->chain_occ) != cudaSuccess) { free_plan(p); return MARKOV_ECUDA; }
    const int ntiles = d.vocab / kTile;
    int g = ntiles / (kChainThreads / 32);
    if (g < 1) g = 1;
    if (g > p->sm_count * p->chain_occ) g = p->sm_count * p->chain_occ;
    p->chain_grid = g;
    p->batch_grid = batch_blocks(d.vocab);
    {
        // the tcgen05 chain: one CTA per SM (at most one per 128-id tile); every
        // CTA's tiles must fit the on-chip chunk budget
        const int T_total = (d.vocab + 127) / 128;
        int g = T_total < p->sm_count ? T_total : p->sm_count;
        const int max_tiles = (T_total + g - 1) / g;
        int occ = 0;
        // (the inverse-CDF exchange reads the CTAs' sums 5 per lane: at most 160 CTAs)
        if (chain_tc_prepare() == cudaSuccess && chain_tc_occupancy(&occ) == cudaSuccess &&
            occ >= 1 && max_tiles * (d.rank / 64) <= chain_tc_max_chunks() && g <= 160) {
            p->tc_ok = true;
            p->tc_grid = g;
        }
        cudaGetLastError();
    }

    p->batch_tc_ok = batch_tc_prepare() == cudaSuccess;
    cudaGetLastError();
    const int Gp = (p->chain_grid + kKeyPad - 1) / kKeyPad * kKeyPad;
    size_t chain_keys = (size_t)kMaxSteps * 2 * kChainRows * Gp;
    size_t batch_keys = (size_t)d.max_rows * p->batch_grid;
    // the per-position path's inverse-CDF weight sums: one per 256 ids and row
    const size_t unit_sums = (size_t)d.max_rows * ((d.vocab + 255) / 256);
    if (batch_keys < unit_sums) batch_keys = unit_sums;
    p->keys_n = chain_keys > batch_keys ? chain_keys : batch_keys;
    p->noise_s0 = d.vocab;
    // fp32 noise of every row for the per-position kernels; the tcgen05 chain
    // reuses the buffer for its 8 noise-bound bytes per (position, id)
    size_t noise_bytes = (size_t)d.max_rows * d.num_steps * d.vocab * sizeof(float);
    const size_t bound_bytes = (size_t)d.num_steps * d.vocab * kChainRows;
    if (p->tc_ok && noise_bytes < bound_bytes) noise_bytes = bound_bytes;
    const int Gtc = p->tc_grid > 0 ? p->tc_grid : 1;
    p->tc_slots_n = (size_t)kMaxSteps * kChainRows * ((Gtc + kKeyPad - 1) / kKeyPad * kKeyPad);
    if (cudaMalloc(&p->noise, noise_bytes) != cudaSuccess ||
        cudaMalloc(&p->keys, p->keys_n * sizeof(uint64_t)) != cudaSuccess ||
        cudaMalloc(&p->sums, p->keys_n * sizeof(uint64_t)) != cudaSuccess ||
        cudaMalloc(&p->ctrl, 8 * sizeof(uint32_t)) != cudaSuccess ||
        cudaMalloc(&p->tc_sums, p->tc_slots_n * sizeof(uint64_t)) != cudaSuccess ||
        cudaMalloc(&p->tok_slots, (size_t)kMaxSteps * kChainRows * sizeof(uint64_t)) != cudaSuccess ||
        cudaMalloc(&p->win_max, kWinMaxN * sizeof(uint64_t)) != cudaSuccess ||
        cudaMalloc(&p->win_cnt, kWinCntN * sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(p->win_max, 0, kWinMaxN * sizeof(uint64_t)) != cudaSuccess ||
        cudaMemset(p->win_cnt, 0, kWinCntN * sizeof(uint32_t)) != cudaSuccess ||
        cudaMalloc(&p->bwin, kBatchWinN * sizeof(uint64_t)) != cudaSuccess ||
        cudaMalloc(&p->bcnt, kBatchCntN * sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(p->bwin, 0, kBatchWinN * sizeof(uint64_t)) != cudaSuccess ||
        cudaMemset(p->bcnt, 0, kBatchCntN * sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(p->tc_sums, 0, p->tc_slots_n * sizeof(uint64_t)) != cudaSuccess ||
        cudaMemset(p->tok_slots, 0, (size_t)kMaxSteps * kChainRows * sizeof(uint64_t)) != cudaSuccess ||
        cudaMemset(p->ctrl, 0, 8 * sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(p->keys, 0, p->keys_n * sizeof(uint64_t)) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_noise, cudaEventDisableTiming) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        free_plan(p);
        return MARKOV_ECUDA;
    }
    *out = p;
    return MARKOV_OK;
}

void markov_plan_destroy(markov_plan *p) {
    if (!p) return;
    DeviceGuard guard(p->d.device);
    cudaDeviceSynchronize();
    free_plan(p);
}

int32_t markov_chain_max_rows(const markov_plan *p) {
    if (!p) return -1;
    return p->d.max_rows < kChainRows ? p->d.max_rows : kChainRows;
}

markov_status markov_plan_set_path(markov_plan *p, markov_path path) {
    if (!p) return MARKOV_EINVAL;
    if (path != MARKOV_PATH_AUTO && path != MARKOV_PATH_CHAIN && path != MARKOV_PATH_BATCH &&
        path != MARKOV_PATH_CHAIN_SIMPLE)
        return MARKOV_EINVAL;
    p->path = path;
    return MARKOV_OK;
}

markov_status markov_noise_fork(markov_plan *p, const int64_t *seeds, const float *temperature,
                                const int64_t *row_state_idx, int32_t rows, void *stream) {
    if (!p || !seeds || !temperature || !row_state_idx) return MARKOV_EINVAL;
    if (rows < 1 || rows > p->d.max_rows) return MARKOV_EINVAL;
    DeviceGuard guard(p->d.device);
    if (!guard.ok) return MARKOV_EDEVICE;
    cudaStream_t main = (cudaStream_t)stream;
    if (cudaEventRecord(p->ev_fork, main) != cudaSuccess ||
        cudaStreamWaitEvent(p->side, p->ev_fork, 0) != cudaSuccess)
        return MARKOV_ECUDA;
    if (launch_noise(seeds, temperature, row_state_idx, rows, p->d.num_steps, p->d.vocab,
                     p->noise, p->noise_s0, 1, p->side) != cudaSuccess)
        return MARKOV_ECUDA;
    if (cudaEventRecord(p->ev_noise, p->side) != cudaSuccess) return MARKOV_ECUDA;
    p->noise_state = 1;
    p->forked_rows = rows;
    return MARKOV_OK;
}

markov_status markov_noise_join(markov_plan *p, void *stream) {
    if (!p) return MARKOV_EINVAL;
    if (p->noise_state != 1) return MARKOV_OK;
    DeviceGuard guard(p->d.device);
    if (!guard.ok) return MARKOV_EDEVICE;
    if (cudaStreamWaitEvent((cudaStream_t)stream, p->ev_noise, 0) != cudaSuccess)
        return MARKOV_ECUDA;
    p->noise_state = 2;
    return MARKOV_OK;
}

markov_status markov_chain_sample(markov_plan *p, const uint16_t *base_logits, int64_t base_s0,
                                  int64_t base_s1, const uint16_t *head, const uint16_t *embed,
                                  const int32_t *anchor_tokens, const float *temperature,
                                  const int64_t *seeds, const int64_t *row_state_idx,
                                  int32_t rows, markov_mode mode, float output_multiplier,
                                  float soft_cap, int64_t *draft_tokens, int64_t tok_s0,
                                  uint16_t *logit_cache, int64_t cache_s0, int64_t cache_s1,
                                  void *stream) {
    return markov_chain_sample_typed(p, base_logits, MARKOV_BF16, base_s0, base_s1, head, embed,
                                     anchor_tokens, temperature, seeds, row_state_idx, rows, mode,
                                     output_multiplier, soft_cap, draft_tokens, tok_s0,
                                     logit_cache, MARKOV_BF16, cache_s0, cache_s1, stream);
}

markov_status markov_chain_sample_typed(markov_plan *p, const void *base_logits,
                                        markov_dtype base_dtype, int64_t base_s0,
                                        int64_t base_s1, const uint16_t *head,
                                        const uint16_t *embed, const int32_t *anchor_tokens,
                                        const float *temperature, const int64_t *seeds,
                                        const int64_t *row_state_idx, int32_t rows,
                                        markov_mode mode, float output_multiplier,
                                        float soft_cap, int64_t *draft_tokens, int64_t tok_s0,
                                        void *logit_cache, markov_dtype cache_dtype,
                                        int64_t cache_s0, int64_t cache_s1, void *stream) {
    if (!p) return MARKOV_EINVAL;
    if ((base_dtype != MARKOV_BF16 && base_dtype != MARKOV_F32) ||
        (cache_dtype != MARKOV_BF16 && cache_dtype != MARKOV_F32))
        return MARKOV_EINVAL;
    const bool base_f32 = base_dtype == MARKOV_F32, cache_f32 = cache_dtype == MARKOV_F32;
    const int64_t cache_es = cache_f32 ? 4 : 2;   // cache element bytes
    const int V = p->d.vocab, r = p->d.rank, N = p->d.num_steps;
    if (!base_logits || !head || !embed || !anchor_tokens || !temperature || !seeds ||
        !row_state_idx || !draft_tokens || !logit_cache)
        return MARKOV_EINVAL;
    if (rows < 1 || rows > p->d.max_rows) return MARKOV_EINVAL;
    if (mode != MARKOV_GUMBEL && mode != MARKOV_INVCDF) return MARKOV_EINVAL;
    if (base_s1 < V || base_s0 < (int64_t)(N - 1) * base_s1 + V) return MARKOV_EINVAL;
    if (cache_s1 < V || cache_s0 < (int64_t)(N - 1) * cache_s1 + V) return MARKOV_EINVAL;
    if (tok_s0 < N) return MARKOV_EINVAL;
    // the cache asserts of the sharded_markov page's sample(): 16-byte
    // aligned pointer and row strides
    if (!aligned16(logit_cache) || (cache_s0 * cache_es) % 16 != 0 ||
        (cache_s1 * cache_es) % 16 != 0)
        return MARKOV_EINVAL;
    if (!aligned16(head) || !aligned16(embed)) return MARKOV_EINVAL;
    if (!std::isfinite(output_multiplier) || std::isnan(soft_cap)) return MARKOV_EINVAL;
    if (p->noise_state != 0 && p->forked_rows != rows) return MARKOV_EINVAL;

    bool chain = rows <= kChainRows;
    if ((p->path == MARKOV_PATH_CHAIN || p->path == MARKOV_PATH_CHAIN_SIMPLE) && !chain)
        return MARKOV_EUNSUPPORTED;
    if (p->path == MARKOV_PATH_BATCH) chain = false;
    // the automatic choice between the chain limit and kChainSliceRows rows
    // in Gumbel mode: one tcgen05 chain launch per 8-row slice (no forked
    // noise: each slice draws its own).  Measured on the 129280 x 256 head:
    // 12 / 16 / 24 rows take 193 / 199 / 300 us this way against 229 / 235 /
    // 328 us for the per-position kernels; in inverse-CDF mode the chain's
    // two-pass selection makes slices slower (9 rows: 381 against 271 us).
    const bool sliced = !chain && p->path == MARKOV_PATH_AUTO && mode == MARKOV_GUMBEL &&
                        rows <= kChainSliceRows && p->tc_ok && p->noise_state == 0;
    if (sliced) chain = true;
    const bool use_tc = chain && p->tc_ok && p->path != MARKOV_PATH_CHAIN_SIMPLE;

    DeviceGuard guard(p->d.device);
    if (!guard.ok) return MARKOV_EDEVICE;
    cudaStream_t s = (cudaStream_t)stream;

    SampleArgs a{};
    a.base = base_f32 ? nullptr : static_cast<const uint16_t *>(base_logits);
    a.base_f = base_f32 ? static_cast<const float *>(base_logits) : nullptr;
    a.base_s0 = base_s0;
    a.base_s1 = base_s1;
    a.head = head;
    a.embed = embed;
    a.anchor = anchor_tokens;
    a.temperature = temperature;
    a.seeds = seeds;
    a.row_state_idx = row_state_idx;
    a.rows = rows;
    a.V = V;
    a.r = r;
    a.N = N;
    a.mode = (int)mode;
    a.tf = make_transform(output_multiplier, soft_cap);
    a.tokens = draft_tokens;
    a.tok_s0 = tok_s0;
    a.cache = cache_f32 ? nullptr : static_cast<uint16_t *>(logit_cache);
    a.cache_f = cache_f32 ? static_cast<float *>(logit_cache) : nullptr;
    a.cache_s0 = cache_s0;
    a.cache_s1 = cache_s1;
    a.noise = p->noise;
    a.noise_s0 = p->noise_s0;
    a.keys = p->keys;
    a.sums = p->sums;
    a.bar_count = p->ctrl;
    a.bar_base = p->ctrl + 1;
    a.status = p->ctrl + 2;
    a.call_counter = p->ctrl + 4;
    a.tc_sums = p->tc_sums;
    a.tok_slots = p->tok_slots;
    a.win_max = p->win_max;
    a.win_cnt = p->win_cnt;
    a.bwin = p->bwin;
    a.bcnt = p->bcnt;
    a.timeout_ns = (uint64_t)p->d.timeout_ms * 1000000ull;

    const bool batch_tc = !chain && p->batch_tc_ok;
    if ((use_tc || batch_tc) && p->tmap_head != head) {
        if (!encode_head_map(&p->tmap, head, V, r)) return MARKOV_ECUDA;
        p->tmap_head = head;
    }
    int launches = 0;
    const int noise_ready = p->noise_state != 0;
    if (p->noise_state == 1) {
        // join the forked noise (in inverse-CDF mode it is unused, but the
        // plan's buffer must not be rewritten while it is being drawn)
        if (cudaStreamWaitEvent(s, p->ev_noise, 0) != cudaSuccess) return MARKOV_ECUDA;
    } else if (p->noise_state == 0 && mode == MARKOV_GUMBEL && !use_tc) {
        // the tcgen05 chain draws its own noise while the head loads
        if (launch_noise(seeds, temperature, row_state_idx, rows, N, V, p->noise, p->noise_s0, 1,
                         s) != cudaSuccess)
            return MARKOV_ECUDA;
        ++launches;
    }
    p->noise_state = 0;

    if (use_tc) {
        a.grid = p->tc_grid;
        for (int b0 = 0; b0 < rows; b0 += kChainRows) {
            // rows [b0, b0 + 8) of the call as one chain launch
            SampleArgs as = a;
            const int64_t bo = (int64_t)b0;
            if (as.base) as.base += bo * base_s0;
            if (as.base_f) as.base_f += bo * base_s0;
            if (as.cache) as.cache += bo * cache_s0;
            if (as.cache_f) as.cache_f += bo * cache_s0;
            as.anchor += b0;
            as.temperature += b0;
            as.seeds += b0;
            as.row_state_idx += b0;
            as.tokens += bo * tok_s0;
            as.rows = rows - b0 < kChainRows ? rows - b0 : kChainRows;
            as.row_base = b0;
            cudaError_t e = launch_chain_tc(as, p->tmap, noise_ready, s);
            if (e == cudaErrorCooperativeLaunchTooLarge) { cudaGetLastError(); return MARKOV_ENOTRESIDENT; }
            if (e != cudaSuccess) { cudaGetLastError(); return MARKOV_ECUDA; }
            ++launches;
        }
        p->last_path = MARKOV_PATH_CHAIN;
    } else if (chain) {
        if (p->chain_occ < 1) return MARKOV_ENOTRESIDENT;
        a.grid = p->chain_grid;
        cudaError_t e = launch_chain(a, s);
        if (e == cudaErrorCooperativeLaunchTooLarge) { cudaGetLastError(); return MARKOV_ENOTRESIDENT; }
        if (e != cudaSuccess) { cudaGetLastError(); return MARKOV_ECUDA; }
        ++launches;
        p->last_path = MARKOV_PATH_CHAIN_SIMPLE;
    } else {
        a.grid = p->batch_grid;
        if (p->batch_dirty) {
            // an earlier call's launches failed part way: start from cleared slots
            if (cudaMemsetAsync(p->bwin, 0, kBatchWinN * sizeof(uint64_t), s) != cudaSuccess ||
                cudaMemsetAsync(p->bcnt, 0, kBatchCntN * sizeof(uint32_t), s) != cudaSuccess)
                return MARKOV_ECUDA;
            p->batch_dirty = false;
        }
        int n = 0;
        cudaError_t e = launch_batch(a, s, &n, batch_tc ? &p->tmap : nullptr, p->sm_count);
        if (e != cudaSuccess) { cudaGetLastError(); p->batch_dirty = true; return MARKOV_ECUDA; }
        launches += n;
        p->last_path = MARKOV_PATH_BATCH;
    }
    p->last_launches = launches;
    return MARKOV_OK;
}

markov_status markov_plan_status(markov_plan *p) {
    if (!p) return MARKOV_EINVAL;
    DeviceGuard guard(p->d.device);
    if (!guard.ok) return MARKOV_EDEVICE;
    if (cudaDeviceSynchronize() != cudaSuccess) { cudaGetLastError(); return MARKOV_ECUDA; }
    uint32_t ctrl[4];
    if (cudaMemcpy(ctrl, p->ctrl, sizeof(ctrl), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MARKOV_ECUDA;
    if (ctrl[2] == 0u) return MARKOV_OK;
    // a launch gave up: clear the status, restart the barrier and call
    // counters, and clear every exchange slot and word
    if (cudaMemset(p->ctrl, 0, 8 * sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(p->tc_sums, 0, p->tc_slots_n * sizeof(uint64_t)) != cudaSuccess ||
        cudaMemset(p->tok_slots, 0, (size_t)kMaxSteps * kChainRows * sizeof(uint64_t)) != cudaSuccess ||
        cudaMemset(p->win_max, 0, kWinMaxN * sizeof(uint64_t)) != cudaSuccess ||
        cudaMemset(p->win_cnt, 0, kWinCntN * sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(p->bwin, 0, kBatchWinN * sizeof(uint64_t)) != cudaSuccess ||
        cudaMemset(p->bcnt, 0, kBatchCntN * sizeof(uint32_t)) != cudaSuccess)
        return MARKOV_ECUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return MARKOV_ECUDA;
    return (markov_status)ctrl[2];
}

markov_status markov_gumbel_noise(const int64_t *seeds, const float *temperature,
                                  const int64_t *row_state_idx, int32_t rows, int32_t num_steps,
                                  int32_t vocab, float *out, int64_t out_s0, void *stream) {
    if (!seeds || !temperature || !row_state_idx || !out) return MARKOV_EINVAL;
    if (rows < 1 || rows > kMaxRows || num_steps < 1 || num_steps > kMaxSteps) return MARKOV_EINVAL;
    if (vocab < 1 || vocab > kMaxVocab || out_s0 < vocab) return MARKOV_EINVAL;
    if (launch_noise(seeds, temperature, row_state_idx, rows, num_steps, vocab, out, out_s0, 1,
                     (cudaStream_t)stream) != cudaSuccess)
        return MARKOV_ECUDA;
    return MARKOV_OK;
}

markov_status markov_device_math(int32_t fn, const float *x, float *y, int64_t n, void *stream) {
    if (fn < 0 || fn > 12 || n < 0 || (n > 0 && (!x || !y)) || (fn == 9 && n % 3 != 0) ||
        (fn == 12 && n % 2 != 0))
        return MARKOV_EINVAL;
    if (launch_device_math(fn, x, y, n, (cudaStream_t)stream) != cudaSuccess) return MARKOV_ECUDA;
    return MARKOV_OK;
}

markov_status markov_plan_inject_status(markov_plan *p, markov_status code, uint32_t where) {
    if (!p || code == MARKOV_OK) return MARKOV_EINVAL;
    DeviceGuard guard(p->d.device);
    if (!guard.ok) return MARKOV_EDEVICE;
    const uint32_t w[2] = {(uint32_t)code, where};
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(p->ctrl + 2, w, sizeof(w), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return MARKOV_ECUDA;
    }
    return MARKOV_OK;
}

int64_t markov_plan_query(const markov_plan *p, int32_t key) {
    if (!p) return -1;
    switch (key) {
        case MARKOV_Q_CHAIN_CTAS: return p->tc_ok ? p->tc_grid : p->chain_grid;
        case MARKOV_Q_RESIDENT_HEAD_BYTES:
            // the tcgen05 chain keeps every head byte on chip across positions
            return p->tc_ok ? (int64_t)p->d.vocab * p->d.rank * 2 : 0;
        case MARKOV_Q_LAST_LAUNCHES: return p->last_launches;
        case MARKOV_Q_LAST_PATH: return p->last_path;
        case MARKOV_Q_SM_COUNT: return p->sm_count;
    }
    return -1;
}

}  // extern "C"
