// internal.h -- structures shared by the C-ABI host code and the kernels.
#pragma once
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace dtm {

constexpr int kMaxSteps = 16;          // draft positions a plan may take
constexpr int kMaxVocab = 262144;      // vocabulary bound
constexpr int kMaxRows = 256;          // rows a plan may take
constexpr int kChainRows = 8;          // rows of one chain launch (MMA N = 8)
constexpr int kChainSliceRows = 24;    // automatic path, Gumbel: tcgen05 chain per 8-row slice up to here
constexpr int kChainThreads = 512;     // threads of a chain CTA (one CTA per SM)
constexpr int kBatchThreads = 256;
constexpr int kTile = 16;              // vocab ids per MMA tile (m16)
constexpr int kKeyPad = 16;            // u64 slots per CTA-key block are padded to 128 B
constexpr int kLineU64 = 16;           // one 128-byte line per exchange word
constexpr int kLineU32 = 32;
constexpr size_t kWinMaxN = (size_t)2 * kMaxSteps * kChainRows * kLineU64;
constexpr size_t kWinCntN = (size_t)2 * kMaxSteps * kLineU32;
// per-position path: a winner word per (position, row) and, per position,
// a done counter per row group of 16 or 32 rows (logits kernel; the first
// kMaxRows / 16 words) and per row (inverse-CDF sum kernel)
constexpr int kBatchCntPerStep = kMaxRows / 16 + kMaxRows;
constexpr size_t kBatchWinN = (size_t)kMaxSteps * kMaxRows;
constexpr size_t kBatchCntN = (size_t)kMaxSteps * kBatchCntPerStep;
constexpr int kCdfRounds = 6;                 // 8-id loads per thread of an inverse-CDF block
constexpr int kCdfIds = kBatchThreads * 8 * kCdfRounds;   // vocab ids per inverse-CDF block

// The output-logit transform (muse_spark markov page, FusedMarkovParams):
// multiplier and cap rounded to fp32, inv_cap = fp32(1) / fp32(cap).
struct Transform {
    int has_transform;
    int has_cap;
    float mult;
    float cap;
    float inv_cap;
};

// Everything one sample call passes to its kernels.
struct SampleArgs {
    const uint16_t *base;
    int64_t base_s0, base_s1;
    const uint16_t *head;
    const uint16_t *embed;
    const int32_t *anchor;
    const float *temperature;
    const int64_t *seeds;
    const int64_t *row_state_idx;
    int rows, V, r, N, mode;
    Transform tf;
    int64_t *tokens;
    int64_t tok_s0;
    uint16_t *cache;
    int64_t cache_s0, cache_s1;
    // fp32 variants (every path): when set, the base logits / the cache are
    // fp32 at these pointers (same strides, in elements) and base / cache are
    // unused
    const float *base_f;
    float *cache_f;
    float *noise;              // [rows * N, V] fp32 Gumbel noise (Gumbel mode)
    int64_t noise_s0;          // row stride of the noise, in floats
    // plan scratch
    uint64_t *keys;            // cross-CTA key / partial slots
    uint64_t *sums;            // cross-CTA inverse-CDF sums
    uint32_t *bar_count;       // grid barrier counter
    uint32_t *bar_base;        // the counter's value at the start of a launch
    uint32_t *status;          // [2]: sticky device status, where it happened
    uint32_t *call_counter;    // calls of the persistent tcgen05 chain so far
    uint64_t *tc_sums;         // [N][8][Gp] inverse-CDF sum slots of the tcgen05 chain
    uint64_t *tok_slots;       // [N][8] inverse-CDF token slots, (id << 32) | epoch
    uint64_t *win_max;         // [2 call parities][N][8 rows] x kLineU64: red.max words
    uint64_t *bwin;            // [kMaxSteps][kMaxRows] per-position path winners (0: none)
    uint32_t *bcnt;            // [kMaxSteps][kBatchCntPerStep] its done counters
    uint32_t *win_cnt;         // [2 call parities][N] x kLineU32: CTAs that reported (the
                               // inverse-CDF chain counts on to 2G for its sums)
    uint64_t timeout_ns;
    int grid;                  // persistent grid size (chain) or vocab blocks (batch)
    int row_base;              // the call's row index of this launch's row 0 (row slices
                               // of the chain): the noise and inverse-CDF hashes take it
};

// Kernel launchers (return the CUDA error of the launch).
// v_offset: the global vocabulary id of column 0 of `out` (a shard's noise)
cudaError_t launch_noise(const int64_t *seeds, const float *temperature,
                         const int64_t *row_state_idx, int rows, int N, int V, float *out,
                         int64_t out_s0, int mode_gumbel_only, cudaStream_t stream, int v_offset = 0);
cudaError_t launch_device_math(int fn, const float *x, float *y, int64_t n, cudaStream_t s);
cudaError_t chain_occupancy(int *blocks_per_sm);
cudaError_t launch_chain(const SampleArgs &a, cudaStream_t stream);
// tmap: the head's TMA descriptor; with it the per-position logits run on
// the tcgen05 kernel (batch_tc.cu) over `sms` multiprocessors, without it on
// the mma.sync kernel
cudaError_t launch_batch(const SampleArgs &a, cudaStream_t stream, int *launches,
                         const CUtensorMap *tmap = nullptr, int sms = 0);
cudaError_t batch_tc_prepare();
size_t batch_tc_smem(int rank);
cudaError_t launch_batch_tc_logits(const SampleArgs &a, const CUtensorMap &tmap, int i, int ctas,
                                   cudaStream_t stream, bool pdl);
int batch_blocks(int V);
size_t chain_tc_smem();
int chain_tc_max_chunks();
cudaError_t chain_tc_prepare();
cudaError_t chain_tc_occupancy(int *blocks_per_sm);
cudaError_t launch_chain_tc(const SampleArgs &a, const CUtensorMap &tmap, int noise_ready,
                            cudaStream_t stream);

}  // namespace dtm
