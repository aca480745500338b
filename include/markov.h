/*
 * markov.h -- C ABI of the GB300 (sm_103a) library for DSpark sequential
 * Markov sampling of speculative draft tokens.
 *
 * The method (sources: the documentation pages
 *   "vllm.models.deepseek_v41.nvidia.specialized_decode.sampling.sharded_markov",
 *   "vllm.models.deepseek_v41.nvidia.ops.fused_markov",
 *   "vllm.models.muse_spark.nvidia.specialized_decode.runtime.markov"):
 * for every request row b and draft position i = 0 .. N-1, with p the
 * anchor token at i = 0 and token i-1 afterwards,
 *   bias  = bf16(markov_head[V, r] . markov_embed[p])            (fp32 sums)
 *   l     = bf16(f32(base[b, i]) + f32(bias)), then optionally
 *           bf16(cap * tanh((l * mult) * (1 / cap)))               (transform)
 *   cache[b, i] = l;  token[b, i] = Gumbel-max of l / T + gumbel, or inverse
 *   CDF of softmax(l / T), argmax at T = 0; lowest NaN id first, lowest id
 *   among equal maxima.
 * (sharded_markov page, module docstring and "Per call" diagram; fused_markov
 * page, module docstring; muse_spark markov page, module docstring,
 * FusedMarkovParams and fused_markov_params.)
 *
 * Conventions for every entry point:
 *   - BF16 tensors are passed as uint16_t bit patterns.
 *   - "device" pointers must be CUDA device memory of the plan's device;
 *     "host" pointers are ordinary (preferably pinned) host memory.
 *   - The caller owns every tensor it passes; the library never frees or
 *     retains them beyond the call's stream work.  A plan owns only its own
 *     scratch, allocated once at creation (so CUDA graphs keep addresses).
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy
 *     default stream.  Calls enqueue work and return without synchronizing,
 *     except markov_plan_status.
 *   - Argument errors are reported synchronously by the return value and
 *     nothing is launched.  Device-side failures (a bounded wait that timed
 *     out) are recorded in a sticky device status word that
 *     markov_plan_status reads; kernels never trap.
 */
#ifndef DTM_MARKOV_H
#define DTM_MARKOV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum markov_status {
    MARKOV_OK = 0,
    MARKOV_EINVAL = 1,          /* bad argument: shape, stride, alignment, range */
    MARKOV_EUNSUPPORTED = 2,    /* valid but outside what this build runs */
    MARKOV_ECUDA = 3,           /* a CUDA runtime call failed */
    MARKOV_ETIMEOUT = 4,        /* an in-kernel bounded wait gave up */
    MARKOV_ENOTRESIDENT = 5,    /* the persistent grid cannot be co-resident */
    MARKOV_EDEVICE = 6          /* wrong or unusable device */
} markov_status;

typedef enum markov_mode {
    MARKOV_GUMBEL = 0,          /* Gumbel-max (sharded_markov page) */
    MARKOV_INVCDF = 1           /* inverse CDF (fused_markov page) */
} markov_mode;

/* Element type of the base logits and of the logits cache (sharded_markov
 * page: the chain kernel is compiled per base and cache dtype, BF16 or fp32). */
typedef enum markov_dtype {
    MARKOV_BF16 = 0,
    MARKOV_F32 = 1
} markov_dtype;

typedef enum markov_path {
    MARKOV_PATH_AUTO = 0,       /* up to markov_chain_max_rows rows: the chain; Gumbel mode
                                   up to 24 rows (no forked noise pending, tcgen05 chain
                                   available): one tcgen05 chain launch per 8-row slice;
                                   else batch */
    MARKOV_PATH_CHAIN = 1,      /* the persistent single-launch chain kernel (tcgen05, head
                                   resident in TMEM and shared memory when it fits) */
    MARKOV_PATH_BATCH = 2,      /* per-position kernels (the larger-batch loop) */
    MARKOV_PATH_CHAIN_SIMPLE = 3 /* the persistent chain with mma.sync bias tiles and the
                                   head re-read from L2 each position: the fallback when
                                   the head does not fit on chip */
} markov_path;

/* Static configuration of a plan.  vocab % 16 == 0 and vocab <= 262144
 * (sharded_markov page, unsupported_reason: V divisible by 16 per rank and
 * bounded); rank a power of two in {64, 128, 256} (muse_spark page,
 * unsupported: a power-of-two-rank w1); 1 <= num_steps <= 16 (a bound on
 * draft positions, unsupported_reason); 1 <= max_rows <= 256.
 * timeout_ms bounds every in-kernel wait (0 selects 100 ms). */
typedef struct markov_desc {
    int32_t vocab;
    int32_t rank;
    int32_t num_steps;
    int32_t max_rows;
    int32_t device;
    int32_t timeout_ms;
} markov_desc;

typedef struct markov_plan markov_plan;

/* Validate `desc`, select the device, and allocate every scratch buffer the
 * plan's calls use (noise [max_rows * N, V] fp32, key and partial-sum slots,
 * barrier and status words, the side stream and its events).  On success
 * *out receives the plan; on failure *out is NULL and nothing is leaked.
 * (sharded_markov page, DSparkShardedMarkovSampler.__init__: persistent
 * buffers allocated once; fused_markov page, FusedMarkovSampler: scratch
 * allocated at init so CUDA graphs keep the addresses.) */
markov_status markov_plan_create(const markov_desc *desc, markov_plan **out);

/* Synchronize the plan's device work and free its scratch.  NULL is a no-op. */
void markov_plan_destroy(markov_plan *plan);

/* Rows a single chain launch takes: 8 (sharded_markov page, module
 * docstring: "up to 8 request rows", the MMA columns). */
int32_t markov_chain_max_rows(const markov_plan *plan);

/* Force the path of later markov_chain_sample calls (testing and
 * benchmarking); MARKOV_PATH_AUTO restores the default.  EINVAL for an
 * unknown path; EUNSUPPORTED is returned later by a call whose rows the
 * forced chain path cannot take. */
markov_status markov_plan_set_path(markov_plan *plan, markov_path path);

/* Draw this call's Gumbel noise on the plan's side stream, ordered after the
 * work already enqueued on `stream`; the next markov_chain_sample on the
 * plan joins it.  seeds [rows] int64, temperature [rows] fp32,
 * row_state_idx [rows] int64 are device pointers and must be the arrays the
 * sample call passes.  The noise depends only on (seed, row, position, vocab
 * id), never on the chain (sharded_markov page, fork_noise and
 * _shard_noise_kernel).  Optional: without it the sample call draws the
 * noise itself on its own stream.  EINVAL if rows > max_rows. */
markov_status markov_noise_fork(markov_plan *plan, const int64_t *seeds,
                                const float *temperature, const int64_t *row_state_idx,
                                int32_t rows, void *stream);

/* Make `stream` wait for the noise of the last markov_noise_fork (the
 * sharded_markov page's join_noise); the next markov_chain_sample must then
 * run on this same stream.  A no-op when no fork is pending. */
markov_status markov_noise_join(markov_plan *plan, void *stream);

/* Draw every live row's N draft tokens and write its logits cache.
 *   base_logits   device, BF16 [rows, N, V]: element (b, i, v) at
 *                 b * base_s0 + i * base_s1 + v; last stride 1.
 *   head, embed   device, BF16 [V, r] contiguous (markov_head / w2 and
 *                 markov_embed / w1).
 *   anchor_tokens device, int32 [rows]: each row's previous token at i = 0.
 *   temperature   device, fp32 [rows]; T > 0 samples, anything else is greedy.
 *   seeds         device, int64 [rows].
 *   row_state_idx device, int64 [rows]; < 0 marks a padding row, which is
 *                 inert: neither its tokens nor its cache are written.
 *   mode          MARKOV_GUMBEL or MARKOV_INVCDF.
 *   output_multiplier, soft_cap: the transform; soft_cap <= 0 means none.
 *                 Both are used as fp32 and inv_cap = fp32(1) / fp32(cap).
 *   draft_tokens  device, int64 [rows, N], element (b, i) at b * tok_s0 + i.
 *   logit_cache   device, BF16 [rows, N, V], element (b, i, v) at
 *                 b * cache_s0 + i * cache_s1 + v; pointer and strides
 *                 16-byte aligned (sharded_markov page, sample: cache asserts).
 * Host-resident inputs and tokens: base_logits, anchor_tokens, temperature,
 * seeds, row_state_idx and draft_tokens may instead be page-locked host
 * memory the device can address (cudaHostAlloc, cudaHostRegister, or a
 * pinned torch CPU tensor); the kernels then read the inputs and write the
 * tokens over the host link during the call, with no staging copy (on
 * GB300 the NVLink-C2C link; the bytes are the same, the results bit for bit
 * those of device-resident arguments).  head, embed and logit_cache must be
 * device memory.  The host must not write the inputs or read the tokens
 * before the call's stream work completes.
 * Rows up to markov_chain_max_rows take one persistent launch; Gumbel calls
 * of up to 24 rows one persistent launch per 8-row slice (the noise hash
 * takes each row's index in the call); larger calls take the per-position
 * kernels (sharded_markov page, module docstring: larger batches take the
 * fused loop).  The path actually taken and its launch count are reported by
 * markov_plan_query.  EINVAL on a bad shape, stride,
 * alignment or mode; ENOTRESIDENT if the persistent grid cannot be
 * co-resident; ECUDA if a launch fails. */
markov_status markov_chain_sample(markov_plan *plan, const uint16_t *base_logits,
                                  int64_t base_s0, int64_t base_s1, const uint16_t *head,
                                  const uint16_t *embed, const int32_t *anchor_tokens,
                                  const float *temperature, const int64_t *seeds,
                                  const int64_t *row_state_idx, int32_t rows,
                                  markov_mode mode, float output_multiplier,
                                  float soft_cap, int64_t *draft_tokens, int64_t tok_s0,
                                  uint16_t *logit_cache, int64_t cache_s0,
                                  int64_t cache_s1, void *stream);

/* markov_chain_sample with the base logits and the cache in either dtype
 * (sharded_markov page: BF16 or fp32 for both; the module docstring's
 * cache_round rounds each logit to the cache's dtype).
 *   base_logits   device, [rows, N, V] of base_dtype, strides in elements.
 *   logit_cache   device, [rows, N, V] of cache_dtype, strides in elements;
 *                 pointer and row strides 16-byte aligned.
 *   With an fp32 cache a logit is fp32(base) + fp32(bf16(head . embed)),
 *   then the transform's fp32 steps when there is one, never rounded to
 *   BF16; with a BF16 cache it is markov_chain_sample's logit (an fp32 base
 *   is added in fp32 before the BF16 rounding).  Keys and tokens follow from
 *   the cached values exactly as in markov_chain_sample.
 * BF16 / BF16 is markov_chain_sample.  Every path takes every dtype pair
 * (each kernel is compiled per base and cache dtype).  Other arguments
 * (host-resident inputs and tokens included) and errors as
 * markov_chain_sample; EINVAL for an unknown dtype. */
markov_status markov_chain_sample_typed(markov_plan *plan, const void *base_logits,
                                        markov_dtype base_dtype, int64_t base_s0,
                                        int64_t base_s1, const uint16_t *head,
                                        const uint16_t *embed, const int32_t *anchor_tokens,
                                        const float *temperature, const int64_t *seeds,
                                        const int64_t *row_state_idx, int32_t rows,
                                        markov_mode mode, float output_multiplier,
                                        float soft_cap, int64_t *draft_tokens, int64_t tok_s0,
                                        void *logit_cache, markov_dtype cache_dtype,
                                        int64_t cache_s0, int64_t cache_s1, void *stream);

/* markov_chain_sample without a plan, for callers that cannot allocate
 * device memory: code running while a CUDA graph is captured on a stream
 * that forbids allocation, servers and plugins that must draw every byte
 * from their own pre-sized pool, processes whose allocator belongs to
 * another runtime.  No counterpart on the documentation pages: it is an
 * addition of this library.
 *   Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   Its scratch (Gumbel noise, cross-CTA slots, barrier and status words)
 *   is one file-scope device array of 33 MiB that every GPU loading the
 *   library holds until the process exits; the calling thread's current
 *   device is used.  The first call on a device looks up that array's
 *   address (cudaGetSymbolAddress); make that first call before any stream
 *   capture.
 *   Arguments, layouts and results are those of markov_chain_sample with
 *   vocab, rank and num_steps given directly; it runs the noise kernel and
 *   the simple persistent chain (the MARKOV_PATH_CHAIN_SIMPLE path), so its
 *   outputs equal that path's bit for bit.
 *   Limits: rows <= 8; in MARKOV_GUMBEL mode also rows * num_steps * vocab
 *   <= 8388608 (the Gumbel noise must fit 32 MiB; inverse-CDF calls draw no
 *   noise and take any vocab up to the library's 262144).  Larger calls
 *   return MARKOV_EUNSUPPORTED before any work is enqueued.  Every call
 *   clears the array's control words on `stream` first.  All calls share the
 *   array, which keeps the last call's contents: calls that may overlap on
 *   the GPU (other streams, other host threads) race and must be serialized
 *   by the caller.
 *   Device-side errors are not reported (reporting needs a plan's
 *   markov_plan_status), so the caller must pass valid device data: every
 *   live row's anchor token in [0, vocab) (an anchor outside it samples from
 *   id 0 and the call still returns MARKOV_OK).  The kernels' bounded waits
 *   give up after a fixed 100 ms; a wait that gives up leaves that call's
 *   outputs incomplete, also unreported. */
markov_status markov_chain_sample_static(int32_t vocab, int32_t rank, int32_t num_steps,
                                         const uint16_t *base_logits, int64_t base_s0,
                                         int64_t base_s1, const uint16_t *head,
                                         const uint16_t *embed, const int32_t *anchor_tokens,
                                         const float *temperature, const int64_t *seeds,
                                         const int64_t *row_state_idx, int32_t rows,
                                         markov_mode mode, float output_multiplier,
                                         float soft_cap, int64_t *draft_tokens, int64_t tok_s0,
                                         uint16_t *logit_cache, int64_t cache_s0,
                                         int64_t cache_s1, void *stream);

/* Synchronize the plan's device and return (then clear) the sticky device
 * status: MARKOV_OK, or MARKOV_ETIMEOUT when a bounded wait gave up, in
 * which case the plan's barrier words are re-zeroed so the next call starts
 * clean.  ECUDA if the device reports an error. */
markov_status markov_plan_status(markov_plan *plan);

/* A static English description of a status code. */
const char *markov_status_string(markov_status status);

/* Gumbel noise, standalone: out[(b * N + i) * out_s0 + v] = -log(-log u) of
 * (seeds[b], b, i, v) for every live row with temperature > 0, v < V.  Rows
 * that are padding or greedy are not written.  Device pointers; the same
 * kernel markov_noise_fork runs (sharded_markov page, _shard_noise_kernel).
 * out_s0 >= V. */
markov_status markov_gumbel_noise(const int64_t *seeds, const float *temperature,
                                  const int64_t *row_state_idx, int32_t rows,
                                  int32_t num_steps, int32_t vocab, float *out,
                                  int64_t out_s0, void *stream);

/* Evaluate the device's own scalar functions element-wise over n floats
 * (device pointers): fn 0 natural log, 1 exp, 2 tanh, 3 Gumbel transform
 * -log(-log x), 4 fp32 -> BF16 round-to-nearest-even (result bits in the
 * low 16 bits of the output word, read as uint32), 5 the same rounding by
 * the packed two-value conversion the tcgen05 chain's epilogue uses (a NaN
 * gives some NaN; 0xDEAD if the two packed halves disagree).  The Gumbel
 * pruning bounds of the tcgen05 chain: fn 6 the noise byte q of a uniform
 * mantissa m < 2^23 passed as the input word's bits (u = (m + 1/2) 2^-23),
 * fn 7 / 8 the upper / lower noise bound of the byte q passed as a float
 * value; fn 9 on triples (l, T, m bits), n a multiple of 3: the Gumbel key's
 * lower bound, its upper bound and the exact key fp32(l / T) + gumbel(u) as
 * the chain computes them.  fn 10 / 11: the low / high 32 bits (read as
 * uint32) of the inverse-CDF integer weight floor(exp(d) 2^40) of
 * d = fp32(l / T) - M <= 0, as every inverse-CDF kernel computes it.  fn 12
 * on pairs (l, T), n even: fp32(l / T) as the inverse-CDF kernels compute
 * it (a product by 1 / T when T is a power of two) and 1 where that product
 * was taken, else 0.  These are the functions the kernels use;
 * exposed so they can be compared bit for bit with an independent
 * implementation, or checked against it as bounds.  EINVAL for an unknown
 * fn. */
markov_status markov_device_math(int32_t fn, const float *x, float *y, int64_t n,
                                 void *stream);

/* Plan facts for reporting: MARKOV_Q_CHAIN_CTAS (persistent grid size),
 * MARKOV_Q_RESIDENT_HEAD_BYTES (head bytes the chain kernel keeps on chip
 * across positions), MARKOV_Q_LAST_LAUNCHES (kernel launches the last
 * sample call enqueued), MARKOV_Q_LAST_PATH (markov_path it took),
 * MARKOV_Q_SM_COUNT.  Returns -1 for an unknown key or a NULL plan. */
enum {
    MARKOV_Q_CHAIN_CTAS = 0,
    MARKOV_Q_RESIDENT_HEAD_BYTES = 1,
    MARKOV_Q_LAST_LAUNCHES = 2,
    MARKOV_Q_LAST_PATH = 3,
    MARKOV_Q_SM_COUNT = 4
};
int64_t markov_plan_query(const markov_plan *plan, int32_t key);

/* Failure detection without a GPU fault (the pages have no counterpart:
 * these are test hooks).
 *
 * markov_plan_inject_status records (code, where) in the plan's sticky
 * device status exactly as a kernel that gave up would (synchronous copy, no
 * kernel runs).  Every later call's kernels see it at their first check and
 * return without computing or writing outputs, until markov_plan_status
 * reports and clears it.  code must be a nonzero markov_status; EINVAL for a
 * NULL plan or a zero code.
 *
 * markov_selftest_wait runs one of the kernels' bounded waits on a wait that
 * nothing can complete, in a one-CTA kernel on `stream`, with a limit of
 * timeout_us microseconds (1 .. 1e6): which 0 is the chain's grid barrier,
 * which 1 an mbarrier wait of the tcgen05 chain.  It synchronizes the stream
 * and returns the status the kernel recorded: MARKOV_ETIMEOUT when the wait
 * gave up as designed, MARKOV_OK if it (wrongly) completed.  The kernel
 * never traps and leaves the context usable.  Its scratch is a static device
 * array, so concurrent calls race. */
markov_status markov_plan_inject_status(markov_plan *plan, markov_status code, uint32_t where);
markov_status markov_selftest_wait(int32_t which, int32_t timeout_us, void *stream);

/* ------------------------------------------------------------------------
 * The vocabulary-sharded chain (sharded_markov page, module docstring and
 * "Per call" diagram), its ranks emulated on one GPU.
 *
 * Rank k of `world` owns rows [k V / world, (k + 1) V / world) of the head.
 * Per draft position every rank computes its shard's logits, writes them
 * into its own cache and into every peer's staging buffer, takes its shard's
 * best key (fp32(l / T) + gumbel, l at T = 0; lowest id among equal keys, a
 * NaN above all) and sends one 64-bit key per (rank, row, position) to every
 * rank's mailbox; the best key of the world is the token on every rank.
 * After the last position each rank copies its peers' columns from its
 * staging buffer into its own cache.  Gumbel-max sampling only, as on the
 * page.  Here the ranks are groups of CTAs of one cooperative launch on the
 * plan's device, each with its own allocations (noise shard, staging buffer,
 * mailbox, CTA key slots); the results equal markov_chain_sample's on the
 * same inputs (the same bias tiles as MARKOV_PATH_CHAIN_SIMPLE: every rank's
 * tokens and full cache are bit-identical to that path's). */
typedef struct markov_shard_plan markov_shard_plan;

/* A sharded plan for `world` ranks (1, 2, 4 or 8): vocab % (16 world) == 0
 * (16-id tiles per rank), rank in {64, 128, 256}, 1 <= num_steps <= 16,
 * 1 <= max_rows <= 8 (the MMA columns), timeout_ms as for markov_plan_create.
 * Allocates every rank's scratch separately.  EINVAL for a bad desc or world;
 * ENOTRESIDENT if no CTA per rank fits. */
markov_status markov_shard_plan_create(const markov_desc *desc, int32_t world,
                                       markov_shard_plan **out);

/* Synchronize and free the plan's scratch.  NULL is a no-op. */
void markov_shard_plan_destroy(markov_shard_plan *plan);

/* CTAs of one sharded launch (world x CTAs per rank); -1 for NULL. */
int32_t markov_shard_plan_ctas(const markov_shard_plan *plan);

/* Synchronize, return and clear the sticky device status of the plan's calls
 * (as markov_plan_status); after an error it also clears the key slots and
 * mailboxes.  A call made while a status is pending writes nothing. */
markov_status markov_shard_plan_status(markov_shard_plan *plan);

/* Sample `rows` request rows (1 <= rows <= max_rows) on every rank.
 *   base_logits   device [rows, N, V] BF16, full vocabulary (each rank reads
 *                 its columns), strides base_s0 >= N base_s1, base_s1 >= V,
 *                 last stride 1;
 *   head_shards   host array of `world` device pointers: rank k's head rows
 *                 [V / world, r] BF16, contiguous, 16-byte aligned;
 *   embed         device [V, r] BF16, contiguous, 16-byte aligned (every
 *                 rank's copy of the embedding table);
 *   anchor_tokens, temperature, seeds, row_state_idx: device [rows] as for
 *                 markov_chain_sample (T = 0 argmax; idx < 0 padding);
 *   draft_tokens  host array of `world` device pointers, rank k's [rows, N]
 *                 int64 output, row stride tok_s0 >= N;
 *   logit_caches  host array of `world` device pointers, rank k's
 *                 [rows, N, V] BF16 output (full vocabulary), 16-byte
 *                 aligned, cache_s0 >= N cache_s1, cache_s1 >= V, both
 *                 multiples of 8.
 * Padding rows are written on no rank.  Asynchronous on `stream`; argument
 * errors return EINVAL with nothing launched; a bounded wait that gives up
 * records MARKOV_ETIMEOUT for markov_shard_plan_status. */
markov_status markov_chain_sample_sharded(markov_shard_plan *plan, const uint16_t *base_logits,
                                          int64_t base_s0, int64_t base_s1,
                                          const uint16_t *const *head_shards,
                                          const uint16_t *embed, const int32_t *anchor_tokens,
                                          const float *temperature, const int64_t *seeds,
                                          const int64_t *row_state_idx, int32_t rows,
                                          float output_multiplier, float soft_cap,
                                          int64_t *const *draft_tokens, int64_t tok_s0,
                                          uint16_t *const *logit_caches, int64_t cache_s0,
                                          int64_t cache_s1, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DTM_MARKOV_H */
