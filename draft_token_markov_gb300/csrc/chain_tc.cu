// chain_tc.cu -- the Blackwell persistent Markov chain kernel: all N draft
// positions of up to 8 request rows in one cooperative launch, with the whole
// Markov head resident on chip across positions.
//
// Sources: sharded_markov page, module docstring (one cooperative kernel per
// shard runs the whole chain and keeps its head rows on chip, so the head is
// read once; up to 8 request rows are the MMA columns; shards agree on each
// position's winner by exchanging one 64-bit (score, index) key; the noise
// is drawn beside the chain) and _shard_noise_kernel (counter-based noise).
// Here the shards are the CTAs of one GPU.
//
// Per CTA: a contiguous run of 128-id vocab tiles (at most 28 chunks of
// [128 ids x 64 K]).  The first 15 chunks live in Tensor Memory as MMA A
// operands (32 columns each), the rest in shared memory in the 128-byte
// swizzled K-major layout the TMA writes.  The 32 free TMEM columns hold two
// 16-column accumulators, and each accumulator takes TWO tiles at once: the
// B operand (the 8 rows' embeddings, N = 16) is read through two views of
// one shared-memory buffer, [E, 0] for the first tile (its bias lands in
// columns 0-7) and [0, E] for the second (columns 8-15); each MMA adds
// exact zeros to the other half.  Measured on GB300: one issuing warp costs
// ~50 cycles per M=128, N=16, K=16 MMA whatever the A source, two issuing
// warps ~25 cycles per MMA together, so two issuers with two tiles per
// accumulator round give the tensor pipe four tiles in flight.
//
// Warp roles (20 warps, 640 threads):
//   0      issues the MMAs of the tiles whose A chunks start in TMEM, two
//          tiles per round into accumulator 0
//   1      the same for the shared-memory tiles, accumulator 1
//   2      lane 0: TMA producer of the head chunks (position 0 only); later
//          positions: the next position's base logits into L2
//   3      lane 0: copies the TMEM-resident chunks from their shared-memory
//          staging slot into TMEM (position 0 only); later: base prefetch
//   4-19   the epilogue: warp 4 + 4c + q reads TMEM lane quarter q of
//          accumulator c / 2, half c % 2 (one tile), so each thread owns one
//          vocab id and all 8 rows; at position 0, before it, the noise
//          bounds of position 0 while the head streams in; after every
//          position, the next position's noise bounds while the winners
//          are exchanged
//   0-3    after each position: the exchange of every row's key with the
//          other CTAs and the staging of markov_embed[token] of rows w and
//          w + 4 as the next position's B operand
// Cross-CTA exchange: every CTA stores its per-row best key, tagged with the
// call's position epoch, into its own slot of a [position][row][CTA] array;
// every CTA polls all slots of its rows until every tag is current and
// takes the maximum (one L2 round trip after the last store, no counter and
// no second read).  Inverse-CDF rows exchange the maximum this way, then
// per-CTA exact integer weight sums (tagged in their top bits); every CTA
// then finds the CTA whose prefix range holds the target and scans that
// CTA's cached logits itself (no third exchange).

#include <cuda.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "gumbel_bounds.cuh"
#include "tc.cuh"

namespace dtm {

namespace {

constexpr int kEpiWarps = 16;             // epilogue warps 4..19
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 128 + kEpiThreads;   // 4 control warps, then the epilogue warps
constexpr int kTmemChunks = 15;           // A chunks in TMEM (32 columns each)
constexpr int kSmemChunks = 13;           // A chunks in shared memory (16 KB each)
constexpr int kMaxChunks = kTmemChunks + kSmemChunks;
constexpr uint32_t kChunkBytes = 128 * 128;   // 128 rows x 64 BF16
constexpr uint32_t kDCol = 480;           // accumulators: columns 480..495, 496..511
constexpr uint32_t kIdesc = tc::idesc_bf16(128, 16);
constexpr uint32_t kSmemHead = kSmemChunks * kChunkBytes;
// B operand: per K-chunk kc an 8-row block E_kc (the rows' embeddings, 128 B
// per row) between zero blocks: [Z][E_0][Z][E_1][Z][E_2][Z][E_3][Z], 1 KB
// each; the view starting at E_kc is [E, 0], the one starting at the zero
// block before it [0, E]
constexpr uint32_t kSmemB = (2 * 4 + 1) * 1024;
constexpr uint32_t kDynSmem = kSmemHead + kSmemB + 1024;   // + alignment slack
constexpr uint32_t kKeyTagMask = 0x3FFFu;   // packed key: ordered key 32 | id 18 | tag 14
constexpr int kSumTagShift = 52;            // sum slots: tag 12 | sum 52

struct Ctl {
    uint64_t full[kSmemChunks];      // TMA landed in slot s
    uint64_t cpdone[kSmemChunks];    // slot s copied into TMEM
    uint64_t accf[2];                // accumulator w holds a finished tile pair
    uint64_t accr[2];                // accumulator w read out by its 8 epilogue warps
    uint64_t fin[2];                 // issuer w's MMAs all complete (exit)
    // Per position parity (a position's values are read while the next
    // one's are written): per row, the CTA's best packed key and, for Gumbel
    // rows, the CTA's threshold (ordered key of the largest key lower bound).
    unsigned long long cbest[2][kChainRows];
    uint32_t lcta[2][kChainRows];
    uint64_t win[kChainRows];
    unsigned long long sum[kChainRows];
    uint64_t wtot[kThreads / 32];    // inverse-CDF scan: per-warp weight totals
    int cstar[kChainRows];           // inverse CDF: the CTA holding the target
    uint64_t rem[kChainRows];        // the target minus the prefix before that CTA
    uint32_t tok[kChainRows];        // the token the scan found
    uint32_t tmem_base;
    uint32_t tmem_ready;             // chunks copied into TMEM so far
    uint32_t abort;
    uint32_t call;                   // the plan's call counter at launch
    int live[kChainRows];
    int sampling[kChainRows];
    float T[kChainRows];
    float invT[kChainRows];          // 1 / T, only for bounds
    uint64_t seed[kChainRows];
    uint64_t hri[kMaxSteps][kChainRows];   // row-step hash of every position
    int64_t prev[kChainRows];
};

__device__ __forceinline__ void fail(Ctl &c, const SampleArgs &a, uint32_t code, uint32_t where) {
    set_status(a.status, code, where);
    c.abort = 1u;
}

// The staging slot of head chunk j and the load's phase in that slot.
// TMEM chunks j < kSmemChunks take slot j (phase 0); the e = ntm -
// kSmemChunks later TMEM chunks reuse the last e slots (phase 1), whose
// first chunks land first; the shared-memory chunks j >= ntm (only when ntm
// = kTmemChunks) stay in slot j - kTmemChunks, after that slot's TMEM
// chunks.  So the loads of shared-memory chunks for the first slots wait
// on early copies and are not queued behind the second TMEM round.
__device__ __forceinline__ void chunk_slot(int j, int ntm, int &slot, uint32_t &phase) {
    const int e = ntm > kSmemChunks ? ntm - kSmemChunks : 0;
    if (j < kSmemChunks && j < ntm) {
        slot = j;
        phase = 0u;
    } else if (j < ntm) {
        slot = j - e;
        phase = 1u;
    } else {
        slot = j - kTmemChunks;
        phase = 1u + (slot >= kSmemChunks - e ? 1u : 0u);
    }
}

// The per-position CTA maxima of one parity back to zero.
__device__ __forceinline__ void clear_position(Ctl &c, int par) {
    for (int b = 0; b < kChainRows; ++b) {
        c.cbest[par][b] = 0ull;
        c.lcta[par][b] = 0u;
    }
}

// This CTA's abort flag (shared memory: cheap enough for hot loops).
__device__ __forceinline__ bool aborted(const Ctl &c) {
    return *(volatile const uint32_t *)&c.abort != 0u;
}

// At a CTA barrier: this CTA's flag, or (thread 0 only, one L2 load, when
// `global` is set) an error another CTA recorded.  The Gumbel positions
// check the global status in their exchange poll instead, off the barrier.
__device__ __forceinline__ bool stop_vote(Ctl &c, const SampleArgs &a, bool global = true) {
    bool s = *(volatile const uint32_t *)&c.abort != 0u;
    if (global && threadIdx.x == 0 && !s && ld_acquire_u32(a.status) != 0u) {
        c.abort = 1u;
        s = true;
    }
    return s;
}

__device__ __forceinline__ uint32_t unpack_id(uint64_t p) {
    return 0x3FFFFu - (uint32_t)((p >> 14) & 0x3FFFFu);
}

// The tiles of CTA `cta` of G: [t0, t1) of T_total 128-id tiles.
__device__ __forceinline__ void cta_tiles(int cta, int G, int T_total, int &t0, int &t1) {
    t0 = (int)((int64_t)cta * T_total / G);
    t1 = (int)((int64_t)(cta + 1) * T_total / G);
}

// Stage 8 elements of markov_embed[p] (16-byte piece `lane` of the row) as
// row b of the B operand's E blocks (K-major, 128-byte swizzle: piece k of
// row b at piece k ^ b).
template <int RANK>
__device__ __forceinline__ void stage_row(uint8_t *b_s, const uint4 v, int b, int lane) {
    const int chunk = lane >> 3, piece = lane & 7;
    *reinterpret_cast<uint4 *>(b_s + (2 * chunk + 1) * 1024 + b * 128 + ((piece ^ b) << 4)) = v;
}

// The noise-bound bytes of position p for this CTA's ids, 8 row bytes per
// id, written by a group of NT threads (thread te takes ids v_begin + te +
// NT j, two at a time so that their hash and log chains overlap).  The
// noise depends on seeds and positions only, so it is drawn off the chain's
// critical path: position 0 by the epilogue warps while the head streams
// in, position p + 1 by the same warps while position p's winners are
// exchanged.  The row loop stays rolled: the kernel's code must fit the
// instruction caches.
template <int NT>
__device__ __forceinline__ void noise_bounds(const Ctl &c, const SampleArgs &a, int p,
                                             uint32_t gum_m, int v_begin, int v_end, int te) {
    uint2 *gq = reinterpret_cast<uint2 *>(a.noise) + (int64_t)p * a.V;
#pragma unroll 1
    for (int v0 = v_begin + te; v0 < v_end; v0 += 2 * NT) {
        uint32_t lo[2] = {0u, 0u}, hi[2] = {0u, 0u};
#pragma unroll 1
        for (int b = 0; b < kChainRows; ++b) {
            if (!((gum_m >> b) & 1u)) continue;
            const uint64_t hb = c.hri[p][b];
            const int sh = 8 * (b & 3);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint32_t qv =
                    quantize_upper(gumbel_upper(dm_splitmix64(hb ^ (uint64_t)(v0 + NT * u)))) << sh;
                lo[u] |= b < 4 ? qv : 0u;
                hi[u] |= b < 4 ? 0u : qv;
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
            if (v0 + NT * u < v_end) gq[v0 + NT * u] = make_uint2(lo[u], hi[u]);
    }
}

// Warm L2 with this CTA's base logits of position p (every live row), one
// 128-byte line per thread of a group of NT threads.
template <int NT>
__device__ __forceinline__ void prefetch_base(const Ctl &c, const SampleArgs &a, int p, int v_begin,
                                              int v_end, int te) {
    const int es = a.base_f ? 4 : 2;   // BF16 or fp32 base logits
#pragma unroll 1
    for (int b = 0; b < a.rows && b < kChainRows; ++b) {
        if (!c.live[b]) continue;
        const int64_t off = b * a.base_s0 + (int64_t)p * a.base_s1;
        const uint8_t *row = a.base_f ? reinterpret_cast<const uint8_t *>(a.base_f + off)
                                      : reinterpret_cast<const uint8_t *>(a.base + off);
        for (int64_t o = (int64_t)v_begin * es + te * 128; o < (int64_t)v_end * es; o += NT * 128)
            tc::prefetch_l2(row + o);
    }
}

// The output-logit transform of two packed cached logits (out of line: only
// soft-capped heads take it, and its tanh is long).
__device__ __noinline__ uint32_t transform_pair(uint32_t lp, const Transform &tf) {
    float y0 = __fmul_rn(__uint_as_float(lp << 16), tf.mult);
    float y1 = __fmul_rn(__uint_as_float(lp & 0xffff0000u), tf.mult);
    if (tf.has_cap) {
        y0 = __fmul_rn(tf.cap, dm_tanh(__fmul_rn(y0, tf.inv_cap)));
        y1 = __fmul_rn(tf.cap, dm_tanh(__fmul_rn(y1, tf.inv_cap)));
    }
    return bf16x2_rn(y0, y1);
}

// The output-logit transform of one fp32 logit, kept in fp32 (fp32 caches).
__device__ __noinline__ float transform_f32(float s, const Transform &tf) {
    float y = __fmul_rn(s, tf.mult);
    if (tf.has_cap) y = __fmul_rn(tf.cap, dm_tanh(__fmul_rn(y, tf.inv_cap)));
    return y;
}

// Tiles of issuer w: [0, n0) for issuer 0 (their first chunk is in TMEM),
// [n0, nt) for issuer 1; each round takes two of them (a pair).
__device__ __forceinline__ int issuer_first(int w, int n0) { return w == 0 ? 0 : n0; }
__device__ __forceinline__ int issuer_last(int w, int n0, int nt) { return w == 0 ? n0 : nt; }

// The MMAs of issuer W (warp W) at position i: per round a tile pair (ta,
// tb) into accumulator W, ta through the [E, 0] view of B (columns 0-7) and
// tb through [0, E] (columns 8-15); per tile, K chunk by K chunk, 4 MMAs
// of K = 16, with A in TMEM (chunk j < kTmemChunks) or in shared memory.
// The first MMA of ta starts the accumulator (its [E, 0] view also zeroes
// tb's half), all others accumulate.  The whole warp runs the loop and one
// elected lane issues.  Position 0 awaits each chunk as the head streams in.
template <int RANK>
__device__ __forceinline__ void issue_tiles(Ctl &c, const SampleArgs &a, const uint32_t tmem, const int W,
                                            const int i, const int n0, const int nt, const int ntm,
                                            const uint32_t b_sa, const uint32_t head_sa,
                                            const uint64_t timeout, uint32_t &uses) {
    constexpr int cpt = RANK / 64;
    const int lane = threadIdx.x & 31;
    const uint32_t d = tmem + kDCol + 16u * (uint32_t)W;
    const uint64_t bdesc0 = tc::sw128_desc(b_sa), adesc0 = tc::sw128_desc(head_sa);
    const int first = issuer_first(W, n0), last = issuer_last(W, n0, nt);
#pragma unroll 1
    for (int ta = first; ta < last; ta += 2) {
        if (__any_sync(0xffffffffu, aborted(c))) break;
        bool freed = true;
        if (uses > 0)
            freed = tc::mbar_wait(tc::smem_u32(&c.accr[W]), (uses - 1) & 1u, tc::now_ns() + timeout);
        if (!__all_sync(0xffffffffu, freed)) {
            if (lane == 0) fail(c, a, 4u, 0x1000u + i);
            break;
        }
        tc::fence_after_sync();
        bool ok = true;
        const int ntile = ta + 1 < last ? 2 : 1;
#pragma unroll 1
        for (int h = 0; h < ntile && ok; ++h) {
            const int k = ta + h;
            // [E, 0] starts at E_kc (block 2 kc + 1), [0, E] at block 2 kc
            const uint64_t bview = bdesc0 + (uint64_t)(h == 0 ? (1024 >> 4) : 0);
#pragma unroll 1
            for (int kc = 0; kc < cpt; ++kc) {
                const int j = k * cpt + kc;
                if (i == 0) {
                    const uint64_t dl = tc::now_ns() + timeout;
                    if (j < kTmemChunks) {
                        while (*(volatile uint32_t *)&c.tmem_ready <= (uint32_t)j) {
                            if (tc::now_ns() > dl || aborted(c)) { ok = false; break; }
                        }
                        tc::fence_after_sync();
                    } else {
                        // a parity wait only tells phases apart one at a time:
                        // every earlier load of this slot (the TMEM chunks
                        // staged in it) must be complete first
                        while (*(volatile uint32_t *)&c.tmem_ready < (uint32_t)ntm) {
                            if (tc::now_ns() > dl || aborted(c)) { ok = false; break; }
                        }
                        int s;
                        uint32_t u;
                        chunk_slot(j, ntm, s, u);
                        if (ok) ok = tc::mbar_wait(tc::smem_u32(&c.full[s]), u & 1u, dl);
                    }
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) {
                        if (lane == 0) fail(c, a, 4u, 0x2000u + j);
                        break;
                    }
                }
                // descriptors advance by (bytes >> 4) in their address field
                const uint64_t bd = bview + (uint64_t)((kc * 2048) >> 4);
                const uint32_t acc0 = (h == 0 && kc == 0) ? 0u : 1u;
                if (j < kTmemChunks) {
                    const uint32_t at = tmem + 32u * (uint32_t)j;
                    tc::mma_tmemA_elect(d, at, bd, kIdesc, acc0);
                    tc::mma_tmemA_elect(d, at + 8u, bd + 2u, kIdesc, 1u);
                    tc::mma_tmemA_elect(d, at + 16u, bd + 4u, kIdesc, 1u);
                    tc::mma_tmemA_elect(d, at + 24u, bd + 6u, kIdesc, 1u);
                } else {
                    const uint64_t ad = adesc0 + (uint64_t)(((uint32_t)(j - kTmemChunks) * kChunkBytes) >> 4);
                    tc::mma_smemA_elect(d, ad, bd, kIdesc, acc0);
                    tc::mma_smemA_elect(d, ad + 2u, bd + 2u, kIdesc, 1u);
                    tc::mma_smemA_elect(d, ad + 4u, bd + 4u, kIdesc, 1u);
                    tc::mma_smemA_elect(d, ad + 6u, bd + 6u, kIdesc, 1u);
                }
            }
        }
        if (!ok) break;
        tc::commit_elect(tc::smem_u32(&c.accf[W]));
        ++uses;
    }
    __syncwarp();
}

// The exact Gumbel key of survivor (id v, row b, cached logit lf) folded
// into the CTA's best key of that row (shared-memory atomic maximum).
__device__ __forceinline__ void survivor_key(Ctl &c, int i, uint32_t v, int b, float lf) {
    const uint64_t h = dm_splitmix64(c.hri[i][b] ^ (uint64_t)v);
    const uint32_t o = ordered_key(exact_key(lf, c.T[b], h));
    atomicMax(&c.cbest[i & 1][b], ((unsigned long long)o << 32) | ((unsigned long long)(0x3FFFFu - v) << 14));
}

// Two upper bounds as FP16 pair, rounded toward +inf (still upper bounds;
// NaN stays NaN, beyond the FP16 range becomes +inf).
__device__ __forceinline__ __half2 half2_up(float lo, float hi) {
    return __halves2half2(__float2half_ru(lo), __float2half_ru(hi));
}

// The epilogue of one position, run by the 16 warps 4-19: warp 4 + 4 cm + q
// serves accumulator W = cm / 2, half hh = cm % 2 (the pair's first or
// second tile), TMEM lane quarter q (the only lanes a warp may read), so
// each thread owns one id per tile and all 8 rows (the tile's 8 columns).
//
// Pass 1, per tile as its bias arrives: the cached logits (two rows per
// packed BF16 conversion), written out; for rows whose key is exact here
// (greedy rows, inverse-CDF rows) the running maximum key with the lowest
// id; for Gumbel rows a lower and an upper bound on every id's key (logit
// / T plus the ends of the id's noise byte), keeping the largest lower
// bound and, per queued tile, the upper bounds as FP16 rounded up.  Pass 2,
// after the warp's last tile (so that no exact key delays an accumulator's
// hand-back): every value of the CTA's threshold (the largest lower bound
// contributed so far) is a lower bound on the CTA's best key, so only ids
// whose upper bound reaches it can be that best; their lanes compute their
// exact keys.  The CTA's maximum (and the token) is exactly that of keys
// computed for every id.  Leaves the CTA's per-row best packed key in
// c.cbest[i & 1] (zeroed, with c.lcta, before the position).  `gum_any`
// (some row is a Gumbel row) is CTA-uniform.
template <int RANK, bool kCdf, int DT>
__device__ __forceinline__ void epilogue(Ctl &c, const SampleArgs &a, const uint32_t tmem,
                                         const int i, const int t0, const int n0, const int nt,
                                         const bool gum_any, const uint64_t timeout, uint32_t &dcount) {
    // tiles a warp may see per position: 2 at rank 256 (the pass-2 queue is
    // kept in registers), more at smaller ranks (read back from L2)
    constexpr bool kRegs = RANK == 256;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ew = warp - 4, q = warp & 3, cm = ew >> 2, W = cm >> 1, hh = cm & 1;
    const int first = issuer_first(W, n0), last = issuer_last(W, n0, nt);
    const int V = a.V;
    const int par = i & 1;
    uint32_t live_m = 0u, samp_m = 0u, div_m = 0u;   // bit b = row b
#pragma unroll
    for (int b = 0; b < kChainRows; ++b) {
        live_m |= c.live[b] ? (1u << b) : 0u;
        samp_m |= c.sampling[b] ? (1u << b) : 0u;
        div_m |= (c.sampling[b] && c.T[b] != 1.0f) ? (1u << b) : 0u;
    }
    // Gumbel rows get the bound treatment; inverse-CDF rows divide by T
    const uint32_t gum_m = kCdf ? 0u : (samp_m & live_m);
    div_m = kCdf ? (div_m & live_m) : 0u;
    const uint2 *gq = reinterpret_cast<const uint2 *>(a.noise) + (int64_t)i * V;
    // DT bit 0: fp32 base logits, bit 1: fp32 cache (else BF16)
    constexpr bool kBaseF32 = (DT & 1) != 0, kCacheF32 = (DT & 2) != 0;
    const int64_t bofs = (int64_t)i * a.base_s1;
    const int64_t cofs = (int64_t)i * a.cache_s1;
    const uint16_t *base_i = kBaseF32 ? nullptr : a.base + bofs;
    const float *base_fi = kBaseF32 ? a.base_f + bofs : nullptr;
    uint16_t *cache_i = kCacheF32 ? nullptr : a.cache + cofs;
    float *cache_fi = kCacheF32 ? a.cache_f + cofs : nullptr;

    // exact-key rows: the best ordered key and its id; Gumbel rows: the
    // largest key lower bound (float bits) in bo
    uint32_t bo[kChainRows], bv[kChainRows];
#pragma unroll
    for (int b = 0; b < kChainRows; ++b) {
        bo[b] = ((gum_m >> b) & 1u) ? 0xff800000u : 0u;
        bv[b] = 0u;
    }
    // the last 2 tiles' packed logits and FP16 key upper bounds, newest first
    uint32_t k0[4] = {0u, 0u, 0u, 0u}, k1[4] = {0u, 0u, 0u, 0u};
    __half2 u0[4], u1[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) u0[j] = u1[j] = __float2half2_rn(0.0f);
    // the next tile's base logits: fp32 bits per row, or BF16 pairs (rows
    // 2j, 2j + 1 in the low / high half of word j)
    constexpr int kNB = kBaseF32 ? kChainRows : kChainRows / 2;
    uint32_t nb[kNB];
    uint2 nq;
    auto load_tile = [&](int k, uint32_t (&bb)[kNB], uint2 &qq) {
        const int v = (t0 + k) * 128 + q * 32 + lane;
        const bool ok2 = k < last && v < V;
        if (kBaseF32) {
#pragma unroll
            for (int b = 0; b < kChainRows; ++b)
                bb[b % kNB] = (ok2 && ((live_m >> b) & 1u)) ? __float_as_uint(__ldg(base_fi + b * a.base_s0 + v)) : 0u;
        } else {
#pragma unroll
            for (int j = 0; j < kChainRows / 2; ++j) {
                const uint32_t lo = (ok2 && ((live_m >> (2 * j)) & 1u)) ? (uint32_t)__ldg(base_i + (2 * j) * a.base_s0 + v) : 0u;
                const uint32_t hi = (ok2 && ((live_m >> (2 * j + 1)) & 1u)) ? (uint32_t)__ldg(base_i + (2 * j + 1) * a.base_s0 + v) : 0u;
                bb[j] = lo | (hi << 16);
            }
        }
        qq = (ok2 && gum_m != 0u) ? __ldcg(gq + v) : make_uint2(0u, 0u);
    };
    load_tile(first + hh, nb, nq);
    bool ok = true;
    int ntw = 0;   // tiles this warp processed
#pragma unroll 1
    for (int ta = first; ta < last; ta += 2) {
        const int k = ta + hh;
        const bool has = k < last;
        uint32_t cb[kNB];
#pragma unroll
        for (int b = 0; b < kNB; ++b) cb[b] = nb[b];
        const uint2 cq = nq;
        load_tile(k + 2, nb, nq);
        if (lane == 0)
            ok = tc::mbar_wait(tc::smem_u32(&c.accf[W]), dcount & 1u, tc::now_ns() + timeout);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            if (lane == 0) fail(c, a, 4u, 0x6000u + i);
            break;
        }
        ++dcount;
        tc::fence_after_sync();
        uint32_t r[8];
        if (has) {
            tc::ld_32x32b_x8(tmem + ((uint32_t)(q * 32) << 16) + kDCol + 16u * W + 8u * hh, r);
            tc::wait_ld();
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&c.accr[W]));
        if (!has) continue;
        // nothing that waits on this tile's base loads may be scheduled
        // before the accumulator is handed back
#pragma unroll
        for (int b = 0; b < kNB; ++b) asm volatile("" : "+r"(cb[b]));
#pragma unroll
        for (int b = 0; b < 8; ++b) asm volatile("" : "+r"(r[b]));
        const int v = (t0 + k) * 128 + q * 32 + lane;
        const bool valid = v < V;
        // bias = bf16(sum); logit = cache_round(f32(base) + f32(bias)), two
        // rows a time (BF16 caches: packed; fp32 caches: kept in fp32)
        uint32_t lp[4];
        float lf8[kChainRows];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t bb = bf16x2_rn(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
            const float b0 = kBaseF32 ? __uint_as_float(cb[(2 * j) % kNB]) : __uint_as_float(cb[j % kNB] << 16);
            const float b1 = kBaseF32 ? __uint_as_float(cb[(2 * j + 1) % kNB])
                                      : __uint_as_float(cb[j % kNB] & 0xffff0000u);
            const float s0 = __fadd_rn(b0, __uint_as_float(bb << 16));
            const float s1 = __fadd_rn(b1, __uint_as_float(bb & 0xffff0000u));
            if (kCacheF32) {
                lf8[2 * j] = s0;
                lf8[2 * j + 1] = s1;
            } else {
                lp[j] = bf16x2_rn(s0, s1);
            }
        }
        if (kCacheF32) {
            if (a.tf.has_transform) {
#pragma unroll
                for (int b = 0; b < kChainRows; ++b) lf8[b] = transform_f32(lf8[b], a.tf);
            }
#pragma unroll
            for (int b = 0; b < kChainRows; ++b)
                if (valid && ((live_m >> b) & 1u)) cache_fi[b * a.cache_s0 + v] = lf8[b];
        } else {
            if (a.tf.has_transform) {
#pragma unroll
                for (int j = 0; j < 4; ++j) lp[j] = transform_pair(lp[j], a.tf);
            }
#pragma unroll
            for (int b = 0; b < kChainRows; ++b) {
                lf8[b] = __uint_as_float((b & 1) ? (lp[b >> 1] & 0xffff0000u) : (lp[b >> 1] << 16));
                if (valid && ((live_m >> b) & 1u))
                    cache_i[b * a.cache_s0 + v] = (uint16_t)(lp[b >> 1] >> (16 * (b & 1)));
            }
        }
        float ku[kChainRows];
#pragma unroll
        for (int b = 0; b < kChainRows; ++b) {
            const float lf = lf8[b];
            ku[b] = 0.0f;
            if ((gum_m >> b) & 1u) {
                const uint32_t qb = ((b < 4 ? cq.x : cq.y) >> (8 * (b & 3))) & 0xffu;
                const float kl = key_lower(lf, c.invT[b], qb);
                bo[b] = (valid && kl > __uint_as_float(bo[b])) ? __float_as_uint(kl) : bo[b];
                ku[b] = key_upper(lf, c.invT[b], qb);
            } else if ((live_m >> b) & 1u) {
                float key = lf;
                if (kCdf && ((div_m >> b) & 1u)) key = __fdiv_rn(lf, c.T[b]);
                const uint32_t o = ordered_key(key);
                const bool better = valid && o > bo[b];
                bo[b] = better ? o : bo[b];
                bv[b] = better ? (uint32_t)v : bv[b];
            }
        }
        if (kRegs && gum_m != 0u) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (!kCacheF32) {
                    k1[j] = k0[j];
                    k0[j] = lp[j];
                }
                u1[j] = u0[j];
                u0[j] = half2_up(ku[2 * j], ku[2 * j + 1]);
            }
        }
        ++ntw;
    }
    // rows with exact keys: the warp's best into the CTA's
#pragma unroll
    for (int b = 0; b < kChainRows; ++b) {
        if (((gum_m >> b) & 1u) || !((live_m >> b) & 1u)) continue;
        const uint64_t pk =
            bo[b] != 0u ? (((uint64_t)bo[b] << 32) | ((uint64_t)(0x3FFFFu - bv[b]) << 14)) : 0ull;
        const uint64_t m = tc::warp_max_u64(pk);
        if (lane == 0 && m != 0ull) atomicMax(&c.cbest[par][b], (unsigned long long)m);
    }
    if (!gum_any) return;

    // ---- pass 2 (Gumbel rows), with no CTA barrier: the warp's threshold
    // (its largest lower bound) goes into the CTA's (shared-memory maximum),
    // and the CTA's threshold as it stands then (every value in it is a
    // lower bound on the CTA's best key, and it already holds this warp's)
    // selects the ids whose upper bound reaches it; their lanes compute
    // their exact keys.  A group that finishes its tiles early does this
    // while the others still work on theirs.
    uint32_t lw = 0u;   // lane b < 8: ordered warp threshold of row b
#pragma unroll
    for (int b = 0; b < kChainRows; ++b) {
        const uint32_t m =
            __reduce_max_sync(0xffffffffu, ((gum_m >> b) & 1u) ? ordered_key(__uint_as_float(bo[b])) : 0u);
        lw = lane == b ? m : lw;
    }
    if (ok && ntw > 0 && lane < kChainRows && lw != 0u) atomicMax(&c.lcta[par][lane], lw);
    __syncwarp();
    float Lc[kChainRows];
#pragma unroll
    for (int b = 0; b < kChainRows; ++b) {
        const uint32_t o = *(volatile uint32_t *)&c.lcta[par][b];
        // no bound recorded (no valid id): nothing can survive
        Lc[b] = o != 0u ? key_from_ordered(o) : __uint_as_float(0x7f800000u);
    }
    if (kRegs && ok) {
        uint32_t cand = 0u;   // bit 8 r + b: queued tile r (newest first), row b survives
        __half2 L[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            L[j] = __halves2half2(__float2half_rd(Lc[2 * j]), __float2half_rd(Lc[2 * j + 1]));
        auto slot = [&](int r, const __half2 (&uu)[4]) {
            const int k = first + hh + 2 * (ntw - 1 - r);
            const int v = (t0 + k) * 128 + q * 32 + lane;
            if (r < ntw && v < V) {
                uint32_t b8 = 0u;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t mj = __hgeu2_mask(uu[j], L[j]);
                    b8 |= ((mj & 1u) | ((mj >> 15) & 2u)) << (2 * j);
                }
                cand |= (b8 & gum_m) << (8 * r);
            }
        };
        slot(0, u0);
        slot(1, u1);
        while (cand != 0u) {
            const int bit = __ffs(cand) - 1;
            cand &= cand - 1u;
            const int r = bit >> 3, b = bit & 7;
            const int k = first + hh + 2 * (ntw - 1 - r);
            const uint32_t v = (uint32_t)((t0 + k) * 128 + q * 32 + lane);
            float lf;
            if (kCacheF32) {
                // an fp32 cache's logit, read back (this thread wrote it)
                lf = cache_fi[b * a.cache_s0 + v];
            } else {
                const uint32_t pr = r == 0 ? k0[b >> 1] : k1[b >> 1];
                lf = __uint_as_float(((pr >> (16 * (b & 1))) & 0xffffu) << 16);
            }
            survivor_key(c, i, v, b, lf);
        }
    }
    if (!kRegs && ok) {
        // more tiles than registers hold (small ranks): the cached logits and
        // noise bytes are read back (L2) tile by tile, exact bounds
#pragma unroll 1
        for (int r = 0; r < ntw; ++r) {
            const int k = first + hh + 2 * r;
            const int v = (t0 + k) * 128 + q * 32 + lane;
            if (v >= V) continue;
            const uint2 qq = __ldcg(gq + v);
#pragma unroll
            for (int b = 0; b < kChainRows; ++b) {
                if (!((gum_m >> b) & 1u)) continue;
                const float lf = kCacheF32 ? __ldcg(cache_fi + b * a.cache_s0 + v)
                                           : __uint_as_float((uint32_t)__ldcg(cache_i + b * a.cache_s0 + v) << 16);
                const uint32_t qb = ((b < 4 ? qq.x : qq.y) >> (8 * (b & 3))) & 0xffu;
                if (!(key_upper(lf, c.invT[b], qb) < Lc[b])) survivor_key(c, i, (uint32_t)v, b, lf);
            }
        }
    }
}

// Poll the [G] tagged key slots of rows b0 and b1 (slot arrays s0, s1;
// a row whose `use` bit is clear is skipped) until every CTA's key carries
// `tag`; the warp's maximum packed key of each row.  Both rows' loads are in
// flight together.  False after the deadline or when another CTA has
// recorded an error.
__device__ __forceinline__ bool poll_rows(const uint64_t *s0, const uint64_t *s1, uint32_t use, int G,
                                          uint32_t tag, uint64_t deadline, const SampleArgs &a,
                                          uint64_t &out0, uint64_t &out1) {
    const int lane = threadIdx.x & 31;
    for (uint32_t spin = 0;; ++spin) {
        bool fresh = true;
        uint64_t m0 = 0ull, m1 = 0ull;
        for (int cc = lane; cc < G; cc += 32) {
            if (use & 1u) {
                const uint64_t k = tc::ld_relaxed_u64(s0 + cc);
                fresh = fresh && (uint32_t)(k & kKeyTagMask) == tag;
                m0 = k > m0 ? k : m0;
            }
            if (use & 2u) {
                const uint64_t k = tc::ld_relaxed_u64(s1 + cc);
                fresh = fresh && (uint32_t)(k & kKeyTagMask) == tag;
                m1 = k > m1 ? k : m1;
            }
        }
        if (__all_sync(0xffffffffu, fresh)) {
            out0 = tc::warp_max_u64(m0) & ~(uint64_t)kKeyTagMask;
            out1 = tc::warp_max_u64(m1) & ~(uint64_t)kKeyTagMask;
            return true;
        }
        if ((spin & 15u) == 15u) {
            const bool bad = tc::now_ns() > deadline || ld_acquire_u32(a.status) != 0u;
            if (__any_sync(0xffffffffu, bad)) return false;
        }
    }
}

// The exact integer weight floor(exp(fp32(l / T) - M) 2^40) of one cached
// logit (inverse CDF; a logit of -inf or one far below M weighs 0).
__device__ __forceinline__ uint64_t cdf_weight(float l, float T, float M) {
    const float x = __fdiv_rn(l, T);
    return (uint64_t)__float2ull_rz(__fmul_rn(dm_exp(__fsub_rn(x, M)), 0x1p40f));
}

template <int DT>
__device__ __forceinline__ float cached_logit(const SampleArgs &a, int64_t row_ofs, int v) {
    return (DT & 2) ? __ldcg(a.cache_f + row_ofs + v)
                    : dm_bf16_f32((uint32_t)__ldcg(a.cache + row_ofs + v));
}

}  // namespace

// MODE 0: Gumbel and greedy rows; MODE 1: inverse-CDF and greedy rows (one
// kernel per mode keeps each kernel's code smaller).
template <int RANK, int MODE, int DT>
__global__ void __launch_bounds__(kThreads, 1)
chain_tc_kernel(const SampleArgs a, const __grid_constant__ CUtensorMap tmap, int noise_ready) {
    constexpr int cpt = RANK / 64;                 // K-chunks per 128-id tile
    extern __shared__ uint8_t dsm_raw[];
    __shared__ Ctl c;
    uint8_t *dsm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t *head_s = dsm;
    uint8_t *b_s = dsm + kSmemHead;
    const uint32_t head_sa = tc::smem_u32(head_s), b_sa = tc::smem_u32(b_s);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = gridDim.x, cta = blockIdx.x;
    const int R = a.rows, N = a.N, V = a.V;
    const int T_total = (V + 127) / 128;
    int t0, t1;
    cta_tiles(cta, G, T_total, t0, t1);
    const int nt = t1 - t0;
    const int nch = nt * cpt;
    const int ntm = nch < kTmemChunks ? nch : kTmemChunks;
    // issuer 0 takes the tiles whose first chunk is in TMEM
    const int n0 = nt < (kTmemChunks + cpt - 1) / cpt ? nt : (kTmemChunks + cpt - 1) / cpt;
    const int v_begin = t0 * 128;
    const int v_end = t1 * 128 < V ? t1 * 128 : V;
    const int Gp = (G + kKeyPad - 1) / kKeyPad * kKeyPad;

    // ------------------------------------------------------------ set-up
    if (tid == 0) {
        for (int s = 0; s < kSmemChunks; ++s) {
            tc::mbar_init(tc::smem_u32(&c.full[s]), 1);
            tc::mbar_init(tc::smem_u32(&c.cpdone[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(tc::smem_u32(&c.accf[b]), 1);
            tc::mbar_init(tc::smem_u32(&c.accr[b]), 8);   // 2 halves x 4 lane quarters
            tc::mbar_init(tc::smem_u32(&c.fin[b]), 1);
        }
        tc::mbar_init_fence();
        c.tmem_ready = 0u;
        clear_position(c, 0);

        c.abort = ld_acquire_u32(a.status) != 0u ? 1u : 0u;
        c.call = *(volatile const uint32_t *)a.call_counter;
    }
    if (tid < kChainRows) {
        const int b = tid;
        const bool live = b < R && a.row_state_idx[b] >= 0;
        c.live[b] = live;
        const float T = live ? a.temperature[b] : 0.0f;
        c.T[b] = T;
        c.sampling[b] = live && samples(T);
        c.seed[b] = live ? (uint64_t)a.seeds[b] : 0ull;
        c.invT[b] = samples(T) ? 1.0f / T : 1.0f;
        int64_t p = live ? (int64_t)a.anchor[b] : 0;
        if (p < 0 || p >= V) {
            set_status(a.status, 1u /* MARKOV_EINVAL */, 0x100u + b);
            p = 0;
        }
        c.prev[b] = p;
    }
    for (int o = tid * 16; o < (int)kSmemB; o += kThreads * 16)
        *reinterpret_cast<uint4 *>(b_s + o) = make_uint4(0u, 0u, 0u, 0u);
    if (warp == 0) tc::tmem_alloc(tc::smem_u32(&c.tmem_base), 512);
    __syncthreads();
    if (tid < N * kChainRows) {
        const int b = tid % kChainRows, i2 = tid / kChainRows;
        c.hri[i2][b] = dm_row_step_hash(c.seed[b], (uint32_t)(a.row_base + b), (uint32_t)i2);
    }
    if (warp < kChainRows && c.live[warp] && lane < RANK / 8)
        stage_row<RANK>(b_s, *reinterpret_cast<const uint4 *>(a.embed + c.prev[warp] * RANK + 8 * lane),
                        warp, lane);
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = c.tmem_base;
    const uint64_t timeout = a.timeout_ns;
    uint32_t gum_mask = 0u;   // Gumbel rows (sampling rows of the Gumbel mode)
#pragma unroll
    for (int b = 0; b < kChainRows; ++b) gum_mask |= c.sampling[b] ? (1u << b) : 0u;
    if (MODE != 0) gum_mask = 0u;
    const bool gum_any = gum_mask != 0u;

    // per-role persistent state
    uint32_t uses = 0;          // issuer: tile pairs issued into its accumulator
    uint32_t dcount = 0;        // epilogue: tile pairs consumed from its accumulator
    uint32_t issued[kSmemChunks];   // producer: loads issued per slot
#pragma unroll
    for (int s = 0; s < kSmemChunks; ++s) issued[s] = 0u;

    bool stop = __syncthreads_or(c.abort != 0u);
    for (int i = 0; i < N && !stop; ++i) {
        // ------------------------------------- phase A: MMA and epilogue
        if (warp < 2) {
            issue_tiles<RANK>(c, a, tmem, warp, i, n0, nt, ntm, b_sa, head_sa, timeout, uses);
        } else if (warp < 4 && i > 0) {
            // warps 2 and 3 after the head load: the next position's base
            // logits into L2, off the chain's critical path
            if (i + 1 < N) prefetch_base<64>(c, a, i + 1, v_begin, v_end, tid - 64);
        } else if (warp == 2) {
            if (lane == 0 && i == 0) {
                for (int j = 0; j < nch; ++j) {
                    if (aborted(c)) break;
                    int s;
                    uint32_t ph;
                    chunk_slot(j, ntm, s, ph);
                    bool ok = true;
                    const uint64_t dl = tc::now_ns() + timeout;
                    // the slot's previous (TMEM) chunk has been copied out:
                    // copy number ph - 1 of this slot
                    if (ph > 0u) ok = tc::mbar_wait(tc::smem_u32(&c.cpdone[s]), (ph - 1u) & 1u, dl);
                    if (!ok) { fail(c, a, 4u, 0x3000u + j); break; }
                    const uint32_t bar = tc::smem_u32(&c.full[s]);
                    tc::mbar_expect_tx(bar, kChunkBytes);
                    tc::tma_load_2d(head_sa + s * kChunkBytes, &tmap, (j % cpt) * 64,
                                    (t0 + j / cpt) * 128, bar);
                    ++issued[s];
                }
            }
            __syncwarp();
        } else if (warp == 3) {
            if (lane == 0 && i == 0) {
                // chunk j's copy is issued as soon as its load lands; its
                // completion is awaited only after the next copy is issued,
                // so the copies' latency overlaps the loads' (unless both
                // chunks share a slot: a parity wait sees one phase at a time)
                bool early = false;
                for (int j = 0; j <= ntm; ++j) {
                    if (aborted(c)) break;
                    int sp = 0;
                    uint32_t pp = 0u;
                    if (j > 0) chunk_slot(j - 1, ntm, sp, pp);
                    if (j < ntm) {
                        int s;
                        uint32_t ph;
                        chunk_slot(j, ntm, s, ph);
                        if (!tc::mbar_wait(tc::smem_u32(&c.full[s]), ph & 1u, tc::now_ns() + timeout)) {
                            fail(c, a, 4u, 0x4000u + j);
                            break;
                        }
                        if (j > 0 && sp == s) {
                            // (already complete: this load waited for it)
                            if (!tc::mbar_wait(tc::smem_u32(&c.cpdone[sp]), pp & 1u, tc::now_ns() + timeout)) {
                                fail(c, a, 4u, 0x5000u + j - 1);
                                break;
                            }
                            tc::fence_before_sync();
                            *(volatile uint32_t *)&c.tmem_ready = (uint32_t)j;
                            early = true;
                        }
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            tc::cp_128x256b(tmem + 32u * j + 8u * ks,
                                            tc::sw128_desc(head_sa + s * kChunkBytes + 32 * ks));
                        tc::commit(tc::smem_u32(&c.cpdone[s]));
                    }
                    if (j > 0 && !early) {
                        // chunk j - 1, in another slot than chunk j's
                        if (!tc::mbar_wait(tc::smem_u32(&c.cpdone[sp]), pp & 1u, tc::now_ns() + timeout)) {
                            fail(c, a, 4u, 0x5000u + j - 1);
                            break;
                        }
                        tc::fence_before_sync();
                        *(volatile uint32_t *)&c.tmem_ready = (uint32_t)j;
                    }
                    early = false;
                }
            }
            __syncwarp();
        } else {
            // warps 4..19: at position 0 the noise bounds of position 0 and the
            // base logits into L2 while the head streams in; then the epilogue
            if (i == 0) {
                const int te = tid - 128;
                prefetch_base<kEpiThreads>(c, a, 0, v_begin, v_end, te);
                if (MODE == 0 && gum_any) {
                    noise_bounds<kEpiThreads>(c, a, 0, gum_mask, v_begin, v_end, te);
                    asm volatile("bar.sync 2, %0;" ::"n"(kEpiThreads) : "memory");
                }
                if (N > 1) prefetch_base<kEpiThreads>(c, a, 1, v_begin, v_end, te);
            }
            epilogue<RANK, MODE == 1, DT>(c, a, tmem, i, t0, n0, nt, gum_any, timeout, dcount);
        }
        stop = __syncthreads_or(stop_vote(c, a, MODE != 0));
        if (stop) break;

        // ------------------------------- phase B: agree on every row's winner
        const uint32_t epoch = c.call * (uint32_t)kMaxSteps + (uint32_t)i + 1u;
        const uint32_t tag = epoch & kKeyTagMask;
        uint64_t *slots_i = a.tc_keys + (size_t)i * kChainRows * Gp;   // [row][Gp]
        if (warp < 4) {
            // warp 0 lane b stores row b's best key, tagged; lanes of warp 1
            // warm L2 with this CTA's candidates' embedding rows (the winning
            // CTA's prefetch serves every CTA's gather); warps 0-3 poll rows
            // w and w + 4
            if (warp == 0 && lane < kChainRows && c.live[lane])
                tc::st_relaxed_u64(slots_i + (size_t)lane * Gp + cta,
                                   ((uint64_t)c.cbest[i & 1][lane] & ~(uint64_t)kKeyTagMask) | tag);
            if (warp == 1 && lane < kChainRows && c.live[lane] && i + 1 < N) {
                const uint64_t m = c.cbest[i & 1][lane];
                const uint32_t id = unpack_id(m);
                if (m != 0ull && id < (uint32_t)V) {
                    const uint8_t *er = reinterpret_cast<const uint8_t *>(a.embed + (int64_t)id * RANK);
#pragma unroll
                    for (int o = 0; o < RANK * 2; o += 128) tc::prefetch_l2(er + o);
                }
            }
            const uint32_t use = (c.live[warp] ? 1u : 0u) | (c.live[warp + 4] ? 2u : 0u);
            if (use != 0u) {
                uint64_t w0 = 0ull, w1 = 0ull;
                if (!poll_rows(slots_i + (size_t)warp * Gp, slots_i + (size_t)(warp + 4) * Gp, use, G, tag,
                               tc::now_ns() + timeout, a, w0, w1)) {
                    if (lane == 0) fail(c, a, 4u, 0x7000u + i);
                    w0 = w1 = 0ull;
                }
                if (lane == 0) {
                    c.win[warp] = w0;
                    c.win[warp + 4] = w1;
                }
            }
        }
        if (MODE == 0) {
            if (warp < 4) {
                __syncwarp();
                // warps 0-3 stage rows w and w + 4: both gathers in flight at once
                const int rb2[2] = {warp, warp + 4};
                uint32_t idr[2];
                uint4 ev[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int b = rb2[h];
                    uint32_t id = unpack_id(c.win[b]);
                    if (c.live[b] && (c.win[b] == 0ull || id >= (uint32_t)V)) {
                        // no CTA reported a key for a live row (or the poll
                        // gave up): never index embed with it
                        if (lane == 0 && !aborted(c)) fail(c, a, 6u /* MARKOV_EDEVICE */, 0xB000u + i);
                        id = 0u;
                    }
                    idr[h] = c.live[b] ? id : 0u;
                    ev[h] = make_uint4(0u, 0u, 0u, 0u);
                    if (c.live[b] && i + 1 < N && lane < RANK / 8)
                        ev[h] = *reinterpret_cast<const uint4 *>(a.embed + (int64_t)idr[h] * RANK + 8 * lane);
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int b = rb2[h];
                    if (!c.live[b]) continue;
                    if (lane == 0) {
                        c.prev[b] = (int64_t)idr[h];
                        if (cta == 0) a.tokens[b * a.tok_s0 + i] = (int64_t)idr[h];
                    }
                    if (i + 1 < N && lane < RANK / 8) stage_row<RANK>(b_s, ev[h], b, lane);
                }
                // the control warps alone close the position: the next MMAs
                // need only the staged B operand
                tc::fence_proxy_async_smem();
                tc::fence_before_sync();
                asm volatile("bar.sync 4, 128;" ::: "memory");
                tc::fence_after_sync();
            } else if (i + 1 < N) {
                // the epilogue warps clear the next position's CTA maxima (their
                // last reader finished before this position's phase-A barrier),
                // draw its noise bounds while the winners are exchanged and the
                // next MMAs start, and go straight on to the next epilogue (no
                // CTA barrier between; their own barrier orders the clearing
                // before the next position's atomics)
                if (tid == 128) clear_position(c, (i + 1) & 1);
                if (gum_any) noise_bounds<kEpiThreads>(c, a, i + 1, gum_mask, v_begin, v_end, tid - 128);
                asm volatile("bar.sync 2, %0;" ::"n"(kEpiThreads) : "memory");
            }
            // an error seen by the control warps stops the CTA at the next
            // position's phase-A barrier
        } else {
            stop = __syncthreads_or(stop_vote(c, a));
            if (stop) break;

            // inverse CDF: rows whose maximum M is finite need the exact integer
            // weight sums floor(exp(x - M) 2^40); every CTA learns every CTA's
            // sum, finds the CTA whose prefix range holds mulhi64(H, S) and
            // scans that CTA's cached logits for the token
            uint32_t cdf_m = 0u;
#pragma unroll
            for (int b = 0; b < kChainRows; ++b) {
                if (b >= R || !c.sampling[b]) continue;
                const uint32_t o = (uint32_t)(c.win[b] >> 32);
                if (o != 0xffffffffu && !isinf(key_from_ordered(o))) cdf_m |= 1u << b;
            }
            if (cdf_m != 0u) {
                const uint32_t stag = epoch & 0xFFFu;
                if (tid < kChainRows) c.sum[tid] = 0ull;
                __syncthreads();
                // 4 rows a time: every cached logit of the group is loaded
                // before any weight, so the rows share one read latency
                constexpr int kMaxIds = kMaxChunks / cpt * 128;
                constexpr int kPT = (kMaxIds + kThreads - 1) / kThreads;   // ids per thread
                constexpr int kGR = RANK == 64 ? 2 : 4;
                for (int b0 = 0; b0 < kChainRows; b0 += kGR) {
                    if (!((cdf_m >> b0) & ((1u << kGR) - 1u))) continue;
                    float xs[kGR][kPT];
#pragma unroll
                    for (int rr = 0; rr < kGR; ++rr) {
                        const int b = b0 + rr;
                        const int64_t crow = b * a.cache_s0 + (int64_t)i * a.cache_s1;
#pragma unroll
                        for (int kk = 0; kk < kPT; ++kk) {
                            const int v = v_begin + tid + kk * kThreads;
                            xs[rr][kk] = ((cdf_m >> b) & 1u) && v < v_end ? cached_logit<DT>(a, crow, v) : 0.0f;
                        }
                    }
#pragma unroll
                    for (int rr = 0; rr < kGR; ++rr) {
                        const int b = b0 + rr;
                        if (!((cdf_m >> b) & 1u)) continue;
                        const float M = key_from_ordered((uint32_t)(c.win[b] >> 32));
                        uint64_t part = 0ull;
#pragma unroll
                        for (int kk = 0; kk < kPT; ++kk) {
                            if (v_begin + tid + kk * kThreads >= v_end) break;
                            part += cdf_weight(xs[rr][kk], c.T[b], M);
                        }
#pragma unroll
                        for (int o2 = 16; o2 > 0; o2 >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o2);
                        if (lane == 0) atomicAdd(&c.sum[b], (unsigned long long)part);
                    }
                }
                __syncthreads();
                // publish (release: this CTA's cache writes are visible to a
                // CTA that reads the tagged sum)
                if (tid < kChainRows && ((cdf_m >> tid) & 1u)) {
                    uint64_t *sl = a.tc_sums + ((size_t)i * kChainRows + tid) * Gp + cta;
                    const uint64_t w = c.sum[tid] | ((uint64_t)stag << kSumTagShift);
                    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(sl), "l"(w) : "memory");
                }
                // warp b: every CTA's sum of row b, the total S, the target
                // t = mulhi64(H, S) and the CTA whose prefix range holds it
                if (warp < kChainRows && ((cdf_m >> warp) & 1u)) {
                    const int b = warp;
                    const uint64_t *sl = a.tc_sums + ((size_t)i * kChainRows + b) * Gp;
                    constexpr int kPer = 5;   // CTAs per lane (G <= 160)
                    const int c0 = lane * kPer;
                    uint64_t s5[kPer];
                    const uint64_t dl = tc::now_ns() + timeout;
                    bool okp = true;
                    for (uint32_t spin = 0;; ++spin) {
                        bool fresh = true;
#pragma unroll
                        for (int u = 0; u < kPer; ++u) {
                            s5[u] = 0ull;
                            if (c0 + u < G) {
                                const uint64_t w = tc::ld_relaxed_u64(sl + c0 + u);
                                fresh = fresh && (uint32_t)(w >> kSumTagShift) == stag;
                                s5[u] = w & ((1ull << kSumTagShift) - 1ull);
                            }
                        }
                        if (__all_sync(0xffffffffu, fresh)) break;
                        if ((spin & 15u) == 15u &&
                            __any_sync(0xffffffffu, tc::now_ns() > dl || ld_acquire_u32(a.status) != 0u)) {
                            okp = false;
                            break;
                        }
                    }
                    if (!okp) {
                        if (lane == 0) fail(c, a, 4u, 0x8000u + i);
                    } else {
                        // acquire: the cache writes of the CTAs whose sums were read
                        asm volatile("fence.acq_rel.gpu;" ::: "memory");
                        uint64_t mine = 0ull;
#pragma unroll
                        for (int u = 0; u < kPer; ++u) mine += s5[u];
                        uint64_t incl = mine;
#pragma unroll
                        for (int o2 = 1; o2 < 32; o2 <<= 1) {
                            const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o2);
                            if (lane >= o2) incl += y;
                        }
                        const uint64_t S = __shfl_sync(0xffffffffu, incl, 31);
                        const uint64_t t = __umul64hi(dm_cdf_hash(c.hri[i][b]), S);
                        uint64_t run = incl - mine;
                        if (run <= t && t < run + mine) {
#pragma unroll
                            for (int u = 0; u < kPer; ++u) {
                                if (c0 + u < G && run <= t && t < run + s5[u]) {
                                    c.cstar[b] = c0 + u;
                                    c.rem[b] = t - run;
                                }
                                run += s5[u];
                            }
                        }
                    }
                }
                stop = __syncthreads_or(stop_vote(c, a));
                if (stop) break;
                // every CTA scans the target CTA's ids of each row itself: the
                // threads split into 4 groups of 5 warps, one row per group
                constexpr int kGroupWarps = (kThreads / 32) / 4;
                constexpr int kGroupThreads = kGroupWarps * 32;
                constexpr int kScanPer = (kMaxIds + kGroupThreads - 1) / kGroupThreads;
                const int grp = warp / kGroupWarps, gt = tid - grp * kGroupThreads;
                for (int b0 = 0; b0 < kChainRows; b0 += 4) {
                    if (!((cdf_m >> b0) & 0xFu)) continue;
                    const int b = b0 + grp;
                    const bool mine_row = (cdf_m >> b) & 1u;
                    int u0 = 0, per = 0;
                    float xs[kScanPer];
                    uint64_t wsum = 0ull;
                    if (mine_row) {
                        int s0, s1;
                        cta_tiles(c.cstar[b], G, T_total, s0, s1);
                        u0 = s0 * 128;
                        const int u1 = s1 * 128 < V ? s1 * 128 : V;
                        per = (u1 - u0 + kGroupThreads - 1) / kGroupThreads;
                        const int64_t crow = b * a.cache_s0 + (int64_t)i * a.cache_s1;
                        const int my0 = u0 + gt * per;
#pragma unroll
                        for (int kk = 0; kk < kScanPer; ++kk)
                            xs[kk] = (kk < per && my0 + kk < u1) ? cached_logit<DT>(a, crow, my0 + kk)
                                                                 : __uint_as_float(0xff800000u);
                        const float M = key_from_ordered((uint32_t)(c.win[b] >> 32));
#pragma unroll
                        for (int kk = 0; kk < kScanPer; ++kk)
                            if (kk < per) wsum += cdf_weight(xs[kk], c.T[b], M);
                    }
                    uint64_t incl = wsum;
#pragma unroll
                    for (int o2 = 1; o2 < 32; o2 <<= 1) {
                        const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o2);
                        if (lane >= o2) incl += y;
                    }
                    if (lane == 31) c.wtot[warp] = incl;
                    __syncthreads();
                    if (mine_row) {
                        uint64_t run = incl - wsum;
                        for (int w2 = grp * kGroupWarps; w2 < warp; ++w2) run += c.wtot[w2];
                        const uint64_t t = c.rem[b];
                        if (run <= t && t < run + wsum) {
                            const float M = key_from_ordered((uint32_t)(c.win[b] >> 32));
                            for (int kk = 0; kk < kScanPer && kk < per; ++kk) {
                                run += cdf_weight(xs[kk], c.T[b], M);
                                if (run > t) {
                                    c.tok[b] = (uint32_t)(u0 + gt * per + kk);
                                    break;
                                }
                            }
                        }
                    }
                    __syncthreads();
                }
                if (tid < kChainRows && ((cdf_m >> tid) & 1u))
                    c.win[tid] = (c.win[tid] & 0xffffffff00000000ull) | ((uint64_t)(0x3FFFFu - c.tok[tid]) << 14);
                __syncthreads();
            }

            // ------------------------- the token, and the next position's B operand
            if (warp < kChainRows && c.live[warp]) {
                const int b = warp;
                uint32_t id = unpack_id(c.win[b]);
                if (c.sampling[b]) {
                    const uint32_t o = (uint32_t)(c.win[b] >> 32);
                    if (o != 0xffffffffu && key_from_ordered(o) == __uint_as_float(0xff800000u)) id = 0u;
                }
                if (c.win[b] == 0ull || id >= (uint32_t)V) {
                    if (lane == 0 && !aborted(c)) fail(c, a, 6u /* MARKOV_EDEVICE */, 0xB100u + i);
                    id = 0u;
                }
                if (lane == 0) {
                    c.prev[b] = (int64_t)id;
                    if (cta == 0) a.tokens[b * a.tok_s0 + i] = (int64_t)id;
                }
                if (i + 1 < N && lane < RANK / 8)
                    stage_row<RANK>(b_s, *reinterpret_cast<const uint4 *>(a.embed + (int64_t)id * RANK + 8 * lane),
                                    b, lane);
            }
            // the next position's CTA maxima (last read before this
            // position's phase-A barrier)
            if (tid == 128 && i + 1 < N) clear_position(c, (i + 1) & 1);
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            stop = __syncthreads_or(stop_vote(c, a));
            tc::fence_after_sync();
        }
    }

    // --------------------------------------------------------------- exit
    // every async operation of this CTA completes before TMEM is released
    if (warp < 2) {
        __syncwarp();
        tc::commit_elect(tc::smem_u32(&c.fin[warp]));
        tc::mbar_wait(tc::smem_u32(&c.fin[warp]), 0u, tc::now_ns() + 1000000000ull);
    }
    if (warp == 2 && lane == 0) {
        for (int s = 0; s < kSmemChunks; ++s) {
            if (issued[s] == 0u) continue;
            tc::mbar_wait(tc::smem_u32(&c.full[s]), (issued[s] - 1u) & 1u,
                          tc::now_ns() + 1000000000ull);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
    if (cta == 0 && tid == 0 && !aborted(c) && ld_acquire_u32(a.status) == 0u)
        *(volatile uint32_t *)a.call_counter = c.call + 1u;
}

size_t chain_tc_smem() { return kDynSmem; }

int chain_tc_max_chunks() { return kMaxChunks; }

// One kernel per (rank, mode, base / cache dtypes).
template <int RANK>
static const void *tc_kernel_for(int mode, int dt) {
    switch (mode * 4 + dt) {
        case 0: return (const void *)chain_tc_kernel<RANK, 0, 0>;
        case 1: return (const void *)chain_tc_kernel<RANK, 0, 1>;
        case 2: return (const void *)chain_tc_kernel<RANK, 0, 2>;
        case 3: return (const void *)chain_tc_kernel<RANK, 0, 3>;
        case 4: return (const void *)chain_tc_kernel<RANK, 1, 0>;
        case 5: return (const void *)chain_tc_kernel<RANK, 1, 1>;
        case 6: return (const void *)chain_tc_kernel<RANK, 1, 2>;
        default: return (const void *)chain_tc_kernel<RANK, 1, 3>;
    }
}

static const void *tc_kernel(int r, int mode, int dt) {
    switch (r) {
        case 64: return tc_kernel_for<64>(mode, dt);
        case 128: return tc_kernel_for<128>(mode, dt);
        case 256: return tc_kernel_for<256>(mode, dt);
        default: return nullptr;
    }
}

cudaError_t chain_tc_prepare() {
    cudaError_t e = cudaSuccess;
    for (int r : {64, 128, 256})
        for (int mode = 0; mode < 2; ++mode)
            for (int dt = 0; dt < 4; ++dt) {
                e = cudaFuncSetAttribute(tc_kernel(r, mode, dt),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynSmem);
                if (e != cudaSuccess) return e;
            }
    return e;
}

cudaError_t chain_tc_occupancy(int *blocks_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, chain_tc_kernel<256, 0, 0>,
                                                         kThreads, kDynSmem);
}

cudaError_t launch_chain_tc(const SampleArgs &a, const CUtensorMap &tmap, int noise_ready,
                            cudaStream_t stream) {
    void *args[] = {(void *)&a, (void *)&tmap, (void *)&noise_ready};
    const int dt = (a.base_f ? 1 : 0) | (a.cache_f ? 2 : 0);
    const void *fn = tc_kernel(a.r, a.mode == 1 ? 1 : 0, dt);
    if (!fn) return cudaErrorInvalidValue;
    return cudaLaunchCooperativeKernel(fn, dim3(a.grid), dim3(kThreads), args, kDynSmem, stream);
}

}  // namespace dtm
