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
// swizzled K-major layout the TMA writes; two 16-column TMEM accumulators
// take the bias tiles.  Measured on GB300: an M=128, N=16, K=16 BF16 MMA
// costs ~9 cycles with A in TMEM (enough issuing threads) and ~39 with A in
// shared memory (bandwidth), and all MMA paths share one tensor pipe, so TMEM
// holds as much of the head as fits.
//
// Warp roles (20 warps, 640 threads):
//   0, 1   the MMAs of the even / odd tiles into accumulator 0 / 1 (one
//          elected lane each, one shared copy of the issue loop)
//   2      lane 0: TMA producer of the head chunks (position 0 only); later
//          positions: the next position's base logits into L2, and during
//          each exchange this CTA's candidate embedding rows into L2
//   3      lane 0: copies the TMEM-resident chunks from their shared-memory
//          staging slot into TMEM (position 0 only); later: base prefetch
//   4-19   the epilogue (warps 4-11 accumulator 0, 12-19 accumulator 1;
//          inverse-CDF calls of at most 4 rows: the two row halves of each
//          accumulator's warps take its tiles in turn); at position 0,
//          before it, the noise bounds of position 0 while the head streams
//          in; after every position, the next position's noise bounds while
//          the winners are exchanged
//   0-3    after each position: warp 0 exchanges every row's key with the
//          other CTAs, and warps 0-3 stage markov_embed[token] of rows w and
//          w + 4 as the next position's B operand
// Cross-CTA exchange (Gumbel and greedy rows): each CTA folds its per-row
// best key into one word per (position, row) with red.max and then adds 1
// to the position's counter (release); one thread per CTA polls the
// counter (acquire, bounded) until all CTAs have counted and reads the
// winners.  Inverse-CDF rows take their maxima the same way, then count
// their per-CTA weight sums (one slot per CTA) on the same counter up to 2G;
// the CTA whose prefix range holds the target scans for the token and
// publishes it in a word tagged with the call's epoch.

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
constexpr int kRowsT = 4;                 // rows per epilogue thread
constexpr int kTmemChunks = 15;           // A chunks in TMEM (32 columns each)
constexpr int kSmemChunks = 13;           // A chunks in shared memory (16 KB each)
constexpr int kMaxChunks = kTmemChunks + kSmemChunks;
constexpr uint32_t kChunkBytes = 128 * 128;   // 128 rows x 64 BF16
constexpr uint32_t kDCol = 480;           // accumulators: columns 480..495, 496..511
constexpr uint32_t kBChunkBytes = 16 * 128;   // B operand: 16 rows x 64 BF16 per K-chunk
constexpr uint32_t kIdesc = tc::idesc_bf16(128, 16);
constexpr uint32_t kSmemHead = kSmemChunks * kChunkBytes;
constexpr uint32_t kSmemB = 4 * kBChunkBytes;
constexpr uint32_t kDynSmem = kSmemHead + kSmemB + 1024;   // + alignment slack

struct Ctl {
    uint64_t full[kSmemChunks];      // TMA landed in slot s
    uint64_t cpdone[kSmemChunks];    // slot s copied into TMEM
    uint64_t dfull[2][2];            // accumulator b holds a finished tile (index 1: the
                                     // odd tiles when the epilogue halves take turns)
    uint64_t dfree[2];               // accumulator b read out by its epilogue
    uint64_t fin[2];                 // issuer b's MMAs all complete (exit)
    uint64_t bstaged;                // the next position's B operand is staged
    uint64_t sdone;                  // the shared-memory tile's bias is in sbias
    // Per position parity (a position's values are read while the next
    // one's are written): per row, the CTA's best packed key and, for Gumbel
    // rows, the CTA's threshold (ordered key of the largest key lower
    // bound); the Gumbel survivor list and its length.
    float sbias[128][kChainRows];    // the last tile's bias sums (mma.sync path)
    unsigned long long cbest[2][kChainRows];
    uint32_t lcta[2][kChainRows];
    uint64_t win[kChainRows];
    unsigned long long sum[kChainRows];
    uint64_t wsum[kChainRows][kEpiThreads / 32];   // inverse CDF: per-row, per-epilogue-warp weight totals
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
__device__ __forceinline__ bool aborted(const Ctl &c, const SampleArgs &) {
    return *(volatile const uint32_t *)&c.abort != 0u;
}

// At a CTA barrier: this CTA's abort flag.  An error another CTA recorded
// reaches this one through its exchange polls, which watch the global
// status off the barriers (a status load here would put an L2 round trip on
// every barrier).
__device__ __forceinline__ bool stop_vote(Ctl &c) {
    return *(volatile const uint32_t *)&c.abort != 0u;
}

// packed key: ordered key (32) | 0x3FFFF - id (18) | epoch tag (14)
__device__ __forceinline__ uint32_t unpack_id(uint64_t p) {
    return 0x3FFFFu - (uint32_t)((p >> 14) & 0x3FFFFu);
}

// Row b's maximum over all CTAs' slots, once every slot carries `tag`.  A
// round issues all of its loads before it looks at any (a compile-time
// bound: with a loop over the runtime CTA count the loads went out one L2
// round trip apart, and a round took microseconds).
constexpr int kMaxGrid = 160;             // CTAs the exchanges take
}  // namespace

namespace {

// Stage markov_embed[p] as row b of the B operand (16 rows x RANK, K-major,
// 128-byte swizzle, one 2 KB block per 64-element K-chunk).
template <int RANK>
__device__ __forceinline__ void stage_embed(uint8_t *b_s, const uint16_t *__restrict__ embed,
                                            int64_t p, int b, int lane) {
    if (lane < RANK / 8) {
        const uint4 v = *reinterpret_cast<const uint4 *>(embed + p * RANK + 8 * lane);
        const int chunk = lane >> 3, piece = lane & 7;
        *reinterpret_cast<uint4 *>(b_s + chunk * kBChunkBytes + b * 128 + ((piece ^ b) << 4)) = v;
    }
}

}  // namespace

namespace {


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

// The output-logit transform of two packed cached logits.
__device__ __forceinline__ uint32_t transform_pair_inl(uint32_t lp, const Transform &tf) {
    float y0 = __fmul_rn(__uint_as_float(lp << 16), tf.mult);
    float y1 = __fmul_rn(__uint_as_float(lp & 0xffff0000u), tf.mult);
    if (tf.has_cap) {
        y0 = __fmul_rn(tf.cap, dm_tanh(__fmul_rn(y0, tf.inv_cap)));
        y1 = __fmul_rn(tf.cap, dm_tanh(__fmul_rn(y1, tf.inv_cap)));
    }
    return bf16x2_rn(y0, y1);
}

// The same out of line, for the Gumbel kernels (whose code is large already;
// the inverse-CDF kernels take it inline, where the two pairs' tanh chains
// overlap).
__device__ __noinline__ uint32_t transform_pair(uint32_t lp, const Transform &tf) {
    return transform_pair_inl(lp, tf);
}

// The output-logit transform of one fp32 logit, kept in fp32 (fp32 caches).
__device__ __noinline__ float transform_f32(float s, const Transform &tf) {
    float y = __fmul_rn(s, tf.mult);
    if (tf.has_cap) y = __fmul_rn(tf.cap, dm_tanh(__fmul_rn(y, tf.inv_cap)));
    return y;
}

// The MMAs of accumulator W (issued by warp W): tiles W, W + 2, ...; per
// tile, K chunk by K chunk, 4 MMAs of K = 16 each, with A in TMEM (chunk j
// < kTmemChunks) or in shared memory.  The whole warp runs the loop and one
// elected lane issues.  Both warps run one copy of this code, kept small:
// the kernel's code is far larger than the SM's instruction caches, and an
// unrolled issue loop (16 KB per copy) measured several times slower inside
// the kernel than alone, its fetches competing with the epilogue's.
// Position 0 awaits each chunk as the head streams in.
template <int RANK>
__device__ __forceinline__ void issue_tiles(Ctl &c, const SampleArgs &a, const uint32_t tmem, const int W,
                                            const int i, const int nt, const int ntm,
                                            const uint32_t b_sa, const uint32_t head_sa,
                                            const uint64_t timeout, const bool alt, uint32_t &uses) {
    constexpr int cpt = RANK / 64;
    const int lane = threadIdx.x & 31;
    const uint32_t d = tmem + kDCol + 16u * (uint32_t)W;
    const uint64_t bdesc0 = tc::sw128_desc(b_sa), adesc0 = tc::sw128_desc(head_sa);
#pragma unroll 1
    for (int k = W; k < nt; k += 2) {
        if (__any_sync(0xffffffffu, aborted(c, a))) break;
        bool freed = true;
        if (uses > 0)
            freed = tc::mbar_wait_for(tc::smem_u32(&c.dfree[W]), (uses - 1) & 1u, timeout);
        if (!__all_sync(0xffffffffu, freed)) {
            if (lane == 0) fail(c, a, 4u, 0x1000u + i);
            break;
        }
        tc::fence_after_sync();
        bool ok = true;
#pragma unroll 1
        for (int kc = 0; kc < cpt; ++kc) {
            const int j = k * cpt + kc;
            if (i == 0) {
                const uint64_t dl = tc::now_ns() + timeout;
                if (j < kTmemChunks) {
                    while (*(volatile uint32_t *)&c.tmem_ready <= (uint32_t)j) {
                        if (tc::now_ns() > dl || aborted(c, a)) { ok = false; break; }
                    }
                    tc::fence_after_sync();
                } else {
                    // a parity wait only tells phases apart one at a time:
                    // every earlier load of this slot (the TMEM chunks
                    // staged in it) must be complete first
                    while (*(volatile uint32_t *)&c.tmem_ready < (uint32_t)ntm) {
                        if (tc::now_ns() > dl || aborted(c, a)) { ok = false; break; }
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
            const uint64_t bd = bdesc0 + (uint64_t)((kc * kBChunkBytes) >> 4);
            const uint32_t acc0 = kc == 0 ? 0u : 1u;
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
        if (!ok) break;
        tc::commit_elect(tc::smem_u32(&c.dfull[W][alt ? ((k - W) >> 1) & 1 : 0]));
        ++uses;
    }
    __syncwarp();
}

// The bias sums of tile `kt` (its 4 K chunks in shared memory, 128-byte
// swizzled K-major as the TMA wrote them) for ids 16 m .. 16 m + 15 and the
// 8 rows, by one warp: 16 mma.sync m16n8k16 (BF16 in, fp32 sums) with
// fragments from ldmatrix, into c.sbias.  The sums' order differs from the
// tcgen05 tiles' only in the last bit of a few fp32 sums.
template <int RANK>
__device__ __forceinline__ void simt_tile(Ctl &c, int kt, int ntm, int m, uint32_t b_sa,
                                          uint32_t head_sa) {
    constexpr int cpt = RANK / 64;
    const int lane = threadIdx.x & 31;
    float d0 = 0.0f, d1 = 0.0f, d2 = 0.0f, d3 = 0.0f;
    const int mi = lane >> 3;                       // ldmatrix.x4: matrix of this lane's address
    const int ra = 16 * m + (mi & 1) * 8 + (lane & 7);   // A row (id within the tile)
    const int nb = lane & 7, hb = (lane >> 3) & 1;       // ldmatrix.x2: B row, K half
#pragma unroll 1
    for (int kc = 0; kc < cpt; ++kc) {
        int slot;
        uint32_t ph;
        chunk_slot(kt * cpt + kc, ntm, slot, ph);
        const uint32_t sa = head_sa + (uint32_t)slot * kChunkBytes + (uint32_t)ra * 128u;
        const uint32_t sb = b_sa + (uint32_t)kc * kBChunkBytes + (uint32_t)nb * 128u;
#pragma unroll
        for (int sub = 0; sub < 4; ++sub) {
            const uint32_t ua = (uint32_t)(2 * sub + (mi >> 1)) ^ (uint32_t)(ra & 7);
            const uint32_t ub = (uint32_t)(2 * sub + hb) ^ (uint32_t)nb;
            uint32_t a0, a1, a2, a3, b0, b1;
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                         : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                         : "r"(sa + (ua << 4)));
            asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                         : "=r"(b0), "=r"(b1)
                         : "r"(sb + (ub << 4)));
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
                "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
        }
    }
    const int id = 16 * m + (lane >> 2), col = (lane & 3) * 2;
    c.sbias[id][col] = d0;
    c.sbias[id][col + 1] = d1;
    c.sbias[id + 8][col] = d2;
    c.sbias[id + 8][col + 1] = d3;
}

// The exact key of Gumbel survivor (id v, row b, cached logit lf) folded
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

// The epilogue of one position, run by the 16 warps 4-19: warp 4 + ew
// serves accumulator wg = ew / 8 (the even / odd tiles), TMEM lane quarter
// q = warp % 4 (the only lanes a warp may read) and rows rb..rb+3, rb =
// 4 ((ew / 4) % 2), so each thread owns one id per tile and 4 of the 8 rows
// (the MMA's N columns).  Two warps per lane quarter halve every thread's
// dependent chains, which bound this code.
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
                                         const int i, const int t0, const int nt, const int nts,
                                         const int ntm, const uint32_t b_sa, const uint32_t head_sa,
                                         const bool gum_any, const uint64_t timeout, uint32_t &dcount) {
    constexpr int cpt = RANK / 64;
    constexpr int kTilesWG = (kMaxChunks / cpt + 1) / 2;   // tiles per group, at most
    constexpr bool kRegs = kTilesWG <= 4;                  // pass-2 tiles kept in registers
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ew = warp - 4, wg = ew >> 3, q = warp & 3, hr = (ew >> 2) & 1;
    // inverse-CDF calls of at most 4 rows: the warps of both row halves take
    // rows 0-3 of the group's tiles in turn (half hr the tiles wg + 2 u with
    // u % 2 == hr, their own full barrier and 4 hand-back arrivals a tile)
    // instead of the second half idling while the first does every tile
    const bool alt = kCdf && a.rows <= kRowsT;
    const int rb = alt ? 0 : kRowsT * hr;
    const int V = a.V;
    const int par = i & 1;
    uint32_t live_m = 0u, samp_m = 0u, div_m = 0u;   // this thread's 4 rows, bit j = row rb + j
#pragma unroll
    for (int j = 0; j < kRowsT; ++j) {
        live_m |= c.live[rb + j] ? (1u << j) : 0u;
        samp_m |= c.sampling[rb + j] ? (1u << j) : 0u;
        div_m |= (c.sampling[rb + j] && c.T[rb + j] != 1.0f) ? (1u << j) : 0u;
    }
    // Gumbel rows get the bound treatment; inverse-CDF rows divide by T
    const uint32_t gum_m = kCdf ? 0u : (samp_m & live_m);
    div_m = kCdf ? (div_m & live_m) : 0u;
    const uint32_t *gq = reinterpret_cast<const uint32_t *>(a.noise) + ((int64_t)i * V) * 2 + hr;
    // DT bit 0: fp32 base logits, bit 1: fp32 cache (else BF16)
    constexpr bool kBaseF32 = (DT & 1) != 0, kCacheF32 = (DT & 2) != 0;
    const int64_t bofs = (int64_t)i * a.base_s1 + rb * a.base_s0;
    const int64_t cofs = (int64_t)i * a.cache_s1 + rb * a.cache_s0;
    const uint16_t *base_i = kBaseF32 ? nullptr : a.base + bofs;
    const float *base_fi = kBaseF32 ? a.base_f + bofs : nullptr;
    uint16_t *cache_i = kCacheF32 ? nullptr : a.cache + cofs;
    float *cache_fi = kCacheF32 ? a.cache_f + cofs : nullptr;

    uint32_t bo[kRowsT], bv[kRowsT];   // best ordered (exact) key and its id
    float lbm[kRowsT], invT[kRowsT];   // Gumbel rows: largest key lower bound
#pragma unroll
    for (int j = 0; j < kRowsT; ++j) {
        bo[j] = 0u;
        bv[j] = 0u;
        lbm[j] = __uint_as_float(0xff800000u);
        invT[j] = c.invT[rb + j];
    }
    // the last 4 tiles' packed logits and FP16 key upper bounds (rows j, j+1)
    // newest first
    uint32_t k0[2] = {0u, 0u}, k1[2] = {0u, 0u}, k2[2] = {0u, 0u}, k3[2] = {0u, 0u};
    __half2 u0[2], u1[2], u2[2], u3[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) u0[j] = u1[j] = u2[j] = u3[j] = __float2half2_rn(0.0f);
    uint32_t nb[kRowsT];
    uint32_t nq;
    auto load_tile = [&](int k, uint32_t (&bb)[kRowsT], uint32_t &qq) {
        const int v = (t0 + k) * 128 + q * 32 + lane;
        const bool ok2 = k < nt && v < V;
#pragma unroll
        for (int j = 0; j < kRowsT; ++j)
            bb[j] = (ok2 && ((live_m >> j) & 1u))
                        ? (kBaseF32 ? __float_as_uint(__ldg(base_fi + j * a.base_s0 + v))
                                    : (uint32_t)__ldg(base_i + j * a.base_s0 + v))
                        : 0u;
        qq = (ok2 && gum_m != 0u) ? __ldcg(gq + 2 * v) : 0u;
    };
    load_tile(alt ? wg + 2 * hr : wg, nb, nq);
    bool ok = true;
    if (nts >= 0 && wg == 1) {
        // group 1, before its first tile: the bias of tile nts, 16 ids per
        // warp, with mma.sync (m16n8k16, fp32 sums) from the tile's shared-
        // memory A chunks and the staged B rows, into sbias
        bool st = true;
        if (lane == 0)
            st = tc::mbar_wait_for(tc::smem_u32(&c.bstaged), (uint32_t)(i - 1) & 1u, timeout);
        st = __shfl_sync(0xffffffffu, st, 0);
        if (!st) {
            if (lane == 0) fail(c, a, 4u, 0xC000u + i);
        } else {
            simt_tile<RANK>(c, nts, ntm, ew - 8, b_sa, head_sa);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&c.sdone));
    }
    int ntw = 0;   // tiles this warp processed
#pragma unroll 1
    for (int k = wg; k < nt; k += 2) {
        if (alt && (((k - wg) >> 1) & 1) != hr) continue;
        uint32_t cb[kRowsT];
#pragma unroll
        for (int j = 0; j < kRowsT; ++j) cb[j] = nb[j];
        const uint32_t cq = nq;
        load_tile(alt ? k + 4 : k + 2, nb, nq);
        if (__shfl_sync(0xffffffffu, lane == 0 ? aborted(c, a) : false, 0)) {
            ok = false;
            break;
        }
        uint32_t r[4];
        if (k == nts) {
            // the mma.sync tile (group 0's last): its bias from sbias
            if (lane == 0)
                ok = tc::mbar_wait_for(tc::smem_u32(&c.sdone), (uint32_t)(i - 1) & 1u, timeout);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) fail(c, a, 4u, 0xD000u + i);
                break;
            }
            const float4 sb = *reinterpret_cast<const float4 *>(&c.sbias[q * 32 + lane][rb]);
            r[0] = __float_as_uint(sb.x);
            r[1] = __float_as_uint(sb.y);
            r[2] = __float_as_uint(sb.z);
            r[3] = __float_as_uint(sb.w);
        } else {
            if (lane == 0)
                ok = tc::mbar_wait_for(tc::smem_u32(&c.dfull[wg][alt ? hr : 0]), dcount & 1u, timeout);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) fail(c, a, 4u, 0x6000u + i);
                break;
            }
            ++dcount;
            tc::fence_after_sync();
            tc::ld_32x32b_x4(tmem + ((uint32_t)(q * 32) << 16) + kDCol + 16u * wg + (uint32_t)rb, r);
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&c.dfree[wg]));
        }
        // nothing that waits on this tile's base loads may be scheduled
        // before the accumulator is handed back
#pragma unroll
        for (int j = 0; j < kRowsT; ++j) asm volatile("" : "+r"(cb[j]));
        asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]));
        const int v = (t0 + k) * 128 + q * 32 + lane;
        const bool valid = v < V;
        // bias = bf16(sum); logit = cache_round(f32(base) + f32(bias)), two
        // rows a time (BF16 caches: packed; fp32 caches: kept in fp32)
        uint32_t lp[2];
        float lf4[kRowsT];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t bb = bf16x2_rn(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
            const float b0 = kBaseF32 ? __uint_as_float(cb[2 * j]) : __uint_as_float(cb[2 * j] << 16);
            const float b1 = kBaseF32 ? __uint_as_float(cb[2 * j + 1]) : __uint_as_float(cb[2 * j + 1] << 16);
            const float s0 = __fadd_rn(b0, __uint_as_float(bb << 16));
            const float s1 = __fadd_rn(b1, __uint_as_float(bb & 0xffff0000u));
            if (kCacheF32) {
                lf4[2 * j] = s0;
                lf4[2 * j + 1] = s1;
            } else {
                lp[j] = bf16x2_rn(s0, s1);
            }
        }
        if (kCacheF32) {
            if (a.tf.has_transform) {
#pragma unroll
                for (int j = 0; j < kRowsT; ++j) lf4[j] = transform_f32(lf4[j], a.tf);
            }
#pragma unroll
            for (int j = 0; j < kRowsT; ++j)
                if (valid && ((live_m >> j) & 1u)) cache_fi[j * a.cache_s0 + v] = lf4[j];
        } else {
            if (a.tf.has_transform) {
                if (kCdf) {
                    lp[0] = transform_pair_inl(lp[0], a.tf);
                    lp[1] = transform_pair_inl(lp[1], a.tf);
                } else {
                    lp[0] = transform_pair(lp[0], a.tf);
                    lp[1] = transform_pair(lp[1], a.tf);
                }
            }
#pragma unroll
            for (int j = 0; j < kRowsT; ++j) {
                lf4[j] = __uint_as_float((j & 1) ? (lp[j >> 1] & 0xffff0000u) : (lp[j >> 1] << 16));
                if (valid && ((live_m >> j) & 1u))
                    cache_i[j * a.cache_s0 + v] = (uint16_t)(lp[j >> 1] >> (16 * (j & 1)));
            }
        }
        float ku[kRowsT];
#pragma unroll
        for (int j = 0; j < kRowsT; ++j) {
            const float lf = lf4[j];
            ku[j] = 0.0f;
            if ((gum_m >> j) & 1u) {
                const uint32_t qb = (cq >> (8 * j)) & 0xffu;
                const float kl = key_lower(lf, invT[j], qb);
                lbm[j] = (valid && kl > lbm[j]) ? kl : lbm[j];
                ku[j] = key_upper(lf, invT[j], qb);
            } else if ((live_m >> j) & 1u) {
                float key = lf;
                if (kCdf && ((div_m >> j) & 1u)) key = __fdiv_rn(lf, c.T[rb + j]);
                const uint32_t o = ordered_key(key);
                const bool better = valid && o > bo[j];
                bo[j] = better ? o : bo[j];
                bv[j] = better ? (uint32_t)v : bv[j];
            }
        }
        if (kRegs && gum_m != 0u) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                if (!kCacheF32) {
                    k3[j] = k2[j];
                    k2[j] = k1[j];
                    k1[j] = k0[j];
                    k0[j] = lp[j];
                }
                u3[j] = u2[j];
                u2[j] = u1[j];
                u1[j] = u0[j];
                u0[j] = half2_up(ku[2 * j], ku[2 * j + 1]);
            }
        }
        ++ntw;
    }
    // rows with exact keys: the warp's best into the CTA's
#pragma unroll
    for (int j = 0; j < kRowsT; ++j) {
        if ((gum_m >> j) & 1u) continue;
        const uint64_t pk =
            bo[j] != 0u ? (((uint64_t)bo[j] << 32) | ((uint64_t)(0x3FFFFu - bv[j]) << 14)) : 0ull;
        const uint64_t m = tc::warp_max_u64(pk);
        if (lane == 0 && m != 0ull) atomicMax(&c.cbest[par][rb + j], (unsigned long long)m);
    }
    if (!gum_any) return;

    // ---- pass 2 (Gumbel rows), with no CTA barrier: the warp's threshold
    // (its largest lower bound) goes into the CTA's (shared-memory maximum),
    // and the CTA's threshold as it stands then (every value in it is a
    // lower bound on the CTA's best key, and it already holds this warp's)
    // selects the ids whose upper bound reaches it; their lanes compute
    // their exact keys.  A group that finishes its tiles early does this
    // while the other still works on its last tile.
    uint32_t lw = 0u;   // lane j < 4: ordered warp threshold of row rb + j
#pragma unroll
    for (int j = 0; j < kRowsT; ++j) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, ((gum_m >> j) & 1u) ? ordered_key(lbm[j]) : 0u);
        lw = lane == j ? m : lw;
    }
    if (ok && ntw > 0 && lane < kRowsT && lw != 0u) atomicMax(&c.lcta[par][rb + lane], lw);
    __syncwarp();
    float Lc[kRowsT];
#pragma unroll
    for (int j = 0; j < kRowsT; ++j) {
        const uint32_t o = *(volatile uint32_t *)&c.lcta[par][rb + j];
        // no bound recorded (no valid id): nothing can survive
        Lc[j] = o != 0u ? key_from_ordered(o) : __uint_as_float(0x7f800000u);
    }
    if (kRegs && ok) {
        uint32_t cand = 0u;   // bit 4 r + j: queued tile r (newest first), row rb + j survives
        const __half2 L01 = __halves2half2(__float2half_rd(Lc[0]), __float2half_rd(Lc[1]));
        const __half2 L23 = __halves2half2(__float2half_rd(Lc[2]), __float2half_rd(Lc[3]));
        auto slot = [&](int r, const __half2 (&uu)[2]) {
            const int k = wg + 2 * (ntw - 1 - r);
            const int v = (t0 + k) * 128 + q * 32 + lane;
            if (r < ntw && v < V) {
                const uint32_t m01 = __hgeu2_mask(uu[0], L01), m23 = __hgeu2_mask(uu[1], L23);
                const uint32_t b4 = (m01 & 1u) | ((m01 >> 15) & 2u) | ((m23 & 1u) << 2) | ((m23 >> 13) & 8u);
                cand |= (b4 & gum_m) << (4 * r);
            }
        };
        slot(0, u0);
        slot(1, u1);
        slot(2, u2);
        slot(3, u3);
        while (cand != 0u) {
            const int bit = __ffs(cand) - 1;
            cand &= cand - 1u;
            const int r = bit >> 2, j = bit & 3;
            const int k = wg + 2 * (ntw - 1 - r);
            const uint32_t v = (uint32_t)((t0 + k) * 128 + q * 32 + lane);
            float lf;
            if (kCacheF32) {
                // an fp32 cache's logit, read back (this thread wrote it)
                lf = cache_fi[j * a.cache_s0 + v];
            } else {
                const uint32_t pr = (j < 2) ? (r == 0 ? k0[0] : r == 1 ? k1[0] : r == 2 ? k2[0] : k3[0])
                                            : (r == 0 ? k0[1] : r == 1 ? k1[1] : r == 2 ? k2[1] : k3[1]);
                lf = __uint_as_float(((pr >> (16 * (j & 1))) & 0xffffu) << 16);
            }
            survivor_key(c, i, v, rb + j, lf);
        }
    }
    if (!kRegs && ok) {
        // more tiles than registers hold (small ranks): the cached logits and
        // noise bytes are read back (L2) tile by tile, exact bounds
#pragma unroll 1
        for (int r = 0; r < ntw; ++r) {
            const int k = wg + 2 * r;
            const int v = (t0 + k) * 128 + q * 32 + lane;
            if (v >= V) continue;
            const uint32_t qq = __ldcg(gq + 2 * v);
#pragma unroll
            for (int j = 0; j < kRowsT; ++j) {
                if (!((gum_m >> j) & 1u)) continue;
                const float lf = kCacheF32 ? __ldcg(cache_fi + j * a.cache_s0 + v)
                                           : __uint_as_float((uint32_t)__ldcg(cache_i + j * a.cache_s0 + v) << 16);
                if (!(key_upper(lf, invT[j], (qq >> (8 * j)) & 0xffu) < Lc[j]))
                    survivor_key(c, i, (uint32_t)v, rb + j, lf);
            }
        }
    }
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
    const int t0 = (int)((int64_t)cta * T_total / G);
    const int t1 = (int)((int64_t)(cta + 1) * T_total / G);
    const int nt = t1 - t0;
    const int nch = nt * cpt;
    const int ntm = nch < kTmemChunks ? nch : kTmemChunks;
    const int v_begin = t0 * 128;
    const int v_end = t1 * 128 < V ? t1 * 128 : V;
    const int Gp = (G + kKeyPad - 1) / kKeyPad * kKeyPad;
    // the epilogue halves take the tiles in turn (inverse CDF, at most 4 rows)
    const bool alt = MODE == 1 && R <= kRowsT;

    // ------------------------------------------------------------ set-up
    if (tid == 0) {
        for (int s = 0; s < kSmemChunks; ++s) {
            tc::mbar_init(tc::smem_u32(&c.full[s]), 1);
            tc::mbar_init(tc::smem_u32(&c.cpdone[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(tc::smem_u32(&c.dfull[b][0]), 1);
            tc::mbar_init(tc::smem_u32(&c.dfull[b][1]), 1);
            tc::mbar_init(tc::smem_u32(&c.dfree[b]), alt ? kEpiWarps / 4 : kEpiWarps / 2);
            tc::mbar_init(tc::smem_u32(&c.fin[b]), 1);
        }
        tc::mbar_init(tc::smem_u32(&c.bstaged), 1);
        tc::mbar_init(tc::smem_u32(&c.sdone), kEpiWarps / 2);
        tc::mbar_init_fence();
        c.tmem_ready = 0u;
        clear_position(c, 0);

        c.abort = ld_acquire_u32(a.status) != 0u ? 1u : 0u;
        c.call = *(volatile const uint32_t *)a.call_counter;
    }
    if (tid < kChainRows) {
        const int b = tid;
        // the row's four arguments in one round trip (not each behind the
        // row_state_idx test)
        int64_t idx = -1, seed = 0;
        float T = 0.0f;
        int32_t anc = 0;
        if (b < R) {
            idx = a.row_state_idx[b];
            T = a.temperature[b];
            seed = a.seeds[b];
            anc = a.anchor[b];
        }
        const bool live = idx >= 0;
        if (!live) T = 0.0f;
        c.live[b] = live;
        c.T[b] = T;
        c.sampling[b] = live && samples(T);
        c.seed[b] = live ? (uint64_t)seed : 0ull;
        c.invT[b] = samples(T) ? 1.0f / T : 1.0f;
        int64_t p = live ? (int64_t)anc : 0;
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
    if (cta == 0 && tid < kMaxSteps * kChainRows) {
        // the next call's exchange words (the other call parity; the previous
        // call, which used them, has completed): back to zero
        const size_t np = (size_t)((c.call + 1u) & 1u);
        a.win_max[(np * kMaxSteps * kChainRows + tid) * kLineU64] = 0ull;
        if (tid < kMaxSteps) a.win_cnt[(np * kMaxSteps + tid) * kLineU32] = 0u;
    }
    if (warp < kChainRows && c.live[warp]) stage_embed<RANK>(b_s, a.embed, c.prev[warp], warp, lane);
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
    uint32_t uses = 0;          // issuer: tiles issued into its accumulator
    uint32_t dcount = 0;        // epilogue: tiles consumed from its accumulator
    uint32_t issued[kSmemChunks];   // producer: loads issued per slot
#pragma unroll
    for (int s = 0; s < kSmemChunks; ++s) issued[s] = 0u;

    bool stop = __syncthreads_or(c.abort != 0u);
    for (int i = 0; i < N && !stop; ++i) {
        // A CTA with the full 7 tiles of rank 256 takes its last tile's bias
        // through mma.sync in the epilogue warps after position 0: the
        // tcgen05 tiles then pair up in 3 rounds of the two accumulators
        // instead of 4.  (Its A chunks are in shared memory.)
        const int nts = (MODE == 0 && RANK == 256 && nt == kMaxChunks / cpt && i > 0) ? nt - 1 : -1;
        // ------------------------------------- phase A: MMA and epilogue
        if (warp < 2) {
            issue_tiles<RANK>(c, a, tmem, warp, i, nts >= 0 ? nts : nt, ntm, b_sa, head_sa, timeout, alt, uses);
        } else if (warp < 4 && i > 0) {
            // warps 2 and 3 after the head load: the next position's base
            // logits into L2, off the chain's critical path
            if (i + 1 < N) prefetch_base<64>(c, a, i + 1, v_begin, v_end, tid - 64);
        } else if (warp == 2) {
            if (lane == 0 && i == 0) {
                for (int j = 0; j < nch; ++j) {
                    if (aborted(c, a)) break;
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
                    if (aborted(c, a)) break;
                    int sp = 0;
                    uint32_t pp = 0u;
                    if (j > 0) chunk_slot(j - 1, ntm, sp, pp);
                    if (j < ntm) {
                        int s;
                        uint32_t ph;
                        chunk_slot(j, ntm, s, ph);
                        if (!tc::mbar_wait_for(tc::smem_u32(&c.full[s]), ph & 1u, timeout)) {
                            fail(c, a, 4u, 0x4000u + j);
                            break;
                        }
                        if (j > 0 && sp == s) {
                            // (already complete: this load waited for it)
                            if (!tc::mbar_wait_for(tc::smem_u32(&c.cpdone[sp]), pp & 1u, timeout)) {
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
                        if (!tc::mbar_wait_for(tc::smem_u32(&c.cpdone[sp]), pp & 1u, timeout)) {
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
            if (MODE == 1)
                epilogue<RANK, true, DT>(c, a, tmem, i, t0, nt, -1, ntm, b_sa, head_sa, false, timeout, dcount);
            else
                epilogue<RANK, false, DT>(c, a, tmem, i, t0, nt, nts, ntm, b_sa, head_sa, gum_any, timeout, dcount);
        }
        stop = __syncthreads_or(stop_vote(c));
        if (stop) break;

        // ------------------------------- phase B: agree on every row's winner
        const uint32_t epoch = c.call * (uint32_t)kMaxSteps + (uint32_t)i + 1u;
        if (MODE == 0) {
            // Gumbel and greedy rows: warp 0 reports this CTA's best key per
            // row and collects the winners; warps 0-3 stage the winners'
            // embeddings (rows w and w + 4) as the next B operand.  Every CTA
            // folds its keys into one word per (position, row) with red.max
            // and then adds 1 to the position's counter (release); lane 0
            // waits until all G CTAs have counted (acquire) and reads the 8
            // words: one polled word per CTA keeps the L2 traffic low.  The
            // words of one call parity are zeroed by the previous call.
            if (warp == 0 || warp == 2) {
                if (warp == 0) {
                    // lane b < 8: row b's best key in this CTA
                    const size_t par = (size_t)(c.call & 1u);
                    uint64_t *wm = a.win_max + ((par * kMaxSteps + i) * kChainRows) * kLineU64;
                    uint32_t *wc = a.win_cnt + (par * kMaxSteps + i) * kLineU32;
                    // lane b < 8 folds row b's best key in (one instruction for
                    // all rows); the warp barrier orders the reds before lane
                    // 0's release
                    if (lane < kChainRows && c.live[lane])
                        tc::red_max_u64(wm + lane * kLineU64, (uint64_t)c.cbest[i & 1][lane]);
                    __syncwarp();
                    if (lane == 0) {
                        bool ok = true;
                        tc::red_release_add_u32(wc, 1u);
                        const uint64_t dl = tc::now_ns() + timeout;
                        for (uint32_t spin = 0;; ++spin) {
                            if ((int32_t)(ld_acquire_u32(wc) - (uint32_t)G) >= 0) break;
                            if ((spin & 15u) == 15u &&
                                (tc::now_ns() > dl || ld_acquire_u32(a.status) != 0u)) {
                                ok = false;
                                break;
                            }
                        }
                        if (ok) {
                            // all 8 loads in flight before any result is used
                            uint64_t w8[kChainRows];
#pragma unroll
                            for (int b = 0; b < kChainRows; ++b)
                                w8[b] = c.live[b] ? tc::ld_relaxed_u64(wm + b * kLineU64) : 0ull;
#pragma unroll
                            for (int b = 0; b < kChainRows; ++b) c.win[b] = w8[b];
                        } else {
                            fail(c, a, 4u, 0x7000u + i);
                        }
                    }
                    __syncwarp();
                } else if (lane < kChainRows && c.live[lane]) {
                    // warp 2: this CTA's candidate of row b = lane into L2
                    // while the winners are agreed (the winning CTA's
                    // prefetch serves every CTA's staging gather)
                    const uint64_t m = c.cbest[i & 1][lane];
                    const uint32_t id = unpack_id(m);
                    if (m != 0ull && id < (uint32_t)V && i + 1 < N) {
                        const uint8_t *er = reinterpret_cast<const uint8_t *>(a.embed + (int64_t)id * RANK);
#pragma unroll
                        for (int o = 0; o < RANK * 2; o += 128) tc::prefetch_l2(er + o);
                    }
                }
            }
            if (warp < 4) {
                asm volatile("bar.sync 3, 128;" ::: "memory");
                // warps 0-3 stage rows w and w + 4: both gathers in flight at once
                const int rb2[2] = {warp, warp + 4};
                uint32_t idr[2];
                uint4 ev[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int b = rb2[h];
                    uint32_t id = unpack_id(c.win[b]);
                    if (c.live[b] && id >= (uint32_t)V) {
                        // no CTA reported a key for a live row: an internal
                        // error; never index embed with it
                        if (lane == 0) fail(c, a, 6u /* MARKOV_EDEVICE */, 0xB000u + i);
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
                    if (i + 1 < N && lane < RANK / 8) {
                        const int chunk = lane >> 3, piece = lane & 7;
                        *reinterpret_cast<uint4 *>(b_s + chunk * kBChunkBytes + b * 128 + ((piece ^ b) << 4)) = ev[h];
                    }
                }
            }
            if (warp < 4) {
                // the control warps alone close the position: the next MMAs
                // need only the staged B operand
                tc::fence_proxy_async_smem();
                tc::fence_before_sync();
                asm volatile("bar.sync 4, 128;" ::: "memory");
                tc::fence_after_sync();
                // the epilogue warps' mma.sync tile reads the staged rows too
                if (tid == 0 && i + 1 < N) tc::mbar_arrive(tc::smem_u32(&c.bstaged));
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
        } else {
            // the rows' maxima as in Gumbel mode: red.max into one word per
            // (position, row), a release-add on the position's counter, one
            // polled word per CTA, then the 8 words
            if (warp == 0) {
                const size_t par = (size_t)(c.call & 1u);
                uint64_t *wm = a.win_max + ((par * kMaxSteps + i) * kChainRows) * kLineU64;
                uint32_t *wc = a.win_cnt + (par * kMaxSteps + i) * kLineU32;
                if (lane < kChainRows && c.live[lane])
                    tc::red_max_u64(wm + lane * kLineU64, (uint64_t)c.cbest[i & 1][lane]);
                __syncwarp();
                if (lane == 0) {
                    bool ok = true;
                    tc::red_release_add_u32(wc, 1u);
                    const uint64_t dl = tc::now_ns() + timeout;
                    for (uint32_t spin = 0;; ++spin) {
                        if ((int32_t)(ld_acquire_u32(wc) - (uint32_t)G) >= 0) break;
                        if ((spin & 15u) == 15u && (tc::now_ns() > dl || ld_acquire_u32(a.status) != 0u)) {
                            ok = false;
                            break;
                        }
                    }
                    if (ok) {
                        uint64_t w8[kChainRows];
#pragma unroll
                        for (int b = 0; b < kChainRows; ++b)
                            w8[b] = c.live[b] ? tc::ld_relaxed_u64(wm + b * kLineU64) : 0ull;
#pragma unroll
                        for (int b = 0; b < kChainRows; ++b) c.win[b] = w8[b];
                    } else {
                        fail(c, a, 4u, 0x7000u + i);
                    }
                }
                __syncwarp();
            } else if (warp == 2 && lane < kChainRows && c.live[lane]) {
                // this CTA's candidates into L2 (the winning CTA's prefetch
                // serves every CTA's gather of a greedy row's token)
                const uint64_t m = c.cbest[i & 1][lane];
                const uint32_t id = unpack_id(m);
                if (m != 0ull && id < (uint32_t)V && i + 1 < N) {
                    const uint8_t *er = reinterpret_cast<const uint8_t *>(a.embed + (int64_t)id * RANK);
#pragma unroll
                    for (int o = 0; o < RANK * 2; o += 128) tc::prefetch_l2(er + o);
                }
            }
            // the inverse-CDF weights need the maxima, but fp32(x / T) of the
            // CTA's cached logits does not: the epilogue warps (thread
            // et = tid - 128 takes the contiguous ids [c0, c1)) load and
            // divide them for the first kGR sampling rows while the maxima
            // are exchanged, and keep them in registers for the weight pass
            // and the owner's scan
            constexpr int kMaxIds = (kTmemChunks + kSmemChunks) / (RANK / 64) * 128;
            constexpr int kPT = (kMaxIds + kEpiThreads - 1) / kEpiThreads;   // ids per thread
            constexpr int kGR = RANK == 64 ? 2 : 4;
            const int et = tid - 128;
            const int chunk = (v_end - v_begin + kEpiThreads - 1) / kEpiThreads;
            const int c0 = v_begin + et * chunk;
            const int c1 = c0 + chunk < v_end ? c0 + chunk : v_end;
            float q0[kGR][kPT];
            if (warp >= 4) {
#pragma unroll
                for (int r = 0; r < kGR; ++r) {
                    const bool s_r = r < R && c.sampling[r];
                    const float T = c.T[r];
                    const bool p2 = dm_pow2_temperature(T);
                    const float rT = p2 ? __frcp_rn(T) : 0.0f;
                    const int64_t crow = r * a.cache_s0 + (int64_t)i * a.cache_s1;
#pragma unroll
                    for (int k = 0; k < kPT; ++k) {
                        float x = 0.0f;
                        if (s_r && c0 + k < c1)
                            x = (DT & 2) ? a.cache_f[crow + c0 + k] : dm_bf16_f32(a.cache[crow + c0 + k]);
                        q0[r][k] = p2 ? dm_div_T<true>(x, T, rT) : dm_div_T<false>(x, T, 0.0f);
                    }
                }
            }
            stop = __syncthreads_or(stop_vote(c));
            if (stop) break;

            // inverse CDF: rows whose maximum M is finite need the exact integer
            // weight sums floor(exp(x - M) 2^40), then the CTA whose prefix range
            // holds mulhi64(H, S) scans its ids for the token
            bool cdf_any = false;
            if (MODE == 1) {
                for (int b = 0; b < R && b < kChainRows; ++b) {
                    if (!c.sampling[b]) continue;
                    const uint32_t o = (uint32_t)(c.win[b] >> 32);
                    const float M = key_from_ordered(o);
                    if (o != 0xffffffffu && !isinf(M)) cdf_any = true;
                }
            }
            if (cdf_any) {
                const uint32_t tag32 = epoch;
                // the epilogue threads' weights: per row a register total
                // (mine) and per warp a shared-memory total (c.wsum), so the
                // owning warp and thread are found with no block barrier and
                // no second pass over the range
                uint64_t mine[kChainRows];
#pragma unroll
                for (int b = 0; b < kChainRows; ++b) mine[b] = 0ull;
                if (warp >= 4) {
                    const int ew = warp - 4;
#pragma unroll
                    for (int b = 0; b < kChainRows; ++b) {
                        if (b >= R) break;
                        const uint32_t o = (uint32_t)(c.win[b] >> 32);
                        const bool use = c.sampling[b] && o != 0xffffffffu && !isinf(key_from_ordered(o));
                        uint64_t part = 0ull;
                        if (use) {
                            const float M = key_from_ordered(o);
                            if (b < kGR) {
#pragma unroll
                                for (int k = 0; k < kPT; ++k)
                                    if (c0 + k < c1) part += dm_cdf_weight(__fsub_rn(q0[b < kGR ? b : 0][k], M));
                            } else {
                                // rows past the first kGR: load and divide now
                                const float T = c.T[b];
                                const int64_t crow = b * a.cache_s0 + (int64_t)i * a.cache_s1;
                                float xs[kPT];
#pragma unroll
                                for (int k = 0; k < kPT; ++k)
                                    xs[k] = (c0 + k < c1) ? ((DT & 2) ? a.cache_f[crow + c0 + k]
                                                                      : dm_bf16_f32(a.cache[crow + c0 + k]))
                                                          : 0.0f;
#pragma unroll
                                for (int k = 0; k < kPT; ++k)
                                    if (c0 + k < c1) part += dm_cdf_weight(__fsub_rn(__fdiv_rn(xs[k], T), M));
                            }
                        }
                        mine[b] = part;
                        if (__any_sync(0xffffffffu, use)) {
#pragma unroll
                            for (int o2 = 16; o2 > 0; o2 >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o2);
                            if (lane == 0) c.wsum[b][ew] = part;
                        }
                    }
                }
                __syncthreads();
                // each row's CTA sum into slot (position, row, CTA), then a
                // release-add on the position's counter, which the maxima
                // took to G and the sums take on to 2G: once a CTA reads 2G
                // every slot of the position holds this call's sum
                const size_t par = (size_t)(c.call & 1u);
                uint32_t *wc = a.win_cnt + (par * kMaxSteps + i) * kLineU32;
                if (warp == 0) {
                    if (lane < kChainRows) {
                        const int b = lane;
                        uint64_t s = 0ull;
                        if (b < R && c.sampling[b]) {
#pragma unroll
                            for (int w = 0; w < kEpiThreads / 32; ++w) s += c.wsum[b][w];
                            tc::st_relaxed_u64(a.tc_sums + ((int64_t)i * kChainRows + b) * Gp + cta, s);
                        }
                        c.sum[b] = s;
                    }
                    __syncwarp();
                    if (lane == 0) tc::red_release_add_u32(wc, 1u);
                }
                // every CTA learns every row's total and its own prefix: per
                // row one warp, whose lane 0 polls the counter and whose lanes
                // then read the row's slots together
                __shared__ uint64_t s_tot[kChainRows], s_pre[kChainRows];
                if (warp < kChainRows && warp < R && c.sampling[warp]) {
                    const int b = warp;
                    const uint32_t o = (uint32_t)(c.win[b] >> 32);
                    const float M = key_from_ordered(o);
                    if (o != 0xffffffffu && !isinf(M)) {
                        bool ok = true;
                        if (lane == 0) {
                            const uint64_t dl = tc::now_ns() + timeout;
                            for (uint32_t spin = 0;; ++spin) {
                                if ((int32_t)(ld_acquire_u32(wc) - 2u * (uint32_t)G) >= 0) break;
                                if ((spin & 15u) == 15u && (tc::now_ns() > dl || ld_acquire_u32(a.status) != 0u)) {
                                    ok = false;
                                    break;
                                }
                            }
                        }
                        __syncwarp();
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        if (!ok) {
                            if (lane == 0) fail(c, a, 4u, 0x8000u + i);
                        } else {
                            const uint64_t *sl = a.tc_sums + ((int64_t)i * kChainRows + b) * Gp;
                            constexpr int kPer = kMaxGrid / 32;
                            uint64_t s5[kPer];
#pragma unroll
                            for (int u = 0; u < kPer; ++u)
                                s5[u] = lane + 32 * u < G ? tc::ld_relaxed_u64(sl + lane + 32 * u) : 0ull;
                            uint64_t tot = 0ull, pre = 0ull;
#pragma unroll
                            for (int u = 0; u < kPer; ++u) {
                                tot += s5[u];
                                if (lane + 32 * u < cta) pre += s5[u];
                            }
#pragma unroll
                            for (int o2 = 16; o2 > 0; o2 >>= 1) {
                                tot += __shfl_xor_sync(0xffffffffu, tot, o2);
                                pre += __shfl_xor_sync(0xffffffffu, pre, o2);
                            }
                            if (lane == 0) { s_tot[b] = tot; s_pre[b] = pre; }
                        }
                    }
                }
                stop = __syncthreads_or(stop_vote(c));
                if (stop) break;
                // the CTA whose prefix range holds the target: its warp whose
                // range holds it, then that warp's thread, scans its own ids
                // (the first kGR rows from the registers)
                if (warp >= 4) {
                    const int ew = warp - 4;
#pragma unroll
                    for (int b = 0; b < kChainRows; ++b) {
                        if (b >= R || !c.sampling[b]) continue;
                        const uint32_t o = (uint32_t)(c.win[b] >> 32);
                        const float M = key_from_ordered(o);
                        if (o == 0xffffffffu || isinf(M)) continue;
                        const uint64_t S = s_tot[b], P = s_pre[b], Sc = c.sum[b];
                        const uint64_t target = __umul64hi(dm_cdf_hash(c.hri[i][b]), S);
                        if (!(P <= target && target < P + Sc)) continue;
                        const uint64_t t = target - P;
                        uint64_t wpre = 0ull;
                        for (int w = 0; w < ew; ++w) wpre += c.wsum[b][w];
                        const uint64_t ws = c.wsum[b][ew];
                        if (!(ws && wpre <= t && t < wpre + ws)) continue;
                        uint64_t incl = mine[b];
#pragma unroll
                        for (int o2 = 1; o2 < 32; o2 <<= 1) {
                            const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o2);
                            if (lane >= o2) incl += y;
                        }
                        uint64_t run = wpre + incl - mine[b];
                        if (mine[b] && run <= t && t < run + mine[b]) {
                            const int64_t crow = b * a.cache_s0 + (int64_t)i * a.cache_s1;
                            for (int k = 0; k < kPT; ++k) {
                                const int v = c0 + k;
                                if (v >= c1) break;
                                float x;
                                if (b < kGR) {
                                    x = q0[b < kGR ? b : 0][k];
                                } else {
                                    const float xc = (DT & 2) ? a.cache_f[crow + v] : dm_bf16_f32(a.cache[crow + v]);
                                    x = __fdiv_rn(xc, c.T[b]);
                                }
                                run += dm_cdf_weight(__fsub_rn(x, M));
                                if (run > t) {
                                    tc::st_relaxed_u64(a.tok_slots + (int64_t)i * kChainRows + b,
                                                       ((uint64_t)v << 32) | tag32);
                                    break;
                                }
                            }
                        }
                    }
                }
                // everyone learns the tokens the owners found
                if (warp < kChainRows && c.sampling[warp] && lane == 0) {
                    const int b = warp;
                    const uint32_t o = (uint32_t)(c.win[b] >> 32);
                    const float M = key_from_ordered(o);
                    if (o != 0xffffffffu && !isinf(M)) {
                        const uint64_t *slot = a.tok_slots + (int64_t)i * kChainRows + b;
                        const uint64_t dl = tc::now_ns() + timeout;
                        uint64_t t = 0ull;
                        for (uint32_t spin = 0;; ++spin) {
                            t = tc::ld_relaxed_u64(slot);
                            if ((uint32_t)t == tag32) break;
                            if ((spin & 15u) == 15u && (tc::now_ns() > dl || ld_acquire_u32(a.status) != 0u)) {
                                fail(c, a, 4u, 0x9000u + i);
                                break;
                            }
                        }
                        const uint32_t v = (uint32_t)(t >> 32);
                        if ((uint32_t)t == tag32 && v < (uint32_t)V)
                            c.win[b] = (c.win[b] & 0xffffffff00000000ull) |
                                       ((uint64_t)(0x3FFFFu - v) << 14);
                        else if ((uint32_t)t == tag32)
                            fail(c, a, 6u, 0xA000u + i);
                    }
                }
                stop = __syncthreads_or(stop_vote(c));
                if (stop) break;
            }

            // ------------------------- the token, and the next position's B operand
            if (warp < kChainRows && c.live[warp]) {
                const int b = warp;
                uint32_t id = unpack_id(c.win[b]);
                if (MODE == 1 && c.sampling[b]) {
                    const uint32_t o = (uint32_t)(c.win[b] >> 32);
                    if (o != 0xffffffffu && key_from_ordered(o) == __uint_as_float(0xff800000u)) id = 0u;
                }
                if (id >= (uint32_t)V) {
                    if (lane == 0) fail(c, a, 6u /* MARKOV_EDEVICE */, 0xB100u + i);
                    id = 0u;
                }
                if (lane == 0) {
                    c.prev[b] = (int64_t)id;
                    if (cta == 0) a.tokens[b * a.tok_s0 + i] = (int64_t)id;
                }
                if (i + 1 < N) stage_embed<RANK>(b_s, a.embed, (int64_t)id, b, lane);
            }
            // the next position's CTA maxima (last read before this
            // position's phase-A barrier)
            if (tid == 128 && i + 1 < N) clear_position(c, (i + 1) & 1);
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            stop = __syncthreads_or(stop_vote(c));
            tc::fence_after_sync();
        }
    }

    // --------------------------------------------------------------- exit
    // every async operation of this CTA completes before TMEM is released
    if (warp < 2) {
        __syncwarp();
        tc::commit_elect(tc::smem_u32(&c.fin[warp]));
        tc::mbar_wait_for(tc::smem_u32(&c.fin[warp]), 0u, 1000000000ull);
    }
    if (warp == 2 && lane == 0) {
        for (int s = 0; s < kSmemChunks; ++s) {
            if (issued[s] == 0u) continue;
            tc::mbar_wait_for(tc::smem_u32(&c.full[s]), (issued[s] - 1u) & 1u, 1000000000ull);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
    if (cta == 0 && tid == 0 && !aborted(c, a) && ld_acquire_u32(a.status) == 0u)
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
