// static_scratch.cu -- markov_chain_sample_static: the persistent chain for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs while a CUDA graph is
// being captured on a stream that forbids allocation, inference servers and
// plugins that must take every byte from their own pre-sized pool, and
// processes whose allocator is owned by another runtime.  This entry point
// takes no plan and allocates nothing.  Its scratch (the Gumbel noise, the
// cross-CTA key and sum slots, the barrier and status words) lives in one
// file-scope __device__ array of kStaticScratchBytes, which every GPU that
// loads the library holds until the process exits.
//
// It runs the same kernels as markov_chain_sample's simple chain path (the
// noise kernel, then the persistent mma.sync chain), so its outputs are
// identical to that path's.
#include <mutex>

#include "../../include/markov.h"
#include "internal.h"

namespace dtm {
namespace {

// Layout of the static scratch: control words, key slots, sum slots, noise.
constexpr size_t kCtrlBytes = 256;
constexpr int kMaxGridPad = 160;                           // padded CTA count
constexpr size_t kSlotBytes = (size_t)kMaxSteps * 2 * kChainRows * kMaxGridPad * 8;
constexpr size_t kNoiseBytes = (size_t)32 << 20;           // rows * N * V fp32 noise values
constexpr size_t kStaticScratchBytes = kCtrlBytes + 2 * kSlotBytes + kNoiseBytes;

__device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char *g_addr[kMaxDevices];   // device address of g_scratch per device
int g_sms[kMaxDevices];
int g_occ[kMaxDevices];

// Once per device, with that device current: the array's device address and
// the co-residency of the chain kernel.
markov_status setup(int dev, unsigned char **addr, int *sms, int *occ) {
    if (dev < 0 || dev >= kMaxDevices) return MARKOV_EDEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return MARKOV_ECUDA;
        }
        int n = 0, o = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            chain_occupancy(&o) != cudaSuccess) {
            cudaGetLastError();
            return MARKOV_ECUDA;
        }
        g_sms[dev] = n;
        g_occ[dev] = o;
        g_addr[dev] = static_cast<unsigned char *>(p);
    }
    *addr = g_addr[dev];
    *sms = g_sms[dev];
    *occ = g_occ[dev];
    return MARKOV_OK;
}

}  // namespace
}  // namespace dtm

using namespace dtm;

extern "C" markov_status markov_chain_sample_static(
    int32_t vocab, int32_t rank, int32_t num_steps, const uint16_t *base_logits, int64_t base_s0,
    int64_t base_s1, const uint16_t *head, const uint16_t *embed, const int32_t *anchor_tokens,
    const float *temperature, const int64_t *seeds, const int64_t *row_state_idx, int32_t rows,
    markov_mode mode, float output_multiplier, float soft_cap, int64_t *draft_tokens,
    int64_t tok_s0, uint16_t *logit_cache, int64_t cache_s0, int64_t cache_s1, void *stream) {
    const int V = vocab, r = rank, N = num_steps;
    if (V <= 0 || V % kTile != 0 || V > kMaxVocab) return MARKOV_EINVAL;
    if (r != 64 && r != 128 && r != 256) return MARKOV_EINVAL;
    if (N < 1 || N > kMaxSteps) return MARKOV_EINVAL;
    if (!base_logits || !head || !embed || !anchor_tokens || !temperature || !seeds ||
        !row_state_idx || !draft_tokens || !logit_cache)
        return MARKOV_EINVAL;
    if (rows < 1) return MARKOV_EINVAL;
    if (rows > kChainRows) return MARKOV_EUNSUPPORTED;          // one chain launch only
    if (mode != MARKOV_GUMBEL && mode != MARKOV_INVCDF) return MARKOV_EINVAL;
    if (base_s1 < V || base_s0 < (int64_t)(N - 1) * base_s1 + V) return MARKOV_EINVAL;
    if (cache_s1 < V || cache_s0 < (int64_t)(N - 1) * cache_s1 + V) return MARKOV_EINVAL;
    if (tok_s0 < N) return MARKOV_EINVAL;
    if ((reinterpret_cast<uintptr_t>(logit_cache) & 15u) || (cache_s0 * 2) % 16 ||
        (cache_s1 * 2) % 16)
        return MARKOV_EINVAL;
    if ((reinterpret_cast<uintptr_t>(head) & 15u) || (reinterpret_cast<uintptr_t>(embed) & 15u))
        return MARKOV_EINVAL;
    if (!(output_multiplier == output_multiplier) || output_multiplier - output_multiplier != 0.0f ||
        soft_cap != soft_cap)
        return MARKOV_EINVAL;
    // the static scratch bounds: the Gumbel noise of every row and position
    // (inverse-CDF calls draw none)
    if (mode == MARKOV_GUMBEL && (size_t)rows * N * V * sizeof(float) > kNoiseBytes)
        return MARKOV_EUNSUPPORTED;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MARKOV_EDEVICE;
    unsigned char *base = nullptr;
    int sms = 0, occ = 0;
    markov_status st = setup(dev, &base, &sms, &occ);
    if (st != MARKOV_OK) return st;
    if (occ < 1) return MARKOV_ENOTRESIDENT;
    int grid = (V / kTile) / (kChainThreads / 32);
    if (grid < 1) grid = 1;
    if (grid > sms * occ) grid = sms * occ;
    if ((grid + kKeyPad - 1) / kKeyPad * kKeyPad > kMaxGridPad) return MARKOV_EUNSUPPORTED;

    cudaStream_t s = (cudaStream_t)stream;
    uint32_t *ctrl = reinterpret_cast<uint32_t *>(base);
    // every call starts from cleared barrier counters and status
    if (cudaMemsetAsync(ctrl, 0, kCtrlBytes, s) != cudaSuccess) return MARKOV_ECUDA;

    SampleArgs a{};
    a.base = base_logits;
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
    a.tf.mult = output_multiplier;
    a.tf.has_cap = soft_cap > 0.0f;
    a.tf.cap = a.tf.has_cap ? soft_cap : 1.0f;
    a.tf.inv_cap = a.tf.has_cap ? 1.0f / a.tf.cap : 1.0f;
    a.tf.has_transform = (output_multiplier != 1.0f) || a.tf.has_cap;
    a.tokens = draft_tokens;
    a.tok_s0 = tok_s0;
    a.cache = logit_cache;
    a.cache_s0 = cache_s0;
    a.cache_s1 = cache_s1;
    a.keys = reinterpret_cast<uint64_t *>(base + kCtrlBytes);
    a.sums = reinterpret_cast<uint64_t *>(base + kCtrlBytes + kSlotBytes);
    a.noise = reinterpret_cast<float *>(base + kCtrlBytes + 2 * kSlotBytes);
    a.noise_s0 = V;
    a.bar_count = ctrl;
    a.bar_base = ctrl + 1;
    a.status = ctrl + 2;
    a.timeout_ns = 100ull * 1000000ull;
    a.grid = grid;
    if (mode == MARKOV_GUMBEL &&
        launch_noise(seeds, temperature, row_state_idx, rows, N, V, a.noise, a.noise_s0, 1, s) !=
            cudaSuccess) {
        cudaGetLastError();
        return MARKOV_ECUDA;
    }
    cudaError_t e = launch_chain(a, s);
    if (e == cudaErrorCooperativeLaunchTooLarge) { cudaGetLastError(); return MARKOV_ENOTRESIDENT; }
    if (e != cudaSuccess) { cudaGetLastError(); return MARKOV_ECUDA; }
    return MARKOV_OK;
}
