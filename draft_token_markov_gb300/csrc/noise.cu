// noise.cu -- counter-based Gumbel noise, and the device-math probe kernel.
//
// The noise of (row b, position i, vocab id v) is -log(-log u) with u the top
// 23 bits of splitmix64(h_bi ^ v), h_bi = sm(sm(sm(seed_b) ^ b) ^ i).  It
// depends on the seeds and positions only, never on the chain, so it can be
// drawn on a side stream before the chain runs (sharded_markov page,
// fork_noise and _shard_noise_kernel).  The kernel is ALU bound: one 64-bit
// hash and two logarithms per element; each thread makes 4 consecutive ids
// and stores them as one 16-byte vector.  A vocabulary shard's noise is the
// same hash of the global id (v_offset + the shard's column).
#include "common.cuh"
#include "gumbel_bounds.cuh"

namespace dtm {

constexpr int kNoiseThreads = 256;
constexpr int kNoisePerThread = 4;

__global__ void __launch_bounds__(kNoiseThreads)
noise_kernel(const int64_t *__restrict__ seeds, const float *__restrict__ temperature,
             const int64_t *__restrict__ row_state_idx, int N, int V, float *__restrict__ out,
             int64_t out_s0, int v_offset) {
    const int sample = blockIdx.y;          // b * N + i
    const int b = sample / N;
    const int i = sample - b * N;
    if (row_state_idx[b] < 0 || !samples(temperature[b])) return;
    const uint64_t hri = dm_row_step_hash((uint64_t)seeds[b], (uint32_t)b, (uint32_t)i);
    float *dst = out + (int64_t)sample * out_s0;
    const int stride = gridDim.x * kNoiseThreads * kNoisePerThread;
    for (int v0 = (blockIdx.x * kNoiseThreads + threadIdx.x) * kNoisePerThread; v0 < V;
         v0 += stride) {
        float g[kNoisePerThread];
#pragma unroll
        for (int j = 0; j < kNoisePerThread; ++j) g[j] = dm_gumbel(hri, (uint32_t)(v_offset + v0 + j));
        if (v0 + kNoisePerThread <= V && ((reinterpret_cast<uintptr_t>(dst + v0) & 15u) == 0u)) {
            *reinterpret_cast<float4 *>(dst + v0) = make_float4(g[0], g[1], g[2], g[3]);
        } else {
            for (int j = 0; j < kNoisePerThread && v0 + j < V; ++j) dst[v0 + j] = g[j];
        }
    }
}

cudaError_t launch_noise(const int64_t *seeds, const float *temperature,
                         const int64_t *row_state_idx, int rows, int N, int V, float *out,
                         int64_t out_s0, int /*mode_gumbel_only*/, cudaStream_t stream, int v_offset) {
    int per_block = kNoiseThreads * kNoisePerThread;
    int bx = (V + per_block - 1) / per_block;
    if (bx > 65535) bx = 65535;
    dim3 grid(bx, rows * N);
    noise_kernel<<<grid, kNoiseThreads, 0, stream>>>(seeds, temperature, row_state_idx, N, V,
                                                      out, out_s0, v_offset);
    return cudaGetLastError();
}

__global__ void device_math_kernel(int fn, const float *__restrict__ x, float *__restrict__ y,
                                   int64_t n) {
    if (fn == 9) {
        // Gumbel key bounds on triples (l, T, uniform mantissa m as bits):
        // the key's lower bound, its upper bound (from m's noise byte and
        // the rounded 1 / T, as the chain computes them) and the exact key
        for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; 3 * t + 2 < n;
             t += (int64_t)gridDim.x * blockDim.x) {
            const float l = x[3 * t], T = x[3 * t + 1];
            const uint64_t h = (uint64_t)(__float_as_uint(x[3 * t + 2]) & 0x7fffffu) << 41;
            const uint32_t q = quantize_upper(gumbel_upper(h));
            const float invT = __fdiv_rn(1.0f, T);
            y[3 * t] = key_lower(l, invT, q);
            y[3 * t + 1] = key_upper(l, invT, q);
            y[3 * t + 2] = exact_key(l, T, h);
        }
        return;
    }
    if (fn == 12) {
        // pairs (x, T): fp32(x / T) as the inverse-CDF kernels take it, and
        // whether T took the power-of-two product
        for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; 2 * t + 1 < n;
             t += (int64_t)gridDim.x * blockDim.x) {
            const float v = x[2 * t], T = x[2 * t + 1];
            const bool p2 = dm_pow2_temperature(T);
            y[2 * t] = p2 ? dm_div_T<true>(v, T, __frcp_rn(T)) : dm_div_T<false>(v, T, 0.0f);
            y[2 * t + 1] = p2 ? 1.0f : 0.0f;
        }
        return;
    }
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
         j += (int64_t)gridDim.x * blockDim.x) {
        float v = x[j];
        float r;
        switch (fn) {
            case 6:
                // the noise byte of the uniform mantissa m (x holds m's bits)
                r = (float)quantize_upper(gumbel_upper((uint64_t)(__float_as_uint(v) & 0x7fffffu) << 41));
                break;
            case 10: r = __uint_as_float((uint32_t)dm_cdf_weight(v)); break;
            case 11: r = __uint_as_float((uint32_t)(dm_cdf_weight(v) >> 32)); break;
            case 7: r = dequantize_upper((uint32_t)v); break;
            case 8: r = dequantize_lower((uint32_t)v); break;
            case 0: r = dm_log(v); break;
            case 1: r = dm_exp(v); break;
            case 2: r = dm_tanh(v); break;
            case 3: r = -dm_log(-dm_log(v)); break;
            case 4: r = __uint_as_float(dm_bf16_bits(v)); break;
            default: {
                // the packed conversion of the tcgen05 epilogue: both halves
                // must agree (0xDEAD, not a NaN, flags a disagreement)
                const uint32_t p = bf16x2_rn(v, v);
                r = __uint_as_float((p & 0xffffu) == (p >> 16) ? (p & 0xffffu) : 0xDEADu);
                break;
            }
        }
        y[j] = r;
    }
}

cudaError_t launch_device_math(int fn, const float *x, float *y, int64_t n, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 65536) blocks = 65536;
    device_math_kernel<<<(unsigned)blocks, 256, 0, s>>>(fn, x, y, n);
    return cudaGetLastError();
}

}  // namespace dtm
