// mma_tile.cuh -- the mma.sync bias tile of the simple and the sharded
// chains: [16 vocab ids x 8 rows] of head . embed (sharded_markov page,
// module docstring: up to 8 request rows are the columns of the tensor-core
// MMA), BF16 operands, fp32 sums.
#pragma once
#include <cstdint>

namespace dtm {

constexpr int kEPad = 32;   // BF16 elements of padding per staged embed row

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint64_t warp_max_u64_shfl(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

// Bias [16 ids x 8 rows] of tile v0 by mma.m16n8k16.  The reduction index k
// is permuted identically in A and B (a dot product does not depend on the
// order of its terms' pairing): thread (g, t) reads 8 consecutive head
// elements [8t + 32j, +8) of rows v0+g and v0+g+8 with one 16-byte load each
// and the same 8 embed elements of row g; words 0/1 feed the k-step 2j,
// words 2/3 the k-step 2j+1.
template <int RANK>
__device__ __forceinline__ void bias_tile(const uint16_t *__restrict__ head, int v0,
                                          const uint16_t *e_smem, int g, int t, float (&acc)[4]) {
    acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
    const uint16_t *ha = head + (int64_t)(v0 + g) * RANK + 8 * t;
    const uint16_t *hb = ha + 8 * RANK;
    const uint16_t *eb = e_smem + g * (RANK + kEPad) + 8 * t;
#pragma unroll
    for (int j = 0; j < RANK / 32; ++j) {
        uint4 a = ldg_nc_v4(ha + 32 * j);
        uint4 b = ldg_nc_v4(hb + 32 * j);
        uint4 e = *reinterpret_cast<const uint4 *>(eb + 32 * j);
        mma_bf16_16816(acc, a.x, b.x, a.y, b.y, e.x, e.y);
        mma_bf16_16816(acc, a.z, b.z, a.w, b.w, e.z, e.w);
    }
}

}  // namespace dtm
