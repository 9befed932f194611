// sampling.cuh -- the target's temperature-T decoding rule, shared by the
// full-tree and path-only accept kernels: one Philox4x64-10 uniform per node
// and a block scan for the inverse-CDF rescan of one vocabulary chunk.
#pragma once

#include "common.cuh"

namespace ddt {

constexpr int kSampleThreads = 256;

// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two 64x64
// multiplies with the Weyl key schedule.
DDT_DEV void philox4x64_10(uint64_t c[4], uint64_t k0, uint64_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t lo0 = 0xD2E7470EE14C6C93ull * c[0], hi0 = __umul64hi(0xD2E7470EE14C6C93ull, c[0]);
        const uint64_t lo1 = 0xCA5A826395121157ull * c[2], hi1 = __umul64hi(0xCA5A826395121157ull, c[2]);
        const uint64_t x0 = hi1 ^ c[1] ^ k0, x2 = hi0 ^ c[3] ^ k1;
        c[0] = x0; c[1] = lo1; c[2] = x2; c[3] = lo0;
        k0 += 0x9E3779B97F4A7C15ull;
        k1 += 0xBB67AE8584CAA73Bull;
    }
}

DDT_DEV float node_uniform(uint64_t seed, uint64_t step, uint64_t seq, uint64_t node) {
    uint64_t c[4] = {seq, node, 0ull, 0ull};
    philox4x64_10(c, seed, step);
    return (float)(c[0] >> 40) * (1.0f / 16777216.0f);
}

// Block-wide exclusive scan of one float per thread (kSampleThreads); also returns
// the block total.  Fixed shuffle/shared-memory tree: deterministic.
DDT_DEV float block_exclusive_scan(float v, float* s_warp, float& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    float before = 0.f, tot = 0.f;
#pragma unroll
    for (int i = 0; i < kSampleThreads / 32; ++i) {
        const float wv = s_warp[i];
        if (i < warp) before += wv;
        tot += wv;
    }
    total = tot;
    __syncthreads();
    return before + incl - v;
}

}  // namespace ddt
