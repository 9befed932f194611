// chunk.cuh -- one CTA's slice of a vocabulary-sized logit row, held in
// registers.  256 threads each own ITEMS 16-byte vectors; vector slot j of the
// chunk is (it * 256 + tid), so every load instruction of a warp touches 512
// contiguous bytes (fully coalesced).  Elements past the row's end read -inf.
#pragma once

#include "common.cuh"

namespace ddt {

template <bool BF16, int ITEMS>
struct RowChunk {
    static constexpr int THREADS = 256;
    static constexpr int ES = BF16 ? 2 : 4;          // element bytes
    static constexpr int VEC = 16 / ES;               // elements per vector
    static constexpr int SIZE = THREADS * ITEMS * VEC;  // elements per chunk

    uint32_t w[ITEMS][4];

    // Loads elements [c0, c0 + SIZE) of a row that starts at `rowp`.
    // `aligned`: the row start is 16-byte aligned (vector loads allowed).
    DDT_DEV void load(const char* __restrict__ rowp, int c0, int V, bool aligned) {
#pragma unroll
        for (int it = 0; it < ITEMS; ++it) {
            const int e0 = c0 + (it * THREADS + (int)threadIdx.x) * VEC;
            if (aligned && e0 + VEC <= V) {
                const uint4 r = ld_stream_v4(rowp + (size_t)e0 * ES);
                w[it][0] = r.x; w[it][1] = r.y; w[it][2] = r.z; w[it][3] = r.w;
            } else if (BF16) {
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const int e = e0 + 2 * p;
                    const uint32_t lo = (e < V) ? (uint32_t)__ldg((const unsigned short*)rowp + e)
                                                : 0xff80u;
                    const uint32_t hi = (e + 1 < V)
                                            ? (uint32_t)__ldg((const unsigned short*)rowp + e + 1)
                                            : 0xff80u;
                    w[it][p] = lo | (hi << 16);
                }
            } else {
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const int e = e0 + p;
                    w[it][p] = (e < V) ? __ldg((const unsigned int*)rowp + e) : 0xff800000u;
                }
            }
        }
    }

    DDT_DEV float elem(int it, int k) const {
        if (BF16) return (k & 1) ? bf16hi(w[it][k >> 1]) : bf16lo(w[it][k >> 1]);
        return __uint_as_float(w[it][k]);
    }

    DDT_DEV static int index(int c0, int it, int k) {
        return c0 + (it * THREADS + (int)threadIdx.x) * VEC + k;
    }

    // Largest element of this thread and its lowest index (-1 if the thread
    // holds no element of the row).
    DDT_DEV void thread_max(int c0, int V, float& vmax, int& vidx) const {
        vmax = -INFINITY;
        vidx = -1;
#pragma unroll
        for (int it = 0; it < ITEMS; ++it) {
#pragma unroll
            for (int k = 0; k < VEC; ++k) {
                const float x = elem(it, k);
                if (it == 0 && k == 0) {
                    const int e = index(c0, 0, 0);
                    if (e < V) { vmax = x; vidx = e; }
                } else if (x > vmax) {
                    vmax = x;
                    vidx = index(c0, it, k);
                }
            }
        }
    }

    // sum over this thread's elements of 2^((x - ref) * c); -inf elements add 0.
    DDT_DEV float thread_exp_sum(float ref, float c) const {
        float s = 0.f;
        const float off = -ref * c;
#pragma unroll
        for (int it = 0; it < ITEMS; ++it) {
#pragma unroll
            for (int k = 0; k < VEC; ++k) s += fast_exp2(fmaf(elem(it, k), c, off));
        }
        return s;
    }
};

DDT_DEV float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}
DDT_DEV float warp_max(float v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

}  // namespace ddt
