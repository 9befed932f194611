// chunk.cuh -- one CTA's slice of a vocabulary-sized logit row, staged in
// shared memory.  Thread 0 issues one bulk copy (cp.async.bulk, completing on
// an mbarrier) for the 16-byte-aligned body of the slice; the few elements of
// an unaligned row or of a ragged tail are loaded by the threads themselves.
// Elements past the row's end read -inf.  Every thread then reads the slice
// from shared memory as 16-byte vectors.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "sm100.cuh"

namespace ddt {

template <bool BF16, int SIZE_>
struct SmemChunk {
    static constexpr int THREADS = 256;
    static constexpr int SIZE = SIZE_;          // elements per chunk
    static constexpr int ES = BF16 ? 2 : 4;     // element bytes
    static constexpr int VEC = 16 / ES;         // elements per 16-byte vector
    static constexpr int NVEC = SIZE / VEC;     // vectors per chunk
    static constexpr int BYTES = SIZE * ES;
    static_assert(NVEC % THREADS == 0, "whole vectors per thread");

    // Starts staging elements [c0, c0 + SIZE) of the row at `rowp` into `buf`
    // (16-byte aligned, BYTES long).  All threads call it; the data may be used
    // only after wait().  A CTA that issues must wait before it exits.
    DDT_DEV static void issue(uint8_t* buf, uint64_t* bar, const char* rowp, int c0, int V,
                              bool aligned) {
        const int n_in = max(0, min(SIZE, V - c0));             // elements of the row
        const int n_bulk = aligned ? (n_in / VEC) * VEC : 0;    // by the copy engine
        if (threadIdx.x == 0) {
            sm100::mbar_init(bar, 1);
            sm100::mbar_init_fence();
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            if (n_bulk > 0) {
                sm100::mbar_arrive_expect_tx(bar, (uint32_t)(n_bulk * ES));
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                    " [%0], [%1], %2, [%3];" ::"r"(sm100::smem_u32(buf)),
                    "l"(rowp + (size_t)c0 * ES), "r"((uint32_t)(n_bulk * ES)),
                    "r"(sm100::smem_u32(bar))
                    : "memory");
            } else {
                sm100::mbar_arrive(bar);
            }
        }
        for (int i = n_bulk + (int)threadIdx.x; i < SIZE; i += THREADS) {
            if (BF16) {
                const unsigned short v =
                    (i < n_in) ? __ldg((const unsigned short*)rowp + c0 + i) : (unsigned short)0xff80u;
                ((unsigned short*)buf)[i] = v;
            } else {
                const unsigned int v = (i < n_in) ? __ldg((const unsigned int*)rowp + c0 + i)
                                                  : 0xff800000u;
                ((unsigned int*)buf)[i] = v;
            }
        }
    }

    // Waits (bounded) for the staged chunk; returns, uniformly across the CTA,
    // whether it arrived.  Every thread sees the whole chunk afterwards.
    DDT_DEV static bool wait(uint64_t* bar) {
        const bool ok = sm100::mbar_wait(bar, 0, nullptr);
        return __syncthreads_and(ok) != 0;
    }

    // For a ring of stages whose mbarriers (count 1) were initialised once:
    // starts staging the chunk into `buf`, completing on `bar`'s next phase.
    // All threads call it; they fill the unaligned tail themselves, so the
    // stage may be read only after wait() and a CTA barrier.
    DDT_DEV static void issue_ring(uint8_t* buf, uint64_t* bar, const char* rowp, int c0, int V,
                                   bool aligned) {
        const int n_in = max(0, min(SIZE, V - c0));
        const int n_bulk = aligned ? (n_in / VEC) * VEC : 0;
        if (threadIdx.x == 0) {
            sm100::fence_proxy_async_smem();  // earlier generic reads of the stage
            if (n_bulk > 0) {
                sm100::mbar_arrive_expect_tx(bar, (uint32_t)(n_bulk * ES));
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                    " [%0], [%1], %2, [%3];" ::"r"(sm100::smem_u32(buf)),
                    "l"(rowp + (size_t)c0 * ES), "r"((uint32_t)(n_bulk * ES)),
                    "r"(sm100::smem_u32(bar))
                    : "memory");
            } else {
                sm100::mbar_arrive(bar);
            }
        }
        for (int i = n_bulk + (int)threadIdx.x; i < SIZE; i += THREADS) {
            if (BF16) {
                const unsigned short v =
                    (i < n_in) ? __ldg((const unsigned short*)rowp + c0 + i) : (unsigned short)0xff80u;
                ((unsigned short*)buf)[i] = v;
            } else {
                const unsigned int v = (i < n_in) ? __ldg((const unsigned int*)rowp + c0 + i)
                                                  : 0xff800000u;
                ((unsigned int*)buf)[i] = v;
            }
        }
    }

    // Waits (bounded) for the given phase of a ring stage; CTA-uniform result.
    DDT_DEV static bool wait_ring(uint64_t* bar, uint32_t parity) {
        const bool ok = sm100::mbar_wait(bar, parity, nullptr);
        return __syncthreads_and(ok) != 0;
    }

    DDT_DEV static bool load(uint8_t* buf, uint64_t* bar, const char* rowp, int c0, int V,
                             bool aligned) {
        issue(buf, bar, rowp, c0, V, aligned);
        return wait(bar);
    }

    // Vector v of the chunk as 8 (bf16) or 4 (fp32) floats.
    DDT_DEV static void unpack(const uint4& w, float (&x)[VEC]) {
        if (BF16) {
            const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                x[2 * p] = bf16lo(a[p]);
                x[2 * p + 1] = bf16hi(a[p]);
            }
        } else {
            x[0] = __uint_as_float(w.x);
            x[1] = __uint_as_float(w.y);
            x[2] = __uint_as_float(w.z);
            x[3] = __uint_as_float(w.w);
        }
    }

    // a0 + a1 += 2^(x c + off) over the vector's elements (two sums, so that
    // the additions form two independent chains).
    DDT_DEV static void exp_sum(const uint4& w, float c, float off, float& a0, float& a1) {
        const uint32_t a[4] = {w.x, w.y, w.z, w.w};
        if (BF16) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                a0 += fast_exp2(fmaf(bf16lo(a[p]), c, off));
                a1 += fast_exp2(fmaf(bf16hi(a[p]), c, off));
            }
        } else {
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                a0 += fast_exp2(fmaf(__uint_as_float(a[2 * p]), c, off));
                a1 += fast_exp2(fmaf(__uint_as_float(a[2 * p + 1]), c, off));
            }
        }
    }

    // Largest element of a vector (bf16: packed max, two elements per op).
    DDT_DEV static float vmax(const uint4& w) {
        if (BF16) {
            const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&w.x);
            const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w.y);
            const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&w.z);
            const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&w.w);
            const __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
            return fmaxf(__low2float(m), __high2float(m));
        }
        return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)),
                     fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
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
