// segment.cuh -- arithmetic on the 16-byte vectors of a logit segment
// (8 bf16 or 4 fp32 logits each), shared by the streaming kernels.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace ddt {

template <bool BF16, int SEG_BYTES = 4096>
struct Seg {
    static constexpr int ES = BF16 ? 2 : 4;
    static constexpr int VEC = 16 / ES;              // elements per vector
    static constexpr int SIZE = SEG_BYTES / ES;      // elements per segment
    static constexpr uint32_t NEG_INF = BF16 ? 0xff80u : 0xff800000u;

    // element k of a vector (k a compile-time constant in every caller)
    DDT_DEV static float elem(const uint4& w, int k) {
        const uint32_t a[4] = {w.x, w.y, w.z, w.w};
        if (BF16) return (k & 1) ? bf16hi(a[k >> 1]) : bf16lo(a[k >> 1]);
        return __uint_as_float(a[k]);
    }
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
    // element k of a vector, k known only at run time
    DDT_DEV static float elem_dyn(const uint4& w, int k) {
        if (BF16) {
            const uint32_t h = (k < 4) ? ((k < 2) ? w.x : w.y) : ((k < 6) ? w.z : w.w);
            return (k & 1) ? bf16hi(h) : bf16lo(h);
        }
        return __uint_as_float((k < 2) ? ((k == 0) ? w.x : w.y) : ((k == 2) ? w.z : w.w));
    }
    // bit k set where element k >= t (t a value of the element type, so that the
    // bf16 comparison is exact; NaN compares false)
    DDT_DEV static unsigned ge_mask(const uint4& w, float t) {
        if (BF16) {
            const __nv_bfloat162 t2 = __bfloat162bfloat162(__float2bfloat16_rn(t));
            const uint32_t a[4] = {w.x, w.y, w.z, w.w};
            unsigned m = 0u;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const unsigned h = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&a[p]), t2);
                m |= ((h & 1u) | ((h >> 15) & 2u)) << (2 * p);
            }
            return m;
        }
        return (__uint_as_float(w.x) >= t ? 1u : 0u) | (__uint_as_float(w.y) >= t ? 2u : 0u) |
               (__uint_as_float(w.z) >= t ? 4u : 0u) | (__uint_as_float(w.w) >= t ? 8u : 0u);
    }
    // acc += 2^(x c + off) over the vector's elements, two lanes per fp32x2
    // instruction (acc.x and acc.y are two independent partial sums)
    DDT_DEV static void exp_sum2(const uint4& w, float c, float off, float2& acc) {
        const uint32_t a[4] = {w.x, w.y, w.z, w.w};
        if (BF16) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float2 y = ffma2(make_float2(bf16lo(a[p]), bf16hi(a[p])), c, off);
                acc = fadd2(acc, make_float2(fast_exp2(y.x), fast_exp2(y.y)));
            }
        } else {
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                const float2 y =
                    ffma2(make_float2(__uint_as_float(a[2 * p]), __uint_as_float(a[2 * p + 1])), c, off);
                acc = fadd2(acc, make_float2(fast_exp2(y.x), fast_exp2(y.y)));
            }
        }
    }
};

}  // namespace ddt
