// common.cuh -- small device helpers shared by the DDTree kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#define DDT_DEV __device__ __forceinline__

namespace ddt {

constexpr float kLog2e = 1.4426950408889634f;

// Error word codes: high byte = kernel, low bytes = reason.  A kernel that
// meets inconsistent device-side data records a code with atomicCAS (first
// error wins) and skips the offending work; it never dereferences it.
enum : uint32_t {
    ERR_TOPK = 0x01000000u,
    ERR_BUILD = 0x02000000u,
    ERR_ATTN = 0x03000000u,
    ERR_ACCEPT = 0x04000000u,
    ERR_COMMIT = 0x05000000u,
    ERR_SELFTEST = 0x0F000000u,  // ddtree_selftest_wait
    ERR_BAD_PREFIX_LEN = 0x1,
    ERR_BAD_N_NODES = 0x2,
    ERR_BAD_TREE = 0x3,
    ERR_WAIT_TIMEOUT = 0x4,
    ERR_BAD_INPUT = 0x5,
    ERR_PLAN = 0x6,  // a launch plan the kernel cannot carry out (a library bug)
};

DDT_DEV void record_error(uint32_t* err, uint32_t code) {
    if (err) atomicCAS(err, 0u, code);
}

// ---------------------------------------------------------------------------
// Orderable keys: a float maps to a uint32 whose unsigned order is the float
// order (-0.0 is folded onto +0.0 first).  A (value, index) pair maps to a
// uint64 whose maximum is the largest value with the lowest index.
// ---------------------------------------------------------------------------
DDT_DEV uint32_t ord_from_bits(uint32_t b) {
    b = (b == 0x80000000u) ? 0u : b;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
DDT_DEV uint32_t ord_from_float(float f) { return ord_from_bits(__float_as_uint(f)); }
DDT_DEV float float_from_ord(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
DDT_DEV uint64_t value_index_key(float v, uint32_t idx) {
    return ((uint64_t)ord_from_float(v) << 32) | (uint64_t)(0xffffffffu - idx);
}
DDT_DEV float key_value(uint64_t k) { return float_from_ord((uint32_t)(k >> 32)); }
DDT_DEV uint32_t key_index(uint64_t k) { return 0xffffffffu - (uint32_t)k; }

// bf16 bits -> fp32 (exact)
DDT_DEV float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
DDT_DEV float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

DDT_DEV float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

DDT_DEV uint64_t shfl_xor_u64(uint64_t v, int m) {
    uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, m);
    uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), m);
    return ((uint64_t)hi << 32) | lo;
}
DDT_DEV uint64_t shfl_u64(uint64_t v, int src) {
    uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)v, src);
    uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(v >> 32), src);
    return ((uint64_t)hi << 32) | lo;
}
DDT_DEV uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }
DDT_DEV uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }

// Warp-wide bitonic sort of one uint64 per lane, descending (lane 0 = max).
DDT_DEV uint64_t warp_sort_desc(uint64_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            uint64_t o = shfl_xor_u64(v, j);
            bool keep_max = (((lane & k) == 0) == ((lane & j) == 0));
            v = keep_max ? umax64(v, o) : umin64(v, o);
        }
    }
    return v;
}

// Both a and b sorted descending across the warp; returns the 32 largest of
// their union, sorted descending.
DDT_DEV uint64_t warp_merge_desc(uint64_t a, uint64_t b) {
    const int lane = threadIdx.x & 31;
    uint64_t rb = shfl_u64(b, 31 - lane);
    uint64_t v = umax64(a, rb);  // bitonic
#pragma unroll
    for (int j = 16; j > 0; j >>= 1) {
        uint64_t o = shfl_xor_u64(v, j);
        v = ((lane & j) == 0) ? umax64(v, o) : umin64(v, o);
    }
    return v;
}

// 128-bit streaming global load that does not allocate in L1.
DDT_DEV uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Counter ticket for "last CTA finishes the reduction".  Call from one thread
// after the CTA's partial results are stored; returns true in exactly one CTA
// of the `expected` that share the counter, and that CTA resets it to zero.
// The release fence before and the acquire fence after make every other CTA's
// partials visible to the last one.
DDT_DEV bool ticket_is_last(unsigned int* counter, unsigned int expected) {
    __threadfence();
    unsigned int prev = atomicAdd(counter, 1u);
    bool last = (prev + 1u == expected);
    if (last) {
        __threadfence();
        *counter = 0u;
    }
    return last;
}

// Acquire / release accesses at GPU scope, for counters that hand partial
// results from one CTA to another.
DDT_DEV unsigned int ld_acquire_u32(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
DDT_DEV unsigned int atom_add_acq_rel_u32(unsigned int* p, unsigned int v) {
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
DDT_DEV unsigned int atom_or_acq_rel_u32(unsigned int* p, unsigned int v) {
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.or.b32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Two floats rounded to a bf16 pair (lo in the low half).
DDT_DEV uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// Packed fp32x2 arithmetic (two lanes per instruction on sm_100-class GPUs).
DDT_DEV float2 ffma2(float2 a, float b, float c) {
    unsigned long long A, B, C, R;
    asm("mov.b64 %0, {%1, %2};" : "=l"(A) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %1};" : "=l"(B) : "f"(b));
    asm("mov.b64 %0, {%1, %1};" : "=l"(C) : "f"(c));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(R) : "l"(A), "l"(B), "l"(C));
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(R));
    return r;
}
DDT_DEV float2 fadd2(float2 a, float2 b) {
    unsigned long long A, B, R;
    asm("mov.b64 %0, {%1, %2};" : "=l"(A) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(B) : "f"(b.x), "f"(b.y));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(R) : "l"(A), "l"(B));
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(R));
    return r;
}

// K-th largest (with multiplicity) of one uint32 per lane, K in [1, 32];
// warp-collective.  Small K: remove the maximum K-1 times (one reduction, one
// ballot each); larger K: a bitonic sort.
DDT_DEV uint32_t warp_kth_largest(uint32_t v, int K) {
    const int lane = threadIdx.x & 31;
    if (K <= 12) {
        for (int r = 1; r < K; ++r) {
            const uint32_t mx = __reduce_max_sync(0xffffffffu, v);
            const unsigned holders = __ballot_sync(0xffffffffu, v == mx);
            if (lane == __ffs(holders) - 1) v = 0u;
        }
        return __reduce_max_sync(0xffffffffu, v);
    }
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const uint32_t o = __shfl_xor_sync(0xffffffffu, v, j);
            const bool keep_max = (((lane & k) == 0) == ((lane & j) == 0));
            v = keep_max ? max(v, o) : min(v, o);
        }
    }
    return __shfl_sync(0xffffffffu, v, K - 1);
}

// Number of a[0..n) larger than x, for a rank by counting.  a is 16-byte
// aligned shared memory read by every thread of a warp at once (broadcast),
// two keys per load, eight loads in flight.
DDT_DEV int count_larger(const uint64_t* a, int n, uint64_t x) {
    const ulonglong2* a2 = reinterpret_cast<const ulonglong2*>(a);
    const int n2 = n >> 1;
    int r = 0;
#pragma unroll 8
    for (int j = 0; j < n2; ++j) {
        const ulonglong2 v = a2[j];
        r += (v.x > x ? 1 : 0) + (v.y > x ? 1 : 0);
    }
    if (n & 1) r += a[n - 1] > x ? 1 : 0;
    return r;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Kernels are launched so that they may start
// while the previous kernel on the stream is finishing: each one waits
// (pdl_wait) until every earlier kernel on the stream has completed and its
// writes are visible before it reads or writes any global memory, and lets its
// own successor be scheduled (pdl_trigger) only once its main work is done --
// a successor's CTAs waiting on an SM slow the kernel still running there.
// What overlaps is launch latency and CTA start-up, never data.
// ---------------------------------------------------------------------------
DDT_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
DDT_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launches `kernel` with programmatic dependent launch; cluster > 1 groups
// that many consecutive CTAs (along x) into one thread-block cluster.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                      size_t smem, cudaStream_t s, unsigned cluster,
                                      Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
    return launch_pdl_cluster(kernel, grid, block, smem, s, 1u, std::forward<Args>(args)...);
}

}  // namespace ddt
