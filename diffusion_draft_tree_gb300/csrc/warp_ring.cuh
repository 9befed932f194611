// warp_ring.cuh -- one warp's private ring of shared-memory stages for
// streaming a logit row segment by segment.  Lane 0 fills a stage with one
// bulk copy (cp.async.bulk, completing on the stage's own mbarrier) for the
// 16-byte-aligned body of the segment; the lanes load the few elements of an
// unaligned row or a ragged tail themselves; elements past the row's end read
// -inf.  A warp keeps several segments in flight this way without holding them
// in registers, and needs no CTA barrier: only __syncwarp between reading a
// stage and refilling it.
#pragma once

#include "common.cuh"
#include "sm100.cuh"

namespace ddt {

template <bool BF16, int SEG_BYTES, int STAGES>
struct WarpRing {
    static constexpr int ES = BF16 ? 2 : 4;        // element bytes
    static constexpr int VEC = 16 / ES;            // elements per 16-byte vector
    static constexpr int SIZE = SEG_BYTES / ES;    // elements per segment
    static constexpr int VPL = SEG_BYTES / 16 / 32;  // vectors per lane per segment
    static_assert(SEG_BYTES % 512 == 0, "whole vectors per lane");

    uint8_t* buf;   // STAGES x SEG_BYTES, 128-byte aligned, this warp's alone
    uint64_t* bar;  // STAGES mbarriers

    // Lane 0 initialises the barriers (count 1); the warp then may issue.
    DDT_DEV void init() {
        if ((threadIdx.x & 31) == 0) {
            for (int s = 0; s < STAGES; ++s) sm100::mbar_init(&bar[s], 1);
            sm100::mbar_init_fence();
        }
        __syncwarp();
    }

    // Starts filling stage s with elements [e0, e0 + SIZE) of the row at
    // `rowp`.  Every lane calls it, after the warp's last reads of the stage
    // (a __syncwarp in between); the stage may be read after wait().
    DDT_DEV void issue(int s, const char* rowp, int e0, int V, bool aligned) {
        const int lane = threadIdx.x & 31;
        uint8_t* dst = buf + s * SEG_BYTES;
        const int n_in = max(0, min(SIZE, V - e0));
        const int n_bulk = aligned ? (n_in / VEC) * VEC : 0;
        if (lane == 0) {
            sm100::fence_proxy_async_smem();  // the warp's earlier reads of the stage
            if (n_bulk > 0) {
                sm100::mbar_arrive_expect_tx(&bar[s], (uint32_t)(n_bulk * ES));
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                    " [%0], [%1], %2, [%3];" ::"r"(sm100::smem_u32(dst)),
                    "l"(rowp + (size_t)e0 * ES), "r"((uint32_t)(n_bulk * ES)),
                    "r"(sm100::smem_u32(&bar[s]))
                    : "memory");
            } else {
                sm100::mbar_arrive(&bar[s]);
            }
        }
        for (int i = n_bulk + lane; i < SIZE; i += 32) {
            if (BF16) {
                const unsigned short v = (i < n_in)
                    ? __ldg(reinterpret_cast<const unsigned short*>(rowp) + e0 + i)
                    : (unsigned short)0xff80u;
                reinterpret_cast<unsigned short*>(dst)[i] = v;
            } else {
                const unsigned int v = (i < n_in)
                    ? __ldg(reinterpret_cast<const unsigned int*>(rowp) + e0 + i)
                    : 0xff800000u;
                reinterpret_cast<unsigned int*>(dst)[i] = v;
            }
        }
    }

    // Waits (bounded) for the fill of stage s with the given phase parity;
    // warp-uniform result.  Every lane sees the whole stage afterwards.
    DDT_DEV bool wait(int s, uint32_t parity) {
        const bool ok = sm100::mbar_wait(&bar[s], parity, nullptr);
        __syncwarp();
        return __all_sync(0xffffffffu, ok) != 0;
    }

    // This lane's vectors of stage s: vector lane + 32 k is elements
    // [(lane + 32 k) VEC, ...) of the segment.
    DDT_DEV void read(int s, uint4 (&v)[VPL]) const {
        const uint4* p = reinterpret_cast<const uint4*>(buf + s * SEG_BYTES) + (threadIdx.x & 31);
#pragma unroll
        for (int k = 0; k < VPL; ++k) v[k] = p[32 * k];
    }
};

}  // namespace ddt
