// topk.cu -- step 1 of a DDTree round: per-position log-softmax and top-K of
// the draft logits ("Accelerating Speculative Decoding with Block Diffusion
// Draft Trees", §3 marginals q_i; §4.3 log-probabilities; App. A restricted
// prefix set).
//
// One row = one (sequence, draft position), V logits.  A row is split into
// chunks of RowChunk::SIZE elements, one CTA per (chunk, row), so even a single
// sequence fills the GPU.  Each CTA streams its chunk once from HBM into
// registers and then computes, without touching memory again:
//   m_c = max, s_c = sum exp(x - m_c), and its K best (value, index) keys.
// Top-K selection avoids per-element insertion: every warp finds tau_w, the
// K-th largest of its 32 lane maxima (a warp bitonic sort), the CTA takes
// tau = max_w tau_w -- a lower bound on the chunk's K-th largest key -- and only
// elements with key >= tau (typically ~2K of 16K) are appended to a shared
// buffer that warp 0 sorts and merges.  The last CTA of a row (atomic ticket,
// no spinning) merges the chunk partials and writes the row's outputs.
#include "chunk.cuh"
#include "internal.h"

#include "../../include/ddtree.h"

namespace ddt {

namespace {

constexpr int kThreads = 256;
constexpr int kItems = 8;
constexpr int kCandCap = 1024;

struct TopkPartial {
    float m;   // chunk max
    float s;   // sum exp(x - m) over the chunk
    uint64_t keys[DDTREE_MAX_K];
};

template <bool BF16>
__global__ void __launch_bounds__(kThreads)
topk_kernel(const void* __restrict__ logits, int V, int64_t row_stride, int K, int nchunks,
            bool aligned, int32_t* __restrict__ topk_idx, float* __restrict__ topk_logp,
            float* __restrict__ lse, TopkPartial* __restrict__ parts,
            unsigned int* __restrict__ tickets) {
    using Chunk = RowChunk<BF16, kItems>;
    __shared__ uint64_t s_cand[kCandCap];
    __shared__ uint64_t s_sel[DDTREE_MAX_K];
    __shared__ float s_wmax[kThreads / 32], s_wsum[kThreads / 32];
    __shared__ uint64_t s_wtau[kThreads / 32];
    __shared__ int s_cnt;
    __shared__ bool s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int chunk = blockIdx.x, row = blockIdx.y;
    const int c0 = chunk * Chunk::SIZE;
    const char* rowp = (const char*)logits + (size_t)row * (size_t)row_stride * Chunk::ES;
    if (tid == 0) s_cnt = 0;

    Chunk x;
    x.load(rowp, c0, V, aligned);

    // ---- lane maxima, warp thresholds, CTA max ---------------------------
    float vmax;
    int vidx;
    x.thread_max(c0, V, vmax, vidx);
    const uint64_t lane_key = (vidx >= 0) ? value_index_key(vmax, (uint32_t)vidx) : 0ull;
    const uint64_t sorted = warp_sort_desc(lane_key);
    const uint64_t tau_w = shfl_u64(sorted, K - 1);
    const float wmax = warp_max(vmax);
    if (lane == 0) {
        s_wmax[warp] = wmax;
        s_wtau[warp] = tau_w;
    }
    __syncthreads();
    float m = s_wmax[0];
    uint64_t tau = s_wtau[0];
#pragma unroll
    for (int i = 1; i < kThreads / 32; ++i) {
        m = fmaxf(m, s_wmax[i]);
        tau = umax64(tau, s_wtau[i]);
    }

    // ---- sum of exponentials ------------------------------------------------
    const float ref = (m == -INFINITY) ? 0.f : m;
    const float ws = warp_sum(x.thread_exp_sum(ref, kLog2e));
    if (lane == 0) s_wsum[warp] = ws;

    // ---- candidates: keys >= tau ------------------------------------------
    if (lane_key != 0ull && lane_key >= tau) {
        const float tv = key_value(tau);
        const uint32_t ti = key_index(tau);
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
#pragma unroll
            for (int k = 0; k < Chunk::VEC; ++k) {
                const float v = x.elem(it, k);
                const int e = Chunk::index(c0, it, k);
                const bool cand = (tau == 0ull)
                                      ? (e < V)
                                      : (v > tv || (v == tv && (uint32_t)e <= ti));
                if (cand) {
                    const int pos = atomicAdd(&s_cnt, 1);
                    if (pos < kCandCap) s_cand[pos] = value_index_key(v, (uint32_t)e);
                }
            }
        }
    }
    __syncthreads();
    const int cnt = s_cnt;

    uint64_t best = 0ull;  // warp 0: the chunk's top keys, sorted, one per lane
    if (cnt <= kCandCap) {
        if (warp == 0) {
            for (int g = 0; g < cnt; g += 32) {
                const uint64_t v = (g + lane < cnt) ? s_cand[g + lane] : 0ull;
                best = warp_merge_desc(best, warp_sort_desc(v));
            }
        }
    } else {
        // Degenerate ties overflowed the buffer: exact K-round selection over
        // the registers (rare path; correctness only).
        uint64_t prev = ~0ull;
        for (int r = 0; r < K; ++r) {
            uint64_t tb = 0ull;
#pragma unroll
            for (int it = 0; it < kItems; ++it) {
#pragma unroll
                for (int k = 0; k < Chunk::VEC; ++k) {
                    const int e = Chunk::index(c0, it, k);
                    if (e < V) {
                        const uint64_t key = value_index_key(x.elem(it, k), (uint32_t)e);
                        if (key < prev && key > tb) tb = key;
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tb = umax64(tb, shfl_xor_u64(tb, o));
            if (lane == 0) s_cand[warp] = tb;
            __syncthreads();
            uint64_t cb = s_cand[0];
            for (int i = 1; i < kThreads / 32; ++i) cb = umax64(cb, s_cand[i]);
            if (tid == 0) s_sel[r] = cb;
            prev = cb;
            __syncthreads();
        }
        if (warp == 0) best = (lane < K) ? s_sel[lane] : 0ull;
    }

    if (warp != 0) return;

    float S = 0.f;
    if (lane == 0) {
        for (int i = 0; i < kThreads / 32; ++i) S += s_wsum[i];
    }
    S = __shfl_sync(0xffffffffu, S, 0);
    float M = ref;

    if (nchunks > 1) {
        TopkPartial* p = parts + (size_t)row * nchunks + chunk;
        if (lane < K) p->keys[lane] = best;
        if (lane == 0) {
            p->m = m;
            p->s = S;
        }
        __threadfence();
        __syncwarp();
        bool last = false;
        if (lane == 0) last = ticket_is_last(&tickets[row], (unsigned)nchunks);
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last) return;
        // ---- last CTA of the row: merge the chunk partials -----------------
        const TopkPartial* rp = parts + (size_t)row * nchunks;
        best = 0ull;
        float mm = -INFINITY;
        for (int c = lane; c < nchunks; c += 32) mm = fmaxf(mm, __ldcg(&rp[c].m));
        mm = warp_max(mm);
        M = (mm == -INFINITY) ? 0.f : mm;
        float ss = 0.f;
        for (int c = lane; c < nchunks; c += 32)
            ss += __ldcg(&rp[c].s) * fast_exp2((__ldcg(&rp[c].m) - M) * kLog2e);
        S = warp_sum(ss);
        for (int c = 0; c < nchunks; ++c) {
            const uint64_t v = (lane < K) ? __ldcg((const unsigned long long*)&rp[c].keys[lane])
                                          : 0ull;
            best = warp_merge_desc(best, v);
        }
    }
    const float logS = logf(S);
    if (lane < K) {
        const float v = key_value(best);
        topk_idx[(size_t)row * K + lane] = (int32_t)key_index(best);
        topk_logp[(size_t)row * K + lane] = (v - M) - logS;
    }
    if (lane == 0 && lse) lse[row] = M + logS;
}

}  // namespace

int topk_chunks(int V, int dtype) {
    const int size = dtype == DDTREE_BF16 ? RowChunk<true, kItems>::SIZE
                                          : RowChunk<false, kItems>::SIZE;
    return (V + size - 1) / size;
}

size_t topk_workspace_bytes(int rows, int V, int dtype) {
    const int nch = topk_chunks(V, dtype);
    if (nch <= 1) return 0;
    return align_up((size_t)rows * sizeof(unsigned int), 256) +
           (size_t)rows * nch * sizeof(TopkPartial);
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s) {
    const int nch = topk_chunks(a.V, a.dtype);
    const int es = a.dtype == DDTREE_BF16 ? 2 : 4;
    const bool aligned = ((uintptr_t)a.logits % 16 == 0) && ((a.row_stride * es) % 16 == 0);
    unsigned int* tickets = nullptr;
    TopkPartial* parts = nullptr;
    if (nch > 1) {
        tickets = (unsigned int*)a.ws;
        parts = (TopkPartial*)((char*)a.ws + align_up((size_t)a.rows * sizeof(unsigned int), 256));
    }
    dim3 grid(nch, a.rows);
    if (a.dtype == DDTREE_BF16)
        topk_kernel<true><<<grid, kThreads, 0, s>>>(a.logits, a.V, a.row_stride, a.K, nch, aligned,
                                                     a.topk_idx, a.topk_logp, a.lse, parts,
                                                     tickets);
    else
        topk_kernel<false><<<grid, kThreads, 0, s>>>(a.logits, a.V, a.row_stride, a.K, nch,
                                                      aligned, a.topk_idx, a.topk_logp, a.lse,
                                                      parts, tickets);
    return cudaGetLastError();
}

}  // namespace ddt
