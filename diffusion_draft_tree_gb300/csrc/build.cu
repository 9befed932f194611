// build.cu -- step 2 of a DDTree round: the best-first heap ("Accelerating
// Speculative Decoding with Block Diffusion Draft Trees", §4.2: the optimal
// valid tree under the surrogate is the set of the N most probable prefixes;
// §4.3 / App. A: pop the best candidate N times, after each pop offer the
// popped prefix's next sibling and its best child).
//
// One CTA per sequence.  Warp 0 runs the heap: the frontier is a set of 64-bit
// keys spread over the lanes' registers (S slots per lane), so a pop is two
// redux.sync max reductions instead of a sift through memory.  A key packs
//   [63:32] orderable fp32 score   (larger = more probable)
//   [31:27] 31 - depth             (shallower first on equal scores)
//   [26:16] 2047 - parent id       (earlier parent first)
//   [15:10] 63 - rank              (lower rank first)
// so the largest key is the next prefix in the heap's total order and node ids
// come out canonical.  A popped slot is reused by the popped prefix's child;
// siblings are appended round-robin over the lanes.  After the loop the whole
// CTA writes the node arrays and the ancestor-only bitmask in parallel.
#include "common.cuh"
#include "internal.h"

#include "../../include/ddtree.h"

namespace ddt {

namespace {

constexpr int kThreads = 128;

DDT_DEV uint64_t make_key(float score, int depth, int parent, int rank) {
    const uint32_t tie = ((uint32_t)(31 - depth) << 27) | ((uint32_t)(2047 - parent) << 16) |
                         ((uint32_t)(63 - rank) << 10);
    return ((uint64_t)ord_from_float(score) << 32) | tie;
}

template <int S>
__global__ void __launch_bounds__(kThreads)
build_kernel(const float* __restrict__ topk_logp, const int32_t* __restrict__ topk_idx,
             const int32_t* __restrict__ bonus, const int32_t* __restrict__ prefix_len, int L,
             int K, int N, int32_t* __restrict__ parent, int32_t* __restrict__ depth,
             int32_t* __restrict__ rank, int32_t* __restrict__ token, int32_t* __restrict__ pos_id,
             float* __restrict__ score, int32_t* __restrict__ child_count,
             uint32_t* __restrict__ anc_mask, int32_t* __restrict__ n_nodes, uint32_t* err) {
    __shared__ float s_lp[DDTREE_MAX_L * DDTREE_MAX_K];
    __shared__ int s_tok[DDTREE_MAX_L * DDTREE_MAX_K];
    __shared__ int s_par[DDTREE_MAX_N + 1];
    __shared__ int s_dep[DDTREE_MAX_N + 1];
    __shared__ int s_rank[DDTREE_MAX_N + 1];
    __shared__ float s_score[DDTREE_MAX_N + 1];
    __shared__ int s_cc[DDTREE_MAX_N + 1];
    __shared__ int s_n;

    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
    const int LK = L * K;
    pdl_wait();
    for (int i = tid; i < LK; i += kThreads) {
        s_lp[i] = topk_logp[(size_t)b * LK + i];
        s_tok[i] = topk_idx[(size_t)b * LK + i];
    }
    for (int i = tid; i <= N; i += kThreads) s_cc[i] = 0;
    if (tid == 0) {
        s_par[0] = -1; s_dep[0] = 0; s_rank[0] = -1; s_score[0] = 0.f;
    }
    __syncthreads();

    if (tid < 32) {
        uint64_t slot[S];
#pragma unroll
        for (int i = 0; i < S; ++i) slot[i] = 0ull;
        uint64_t best = 0ull;
        int best_i = 0;
        if (N > 0 && lane == 0) {
            slot[0] = make_key(__fadd_rn(0.f, s_lp[0]), 1, 0, 0);
            best = slot[0];
        }
        int n = 0, sib_pos = 1;
        while (n < N) {
            const uint32_t bh = (uint32_t)(best >> 32), bl = (uint32_t)best;
            const uint32_t mh = __reduce_max_sync(0xffffffffu, bh);
            const uint32_t ml = __reduce_max_sync(0xffffffffu, bh == mh ? bl : 0u);
            if (mh == 0u && ml == 0u) break;  // frontier exhausted
            const int winner = __ffs(__ballot_sync(0xffffffffu, bh == mh && bl == ml)) - 1;
            const float sc = float_from_ord(mh);
            const int dp = 31 - (int)(ml >> 27);
            const int pa = 2047 - (int)((ml >> 16) & 0x7ffu);
            const int rk = 63 - (int)((ml >> 10) & 0x3fu);
            const int id = ++n;
            if (lane == 0) {
                s_par[id] = pa; s_dep[id] = dp; s_rank[id] = rk; s_score[id] = sc;
            }
            const uint64_t child = (dp < L) ? make_key(__fadd_rn(sc, s_lp[dp * K]), dp + 1, id, 0)
                                            : 0ull;
            const uint64_t sib = (rk + 1 < K)
                                     ? make_key(__fadd_rn(s_score[pa], s_lp[(dp - 1) * K + rk + 1]),
                                                dp, pa, rk + 1)
                                     : 0ull;
            if (lane == winner) {
#pragma unroll
                for (int i = 0; i < S; ++i)
                    if (i == best_i) slot[i] = child;
                best = 0ull;
#pragma unroll
                for (int i = 0; i < S; ++i)
                    if (slot[i] > best) { best = slot[i]; best_i = i; }
            }
            if (sib != 0ull) {
                const int p = sib_pos++;
                if (lane == (p & 31)) {
                    const int si = p >> 5;
#pragma unroll
                    for (int i = 0; i < S; ++i)
                        if (i == si) slot[i] = sib;
                    if (sib > best) { best = sib; best_i = si; }
                }
            }
            __syncwarp();
        }
        if (lane == 0) s_n = n;
    }
    __syncthreads();
    const int n = s_n;
    for (int c = 1 + tid; c <= n; c += kThreads) atomicAdd(&s_cc[s_par[c]], 1);
    __syncthreads();

    pdl_trigger();
    const int R = N + 1, W = (N + 1 + 31) / 32;
    const int P = prefix_len[b];
    for (int u = tid; u < R; u += kThreads) {
        const size_t o = (size_t)b * R + u;
        if (u <= n) {
            parent[o] = s_par[u];
            depth[o] = s_dep[u];
            rank[o] = s_rank[u];
            token[o] = (u == 0) ? bonus[b] : s_tok[(s_dep[u] - 1) * K + s_rank[u]];
            pos_id[o] = P + s_dep[u];
            score[o] = s_score[u];
            child_count[o] = s_cc[u];
        } else {
            parent[o] = -1; depth[o] = -1; rank[o] = -1; token[o] = -1; pos_id[o] = -1;
            score[o] = -INFINITY;
            child_count[o] = 0;
        }
    }
    // ancestor-only mask: word w of row u collects the bits of u's root path
    // that fall in [32w, 32w+32).
    for (int i = tid; i < R * W; i += kThreads) {
        const int u = i / W, w = i - u * W;
        uint32_t word = 0u;
        if (u <= n) {
            for (int a = u; a >= 0; a = s_par[a])
                if ((a >> 5) == w) word |= 1u << (a & 31);
        }
        anc_mask[(size_t)b * R * W + i] = word;
    }
    if (tid == 0) n_nodes[b] = n;
}

template <int S>
cudaError_t launch_s(const BuildArgs& a, cudaStream_t s) {
    return launch_pdl(build_kernel<S>, dim3(a.B), dim3(kThreads), 0, s, a.topk_logp, a.topk_idx,
                      a.bonus, a.prefix_len, a.L, a.K, a.N, a.parent, a.depth, a.rank, a.token,
                      a.pos_id, a.score, a.child_count, a.anc_mask, a.n_nodes, a.err);
}

}  // namespace

cudaError_t launch_build(const BuildArgs& a, cudaStream_t s) {
    // slots per lane: sibling positions run 0..N, position p lives in slot p / 32
    const int need = (a.N >> 5) + 1;
    if (need <= 1) return launch_s<1>(a, s);
    if (need <= 2) return launch_s<2>(a, s);
    if (need <= 3) return launch_s<3>(a, s);
    if (need <= 5) return launch_s<5>(a, s);
    if (need <= 9) return launch_s<9>(a, s);
    if (need <= 17) return launch_s<17>(a, s);
    return launch_s<33>(a, s);
}

}  // namespace ddt
