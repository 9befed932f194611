// commit.cu -- after the walk: the accepted path joins the KV cache
// ("Accelerating Speculative Decoding with Block Diffusion Draft Trees", §3 and
// §4.1: the bonus token that rooted the tree and the accepted tokens are
// verified, so they become part of the prefix the next round attends to).
//
// One CTA per sequence.  The path rows are node 0 (the root) followed by the
// a = accept_len accepted nodes; row i of the path holds its tokens' keys and
// values for every KV head in the tree K/V and moves to cache position P + i
// (its depth is i, and tree keys were computed at position P + depth).  The
// CTA reads P and the path once, copies (a+1) x Hkv rows of D bf16 for K and
// V with 16-byte accesses, then advances prefix_len[b] to P + a + 1 -- in
// place, which is safe because only this CTA touches sequence b.  HBM-bound;
// algorithmic bytes per sequence 8 (a+1) Hkv D (K and V, read and written).
#include "common.cuh"
#include "internal.h"

#include "../../include/ddtree.h"

namespace ddt {

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
commit_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int64_t cache_cap,
              const uint4* __restrict__ k_tree, const uint4* __restrict__ v_tree,
              const int32_t* __restrict__ accept_len, const int32_t* __restrict__ accepted_nodes,
              int32_t* __restrict__ prefix_len, int L, int N, int Hkv, int D, uint32_t* err) {
    __shared__ int s_rows[DDTREE_MAX_L + 1];
    __shared__ int s_ok;
    __shared__ int64_t s_P;
    __shared__ int s_a;
    const int b = blockIdx.x, tid = threadIdx.x;
    pdl_wait();
    if (tid == 0) {
        const int64_t P = prefix_len[b];
        const int a = accept_len[b];
        s_P = P;
        s_a = a;
        s_ok = (a >= 0 && a <= L && P >= 0 && P + a + 1 <= cache_cap) ? 1 : 0;
        s_rows[0] = 0;
        if (!s_ok) record_error(err, ERR_COMMIT | ERR_BAD_PREFIX_LEN);
    }
    __syncthreads();
    const int a = s_a;
    if (s_ok && tid < a) {
        const int u = accepted_nodes[(size_t)b * L + tid];
        s_rows[tid + 1] = u;
        if (u < 1 || u > N) {
            s_ok = 0;
            record_error(err, ERR_COMMIT | ERR_BAD_TREE);
        }
    }
    __syncthreads();
    pdl_trigger();
    if (!s_ok) return;
    const int64_t P = s_P;
    const int vd = D / 8;                 // 16-byte vectors per row
    const int per_row = Hkv * vd;
    const int R = N + 1;
    const int total = (a + 1) * per_row;
    for (int i = tid; i < total; i += kThreads) {
        const int r = i / per_row, rem = i - r * per_row;
        const int g = rem / vd, c = rem - g * vd;
        const size_t src = (((size_t)b * R + s_rows[r]) * Hkv + g) * vd + c;
        const size_t dst = (((size_t)b * Hkv + g) * (size_t)cache_cap + (size_t)(P + r)) * vd + c;
        k_cache[dst] = __ldg(&k_tree[src]);
        v_cache[dst] = __ldg(&v_tree[src]);
    }
    __syncthreads();
    if (tid == 0) prefix_len[b] = (int32_t)(P + a + 1);
}

}  // namespace

cudaError_t launch_commit(const CommitArgs& a, cudaStream_t s) {
    return launch_pdl(commit_kernel, dim3(a.B), dim3(kThreads), 0, s, (uint4*)a.k_cache,
                      (uint4*)a.v_cache, a.cache_cap, (const uint4*)a.k_tree,
                      (const uint4*)a.v_tree, a.accept_len, a.accepted_nodes, a.prefix_len, a.L,
                      a.N, a.Hkv, a.D, a.err);
}

}  // namespace ddt
