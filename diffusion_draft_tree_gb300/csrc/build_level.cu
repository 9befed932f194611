// build_level.cu -- step 2 of a DDTree round computed level by level.
//
// Algorithm 1 of "Accelerating Speculative Decoding with Block Diffusion Draft
// Trees" (§4.3, App. A) pops the N best prefixes one at a time.  Its result is
// fixed by the priority order alone: the first N prefixes of the restricted
// set in that order (score desc, depth asc, earlier parent, lower rank), in
// that order (§4.2 / App. A: ancestors are at least as probable as their
// descendants, so the top N are prefix-closed).  That set can be built with L
// parallel steps instead of N sequential pops:
//
//   T_0 = {}; for d = 1..L:  T_d = top-N( T_{d-1}  U  children of the
//                                          depth-(d-1) nodes of T_{d-1} )
//
// T_d is the top N among all prefixes of depth <= d (a depth-d prefix in it
// has its parent in it, and that parent is among the top N of depth <= d-1).
// T_1 needs no merge: the root's children are position 1's K tokens, which
// the top-K step already returns in priority order, so it is written directly.
// When T is full, a child must beat its last key, and once the strongest
// parent's best child cannot, no deeper node can enter and the build stops.
// The qualifying children are gathered (in any order), sorted (rank counting
// up to 512 keys, a bitonic network above) and merged into T with a
// rank-by-binary-search merge.  The result -- nodes, their order, fp32 scores
// formed as parent score + log-prob -- is identical to the heap's.
//
// One CTA per sequence (128 threads for budgets up to 64, else 512).  T holds 64-bit keys:
//   [63:32] orderable fp32 score, [31:27] 31 - depth,
//   [26:16] 2046 - parent position (2047 for the root), [15:10] 63 - rank.
// Parent positions refer to T_{d-1} while level d is built and are remapped to
// the new positions when the level ends, through a map that the merges fill in
// (the relative order of survivors, and so every comparison, is unchanged by
// the remap).
#include "common.cuh"
#include "internal.h"

#include "../../include/ddtree.h"

namespace ddt {

namespace {

constexpr int kCandCap = 2048;  // children merged per batch
constexpr int kRankCountMax = 512;  // batches up to this size are ranked by counting

DDT_DEV uint64_t lkey(float score, int depth, int ppos, int rank) {
    return ((uint64_t)ord_from_float(score) << 32) | ((uint32_t)(31 - depth) << 27) |
           ((uint32_t)(2046 - ppos) << 16) | ((uint32_t)(63 - rank) << 10);
}
DDT_DEV float lk_score(uint64_t k) { return float_from_ord((uint32_t)(k >> 32)); }
DDT_DEV int lk_depth(uint64_t k) { return 31 - (int)((uint32_t)k >> 27); }
DDT_DEV int lk_ppos(uint64_t k) { return 2046 - (int)(((uint32_t)k >> 16) & 0x7ffu); }
DDT_DEV int lk_rank(uint64_t k) { return 63 - (int)(((uint32_t)k >> 10) & 0x3fu); }
DDT_DEV uint64_t lk_with_ppos(uint64_t k, int ppos) {
    return (k & ~(0x7ffull << 16)) | ((uint64_t)(2046 - ppos) << 16);
}

// Exclusive scan of one int per thread over the CTA; *total gets the sum.
template <int kThreads>
DDT_DEV int block_scan(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int before = 0, tot = 0;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) {
        const int w = s_warp[i];
        before += (i < warp) ? w : 0;
        tot += w;
    }
    *total = tot;
    __syncthreads();
    return before + incl - v;
}

// Sorts s[0..p2) descending, p2 a power of two <= kCandCap (the buffer is
// zero past the batch, up to kCandCap): a bitonic network with E = 4 keys a
// thread (kThreads = 512), strides below E inside the thread, below 32 E by
// warp shuffles, only the longer strides through shared memory (two barriers
// each, instead of one barrier for every stage).
template <int kThreads>
DDT_DEV void bitonic_desc_regs(uint64_t* s, int p2) {
    constexpr int E = kCandCap / kThreads;
    static_assert(E == 4, "keys a thread");
    const int tid = threadIdx.x;
    uint64_t a[E];
#pragma unroll
    for (int e = 0; e < E; ++e) a[e] = s[tid * E + e];
#pragma unroll 1
    for (int k2 = 2; k2 <= p2; k2 <<= 1) {
#pragma unroll 1
        for (int j = k2 >> 1; j > 0; j >>= 1) {
            if (j < E) {
                uint64_t b[E];
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int i = tid * E + e;
                    const uint64_t q = (j == 1) ? a[e ^ 1] : a[e ^ 2];
                    const bool keep_max = ((i & j) == 0) == ((i & k2) == 0);
                    b[e] = keep_max ? umax64(a[e], q) : umin64(a[e], q);
                }
#pragma unroll
                for (int e = 0; e < E; ++e) a[e] = b[e];
            } else if (j < 32 * E) {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int i = tid * E + e;
                    const uint64_t q = shfl_xor_u64(a[e], j / E);
                    const bool keep_max = ((i & j) == 0) == ((i & k2) == 0);
                    a[e] = keep_max ? umax64(a[e], q) : umin64(a[e], q);
                }
            } else {
                __syncthreads();  // the previous shared stage has been read
#pragma unroll
                for (int e = 0; e < E; ++e) s[tid * E + e] = a[e];
                __syncthreads();
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int i = tid * E + e;
                    const uint64_t q = s[i ^ j];
                    const bool keep_max = ((i & j) == 0) == ((i & k2) == 0);
                    a[e] = keep_max ? umax64(a[e], q) : umin64(a[e], q);
                }
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; ++e) s[tid * E + e] = a[e];
    __syncthreads();
}

// Writes each of the c distinct keys s[0..c) to s[kCandCap/2 + its rank in
// descending order]; M keys a thread, ranked in one pass over the batch.
template <int M, int kThreads>
DDT_DEV void rank_scatter(uint64_t* s, int c) {
    const int tid = threadIdx.x;
    uint64_t kk[M];
    int rk[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const int i = tid + m * kThreads;
        kk[m] = i < c ? s[i] : ~0ull;
        rk[m] = 0;
    }
    const ulonglong2* a2 = reinterpret_cast<const ulonglong2*>(s);
#pragma unroll 4
    for (int j = 0; j < (c >> 1); ++j) {
        const ulonglong2 v = a2[j];
#pragma unroll
        for (int m = 0; m < M; ++m) rk[m] += (v.x > kk[m] ? 1 : 0) + (v.y > kk[m] ? 1 : 0);
    }
    if (c & 1) {
#pragma unroll
        for (int m = 0; m < M; ++m) rk[m] += s[c - 1] > kk[m] ? 1 : 0;
    }
#pragma unroll
    for (int m = 0; m < M; ++m)
        if (tid + m * kThreads < c) s[kCandCap / 2 + rk[m]] = kk[m];
}

// A slot for this lane's item (when `take`) at the end of a shared list whose
// length is *cnt: one atomic per warp.  Every lane of the warp calls it; the
// order of the warps' runs is arbitrary.
DDT_DEV int warp_append_slot(bool take, int* cnt) {
    const unsigned m = __ballot_sync(0xffffffffu, take);
    const int lane = threadIdx.x & 31;
    int base = 0;
    if (lane == 0 && m) base = atomicAdd(cnt, __popc(m));
    base = __shfl_sync(0xffffffffu, base, 0);
    return base + __popc(m & ((1u << lane) - 1u));
}

// Number of keys of the descending array a[0..n) that are larger than x.
DDT_DEV int count_greater(const uint64_t* a, int n, uint64_t x) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] > x) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

template <int kThreads>
__global__ void __launch_bounds__(kThreads)
build_level_kernel(const float* __restrict__ topk_logp, const int32_t* __restrict__ topk_idx,
                   const int32_t* __restrict__ bonus, const int32_t* __restrict__ prefix_len,
                   int L, int K, int N, int32_t* __restrict__ parent, int32_t* __restrict__ depth,
                   int32_t* __restrict__ rank, int32_t* __restrict__ token,
                   int32_t* __restrict__ pos_id, float* __restrict__ score,
                   int32_t* __restrict__ child_count, uint32_t* __restrict__ anc_mask,
                   int32_t* __restrict__ n_nodes) {
    __shared__ uint64_t s_T[2][DDTREE_MAX_N];
    __shared__ int16_t s_orig[2][DDTREE_MAX_N];
    __shared__ __align__(16) uint64_t s_cand[kCandCap];
    __shared__ int16_t s_plist[DDTREE_MAX_N];  // parents: T_{d-1} positions
    __shared__ float s_pscore[DDTREE_MAX_N];   // ... and their scores
    __shared__ int16_t s_map[DDTREE_MAX_N];
    __shared__ float s_lp[DDTREE_MAX_L * DDTREE_MAX_K];
    __shared__ int32_t s_idx[DDTREE_MAX_L * DDTREE_MAX_K];  // tokens, staged with s_lp
    __shared__ int s_flag[2];  // a node of depth d is in T, by level parity
    __shared__ int s_warp[kThreads / 32];
    constexpr int kPosPerThread = DDTREE_MAX_N / kThreads;
    // list lengths, double-buffered so that a counter is reset while its
    // previous value can no longer be read: parents by level, children by batch
    __shared__ int s_np[2], s_nc[2];
    __shared__ int s_fp[2];  // T position of the strongest parent, by level parity

    const int b = blockIdx.x, tid = threadIdx.x;
    const int LK = L * K;
    pdl_wait();
    for (int i = tid; i < LK; i += kThreads) {
        s_lp[i] = topk_logp[(size_t)b * LK + i];
        s_idx[i] = topk_idx[(size_t)b * LK + i];
    }
    const int P = prefix_len[b], bon = bonus[b];  // (read now: used by the outputs)
    if (tid < 2) {
        s_np[tid] = s_nc[tid] = 0;
        s_flag[tid] = 0;
        s_fp[tid] = 0x7fffffff;
    }
    __syncthreads();

    int t = 0, cur = 0, nb = 0;
    // ---- level 1: the root's children (the empty prefix has score 0), which the
    // sorted log-probs already put in priority order (equal log-probs: lower
    // rank first, as in the key) ----
    if (N > 0) {
        t = min(N, K);
        for (int i = tid; i < t; i += kThreads) s_T[cur][i] = lkey(__fadd_rn(0.f, s_lp[i]), 1, -1, i);
        __syncthreads();
    }
    for (int d = 2; d <= L && t > 0; ++d) {
        // ---- parents: the depth-(d-1) nodes of T -----------------------------------
        int npar, first = 0;
        if (t * K > kCandCap) {
            // children in several batches: parents in T order, so that the first
            // batches hold the strongest children and T's last key rises early
            if (tid == 0) s_np[(d + 1) & 1] = 0;
            int f[kPosPerThread];
            int fs = 0;
#pragma unroll
            for (int j = 0; j < kPosPerThread; ++j) {
                const int i = tid * kPosPerThread + j;
                f[j] = (i < t && lk_depth(s_T[cur][i]) == d - 1) ? 1 : 0;
                fs += f[j];
            }
            int tot;
            int pos = block_scan<kThreads>(fs, s_warp, &tot);
#pragma unroll
            for (int j = 0; j < kPosPerThread; ++j) {
                if (f[j]) {
                    s_plist[pos] = (int16_t)(tid * kPosPerThread + j);
                    s_pscore[pos] = lk_score(s_T[cur][tid * kPosPerThread + j]);
                    ++pos;
                }
            }
            npar = tot;
            __syncthreads();
            first = s_plist[0];
        } else {
            // one batch: parents in any order (the children are sorted below)
            if (tid == 0) {
                s_np[(d + 1) & 1] = 0;
                s_fp[(d + 1) & 1] = 0x7fffffff;
            }
            const int tr = (t + kThreads - 1) / kThreads * kThreads;
            for (int i = tid; i < tr; i += kThreads) {
                const uint64_t k = i < t ? s_T[cur][i] : 0ull;
                const bool f = i < t && lk_depth(k) == d - 1;
                const int pos = warp_append_slot(f, &s_np[d & 1]);
                if (f) {
                    s_plist[pos] = (int16_t)i;
                    s_pscore[pos] = lk_score(k);
                }
                const int fm = __reduce_min_sync(0xffffffffu, f ? i : 0x7fffffff);
                if ((tid & 31) == 0 && fm != 0x7fffffff) atomicMin(&s_fp[d & 1], fm);
            }
            __syncthreads();
            npar = s_np[d & 1];
            first = s_fp[d & 1];
        }
        if (npar == 0) break;
        // T is sorted, so its first depth-(d-1) node is the strongest parent, and
        // lkey(its score + the best log-prob, d, position 0, rank 0) bounds every
        // child's key: when that cannot beat a full T's last key, no node of
        // depth >= d enters and the tree is complete.
        if (t == N && lkey(__fadd_rn(lk_score(s_T[cur][first]), s_lp[(d - 1) * K]), d, 0, 0) <=
                          s_T[cur][t - 1])
            break;
        for (int i = tid; i < t; i += kThreads) s_orig[cur][i] = (int16_t)i;

        // ---- children in batches of kCandCap (parent, rank) pairs --------------------
        bool merged = false;
        const int pairs = npar * K;
        const float* lp = s_lp + (d - 1) * K;
        for (int base = 0; base < pairs; base += kCandCap) {
            const bool full = (t == N);
            // a child enters a full T only by beating its last key (keys are a
            // total order, so the batches may come in any parent order)
            const uint64_t theta = full ? s_T[cur][t - 1] : 0ull;
            // pair q = (parent q / K, rank q % K), appended when it can enter T
            // (the batch is sorted below, so the order of the keys is free)
            const int q_end = min(pairs, base + kCandCap);
            const int qr = base + (q_end - base + kThreads - 1) / kThreads * kThreads;
            int* cnt = &s_nc[nb & 1];
            if (tid == 0) s_nc[(nb + 1) & 1] = 0;
            ++nb;
            for (int q = base + tid; q < qr; q += kThreads) {
                uint64_t key = 0ull;
                if (q < q_end) {
                    const int pi = q / K, r = q - pi * K;
                    const float sc = __fadd_rn(s_pscore[pi], lp[r]);
                    const uint64_t k = lkey(sc, d, s_plist[pi], r);
                    if (k > theta) key = k;
                }
                const int pos = warp_append_slot(key != 0ull, cnt);
                if (key != 0ull) s_cand[pos] = key;
            }
            __syncthreads();
            const int c = *cnt;
            if (c == 0) {
                __syncthreads();
                continue;
            }
            // Sort the batch, descending.  Up to 512 keys: each key's rank is
            // counted by its own thread (up to four keys a thread in one pass
            // over the batch) and the key is scattered to that rank in the upper
            // half of the buffer.  Larger batches: a bitonic network padded to a
            // power of two (held in registers, four keys a thread, for the
            // 512-thread variant; in shared memory for the 128-thread one).
            const uint64_t* sorted = s_cand;
            if (c <= kRankCountMax) {
                // (the batch's keys are in place: the count was read after a barrier)
                // up to four keys a thread, counted in one pass over the batch
                if (c <= kThreads) rank_scatter<1, kThreads>(s_cand, c);
                else if (c <= 2 * kThreads) rank_scatter<2, kThreads>(s_cand, c);
                else rank_scatter<(kRankCountMax + kThreads - 1) / kThreads, kThreads>(s_cand, c);
                sorted = s_cand + kCandCap / 2;
                __syncthreads();
            } else {
                int p2 = 1;
                while (p2 < c) p2 <<= 1;
                if constexpr (4 * kThreads == kCandCap) {
                    for (int i = c + tid; i < kCandCap; i += kThreads) s_cand[i] = 0ull;
                    __syncthreads();
                    bitonic_desc_regs<kThreads>(s_cand, p2);
                } else {
                    for (int i = c + tid; i < p2; i += kThreads) s_cand[i] = 0ull;
                    __syncthreads();
                    for (int k2 = 2; k2 <= p2; k2 <<= 1) {
                        for (int j2 = k2 >> 1; j2 > 0; j2 >>= 1) {
                            for (int i = tid; i < p2; i += kThreads) {
                                const int ix = i ^ j2;
                                if (ix > i) {
                                    const uint64_t a = s_cand[i], e = s_cand[ix];
                                    const bool desc = (i & k2) == 0;
                                    if (desc ? (a < e) : (a > e)) {
                                        s_cand[i] = e;
                                        s_cand[ix] = a;
                                    }
                                }
                            }
                            __syncthreads();
                        }
                    }
                }
            }
            // merge T[0..t) and cand[0..c) by output rank; keep the first N
            const int nxt = cur ^ 1;
            for (int i = tid; i < t + c; i += kThreads) {
                if (i < t) {
                    const uint64_t a = s_T[cur][i];
                    const int rk = i + count_greater(sorted, c, a);
                    if (rk < N) {
                        const int o = s_orig[cur][i];
                        s_T[nxt][rk] = a;
                        s_orig[nxt][rk] = (int16_t)o;
                        if (o >= 0) s_map[o] = (int16_t)rk;  // the last merge's position wins
                    }
                } else {
                    const int j = i - t;
                    const uint64_t e = sorted[j];
                    const int rk = j + count_greater(s_T[cur], t, e);
                    if (rk < N) {
                        s_T[nxt][rk] = e;
                        s_orig[nxt][rk] = -1;
                    }
                }
            }
            t = min(N, t + c);
            cur = nxt;
            merged = true;
            __syncthreads();
        }

        // ---- level end: parent positions T_{d-1} -> T_d (s_map was written by the
        // merges: a node of T_{d-1} that survives was moved by every merge, and a
        // dropped one has no descendant in T); stop when nothing reached depth d --
        if (!merged) break;  // no child entered: T is complete
        for (int i = tid; i < t; i += kThreads) {
            const uint64_t k = s_T[cur][i];
            const int pp = lk_ppos(k);
            if (pp >= 0) s_T[cur][i] = lk_with_ppos(k, s_map[pp]);
            if (lk_depth(k) == d) s_flag[d & 1] = 1;
        }
        if (tid == 0) s_flag[(d + 1) & 1] = 0;  // read last a level ago
        __syncthreads();
        if (!s_flag[d & 1]) break;
    }

    pdl_trigger();
    // ---- outputs: node u = position u-1 of T ------------------------------------------
    const int n = t;
    int16_t* s_par = (int16_t*)s_cand;                    // [N+1]
    int* s_cc = (int*)(s_cand + (DDTREE_MAX_N + 8) / 4);  // [N+1]
    for (int u = tid; u <= n; u += kThreads) {
        s_par[u] = (u == 0) ? (int16_t)-1 : (int16_t)(lk_ppos(s_T[cur][u - 1]) + 1);
        s_cc[u] = 0;
    }
    __syncthreads();
    for (int u = 1 + tid; u <= n; u += kThreads) atomicAdd(&s_cc[s_par[u]], 1);
    __syncthreads();
    const int R = N + 1, W = (N + 1 + 31) / 32;
    for (int u = tid; u < R; u += kThreads) {
        const size_t o = (size_t)b * R + u;
        if (u == 0) {
            parent[o] = -1; depth[o] = 0; rank[o] = -1; token[o] = bon; pos_id[o] = P;
            score[o] = 0.f; child_count[o] = s_cc[0];
        } else if (u <= n) {
            const uint64_t k = s_T[cur][u - 1];
            const int dp = lk_depth(k), rk = lk_rank(k);
            parent[o] = s_par[u];
            depth[o] = dp;
            rank[o] = rk;
            token[o] = s_idx[(dp - 1) * K + rk];
            pos_id[o] = P + dp;
            score[o] = lk_score(k);
            child_count[o] = s_cc[u];
        } else {
            parent[o] = -1; depth[o] = -1; rank[o] = -1; token[o] = -1; pos_id[o] = -1;
            score[o] = -INFINITY;
            child_count[o] = 0;
        }
    }
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

}  // namespace

cudaError_t launch_build_level(const BuildArgs& a, cudaStream_t s) {
    // small budgets: fewer threads make each of the level's barriers cheaper
    if (a.N <= 64)
        return launch_pdl(build_level_kernel<128>, dim3(a.B), dim3(128), 0, s, a.topk_logp,
                          a.topk_idx, a.bonus, a.prefix_len, a.L, a.K, a.N, a.parent, a.depth,
                          a.rank, a.token, a.pos_id, a.score, a.child_count, a.anc_mask,
                          a.n_nodes);
    return launch_pdl(build_level_kernel<512>, dim3(a.B), dim3(512), 0, s, a.topk_logp, a.topk_idx,
                      a.bonus, a.prefix_len, a.L, a.K, a.N, a.parent, a.depth, a.rank, a.token,
                      a.pos_id, a.score, a.child_count, a.anc_mask, a.n_nodes);
}

}  // namespace ddt
