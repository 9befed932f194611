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
//
// A level never sorts more children than can enter T.  A child enters a full
// T only by beating its last key; when more children pass that test than the
// CTA has threads and T cannot take them all, the N-th largest key of
// T U children is found first by an exact MSB-first radix select over the
// 64-bit keys (8-bit digits below the bits that all keys share, until at
// most 32 keys are left in the digit that holds it, which one warp sorts), and
// only the children at or above it -- at most N of them, often far fewer --
// are compacted, sorted (rank counting up to 64 keys, per-warp register
// sorts merged pairwise above) and merged into T with a rank-by-binary-search
// merge.  A parent takes part only if its best child can beat a full T's last
// key; the first pass over its children keeps every child's key (zero when it
// cannot enter) in its thread's registers, up to 8 a thread, where the
// select and the compaction read it (past that, every pass recomputes a
// child's key from its parent's score and the position's log-prob).  Once no
// parent takes part, or no child qualifies, the build stops.  The
// result -- nodes, their order, fp32 scores formed as parent score +
// log-prob -- is identical to the heap's.  The outputs are written from T at
// the end; the ancestor bitmask is built row by row in dynamic shared memory
// and leaves with coalesced stores.
//
// One CTA per sequence (128 threads for budgets up to 64, else 512).  T holds 64-bit keys:
//   [63:32] orderable fp32 score, [31:27] 31 - depth,
//   [26:16] 2046 - parent position (2047 for the root), [15:10] 63 - rank.
// Keys of distinct prefixes differ.  Parent positions refer to T_{d-1} while
// level d is built and are remapped to the new positions when the level ends
// (the relative order of survivors, and so every comparison, is unchanged by
// the remap).
#include <mutex>

#include "common.cuh"
#include "internal.h"

#include "../../include/ddtree.h"

namespace ddt {

namespace {

constexpr int kCandCap = 2048;  // survivors (<= DDTREE_MAX_N), then the sorts' second buffer
constexpr int kRankSortMax = 64;  // batches up to this size are ranked by counting
constexpr int kBins = 256;  // radix-select digit: 8 bits
constexpr int kRegKeys = 8;  // child keys a thread keeps in registers over a level
constexpr int kAncWords = 16384;  // ancestor-mask words staged in shared memory at a time

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

DDT_DEV uint64_t warp_max_u64(uint64_t v) {
    const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(v >> 32));
    const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(v >> 32) == hi ? (uint32_t)v : 0u);
    return ((uint64_t)hi << 32) | lo;
}
DDT_DEV uint64_t warp_min_u64(uint64_t v) {
    const uint32_t hi = __reduce_min_sync(0xffffffffu, (uint32_t)(v >> 32));
    const uint32_t lo =
        __reduce_min_sync(0xffffffffu, (uint32_t)(v >> 32) == hi ? (uint32_t)v : 0xffffffffu);
    return ((uint64_t)hi << 32) | lo;
}

// Number of keys of the descending run a[0..run) (run a power of two) larger
// than x: log2(run) probes of a branch-free binary search and a last look.
DDT_DEV int run_count_greater(const uint64_t* a, int run, uint64_t x) {
    int lo = 0;
    for (int step = run >> 1; step > 0; step >>= 1)
        if (a[lo + step - 1] > x) lo += step;
    return lo + (a[lo] > x ? 1 : 0);
}

// Sorts the c distinct keys s[0..c) descending, 32 < c <= E * kThreads; returns
// the buffer that holds the result (s or tmp, each with room for E * kThreads
// keys).  The batch is padded to a power of two P with distinct keys smaller
// than any child's (P - i: a child's key carries its score in the top 32
// bits); every warp sorts runs of 32 in registers (a bitonic network over
// shuffles), then runs are merged pairwise, log2(P / 32) rounds, each key
// moving to its own position in its run plus the number of keys of the
// partner run above it (a binary search), through two buffers.
template <int kThreads, int E>
DDT_DEV const uint64_t* merge_sort_desc(uint64_t* s, uint64_t* tmp, int c) {
    int P = 32;
    while (P < c) P <<= 1;
    uint64_t v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int i = threadIdx.x + e * kThreads;
        v[e] = 0ull;
        if (i < P) v[e] = warp_sort_desc(i < c ? s[i] : (uint64_t)(P - i));
    }
    __syncthreads();  // (every key of s is in a register now)
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int i = threadIdx.x + e * kThreads;
        if (i < P) s[i] = v[e];
    }
    __syncthreads();
    uint64_t* src = s;
    uint64_t* dst = tmp;
    for (int run = 32; run < P; run <<= 1) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int i = threadIdx.x + e * kThreads;
            if (i < P) {
                const int base = i & ~(2 * run - 1), own = i & (run - 1);
                const uint64_t* partner = src + base + ((i & run) ? 0 : run);
                dst[base + own + run_count_greater(partner, run, v[e])] = v[e];
            }
        }
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int i = threadIdx.x + e * kThreads;
            if (i < P) v[e] = dst[i];
        }
        uint64_t* x = src;
        src = dst;
        dst = x;
    }
    return src;
}

// Sorts the c distinct keys s[0..c) (c <= kThreads) descending in place: each
// key's rank is counted by its own thread in one pass over the batch, the key
// is scattered to that rank in tmp, and copied back.  Its shared-memory
// traffic grows as c^2 (every thread reads every key), so it serves small
// batches only.
template <int kThreads>
DDT_DEV void rank_sort(uint64_t* s, uint64_t* tmp, int c) {
    const int tid = threadIdx.x;
    if (tid < c) {
        const uint64_t kk = s[tid];
        int rk = 0;
        const ulonglong2* a2 = reinterpret_cast<const ulonglong2*>(s);
#pragma unroll 4
        for (int j = 0; j < (c >> 1); ++j) {
            const ulonglong2 v = a2[j];
            rk += (v.x > kk ? 1 : 0) + (v.y > kk ? 1 : 0);
        }
        if (c & 1) rk += s[c - 1] > kk ? 1 : 0;
        tmp[rk] = kk;
    }
    __syncthreads();
    if (tid < c) s[tid] = tmp[tid];
    __syncthreads();
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

// Children of a level's parents: pair q = (parent list entry q / K, rank q % K).
// Each thread walks the pairs kThreads apart, advancing (pi, r) without a division.
struct PairWalk {
    int pi, r;
    const int dpi, dr, K;
    DDT_DEV void next() {
        pi += dpi;
        r += dr;
        if (r >= K) {
            r -= K;
            ++pi;
        }
    }
};

// Dynamic shared memory of build_level_kernel: the ancestor-mask staging rows.
constexpr size_t kLevelDynSmem = (size_t)kAncWords * sizeof(uint32_t);

template <int kThreads>
__global__ void __launch_bounds__(kThreads, 1)
build_level_kernel(const float* __restrict__ topk_logp, const int32_t* __restrict__ topk_idx,
                   const int32_t* __restrict__ bonus, const int32_t* __restrict__ prefix_len,
                   int L, int K, int N, int32_t* __restrict__ parent, int32_t* __restrict__ depth,
                   int32_t* __restrict__ rank, int32_t* __restrict__ token,
                   int32_t* __restrict__ pos_id, float* __restrict__ score,
                   int32_t* __restrict__ child_count, uint32_t* __restrict__ anc_mask,
                   int32_t* __restrict__ n_nodes) {
    constexpr int kWarps = kThreads / 32;
    // qualifying children sorted without a select when T overflows by at most this many
    constexpr int kDirect = kThreads;
    __shared__ uint64_t s_T[2][DDTREE_MAX_N];
    __shared__ __align__(16) uint64_t s_cand[kCandCap];
    __shared__ int16_t s_plist[DDTREE_MAX_N];  // live parents: T_{d-1} positions
    __shared__ float s_pscore[DDTREE_MAX_N];   // ... and their scores
    __shared__ int16_t s_map[DDTREE_MAX_N];    // T_{d-1} position -> T_d position
    __shared__ float s_lp[DDTREE_MAX_L * DDTREE_MAX_K];
    __shared__ int32_t s_idx[DDTREE_MAX_L * DDTREE_MAX_K];  // tokens, staged with s_lp
    __shared__ int s_hist[2][kBins];
    __shared__ int s_wcnt[kWarps];
    __shared__ uint64_t s_wmax[kWarps], s_wmin[kWarps];
    __shared__ int s_sel[3];  // select: the digit, keys above it, keys in it
    __shared__ int s_ntie;    // select: keys gathered from a small last digit ...
    __shared__ uint64_t s_tie[32], s_thr;  // ... and the threshold taken among them
    // list lengths, double-buffered by level parity so that a counter is reset
    // only once its previous value can no longer be read: live parents,
    // children kept
    __shared__ int s_np[2], s_nc[2];
    extern __shared__ __align__(16) uint32_t s_anc[];  // [kAncWords] ancestor-mask rows

    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int LK = L * K;
    pdl_wait();
    for (int i = tid; i < LK; i += kThreads) {
        s_lp[i] = topk_logp[(size_t)b * LK + i];
        s_idx[i] = topk_idx[(size_t)b * LK + i];
    }
    const int P = prefix_len[b], bon = bonus[b];  // (read now: used by the outputs)
    if (tid < 2) s_np[tid] = s_nc[tid] = 0;
    __syncthreads();

    int t = 0, cur = 0;
    // ---- level 1: the root's children (the empty prefix has score 0), which the
    // sorted log-probs already put in priority order (equal log-probs: lower
    // rank first, as in the key) ----
    if (N > 0) {
        t = min(N, K);
        for (int i = tid; i < t; i += kThreads) s_T[cur][i] = lkey(__fadd_rn(0.f, s_lp[i]), 1, -1, i);
        __syncthreads();
    }
    const PairWalk walk0{tid / K, tid % K, kThreads / K, kThreads % K, K};
    for (int d = 2; d <= L && t > 0; ++d) {
        const float* lp = s_lp + (d - 1) * K;
        const bool full = (t == N);
        // a child enters a full T only by beating its last key
        const uint64_t theta = full ? s_T[cur][t - 1] : 0ull;
        // ---- live parents: the depth-(d-1) nodes of T whose best child (rank 0,
        // the largest of their children's keys) beats theta, in any order ------
        if (tid == 0) {
            s_np[(d + 1) & 1] = 0;
            s_nc[(d + 1) & 1] = 0;
        }
        const int tr = (t + kThreads - 1) / kThreads * kThreads;
        for (int i = tid; i < tr; i += kThreads) {
            const uint64_t k = i < t ? s_T[cur][i] : 0ull;
            const bool f = i < t && lk_depth(k) == d - 1 &&
                           lkey(__fadd_rn(lk_score(k), lp[0]), d, i, 0) > theta;
            const int pos = warp_append_slot(f, &s_np[d & 1]);
            if (f) {
                s_plist[pos] = (int16_t)i;
                s_pscore[pos] = lk_score(k);
            }
        }
        __syncthreads();
        const int npar = s_np[d & 1];
        if (npar == 0) break;  // no node of depth >= d can enter: T is complete
        const int pairs = npar * K;
        auto key_of = [&](const PairWalk& w) {
            return lkey(__fadd_rn(s_pscore[w.pi], lp[w.r]), d, s_plist[w.pi], w.r);
        };

        // ---- pass 0: the children that can enter T -- counted, their largest and
        // smallest keys, and, when every thread's share fits kRegKeys registers,
        // each child's key (0 when it cannot enter) kept for the passes below ----
        const bool cached = pairs <= kRegKeys * kThreads;
        int cnt = 0;
        uint64_t kmx = 0ull, kmn = ~0ull;
        uint64_t kr[kRegKeys];
        // register slots past jr (the same for the whole CTA) hold no child
        const int jr = (pairs + kThreads - 1) / kThreads;
        if (cached) {
            PairWalk w = walk0;
#pragma unroll
            for (int j = 0; j < kRegKeys; ++j) kr[j] = 0ull;
#pragma unroll
            for (int j = 0; j < kRegKeys; ++j, w.next()) {
                if (j >= jr) break;
                uint64_t k = 0ull;
                if (tid + j * kThreads < pairs) {
                    k = key_of(w);
                    if (k > theta) {
                        ++cnt;
                        kmx = umax64(kmx, k);
                        kmn = umin64(kmn, k);
                    } else {
                        k = 0ull;
                    }
                }
                kr[j] = k;
            }
        } else {
            PairWalk w = walk0;
            for (int q = tid; q < pairs; q += kThreads, w.next()) {
                const uint64_t k = key_of(w);
                if (k > theta) {
                    ++cnt;
                    kmx = umax64(kmx, k);
                    kmn = umin64(kmn, k);
                }
            }
        }
        for (int i = tid; i < 2 * kBins; i += kThreads) (&s_hist[0][0])[i] = 0;
        if (tid == 0) s_ntie = 0;
        cnt = __reduce_add_sync(0xffffffffu, cnt);
        kmx = warp_max_u64(kmx);
        kmn = warp_min_u64(kmn);
        if (lane == 0) {
            s_wcnt[warp] = cnt;
            s_wmax[warp] = kmx;
            s_wmin[warp] = kmn;
        }
        __syncthreads();
        int cp = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) cp += s_wcnt[w];
        if (cp == 0) break;  // no child can enter: T is complete

        // ---- select: when many more children qualify than T can take, the N-th
        // largest key thr of U = T u {qualifying children}, by MSB-first radix
        // select (keys are distinct, so exactly N keys of U are >= thr) ----------
        uint64_t thr = 0ull;
        if (t + cp > N && cp > kDirect) {
            uint64_t umx = s_T[cur][0], umn = s_T[cur][t - 1];
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                umx = umax64(umx, s_wmax[w]);
                umn = umin64(umn, s_wmin[w]);
            }
            // every key of U lies in [umn, umx], so all share the bits above the
            // highest one where those two differ; digits start right below them
            const int hb = 63 - __clzll((long long)(umx ^ umn));
            int wd = hb + 1 < 8 ? hb + 1 : 8, sh = hb + 1 - wd;
            uint64_t pmask = hb >= 63 ? 0ull : (~0ull << (hb + 1));
            uint64_t prefix = umx & pmask;
            int rem = N, buf = 0;  // keys still wanted among those matching prefix
            for (;;) {
                const uint32_t dm = (1u << wd) - 1u;
                for (int i = tid; i < t; i += kThreads) {
                    const uint64_t k = s_T[cur][i];
                    if ((k & pmask) == prefix) atomicAdd(&s_hist[buf][(uint32_t)(k >> sh) & dm], 1);
                }
                if (cached) {
#pragma unroll
                    for (int j = 0; j < kRegKeys; ++j) {
                        if (j >= jr) break;
                        const uint64_t k = kr[j];
                        if (k != 0ull && (k & pmask) == prefix)
                            atomicAdd(&s_hist[buf][(uint32_t)(k >> sh) & dm], 1);
                    }
                } else {
                    PairWalk w = walk0;
                    for (int q = tid; q < pairs; q += kThreads, w.next()) {
                        const uint64_t k = key_of(w);
                        if (k > theta && (k & pmask) == prefix)
                            atomicAdd(&s_hist[buf][(uint32_t)(k >> sh) & dm], 1);
                    }
                }
                __syncthreads();
                if (warp == 0) {
                    // lane l holds digits 255-8l .. 248-8l (descending); the digit
                    // where the count from the top first reaches rem holds the N-th key
                    int cv[8], sum = 0;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        cv[e] = s_hist[buf][kBins - 1 - 8 * lane - e];
                        sum += cv[e];
                    }
                    int incl = sum;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int u = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += u;
                    }
                    int before = incl - sum;
                    if (before < rem && rem <= incl) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            if (before + cv[e] >= rem) {
                                s_sel[0] = kBins - 1 - 8 * lane - e;
                                s_sel[1] = before;
                                s_sel[2] = cv[e];
                                break;
                            }
                            before += cv[e];
                        }
                    }
                } else {
                    for (int i = tid - 32; i < kBins; i += kThreads - 32) s_hist[buf ^ 1][i] = 0;
                }
                __syncthreads();
                rem -= s_sel[1];
                prefix |= (uint64_t)s_sel[0] << sh;
                pmask |= (uint64_t)dm << sh;
                const int h = s_sel[2];
                if (h == rem || sh == 0) {  // the whole digit is wanted
                    thr = prefix;
                    break;
                }
                if (h <= 32) {
                    // few keys left in the digit (often exact score ties that
                    // agree on many more bits): one warp sorts them and the
                    // rem-th largest is the threshold
                    for (int i = tid; i < t; i += kThreads) {
                        const uint64_t k = s_T[cur][i];
                        if ((k & pmask) == prefix) s_tie[atomicAdd(&s_ntie, 1)] = k;
                    }
                    if (cached) {
#pragma unroll
                        for (int j = 0; j < kRegKeys; ++j) {
                            if (j >= jr) break;
                            const uint64_t k = kr[j];
                            if (k != 0ull && (k & pmask) == prefix) s_tie[atomicAdd(&s_ntie, 1)] = k;
                        }
                    } else {
                        PairWalk w = walk0;
                        for (int q = tid; q < pairs; q += kThreads, w.next()) {
                            const uint64_t k = key_of(w);
                            if (k > theta && (k & pmask) == prefix) s_tie[atomicAdd(&s_ntie, 1)] = k;
                        }
                    }
                    __syncthreads();
                    if (warp == 0) {
                        const uint64_t v = warp_sort_desc(lane < h ? s_tie[lane] : 0ull);
                        const uint64_t x = shfl_u64(v, rem - 1);
                        if (lane == 0) s_thr = x;
                    }
                    __syncthreads();
                    thr = s_thr;
                    break;
                }
                wd = sh < 8 ? sh : 8;
                sh -= wd;
                buf ^= 1;
            }
        }

        // ---- compact the children that enter: >= thr (at most max(N, kDirect)) ------
        if (cached) {
#pragma unroll
            for (int j = 0; j < kRegKeys; ++j) {
                if (j >= jr) break;
                const uint64_t k = kr[j];
                const bool take = k != 0ull && k >= thr;
                const int pos = warp_append_slot(take, &s_nc[d & 1]);
                if (take) s_cand[pos] = k;
            }
        } else {
            PairWalk w = walk0;
            const int qr = (pairs + kThreads - 1) / kThreads * kThreads;
            for (int q = tid; q < qr; q += kThreads, w.next()) {
                uint64_t k = 0ull;
                if (q < pairs) {
                    k = key_of(w);
                    if (!(k > theta && k >= thr)) k = 0ull;
                }
                const int pos = warp_append_slot(k != 0ull, &s_nc[d & 1]);
                if (k != 0ull) s_cand[pos] = k;
            }
        }
        __syncthreads();
        const int c = s_nc[d & 1];
        if (c == 0) break;

        // ---- sort them, descending: up to kRankSortMax keys by rank counting, more
        // by warp sorts merged pairwise (two keys a thread past kThreads keys) ----
        const uint64_t* sorted = s_cand;
        if (c <= kRankSortMax) {
            rank_sort<kThreads>(s_cand, s_cand + kCandCap / 2, c);
        } else if (c <= kThreads) {
            sorted = merge_sort_desc<kThreads, 1>(s_cand, s_cand + kCandCap / 2, c);
        } else if constexpr (2 * kThreads <= kCandCap / 2) {
            sorted = merge_sort_desc<kThreads, 2>(s_cand, s_cand + kCandCap / 2, c);
        }

        // ---- merge T[0..t) and the sorted children by output rank; keep the first N
        const int nxt = cur ^ 1;
        for (int i = tid; i < t + c; i += kThreads) {
            if (i < t) {
                const uint64_t a = s_T[cur][i];
                const int rk = i + count_greater(sorted, c, a);
                if (rk < N) {
                    s_T[nxt][rk] = a;
                    s_map[i] = (int16_t)rk;
                }
            } else {
                const int j = i - t;
                const uint64_t e = sorted[j];
                const int rk = j + count_greater(s_T[cur], t, e);
                if (rk < N) s_T[nxt][rk] = e;
            }
        }
        t = min(N, t + c);
        cur = nxt;
        __syncthreads();
        // ---- level end: parent positions T_{d-1} -> T_d (a dropped node has no
        // descendant in T: descendants' keys are smaller) --------------------------
        for (int i = tid; i < t; i += kThreads) {
            const uint64_t k = s_T[cur][i];
            const int pp = lk_ppos(k);
            if (pp >= 0) s_T[cur][i] = lk_with_ppos(k, s_map[pp]);
        }
        __syncthreads();
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
    // Ancestor bitmask, staged in shared memory a block of rows at a time: the
    // rows are zeroed, each node's thread walks its chain once and sets one bit
    // per ancestor in its own row, and the block is copied out with coalesced
    // stores.  Rows past n stay zero.
    uint32_t* am = anc_mask + (size_t)b * R * W;
    const int rows_per = kAncWords / W;
    for (int r0 = 0; r0 < R; r0 += rows_per) {
        const int r1 = min(R, r0 + rows_per), nw = (r1 - r0) * W;
        for (int i = tid; i < nw; i += kThreads) s_anc[i] = 0u;
        __syncthreads();
        for (int u = r0 + tid; u < r1 && u <= n; u += kThreads) {
            uint32_t* row = s_anc + (size_t)(u - r0) * W;
            for (int a = u; a >= 0; a = s_par[a]) row[a >> 5] |= 1u << (a & 31);
        }
        __syncthreads();
        for (int i = tid; i < nw; i += kThreads) am[(size_t)r0 * W + i] = s_anc[i];
        __syncthreads();
    }
    if (tid == 0) n_nodes[b] = n;
}

template <int kThreads>
cudaError_t launch_level(const BuildArgs& a, cudaStream_t s) {
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaGetDevice(&dev);
    std::call_once(once[dev & 63], [&] {
        attr_err[dev & 63] = cudaFuncSetAttribute(build_level_kernel<kThreads>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  (int)kLevelDynSmem);
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    return launch_pdl(build_level_kernel<kThreads>, dim3(a.B), dim3(kThreads),
                      kLevelDynSmem, s, a.topk_logp, a.topk_idx, a.bonus,
                      a.prefix_len, a.L, a.K, a.N, a.parent, a.depth, a.rank, a.token, a.pos_id,
                      a.score, a.child_count, a.anc_mask, a.n_nodes);
}

}  // namespace

cudaError_t launch_build_level(const BuildArgs& a, cudaStream_t s) {
    // small budgets: fewer threads make each of the level's barriers cheaper
    if (a.N <= 64) return launch_level<128>(a, s);
    return launch_level<512>(a, s);
}

}  // namespace ddt
