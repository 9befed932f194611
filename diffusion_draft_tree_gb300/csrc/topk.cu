// topk.cu -- step 1 of a DDTree round: per-position log-softmax and top-K of
// the draft logits ("Accelerating Speculative Decoding with Block Diffusion
// Draft Trees", §3 marginals q_i; §4.3 log-probabilities; App. A restricted
// prefix set).
//
// One row = one (sequence, draft position), V logits, cut into 4 KB segments.
// The flattened (row, segment) list is split into equal chunks, one per warp
// of a single wave, long enough that a row meets at most 32 (or, for long rows
// in small batches, 96) chunks -- its "pieces".  A warp streams its chunk
// through a private ring of shared-memory stages filled by bulk copies two
// segments ahead (no CTA barrier anywhere), and keeps, for the piece of a row
// it is in:
//   - each lane's online (max, sum of exponentials);
//   - the piece's K best (value, index) keys, as a sorted list in shared memory
//     followed by new candidates.  A candidate must beat the bound: the list's
//     K-th key, or the row's shared bound if that is larger (before either
//     exists, the K-th largest lane maximum of the segment, which K distinct
//     elements reach).  Vectors whose maximum is below the bound are skipped
//     whole; a passing vector is re-read from its stage and its qualifying
//     elements placed with a shared-memory add.  Ranking by counting merges
//     the candidates into the list once 32 have gathered, while the list is
//     not yet full, and at the piece's end.
// A piece whose list fills raises the row's shared bound (a key that K
// elements of the row reach), which every piece then filters against.
// At the end of a piece the warp publishes (max, sum) and its K keys, and takes
// the row's ticket; the warp that completes the row merges its pieces: the
// logsumexp from the (max, sum) pairs, the K best by a K-round tournament over
// the pieces' sorted lists (one or three pieces per lane), and leaves the
// row's counter, bound and slots at zero (the workspace is all zero again
// after a call).
#include <algorithm>
#include <mutex>

#include "internal.h"
#include "segment.cuh"
#include "warp_ring.cuh"

#include "../../include/ddtree.h"

namespace ddt {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kSegBytes = 4096;
constexpr int kStages = 3;
constexpr int kRingBytes = kWarps * kStages * kSegBytes;  // 192 KB
constexpr int kSmemBytes = kRingBytes + 128;              // + alignment slack
constexpr int kCap = 96;            // a warp's sorted list (first n) + candidates
// A merging lane holds LISTS pieces of a row (1, or 3 when rows are long
// against the wave: more, shorter pieces), so a row has at most 32 LISTS.
constexpr int kMaxGridWarps = 2560; // warps of the wave (160 SMs), for the workspace bound
constexpr int kMaxV = 1 << 24;      // logits per row (element ids and segment counts fit)
constexpr int kMergeHeads = 4;      // keys of each held piece in registers at a time

// Merges (m, s) pairs: s2 rescaled to the larger maximum (exp base 2^(x c)).
DDT_DEV void ms_combine(float& m, float& s, float m2, float s2, float c) {
    const float mx = fmaxf(m, m2);
    s = (m == -INFINITY ? 0.f : s * fast_exp2((m - mx) * c)) +
        (m2 == -INFINITY ? 0.f : s2 * fast_exp2((m2 - mx) * c));
    m = mx;
}

// A warp's K best keys of the current piece: buf[0, n) sorted descending (the
// list), buf[n, n + cc) unsorted candidates; tkey = the list's K-th key once it
// is full (0 before: every key is larger); rb = a bound on the row's K-th key
// found by any piece of the row.  Keys <= bound() are out.  Every member is
// warp-uniform.
struct KBest {
    uint64_t* buf;  // kCap keys, 16-byte aligned, this warp's alone
    int K, n, cc;
    uint64_t tkey, rb;

    DDT_DEV uint64_t bound() const { return tkey > rb ? tkey : rb; }
    DDT_DEV void reset() {
        n = 0;
        cc = 0;
        tkey = 0ull;
        rb = 0ull;
    }
    // The K largest of list + candidates, sorted, into the list (rank by
    // counting: the keys are distinct, so the ranks are).
    DDT_DEV void reduce() {
        const int lane = threadIdx.x & 31;
        const int t = n + cc;
        __syncwarp();
        const uint64_t k0 = lane < t ? buf[lane] : 0ull;
        const uint64_t k1 = lane + 32 < t ? buf[lane + 32] : 0ull;
        const uint64_t k2 = lane + 64 < t ? buf[lane + 64] : 0ull;
        const int r0 = lane < t ? count_larger(buf, t, k0) : kCap;
        const int r1 = lane + 32 < t ? count_larger(buf, t, k1) : kCap;
        const int r2 = lane + 64 < t ? count_larger(buf, t, k2) : kCap;
        __syncwarp();
        if (r0 < K) buf[r0] = k0;
        if (r1 < K) buf[r1] = k1;
        if (r2 < K) buf[r2] = k2;
        __syncwarp();
        n = min(K, t);
        cc = 0;
        tkey = n == K ? buf[K - 1] : 0ull;
    }
    // Appends `key` of every lane where c holds (warp-collective); makes room
    // first if the buffer could overflow, and then re-tests c against the
    // raised K-th key.
    DDT_DEV void push(bool c, uint64_t key) {
        const int lane = threadIdx.x & 31;
        unsigned b = __ballot_sync(0xffffffffu, c);
        if (!b) return;
        if (n + cc + __popc(b) > kCap) {
            reduce();
            c = c && key > bound();
            b = __ballot_sync(0xffffffffu, c);
        }
        if (c) buf[n + cc + __popc(b & ((1u << lane) - 1u))] = key;
        cc += __popc(b);
    }
};

// Workspace: per row a completion counter and a shared bound; per piece slot (chunk c's piece of
// row r sits at slot c + r) the piece's (max, sum) as a float2 followed by its
// K keys (0 past the piece's element count).
struct TopkWs {
    unsigned int* row_cnt;         // [rows]
    unsigned long long* row_tau;   // [rows] largest piece K-th key so far (0: none)
    uint64_t* slots;               // [nslots][1 + K]
};

struct Cur {  // a warp's position: chunk c, flattened segment i of [., iend)
    long c, i, iend;
    int row, seg;
};

// One wave: warp w of CTA b streams chunks w grid + b + k nw, k = 0, 1, ...
// (spc segments each; the plan makes at most one per warp).
template <bool BF16, int LISTS>
__global__ void __launch_bounds__(kThreads, 1)
topk_kernel(const void* __restrict__ logits, int V, int64_t row_stride, int rows, int nseg,
            long spc, bool aligned, int K, TopkWs ws, int32_t* __restrict__ topk_idx,
            float* __restrict__ topk_logp, float* __restrict__ lse, uint32_t* err) {
    using S = Seg<BF16, kSegBytes>;
    using Ring = WarpRing<BF16, kSegBytes, kStages>;
    constexpr int VEC = S::VEC;
    constexpr int VPL = Ring::VPL;  // vectors per lane per segment
    extern __shared__ __align__(128) uint8_t smem_raw[];  // the warps' rings
    __shared__ __align__(8) uint64_t s_bar[kWarps][kStages];
    __shared__ __align__(16) uint64_t s_buf[kWarps][kCap];
    __shared__ int s_cc[kWarps];  // a warp's next free buffer place (fast path)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long total = (long)rows * nseg;
    const long nchunks = (total + spc - 1) / spc;
    const long nw = (long)gridDim.x * kWarps;
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 127) & ~(uintptr_t)127);
    Ring ring{smem + warp * kStages * kSegBytes, s_bar[warp]};
    ring.init();
    KBest kb{s_buf[warp], K, 0, 0, 0ull, 0ull};
    pdl_wait();

    auto place = [&](Cur& x) -> bool {  // x.c set: its first segment
        if (x.c >= nchunks) return false;
        x.i = x.c * spc;
        x.iend = min(total, x.i + spc);
        x.row = (int)(x.i / nseg);
        x.seg = (int)(x.i - (long)x.row * nseg);
        return true;
    };
    auto next = [&](Cur& x) -> bool {
        if (++x.i < x.iend) {
            if (++x.seg == nseg) {
                ++x.row;
                x.seg = 0;
            }
            return true;
        }
        x.c += nw;
        return place(x);
    };
    // chunks that hold a piece of the row (at most 32 LISTS by the plan)
    auto pieces = [&](int row) -> int {
        return (int)(((long)(row + 1) * nseg - 1) / spc - ((long)row * nseg) / spc + 1);
    };
    auto rowp_of = [&](int row) {
        return (const char*)logits + (size_t)row * (size_t)row_stride * S::ES;
    };
    // The row's result, by the warp that completed it (its count was acquired,
    // so every piece's slot is visible).  Lane p holds pieces p, p + 32, ...
    // (LISTS of them): their (max, sum) and their sorted keys, kMergeHeads of
    // each at a time in registers.  K rounds of a tournament take the largest head (the
    // value word, then the index word, each by one warp reduction); the piece
    // that held it moves to its next key.  Every key of the row's K best is in
    // its piece's list, so the K winners are the row's K best, in order.
    auto merge = [&](int row) {
        const long c_lo = ((long)row * nseg) / spc;
        const int np = pieces(row);
        uint64_t* base = ws.slots + (size_t)(c_lo + row) * (size_t)(1 + K);
        float pm = -INFINITY, ps = 0.f;
        uint64_t hk[LISTS][kMergeHeads];
        int used[LISTS];  // keys of each held piece taken so far
#pragma unroll
        for (int q = 0; q < LISTS; ++q) {
            const int pc = lane + 32 * q;
            const uint64_t* sl = base + (size_t)pc * (1 + K);
#pragma unroll
            for (int i = 0; i < kMergeHeads; ++i)
                hk[q][i] = (pc < np && i < K) ? __ldcg((const unsigned long long*)sl + 1 + i) : 0ull;
            used[q] = 0;
            if (pc < np) {
                const float2 h = __ldcg(reinterpret_cast<const float2*>(sl));
                ms_combine(pm, ps, h.x, h.y, kLog2e);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, pm, o);
            const float so = __shfl_xor_sync(0xffffffffu, ps, o);
            ms_combine(pm, ps, mo, so, kLog2e);
        }
        const float M = (pm == -INFINITY) ? 0.f : pm;
        const float logS = logf(ps);
        for (int r = 0; r < K; ++r) {
            uint64_t best = hk[0][0];
#pragma unroll
            for (int q = 1; q < LISTS; ++q) best = umax64(best, hk[q][0]);
            const uint32_t vw = (uint32_t)(best >> 32);
            const uint32_t vmax = __reduce_max_sync(0xffffffffu, vw);
            const uint32_t iw = (vw == vmax) ? (uint32_t)best : 0u;
            const uint32_t imax = __reduce_max_sync(0xffffffffu, iw);
            const uint64_t key = ((uint64_t)vmax << 32) | imax;
            if (lane == 0) {
                topk_idx[(size_t)row * K + r] = (int32_t)key_index(key);
                topk_logp[(size_t)row * K + r] = (key_value(key) - M) - logS;
            }
#pragma unroll
            for (int q = 0; q < LISTS; ++q) {
                if (hk[q][0] != key) continue;  // (keys are distinct: one piece holds it)
#pragma unroll
                for (int i = 0; i + 1 < kMergeHeads; ++i) hk[q][i] = hk[q][i + 1];
                hk[q][kMergeHeads - 1] = 0ull;
                if (++used[q] % kMergeHeads == 0 && used[q] < K) {  // its next keys
                    const uint64_t* sl = base + (size_t)(lane + 32 * q) * (1 + K) + 1 + used[q];
#pragma unroll
                    for (int i = 0; i < kMergeHeads; ++i)
                        hk[q][i] = used[q] + i < K ? __ldcg((const unsigned long long*)sl + i) : 0ull;
                }
            }
        }
        __syncwarp();
        // the row's slots back to zero, like its counter and bound: a later call
        // of other sizes may place its counters here
        for (int wd = lane; wd < np * (1 + K); wd += 32) base[wd] = 0ull;
        if (lane == 0) {
            if (lse) lse[row] = M + logS;
            ws.row_cnt[row] = 0u;  // ready for the next call
            ws.row_tau[row] = 0ull;
        }
        __syncwarp();
    };

    // Segment by segment through the warp's ring, kStages - 1 ahead.  After a
    // fill that never lands (a bounded wait that timed out) the warp stops
    // issuing, records the error and runs the rest of its protocol on zeros, so
    // every row count still completes (and returns to zero) and the call ends.
    // chunk c goes to CTA c mod grid: every SM streams even when there are
    // fewer chunks than warps
    Cur xi{(long)warp * gridDim.x + blockIdx.x, 0, 0, 0, 0};
    bool hi = place(xi);
    Cur xp = xi;
    bool hp = hi;
    int ni = 0, np = 0;
    bool dead = false;
    // The row's shared bound is fetched with each segment's copy and used when
    // the segment is read: a queue of kStages values (q0 is the segment read
    // next), in registers.
    static_assert(kStages == 3, "the bound queue holds three segments");
    uint64_t q0 = 0ull, q1 = 0ull, q2 = 0ull;
    for (int k = 0; k < kStages - 1 && hi; ++k) {
        ring.issue(ni % kStages, rowp_of(xi.row), xi.seg * S::SIZE, V, aligned);
        (k == 0 ? q0 : q1) = __ldcg(&ws.row_tau[xi.row]);
        ++ni;
        hi = next(xi);
    }
    float m = -INFINITY;                      // the lane's running max of the piece
    float2 acc = make_float2(0.f, 0.f);       // ... and sum of exp(x - m), in two
    float2 acc2 = make_float2(0.f, 0.f);      // independent chains
    while (hp) {
        if (hi && !dead) {  // into the stage read last
            ring.issue(ni % kStages, rowp_of(xi.row), xi.seg * S::SIZE, V, aligned);
            q2 = __ldcg(&ws.row_tau[xi.row]);
            ++ni;
            hi = next(xi);
        }
        const uint64_t rbl = q0;  // this segment's row bound, fetched with its copy
        q0 = q1;
        q1 = q2;
        const int st = np % kStages;
        if (!dead && !ring.wait(st, (uint32_t)((np / kStages) & 1))) {
            dead = true;
            if (lane == 0) record_error(err, ERR_TOPK | ERR_WAIT_TIMEOUT);
        }
        uint4 cur[VPL];
        if (!dead) {
            ring.read(st, cur);
        } else {
#pragma unroll
            for (int k = 0; k < VPL; ++k) cur[k] = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();  // every lane has read the stage: it may be refilled
        ++np;
        const int e0 = xp.seg * S::SIZE;

        // ---- vector maxima; the lane's online (max, sum of exponentials) ----
        float vm[VPL];
        float ms = -INFINITY;
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            vm[k] = S::vmax(cur[k]);
            ms = fmaxf(ms, vm[k]);
        }
        if (ms > m) {
            const float f = fast_exp2((m - ms) * kLog2e);  // 0 while m = -inf
            acc.x *= f;
            acc.y *= f;
            acc2.x *= f;
            acc2.y *= f;
            m = ms;
        }
        if (m != -INFINITY) {
            const float off = -m * kLog2e;
#pragma unroll
            for (int k = 0; k < VPL; k += 2) {
                S::exp_sum2(cur[k], kLog2e, off, acc);
                S::exp_sum2(cur[k + 1], kLog2e, off, acc2);
            }
        }

        // ---- candidates: keys above the bound (the list's K-th key or the
        // row's shared bound; with neither, at or above the K-th largest lane
        // maximum of the segment) ----
        kb.rb = umax64(kb.rb, rbl);
        const uint64_t bnd = kb.bound();
        float tv = bnd != 0ull ? key_value(bnd) : -INFINITY;
        if (bnd == 0ull) {
            const bool real = e0 + lane * VEC < V;  // the lane holds an element
            const uint32_t b = warp_kth_largest(real ? ord_from_float(ms) : 0u, K);
            if (b != 0u) tv = fmaxf(tv, float_from_ord(b));
        }
        unsigned vpm = 0u;  // the lane's vectors that may hold a candidate
#pragma unroll
        for (int k = 0; k < VPL; ++k)
            if (e0 + (lane + 32 * k) * VEC < V && vm[k] >= tv) vpm |= 1u << k;
        if (__any_sync(0xffffffffu, vpm != 0u)) {
            const uint4* stv = reinterpret_cast<const uint4*>(ring.buf + st * kSegBytes) + lane;
            // Fast path: each lane walks its own passing vectors (re-read from the
            // stage, intact until the next iteration refills it) and reserves
            // buffer places with a shared-memory add -- no warp-wide step per
            // candidate.  If the buffer would overflow, nothing of it is kept
            // and the slow path below redoes the step from the same place.
            const int base0 = kb.n + kb.cc;
            if (lane == 0) s_cc[warp] = base0;
            __syncwarp();
            const uint64_t tk = kb.bound();
            bool ovf = false;
            for (unsigned pend = vpm; pend != 0u; pend &= pend - 1u) {
                const int k = __ffs(pend) - 1;
                const uint4 v = stv[32 * k];
                const int ev = e0 + (lane + 32 * k) * VEC;
                // the vector's elements >= tv (one packed comparison per pair),
                // then the key test for those alone (usually one)
                for (unsigned em = S::ge_mask(v, tv); em != 0u; em &= em - 1u) {
                    const int j = __ffs(em) - 1;
                    const uint64_t key = value_index_key(S::elem_dyn(v, j), (uint32_t)(ev + j));
                    if (ev + j >= V || key <= tk) continue;
                    const int pos = atomicAdd(&s_cc[warp], 1);
                    if (pos < kCap) kb.buf[pos] = key;
                    else ovf = true;
                }
            }
            __syncwarp();
            if (!__any_sync(0xffffffffu, ovf)) {
                kb.cc = s_cc[warp] - kb.n;
            } else {
                // Slow path (the buffer would overflow: many ties): key by key,
                // merging whenever the buffer fills; rare, so kept compact.
#pragma unroll 1
                for (int k = 0; k < VPL; ++k) {
                    const uint4 v = stv[32 * k];
                    const int ev = e0 + (lane + 32 * k) * VEC;
                    const bool vp = (vpm >> k) & 1u;
#pragma unroll 1
                    for (int j = 0; j < VEC; ++j) {
                        const float x = S::elem_dyn(v, j);
                        const uint64_t key = value_index_key(x, (uint32_t)(ev + j));
                        kb.push(vp && ev + j < V && x >= tv && key > kb.bound(), key);
                    }
                }
            }
        }
        // merge the candidates once 32 have gathered (and while the list is not
        // yet full): the list's K-th key, and with it the row's bound, rises
        if (kb.cc >= 32 || (kb.n < K && kb.cc > 0)) kb.reduce();
        if (kb.n == K && kb.tkey > kb.rb) {  // a tighter bound for the whole row
            if (lane == 0) atomicMax(&ws.row_tau[xp.row], (unsigned long long)kb.tkey);
            kb.rb = kb.tkey;
        }

        // ---- the row's piece ends: publish, take the row's ticket, and merge
        // the row if this piece completes it ----
        if (xp.seg + 1 == nseg || xp.i + 1 == xp.iend) {
            if (kb.cc > 0) kb.reduce();
            float mw = m, sw = (acc.x + acc.y) + (acc2.x + acc2.y);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float mo = __shfl_xor_sync(0xffffffffu, mw, o);
                const float so = __shfl_xor_sync(0xffffffffu, sw, o);
                ms_combine(mw, sw, mo, so, kLog2e);
            }
            uint64_t* sl = ws.slots + (size_t)(xp.c + xp.row) * (size_t)(1 + K);
            if (lane == 0) *reinterpret_cast<float2*>(sl) = make_float2(mw, sw);
            if (lane < K) sl[1 + lane] = lane < kb.n ? kb.buf[lane] : 0ull;
            __syncwarp();
            // the piece before its count; the other pieces visible to the warp
            // whose count completes the row
            unsigned now = 0u;
            if (lane == 0) now = atom_add_acq_rel_u32(&ws.row_cnt[xp.row], 1u) + 1u;
            now = __shfl_sync(0xffffffffu, now, 0);
            __syncwarp();
            if (now == (unsigned)pieces(xp.row)) merge(xp.row);
            kb.reset();
            m = -INFINITY;
            acc = make_float2(0.f, 0.f);
            acc2 = make_float2(0.f, 0.f);
        }
        hp = next(xp);
    }
    if (dead)  // copies still in flight into the ring: one more bounded wait each
        for (int k = np; k < ni; ++k) ring.wait(k % kStages, (uint32_t)((k / kStages) & 1));
    pdl_trigger();
}

struct Plan {
    int nseg, lists;
    long spc, nchunks;
    int grid;
};

// Streaming multiprocessors of the current device (148 if the query fails).
int num_sms_topk() {
    static int cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

int seg_count(int V, int dtype) {
    const int size = kSegBytes / (dtype == DDTREE_BF16 ? 2 : 4);
    return (V + size - 1) / size;
}

// Equal chunks, one per warp of a one-CTA-per-SM wave, each at least
// (nseg - 1) / (32 LISTS - 1) segments long so that no row has more than
// 32 LISTS pieces; LISTS = 3 only where the 32-piece bound is what limits the
// chunk length (long rows against the wave), since the larger merge costs more.
Plan topk_plan(int rows, int V, int dtype, int sms) {
    Plan p;
    p.nseg = seg_count(V, dtype);
    const long total = (long)rows * p.nseg;
    const long w = (long)std::min(sms, kMaxGridWarps / kWarps) * kWarps;
    // a row meets at most ceil((nseg - 1) / spc) + 1 chunks
    auto spc_for = [&](int lists) {
        const long mp = 32L * lists;
        return std::max({1L, (total + w - 1) / w, (long)(p.nseg - 1 + mp - 2) / (mp - 1)});
    };
    p.lists = spc_for(3) < spc_for(1) ? 3 : 1;
    p.spc = spc_for(p.lists);
    p.nchunks = (total + p.spc - 1) / p.spc;
    p.grid = (int)std::min((long)sms, p.nchunks);
    return p;
}

// Workspace: the row counters and bounds, then one slot per (chunk, row) piece.  Chunk c's
// piece of row r sits at slot c + r < chunks + rows; the plan never makes more
// chunks than segments or than kMaxGridWarps, whatever the device.
struct WsLayout {
    size_t row_cnt, row_tau, slots, total;
};
WsLayout topk_layout(int rows, int V, int dtype, int K) {
    const long total = (long)rows * seg_count(V, dtype);
    const size_t nslots = (size_t)std::min(total, (long)kMaxGridWarps) + (size_t)rows;
    WsLayout l;
    l.row_cnt = 0;
    l.row_tau = align_up((size_t)rows * 4, 256);
    l.slots = align_up(l.row_tau + (size_t)rows * 8, 256);
    l.total = align_up(l.slots + nslots * 8 * (size_t)(1 + K), 256);
    return l;
}

}  // namespace

bool topk_supported(int V, int dtype, int K) {
    (void)dtype;
    return V >= 1 && V <= kMaxV && K >= 1 && K <= DDTREE_MAX_K;
}

size_t topk_workspace_bytes(int rows, int V, int dtype, int K) {
    if (rows <= 0 || V <= 0) return 0;
    return topk_layout(rows, V, dtype, K >= 1 ? K : DDTREE_MAX_K).total;
}

template <bool BF16, int LISTS>
cudaError_t launch_stream(const TopkArgs& a, const Plan& p, bool aligned, TopkWs ws,
                          cudaStream_t s) {
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaGetDevice(&dev);
    std::call_once(once[dev & 63], [&] {
        attr_err[dev & 63] = cudaFuncSetAttribute(
            topk_kernel<BF16, LISTS>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    return launch_pdl(topk_kernel<BF16, LISTS>, dim3(p.grid), dim3(kThreads), (size_t)kSmemBytes, s,
                      a.logits, a.V, a.row_stride, a.rows, p.nseg, p.spc, aligned, a.K, ws,
                      a.topk_idx, a.topk_logp, a.lse, a.err);
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s) {
    const int es = a.dtype == DDTREE_BF16 ? 2 : 4;
    const bool aligned = ((uintptr_t)a.logits % 16 == 0) && ((a.row_stride * es) % 16 == 0);
    const Plan p = topk_plan(a.rows, a.V, a.dtype, num_sms_topk());
    const WsLayout l = topk_layout(a.rows, a.V, a.dtype, a.K);
    char* base = (char*)a.ws;
    const TopkWs ws{(unsigned int*)(base + l.row_cnt), (unsigned long long*)(base + l.row_tau),
                    (uint64_t*)(base + l.slots)};
    if (a.dtype == DDTREE_BF16)
        return p.lists == 3 ? launch_stream<true, 3>(a, p, aligned, ws, s)
                            : launch_stream<true, 1>(a, p, aligned, ws, s);
    return p.lists == 3 ? launch_stream<false, 3>(a, p, aligned, ws, s)
                        : launch_stream<false, 1>(a, p, aligned, ws, s);
}

}  // namespace ddt

// ---------------------------------------------------------------------------
// ddtree_topk_noalloc: the same top-K for callers that may not allocate device
// memory, so cannot supply a workspace.  Its cross-CTA partials and counters
// live in one library-owned array of fixed size instead.
// ---------------------------------------------------------------------------

static __device__ __align__(256) unsigned char g_topk_noalloc_scratch[DDTREE_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevicesNoAlloc = 64;
void* g_noalloc_ptr[kMaxDevicesNoAlloc];
std::mutex g_noalloc_mu;

// Device address of this device's scratch array, looked up on the first call
// made with that device current.  In host code the array's name is only a
// stand-in, so the address must come from cudaGetSymbolAddress.
cudaError_t noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevicesNoAlloc) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_topk_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" ddtree_status ddtree_topk_noalloc(const void* draft_logits, int dtype, int rows, int V,
                                             int64_t row_stride, int K, int32_t* topk_idx,
                                             float* topk_logp, float* lse, void* stream) {
    if (!draft_logits || !topk_idx || !topk_logp) return DDTREE_ERR_INVALID_ARG;
    if (dtype != DDTREE_BF16 && dtype != DDTREE_FP32) return DDTREE_ERR_INVALID_ARG;
    if (rows <= 0 || rows > 65535 || V <= 0 || row_stride < V || K < 1 || K > V)
        return DDTREE_ERR_INVALID_ARG;
    if (K > DDTREE_MAX_K || !ddt::topk_supported(V, dtype, K)) return DDTREE_ERR_UNSUPPORTED;
    if ((uintptr_t)draft_logits % (dtype == DDTREE_BF16 ? 2 : 4)) return DDTREE_ERR_INVALID_ARG;
    if ((uintptr_t)topk_idx % 4 || (uintptr_t)topk_logp % 4 || (lse && (uintptr_t)lse % 4))
        return DDTREE_ERR_INVALID_ARG;
    const size_t need = ddt::topk_workspace_bytes(rows, V, dtype, K);
    if (need > DDTREE_NOALLOC_SCRATCH_BYTES) return DDTREE_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    // (the array starts zeroed and every call leaves its row counters at zero)
    if (need) {
        const cudaError_t e = noalloc_scratch(&scratch);
        if (e != cudaSuccess) return (ddtree_status)ddt::launch_status(e);
    }
    ddt::TopkArgs a{draft_logits, dtype, rows, V, row_stride, K, topk_idx, topk_logp, lse,
                    scratch, ddt::error_word()};
    return (ddtree_status)ddt::launch_status(ddt::launch_topk(a, (cudaStream_t)stream));
}
