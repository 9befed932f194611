// accept.cu -- step 4 of a DDTree round: the target's decoding rule at every
// tree node, then the acceptance walk ("Accelerating Speculative Decoding with
// Block Diffusion Draft Trees", §4.1: walk the tree with the target's decoding
// rule, accept the matched path, the first unmatched target token becomes the
// next bonus; §5 / App. B: temperatures 0 and 1).
//
// One persistent wave streams every live node row once from HBM.  The rows
// are cut into 4 KB segments and the flattened (sequence, node, segment) list
// is grouped into chunks of consecutive segments of one row, dealt round-robin
// to the warps (sixteen per SM).  Each warp streams its segments through its
// own ring of shared-memory stages filled by bulk copies two segments ahead
// (warp_ring.cuh), needs no CTA barrier, and publishes once per chunk:
//   T = 0: the chunk's (max, lowest index), folded into the row's 64-bit
//          slot with one atomicMax;
//   T > 0: the segment's max m_s and s_s = sum 2^((x - m_s) c), c = log2(e)/T
//          (packed two-lane fp32 arithmetic); each chunk is counted on its
//          row, and one sampler warp per CTA (fifteen stream) resolves the
//          inverse-CDF sample of each of its rows once all its chunks are in:
//          the segment in which the running sum crosses U * Z, then that
//          segment rescanned (from L2) in token order.
// The last CTA to finish (atomic ticket over the grid) runs the walks: all its
// threads stage every node's target token, parent and token in shared memory
// in one round of loads, mark each parent's chosen child, then one thread per
// sequence follows the chosen children.
#include <algorithm>
#include <mutex>

#include "chunk.cuh"
#include "internal.h"
#include "sampling.cuh"
#include "segment.cuh"
#include "warp_ring.cuh"

#include "../../include/ddtree.h"

namespace ddt {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kSegBytes = 4096;                 // one warp's unit of work
constexpr int kStages = 3;                      // segments in flight per warp
constexpr int kVpl = kSegBytes / 16 / 32;       // 16-byte vectors per lane per segment
constexpr int kMaxSegs = 1024;                  // per row
constexpr int kRingBytes = kWarps * kStages * kSegBytes;  // 192 KB: one CTA per SM
constexpr int kSmemBytes = kRingBytes + 128;    // (the walks reuse the rings)
constexpr int kChunksPerWarp = 4;  // (ragged_serving T = 1: 133 us at 8, 127 us at 4, 139 us at 2)
constexpr int kRegRounds = 4;                   // rows of <= 128 segments resolve from registers
constexpr unsigned kOrphan = 0x80000000u;       // row count flag: the owner has finished
constexpr uint64_t kLingerNs = 20000;           // a sampler's wait for its last rows

struct AcceptWs {
    unsigned int* row_cnt;        // [B][N+1] chunks done | kOrphan (sampling)
    unsigned int* done;           // CTAs done
    float2* parts;                // [B][N+1][nseg]: (m_s, s_s) (sampling)
    int32_t* tok;                 // [B][N+1] sampled target tokens
    unsigned long long* row_best; // [B][N+1] greedy: max (value, lowest index) key
};


DDT_DEV double shfl_up_f64(double v, int o) {
    return __longlong_as_double(
        (long long)__shfl_up_sync(0xffffffffu, (unsigned long long)__double_as_longlong(v), o));
}

// The inverse-CDF sample of one row (one warp): Z = sum_s s_s 2^((m_s - M) c)
// over the row's segment partials; the segment in which the running sum
// crosses U * Z; that segment rescanned in token order (a lane owns 1/32 of
// it, contiguous).  Returns the token, in every lane.
template <bool BF16>
DDT_DEV int resolve_row(const char* rowp, bool aligned, const float2* parts, int nseg, int V,
                        float c_exp, uint64_t seed, uint64_t step, uint64_t seq, uint64_t node) {
    using S = Seg<BF16>;
    const int lane = threadIdx.x & 31;
    int cs = nseg - 1;
    float tloc = 0.f, mref = 0.f;
    if (nseg <= 32 * kRegRounds) {
        // the row's segment partials in registers (segment lane + 32 j), summed
        // in fp32: with at most 128 terms the rounding of Z and of the running
        // sums stays below 1e-5 Z, the resolution of the per-segment sums
        float2 pr[kRegRounds];
#pragma unroll
        for (int j = 0; j < kRegRounds; ++j) {
            const int s = lane + 32 * j;
            pr[j] = s < nseg ? __ldcg(&parts[s]) : make_float2(-INFINITY, 0.f);
        }
        const float u = node_uniform(seed, step, seq, node);  // while the loads are in flight
        float M = -INFINITY;
#pragma unroll
        for (int j = 0; j < kRegRounds; ++j) M = fmaxf(M, pr[j].x);
        M = warp_max(M);
        float sc[kRegRounds], ct[kRegRounds], Zl = 0.f;
#pragma unroll
        for (int j = 0; j < kRegRounds; ++j) {
            sc[j] = lane + 32 * j < nseg ? fast_exp2((pr[j].x - M) * c_exp) : 0.f;
            ct[j] = pr[j].y * sc[j];
            Zl += ct[j];
        }
        const float target = u * warp_sum(Zl);
        float base = 0.f;
        bool found = false;
#pragma unroll
        for (int j = 0; j < kRegRounds; ++j) {
            if (found || 32 * j >= nseg) continue;
            const int s = 32 * j + lane;
            float incl = ct[j];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            const float before = base + incl - ct[j];
            const bool cross = s < nseg && (before + ct[j] > target || s == nseg - 1);
            const unsigned bal = __ballot_sync(0xffffffffu, cross);
            if (bal) {
                const int src = __ffs(bal) - 1;
                cs = 32 * j + src;
                const float t = sc[j] > 0.f ? (target - before) / sc[j] : 0.f;
                tloc = __shfl_sync(0xffffffffu, t, src);
                mref = __shfl_sync(0xffffffffu, pr[j].x, src);
                found = true;
            }
            base += __shfl_sync(0xffffffffu, incl, 31);
        }
    } else {
        float M = -INFINITY;
        for (int s = lane; s < nseg; s += 32) M = fmaxf(M, __ldcg(&parts[s]).x);
        M = warp_max(M);
        double Z = 0.0;
        for (int s = lane; s < nseg; s += 32) {
            const float2 p = __ldcg(&parts[s]);
            Z += (double)p.y * (double)fast_exp2((p.x - M) * c_exp);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            Z += __longlong_as_double((long long)__shfl_xor_sync(
                0xffffffffu, (unsigned long long)__double_as_longlong(Z), o));
        const double target = (double)node_uniform(seed, step, seq, node) * Z;
        // running sum over segments, 32 at a time, until it passes the target
        double base = 0.0;
        for (int s0 = 0; s0 < nseg; s0 += 32) {
            const int s = s0 + lane;
            double contrib = 0.0, scale = 0.0;
            if (s < nseg) {
                const float2 p = __ldcg(&parts[s]);
                scale = (double)fast_exp2((p.x - M) * c_exp);
                contrib = (double)p.y * scale;
            }
            double incl = contrib;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double t = shfl_up_f64(incl, o);
                if (lane >= o) incl += t;
            }
            const double before = base + incl - contrib;
            const bool cross = s < nseg && (before + contrib > target || s == nseg - 1);
            const unsigned bal = __ballot_sync(0xffffffffu, cross);
            if (bal) {
                const int src = __ffs(bal) - 1;
                cs = s0 + src;
                const float t = scale > 0.0 ? (float)((target - before) / scale) : 0.f;
                tloc = __shfl_sync(0xffffffffu, t, src);
                break;
            }
            base += __shfl_sync(0xffffffffu, incl, 31);
        }
        mref = __ldcg(&parts[cs]).x;
    }
    // rescan segment cs: weights relative to its own maximum; lane l owns
    // elements [l PER, (l + 1) PER) of it, held in registers for both passes
    mref = fmaxf(mref, -3.0e38f);
    constexpr int PER = S::SIZE / 32;
    constexpr int NQ = PER / S::VEC;  // 16-byte vectors per lane
    const int e0 = cs * S::SIZE + lane * PER;
    uint4 q[NQ];
    if (aligned && e0 + PER <= V) {
#pragma unroll
        for (int k = 0; k < NQ; ++k) q[k] = __ldcg(reinterpret_cast<const uint4*>(rowp + (size_t)e0 * S::ES) + k);
    } else {
#pragma unroll
        for (int k = 0; k < NQ; ++k) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (BF16) {
                    const int e = e0 + k * S::VEC + 2 * i;
                    const uint32_t lo = e < V ? (uint32_t)__ldcg(reinterpret_cast<const unsigned short*>(rowp) + e) : 0xff80u;
                    const uint32_t hi = e + 1 < V ? (uint32_t)__ldcg(reinterpret_cast<const unsigned short*>(rowp) + e + 1) : 0xff80u;
                    w[i] = lo | (hi << 16);
                } else {
                    const int e = e0 + k * S::VEC + i;
                    w[i] = e < V ? __ldcg(reinterpret_cast<const unsigned int*>(rowp) + e) : 0xff800000u;
                }
            }
            q[k] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < NQ; ++k)
#pragma unroll
        for (int j = 0; j < S::VEC; ++j) sum += fast_exp2((S::elem(q[k], j) - mref) * c_exp);
    float incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    const float before = incl - sum;
    // owner: the first lane whose running sum passes tloc; if rounding leaves
    // none (tloc at the segment's very end), the last lane with nonzero weight
    const unsigned pass = __ballot_sync(0xffffffffu, sum > 0.f && tloc < before + sum);
    const unsigned nz = __ballot_sync(0xffffffffu, sum > 0.f);
    const int owner = pass ? __ffs(pass) - 1 : (nz ? 31 - __clz(nz) : -1);
    int pick = cs * S::SIZE;
    if (owner >= 0 && lane == owner) {  // its elements again, in token order
        float acc = before;
        int p = -1, lastnz = -1;
#pragma unroll
        for (int k = 0; k < NQ; ++k)
#pragma unroll
            for (int j = 0; j < S::VEC; ++j) {
                const float w = fast_exp2((S::elem(q[k], j) - mref) * c_exp);
                acc += w;
                const int e = e0 + k * S::VEC + j;
                if (p < 0 && acc > tloc) p = e;
                if (w > 0.f) lastnz = e;
            }
        pick = p >= 0 ? p : lastnz;
    }
    return owner >= 0 ? __shfl_sync(0xffffffffu, pick, owner) : pick;
}

// A warp's position in the stream: flattened segment i (row `row`, segment
// `seg` of it) of chunk c, whose segments are [c spc, iend).
struct Cursor {
    long c, i, iend;
    int row, b, u, seg;
};

template <bool BF16, bool SAMPLE>
__global__ void __launch_bounds__(kThreads, 1)
accept_kernel(const void* __restrict__ logits, int V, int64_t row_stride, int nseg, long spc,
              bool aligned, int B, int seq_batch, const int32_t* __restrict__ parent,
              const int32_t* __restrict__ token, const int32_t* __restrict__ n_nodes, int L,
              int N, float c_exp, uint64_t seed, uint64_t step,
              int32_t* __restrict__ target_token, int32_t* __restrict__ accept_len,
              int32_t* __restrict__ accepted_nodes, int32_t* __restrict__ out_tokens,
              int32_t* __restrict__ next_bonus, AcceptWs ws, uint32_t* err) {
    using S = Seg<BF16>;
    using Ring = WarpRing<BF16, kSegBytes, kStages>;
    constexpr int VEC = S::VEC;
    extern __shared__ __align__(128) uint8_t smem_raw[];  // the warps' rings; later the walks
    __shared__ __align__(8) uint64_t s_bar[kWarps][kStages];
    __shared__ bool s_last;
    __shared__ unsigned s_streamed;  // streaming warps of this CTA that are done
    __shared__ int s_nn[kThreads];   // n_nodes of sequences 0 .. kThreads - 1
    // Sampling: the last warp of each CTA samples rows while the others stream.
    constexpr int kStreamers = SAMPLE ? kWarps - 1 : kWarps;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool sampler = SAMPLE && warp == kWarps - 1;
    const int R = N + 1;
    const long total = (long)B * R * nseg;        // segments of the flattened rows
    const long nchunks = (total + spc - 1) / spc;
    const long nw = (long)gridDim.x * kStreamers;
    const long gw = (long)blockIdx.x * kStreamers + warp;
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 127) & ~(uintptr_t)127);
    Ring ring{smem + warp * kStages * kSegBytes, s_bar[warp]};
    ring.init();
    if (tid == 0) s_streamed = 0u;
    __syncthreads();
    pdl_wait();
    // the tree sizes of the first sequences, for the walks (the last CTA's)
    for (int b = tid; b < min(B, kThreads); b += kThreads) s_nn[b] = __ldg(&n_nodes[b]);
    if (blockIdx.x == 0)
        for (int b = tid; b < B; b += kThreads) {
            const int n = __ldg(&n_nodes[b]);
            if (n < 0 || n > N) record_error(err, ERR_ACCEPT | ERR_BAD_N_NODES);
        }

    // Moves x to the first live segment at or after x.i, through this warp's
    // chunks x.c, x.c + nw, ... (segments of dead rows are skipped).
    auto place = [&](Cursor& x) -> bool {
        for (;;) {
            if (x.i >= x.iend) {
                x.c += nw;
                if (x.c >= nchunks) return false;
                x.i = x.c * spc;
                x.iend = min(x.i + spc, total);
            }
            const int row = (int)(x.i / nseg);
            const int b = row / R, u = row - b * R;
            const int n = __ldg(&n_nodes[b]);
            if (n >= 0 && n <= N && u <= n) {
                x.row = row;
                x.b = b;
                x.u = u;
                x.seg = (int)(x.i - (long)row * nseg);
                return true;
            }
            x.i = (long)(row + 1) * nseg;  // a dead row: skip it
        }
    };
    auto first = [&](long c, Cursor& x) -> bool {
        x.c = c;
        x.i = c * spc;
        x.iend = c < nchunks ? min(x.i + spc, total) : x.i;
        if (c >= nchunks) return false;
        return place(x);
    };
    auto next = [&](Cursor& x) -> bool {
        ++x.i;
        if (x.i < x.iend && x.seg + 1 < nseg) {  // the same row: no division, no lookup
            ++x.seg;
            return true;
        }
        return place(x);
    };
    // chunks that hold a piece of the row: each publishes once for it
    auto pieces = [&](int row) -> unsigned {
        return (unsigned)(((long)(row + 1) * nseg - 1) / spc - ((long)row * nseg) / spc + 1);
    };
    auto rowp_of = [&](const Cursor& x) {
        return (const char*)logits + (size_t)x.row * (size_t)row_stride * S::ES;
    };
    // Sampling: the sampler warp of CTA k owns rows k, k + gridDim.x, ... and
    // samples each once all its chunks are counted, polling while its CTA's
    // streaming warps run; rows still open when they are done are orphaned,
    // to be sampled by the warp that completes them.
    int own = (int)min((long)blockIdx.x, (long)B * R);
    auto skip_dead = [&]() {
        while (own < B * R) {
            const int b = own / R, n = __ldg(&n_nodes[b]);
            if (n >= 0 && n <= N && own - b * R <= n) break;
            own += (int)gridDim.x;
        }
        if (own > B * R) own = B * R;
    };
    // The inverse-CDF sample of a completed row.
    // (the caller has acquired the row's count, so every chunk's partials of
    // the row are visible; the token is published by the grid's final ticket)
    auto resolve = [&](int row) {
        const int b = row / R, u = row - b * R;
        const char* rowp = (const char*)logits + (size_t)row * (size_t)row_stride * S::ES;
        const int pick = resolve_row<BF16>(rowp, aligned, ws.parts + (size_t)row * nseg, nseg, V,
                                           c_exp, seed, step, (uint64_t)b, (uint64_t)u);
        if (lane == 0) {
            ws.row_cnt[row] = 0u;  // ready for the next call
            ws.tok[row] = pick;
        }
    };
    // Chunks c = gw, gw + nw, ... segment by segment through the warp's ring,
    // kStages - 1 segments ahead.  A chunk publishes its result once, at its
    // end.  After a fill that never lands (a bounded wait that timed out) the
    // warp stops issuing, records the error and runs the rest of its protocol
    // on empty data, so every count still completes and the call ends.
    Cursor xi{}, xp{};
    bool hi = !sampler && first(gw, xi);
    bool hp = hi;
    xp = xi;
    int ni = 0, np = 0;
    bool dead = false;
    for (int k = 0; k < kStages - 1 && hi; ++k) {
        ring.issue(ni % kStages, rowp_of(xi), xi.seg * S::SIZE, V, aligned);
        ++ni;
        hi = next(xi);
    }
    unsigned long long ckey = 0ull;  // greedy: the chunk's best (value, lowest index) key
    while (hp) {
        if (hi && !dead) {  // into the stage read last
            ring.issue(ni % kStages, rowp_of(xi), xi.seg * S::SIZE, V, aligned);
            ++ni;
            hi = next(xi);
        }
        const int st = np % kStages;
        if (!dead && !ring.wait(st, (uint32_t)((np / kStages) & 1))) {
            dead = true;
            if (lane == 0) record_error(err, ERR_ACCEPT | ERR_WAIT_TIMEOUT);
        }
        uint4 cur[kVpl];
        if (!dead) {
            ring.read(st, cur);
        } else {
#pragma unroll
            for (int k = 0; k < kVpl; ++k) cur[k] = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();  // every lane has read the stage: it may be refilled
        ++np;
        const int e0 = xp.seg * S::SIZE;
        const bool chunk_end = xp.seg + 1 == nseg || xp.i + 1 == xp.iend;  // the row's piece ends
        if (!SAMPLE) {
            // the segment's maximum and its lowest index
            float best = -INFINITY;
            uint4 bv = make_uint4(0, 0, 0, 0);
            int bk = -1;
#pragma unroll
            for (int k = 0; k < kVpl; ++k) {
                const float vm = S::vmax(cur[k]);
                if (vm > best) {
                    best = vm;
                    bv = cur[k];
                    bk = k;
                }
            }
            const float wmax = warp_max(best);
            int first = 0x7fffffff;
            if (bk >= 0 && best == wmax) {
                const int eb = e0 + (lane + 32 * bk) * VEC;
#pragma unroll
                for (int j = VEC - 1; j >= 0; --j)
                    if (S::elem(bv, j) == wmax && eb + j < V) first = eb + j;
            }
            first = __reduce_min_sync(0xffffffffu, first);
            if (first != 0x7fffffff) ckey = umax64(ckey, value_index_key(wmax, (uint32_t)first));
            if (chunk_end) {
                if (lane == 0 && ckey != 0ull) atomicMax(&ws.row_best[xp.row], ckey);
                ckey = 0ull;
            }
        } else {
            // the segment's maximum, then its sum of exponentials against it
            float vm = -INFINITY;
#pragma unroll
            for (int k = 0; k < kVpl; ++k) vm = fmaxf(vm, S::vmax(cur[k]));
            const float m = warp_max(vm);
            float2 acc = make_float2(0.f, 0.f), acc2 = make_float2(0.f, 0.f);
            const float off = -m * c_exp;  // m is finite: every segment holds elements
#pragma unroll
            for (int k = 0; k < kVpl; k += 2) {
                S::exp_sum2(cur[k], c_exp, off, acc);
                if (k + 1 < kVpl) S::exp_sum2(cur[k + 1], c_exp, off, acc2);
            }
            const float ssum = warp_sum((acc.x + acc.y) + (acc2.x + acc2.y));
            if (lane == 0) ws.parts[(size_t)xp.row * nseg + xp.seg] = make_float2(m, ssum);
            if (chunk_end) {
                unsigned now = 0;
                // this chunk's partials before its count; the other chunks'
                // partials visible to the one that completes the row
                if (lane == 0) now = atom_add_acq_rel_u32(&ws.row_cnt[xp.row], 1u) + 1u;
                now = __shfl_sync(0xffffffffu, now, 0);
                __syncwarp();
                // the last chunk of a row whose owner has finished: sample it here
                if (now == (kOrphan | pieces(xp.row))) resolve(xp.row);
            }
        }
        hp = next(xp);
    }
    if (dead)  // copies still in flight into the ring: one more bounded wait each
        for (int k = np; k < ni; ++k) ring.wait(k % kStages, (uint32_t)((k / kStages) & 1));
    if (SAMPLE) {
        if (!sampler) {
            __syncwarp();
            if (lane == 0) atomicAdd(&s_streamed, 1u);
        } else {
            // owned rows as they complete, while this CTA's streamers run
            uint64_t t_done = 0ull;
            for (skip_dead(); own < B * R;) {
                unsigned cnt = 0;
                if (lane == 0) cnt = ld_acquire_u32(&ws.row_cnt[own]);
                cnt = __shfl_sync(0xffffffffu, cnt, 0);
                __syncwarp();  // lane 0's acquire orders every lane's reads of the row
                if (cnt == pieces(own)) {
                    resolve(own);
                    own += (int)gridDim.x;
                    skip_dead();
                    continue;
                }
                // after this CTA's streamers are done, linger a little (bounded)
                // for rows the other CTAs are about to complete
                if (*(volatile unsigned*)&s_streamed == (unsigned)kStreamers) {
                    if (t_done == 0ull) t_done = sm100::globaltimer_ns();
                    else if (sm100::globaltimer_ns() - t_done > kLingerNs) break;
                }
                __nanosleep(256);
            }
            // Owned rows still open are handed to whichever warp completes them:
            // the flag and the count share one word, so exactly one of this warp
            // (the row was complete already) and the completing warp samples it.
            for (; own < B * R; own += (int)gridDim.x, skip_dead()) {
                unsigned old = 0;
                if (lane == 0) old = atom_or_acq_rel_u32(&ws.row_cnt[own], kOrphan);
                old = __shfl_sync(0xffffffffu, old, 0);
                __syncwarp();
                if (old == pieces(own)) resolve(own);
            }
        }
    }
    // the tree arrays the walks read, pulled into L2 (each CTA a slice) while
    // the last CTAs finish
    {
        const long nodes = (long)B * R;
        const long per = (nodes + gridDim.x - 1) / gridDim.x;
        const long lo = blockIdx.x * per, hi2 = min(nodes, lo + per);
        for (long i = lo + tid * 32; i < hi2; i += (long)kThreads * 32) {  // 128-byte lines
            asm volatile("prefetch.global.L2 [%0];" ::"l"(parent + i));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(token + i));
        }
    }
    pdl_trigger();

    // ---- the last CTA to finish walks every sequence ---------------------------
    __syncthreads();
    if (tid == 0) s_last = ticket_is_last(ws.done, gridDim.x);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // Per sequence of a batch, in the idle rings: target token, chosen child,
    // parent and token of every node; then the batch's tree sizes.
    int* s_walk = reinterpret_cast<int*>(smem);  // every warp's ring is idle now
    int* s_n = s_walk + seq_batch * 4 * R;
    for (int b0 = 0; b0 < B; b0 += seq_batch) {
        const int nb_seq = min(seq_batch, B - b0);
        for (int bl = tid; bl < nb_seq; bl += kThreads)
            s_n[bl] = b0 + bl < kThreads ? s_nn[b0 + bl] : __ldcg(&n_nodes[b0 + bl]);
        __syncthreads();
        // every node's target token, parent and token into shared memory, all
        // threads at once (kU nodes, three independent loads each, in flight)
        constexpr int kU = 8;
        for (int i0 = tid; i0 < nb_seq * R; i0 += kU * kThreads) {
            int t[kU], pa[kU], tk[kU];
#pragma unroll
            for (int k = 0; k < kU; ++k) {
                const int i = i0 + k * kThreads;
                const int bl = i / R, u = i - bl * R;
                const bool live = i < nb_seq * R && s_n[bl] >= 0 && s_n[bl] <= N && u <= s_n[bl];
                const size_t r = (size_t)(b0 + bl) * R + u;
                t[k] = pa[k] = tk[k] = -1;
                if (live) {
                    t[k] = SAMPLE ? __ldcg(&ws.tok[r]) : (int)key_index(__ldcg(&ws.row_best[r]));
                    pa[k] = __ldg(&parent[r]);
                    tk[k] = __ldg(&token[r]);
                }
            }
#pragma unroll
            for (int k = 0; k < kU; ++k) {
                const int i = i0 + k * kThreads;
                if (i >= nb_seq * R) continue;
                const int bl = i / R, u = i - bl * R;
                const size_t r = (size_t)(b0 + bl) * R + u;
                const bool valid = s_n[bl] >= 0 && s_n[bl] <= N;
                if (!SAMPLE && valid && u <= s_n[bl]) ws.row_best[r] = 0ull;  // for the next call
                int* w = s_walk + bl * 4 * R;
                w[u] = t[k];
                w[R + u] = -1;
                w[2 * R + u] = pa[k];
                w[3 * R + u] = tk[k];
                if (target_token && valid) target_token[r] = t[k];
            }
        }
        __syncthreads();
        // chosen[p] = the child c of p whose token equals the target's token at p
        for (int i = tid; i < nb_seq * R; i += kThreads) {
            const int bl = i / R, c = i - bl * R;
            if (c == 0 || s_n[bl] < 0 || s_n[bl] > N || c > s_n[bl]) continue;
            int* w = s_walk + bl * 4 * R;
            const int p = w[2 * R + c];
            if (p < 0 || p >= c) {
                record_error(err, ERR_ACCEPT | ERR_BAD_TREE);
                continue;
            }
            if (w[3 * R + c] == w[p]) w[R + p] = c;
        }
        __syncthreads();
        for (int bl = tid; bl < nb_seq; bl += kThreads) {
            const int b = b0 + bl;
            const int n = s_n[bl];
            if (n >= 0 && n <= N) {
                const int* s_tok = s_walk + bl * 4 * R;
                const int* s_ch = s_tok + R;
                int cur_n = 0, len = 0;
                int32_t* acc = accepted_nodes + (size_t)b * L;
                int32_t* ot = out_tokens + (size_t)b * (L + 1);
                while (len < L && s_ch[cur_n] >= 0) {
                    ot[len] = s_tok[cur_n];  // the accepted child's token is the target's
                    cur_n = s_ch[cur_n];
                    acc[len] = cur_n;
                    ++len;
                }
                for (int i = len; i < L; ++i) acc[i] = -1;
                const int bonus = s_tok[cur_n];
                ot[len] = bonus;
                for (int i = len + 1; i <= L; ++i) ot[i] = -1;
                accept_len[b] = len;
                next_bonus[b] = bonus;
            }
        }
        __syncthreads();
    }
}

int num_sms_accept() {
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

int accept_segs(int V, int dtype) {
    const int size = kSegBytes / (dtype == DDTREE_BF16 ? 2 : 4);
    return (V + size - 1) / size;
}

struct WsLayout {
    size_t row_cnt, done, parts, tok, row_best, total;
};

WsLayout accept_layout(int B, int N, int nseg) {
    WsLayout l;
    const size_t R = (size_t)N + 1;
    l.row_cnt = 0;
    l.done = align_up(l.row_cnt + (size_t)B * R * 4, 256);
    l.parts = align_up(l.done + 16, 256);
    l.tok = align_up(l.parts + (size_t)B * R * nseg * sizeof(float2), 256);
    l.row_best = align_up(l.tok + (size_t)B * R * 4, 256);
    l.total = align_up(l.row_best + (size_t)B * R * 8, 256);
    return l;
}

template <bool BF16, bool SAMPLE>
cudaError_t launch_one(const AcceptArgs& a, int nseg, bool aligned, float c_exp, AcceptWs ws,
                       cudaStream_t s) {
    auto kern = accept_kernel<BF16, SAMPLE>;
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaGetDevice(&dev);
    std::call_once(once[dev & 63], [&] {
        attr_err[dev & 63] =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    // the walks stage [tok | chosen] of as many sequences as the rings hold
    const int R = a.N + 1;
    const int seq_batch =
        std::max(1, std::min(a.B, kRingBytes / ((4 * R + 1) * (int)sizeof(int))));
    // One CTA per SM.  The rows' segments, flattened, are cut into equal
    // chunks of spc segments, kChunksPerWarp per warp of the wave, dealt
    // round-robin: every warp streams the same number of segments, and rows
    // complete wave by wave.
    const long segs = (long)a.B * R * nseg;
    const long slots = (long)num_sms_accept();
    const long want = kChunksPerWarp * slots * (SAMPLE ? kWarps - 1 : kWarps);
    const long spc = std::max(1L, (segs + want - 1) / want);
    const long chunks = (segs + spc - 1) / spc;
    const int grid = (int)std::max(1L, std::min(slots, (chunks + kWarps - 1) / kWarps));
    return launch_pdl(kern, dim3(grid), dim3(kThreads), (size_t)kSmemBytes, s, a.logits, a.V,
                      a.row_stride, nseg, spc, aligned, a.B, seq_batch, a.parent, a.token,
                      a.n_nodes, a.L, a.N, c_exp, a.seed, a.step, a.target_token, a.accept_len,
                      a.accepted_nodes, a.out_tokens, a.next_bonus, ws, a.err);
}

}  // namespace

bool accept_supported(int V, int dtype) { return accept_segs(V, dtype) <= kMaxSegs; }

size_t accept_workspace_bytes(int B, int N, int V, int dtype) {
    return accept_layout(B, N, accept_segs(V, dtype)).total;
}

cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s) {
    const int nseg = accept_segs(a.V, a.dtype);
    const WsLayout l = accept_layout(a.B, a.N, nseg);
    char* base = (char*)a.ws;
    AcceptWs ws{(unsigned int*)(base + l.row_cnt), (unsigned int*)(base + l.done),
                (float2*)(base + l.parts), (int32_t*)(base + l.tok),
                (unsigned long long*)(base + l.row_best)};
    const int es = a.dtype == DDTREE_BF16 ? 2 : 4;
    const bool aligned = ((uintptr_t)a.logits % 16 == 0) && ((a.row_stride * es) % 16 == 0);
    const bool sample = a.temperature > 0.f;
    const float c_exp = sample ? kLog2e / a.temperature : 0.f;
    if (a.dtype == DDTREE_BF16)
        return sample ? launch_one<true, true>(a, nseg, aligned, c_exp, ws, s)
                      : launch_one<true, false>(a, nseg, aligned, c_exp, ws, s);
    return sample ? launch_one<false, true>(a, nseg, aligned, c_exp, ws, s)
                  : launch_one<false, false>(a, nseg, aligned, c_exp, ws, s);
}

}  // namespace ddt
