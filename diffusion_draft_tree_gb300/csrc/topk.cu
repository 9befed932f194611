// topk.cu -- step 1 of a DDTree round: per-position log-softmax and top-K of
// the draft logits ("Accelerating Speculative Decoding with Block Diffusion
// Draft Trees", §3 marginals q_i; §4.3 log-probabilities; App. A restricted
// prefix set).
//
// One row = one (sequence, draft position), V logits, split into chunks (32 KB
// = 16384 bf16 or 8192 fp32 logits; 16 KB when that many chunks still fit in
// one wave).  A persistent wave of CTAs streams the (row, chunk) list, each
// CTA a contiguous run of chunks through a ring of shared-memory stages
// filled by bulk copies a few chunks ahead, so HBM is read once and stays
// busy.  Per chunk, each warp makes one pass over its eighth in shared memory:
// every vector's maximum, and each lane's online (max, sum of exponentials).
// The chunk's K best keys need no sort here: every warp sorts the few vector
// maxima of its slice above its K-th largest lane maximum and publishes its K
// largest; tau, the K-th largest of those lists, is the K-th largest vector
// maximum of the chunk -- K distinct elements are >= it -- so the chunk keeps
// only its (value, index) keys >= tau (usually K to 1.5K), together with its
// (m, s) and tau.  Any chunk's tau bounds its row's K-th largest from below,
// so a CTA's later chunks of a row it has already met skip the sorts: they
// keep their keys >= the bound found so far and report it as their tau.  A
// second, PDL-chained kernel (one CTA per row) bounds the row's K-th largest
// by the largest chunk tau, ranks the kept keys above it by counting, and
// forms the logsumexp.
#include <mutex>

#include "chunk.cuh"
#include "internal.h"

#include "../../include/ddtree.h"

namespace ddt {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
// Chunks are 32 KB when there are enough to keep every CTA streaming, else
// 16 KB (twice the CTAs, half the work per warp: lower latency).
constexpr int kChunkBig = 32768, kChunkSmall = 16384;
constexpr int kMaxChunks = 128;  // per row, at the small size
constexpr int kStages = 3;       // chunks in flight per CTA
constexpr int kCtasPerSm = 2;
constexpr int kMergeCand = 1024; // candidates the merge gathers before its slow path

// Warp-wide bitonic sort of one uint32 per lane, descending (lane 0 largest).
DDT_DEV uint32_t warp_sort_desc_u32(uint32_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const uint32_t o = __shfl_xor_sync(0xffffffffu, v, j);
            const bool keep_max = (((lane & k) == 0) == ((lane & j) == 0));
            v = keep_max ? max(v, o) : min(v, o);
        }
    }
    return v;
}

// Merges (m, s) pairs: s2 rescaled to the larger maximum (exp base 2^(x c)).
DDT_DEV void ms_combine(float& m, float& s, float m2, float s2, float c) {
    const float mx = fmaxf(m, m2);
    s = (m == -INFINITY ? 0.f : s * fast_exp2((m - mx) * c)) +
        (m2 == -INFINITY ? 0.f : s2 * fast_exp2((m2 - mx) * c));
    m = mx;
}

// Per chunk, the streaming kernel leaves its (m, s), a bound tau on its K-th
// largest value (as an order key) and every key >= tau -- usually K to 2K of
// them, at most kChunkCand; a chunk with more (degenerate ties) keeps exactly
// its K best, sorted, and sets tau to the K-th.
constexpr int kChunkCand = 64;
struct ChunkOut {
    float m, s;       // max, sum exp(x - m)
    uint32_t tau;     // ord key: the chunk has >= K elements >= it
    int count;        // keys below
    uint64_t keys[kChunkCand];
};

// Exact K best keys of a chunk by K rounds of a CTA-wide maximum below the
// previous one (all threads call it; correctness only, kept out of line).
// Thread 0 writes them to out->keys.
template <typename Chunk>
__device__ __noinline__ void cta_exact_top_k(const uint4* vec, int c0, int V, int K,
                                             uint64_t* s_red, ChunkOut* out) {
    constexpr int VEC = Chunk::VEC;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint64_t prev = ~0ull;
    for (int r = 0; r < K; ++r) {
        uint64_t tb = 0ull;
#pragma unroll 1
        for (int v = tid; v < Chunk::NVEC; v += kThreads) {
            float x[VEC];
            Chunk::unpack(vec[v], x);
            for (int k = 0; k < VEC; ++k) {
                const int e = c0 + v * VEC + k;
                if (e < V) {
                    const uint64_t key = value_index_key(x[k], (uint32_t)e);
                    if (key < prev && key > tb) tb = key;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tb = umax64(tb, shfl_xor_u64(tb, o));
        if (lane == 0) s_red[warp] = tb;
        __syncthreads();
        tb = s_red[0];
        for (int i = 1; i < kWarps; ++i) tb = umax64(tb, s_red[i]);
        if (tid == 0) out->keys[r] = tb;
        prev = tb;
        __syncthreads();
    }
    if (tid == 0) {
        out->count = K;
        out->tau = (uint32_t)(prev >> 32);
    }
}

// Persistent: CTA i handles chunks [i per, (i+1) per) of the flattened
// (row, chunk) list, streaming them through a ring of kStages shared-memory
// stages (bulk copies issued kStages-1 chunks ahead), and writes one ChunkOut
// per chunk.  Warps own eighths of the chunk until the chunk's tau is known.
template <bool BF16, int CHUNK_BYTES>
__global__ void __launch_bounds__(kThreads)
topk_kernel(const void* __restrict__ logits, int V, int64_t row_stride, int K, int nchunks,
            bool aligned, int total, int per, ChunkOut* __restrict__ outs, uint32_t* err) {
    using Chunk = SmemChunk<BF16, CHUNK_BYTES / (BF16 ? 2 : 4)>;
    constexpr int VEC = Chunk::VEC;
    constexpr int VPW = Chunk::NVEC / kWarps;  // vectors per warp
    constexpr int PL = VPW / 32;               // vectors per lane
    extern __shared__ __align__(128) uint8_t s_ring[];  // kStages x Chunk::BYTES
    __shared__ __align__(8) uint64_t s_bar[kStages];
    __shared__ float2 s_wms[kWarps];
    __shared__ uint64_t s_red[kWarps];
    __shared__ int16_t s_vlist[kWarps][Chunk::NVEC / kWarps];  // passing vector ids per warp
    __shared__ uint32_t s_vm[kWarps][32];                      // a warp's top vector maxima
    __shared__ int s_cnt;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int w0 = blockIdx.x * per;
    const int nmine = min(total, w0 + per) - w0;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) sm100::mbar_init(&s_bar[s], 1);
        sm100::mbar_init_fence();
    }
    __syncthreads();
    pdl_wait();
    auto issue = [&](int j) {  // chunk j of this CTA into stage j % kStages
        const int w = w0 + j, row = w / nchunks, chunk = w - row * nchunks;
        Chunk::issue_ring(s_ring + (j % kStages) * Chunk::BYTES, &s_bar[j % kStages],
                          (const char*)logits + (size_t)row * (size_t)row_stride * Chunk::ES,
                          chunk * Chunk::SIZE, V, aligned);
    };
    for (int j = 0; j < kStages - 1 && j < nmine; ++j) issue(j);
    uint32_t tau_run = 0u;  // a bound <= the current row's K-th largest (0: none yet)
    for (int j = 0; j < nmine; ++j) {
        if (j + kStages - 1 < nmine) issue(j + kStages - 1);  // into the stage freed last step
        if (j == nmine - 1) pdl_trigger();
        const int w = w0 + j;
        const int c0 = (w % nchunks) * Chunk::SIZE;
        if (c0 == 0) tau_run = 0u;  // a new row
        ChunkOut* out = outs + w;
        if (tid == 0) s_cnt = 0;
        if (!Chunk::wait_ring(&s_bar[j % kStages], (uint32_t)((j / kStages) & 1))) {
            if (tid == 0) record_error(err, ERR_TOPK | ERR_WAIT_TIMEOUT);
            // A copy never landed.  Give every copy still in flight into this
            // CTA's ring (chunks j .. j+kStages-1) one more bounded wait before
            // the shared memory is released; then leave.
            for (int jj = j; jj < min(nmine, j + kStages); ++jj)
                Chunk::wait_ring(&s_bar[jj % kStages], (uint32_t)((jj / kStages) & 1));
            return;
        }
        const uint4* vec = reinterpret_cast<const uint4*>(s_ring + (j % kStages) * Chunk::BYTES);
        const uint4* vw = vec + warp * VPW;
        const int e_lane = c0 + (warp * VPW + lane) * VEC;  // first element of the lane

        // ---- one pass: vector maxima, and the lane's online (max, sum of exps) ----
        float vmx[PL];
        float mt = -INFINITY, a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = 0; i < PL; ++i) {
            const uint4 v = vw[lane + 32 * i];
            const float vm = Chunk::vmax(v);
            vmx[i] = vm;
            if (vm > mt) {
                const float f = fast_exp2((mt - vm) * kLog2e);  // 0 while mt = -inf
                a0 *= f;
                a1 *= f;
                mt = vm;
            }
            if (mt != -INFINITY) Chunk::exp_sum(v, kLog2e, -mt * kLog2e, a0, a1);
        }
        float m_w = mt, s_w = a0 + a1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, m_w, o);
            const float so = __shfl_xor_sync(0xffffffffu, s_w, o);
            ms_combine(m_w, s_w, mo, so, kLog2e);
        }
        if (lane == 0) s_wms[warp] = make_float2(m_w, s_w);

        // The chunk's keys >= tv, from the vectors whose maximum reaches it: their
        // ids are compacted per warp first (a ballot per vector row), so each
        // passing vector is unpacked by one lane instead of the whole warp
        // stepping through every row in which any lane passes.  Counts them in
        // s_cnt; stores the first kChunkCand.
        auto gather = [&](float tv) {
            int nv = 0;
#pragma unroll
            for (int i = 0; i < PL; ++i) {
                const unsigned bal = __ballot_sync(0xffffffffu, vmx[i] >= tv);
                if (vmx[i] >= tv) s_vlist[warp][nv + __popc(bal & ((1u << lane) - 1u))] = (int16_t)(lane + 32 * i);
                nv += __popc(bal);
            }
            __syncwarp();
            for (int b0 = 0; b0 < nv; b0 += 32) {
                const int v = b0 + lane < nv ? s_vlist[warp][b0 + lane] : -1;
                float x[VEC];
                int mine = 0;
                const int e = c0 + (warp * VPW + v) * VEC;
                if (v >= 0) {
                    Chunk::unpack(vw[v], x);
#pragma unroll
                    for (int k = 0; k < VEC; ++k) mine += (x[k] >= tv && e + k < V) ? 1 : 0;
                }
                int incl = mine;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                int wbase = 0;
                if (lane == 31 && incl > 0) wbase = atomicAdd(&s_cnt, incl);
                wbase = __shfl_sync(0xffffffffu, wbase, 31);
                if (mine) {
                    int pos = wbase + incl - mine;
#pragma unroll
                    for (int k = 0; k < VEC; ++k) {
                        if (x[k] >= tv && e + k < V) {
                            if (pos < kChunkCand) out->keys[pos] = value_index_key(x[k], (uint32_t)(e + k));
                            ++pos;
                        }
                    }
                }
            }
        };

        // A later chunk of the row this CTA already met: every key below tau_run
        // (an earlier chunk's bound) is out of the row's K best, so the chunk
        // keeps its keys >= tau_run and reports tau_run as its bound -- valid for
        // the merge, which needs only a bound <= the row's K-th largest and every
        // key >= it.  Too many such keys: the chunk takes the full path below.
        bool cheap = false;
        int cnt = 0;
        if (tau_run != 0u) {
            gather(float_from_ord(tau_run));
            __syncthreads();
            cnt = s_cnt;
            cheap = cnt <= kChunkCand;
            if (!cheap) {
                __syncthreads();  // every thread has read the count
                if (tid == 0) s_cnt = 0;
            }
        }
        uint32_t tau = tau_run;
        if (!cheap) {
            // The warp's K largest vector maxima (K distinct elements), descending,
            // into s_vm[warp]: the vector maxima at or above the K-th largest lane
            // maximum (usually K to 3K) sorted by the warp; if there are too many,
            // K copies of that lane bound (still K elements >= each).
            {
                const uint32_t tau_l = warp_kth_largest(e_lane < V ? ord_from_float(mt) : 0u, K);
                const float tl = (tau_l == 0u) ? -INFINITY : float_from_ord(tau_l);
                int nm = 0;
#pragma unroll
                for (int i = 0; i < PL; ++i) {
                    const bool in = vmx[i] >= tl && e_lane + 32 * i * VEC < V;
                    const unsigned bal = __ballot_sync(0xffffffffu, in);
                    const int at = nm + __popc(bal & ((1u << lane) - 1u));
                    if (in && at < 32) s_vm[warp][at] = ord_from_float(vmx[i]);
                    nm += __popc(bal);
                }
                __syncwarp();
                uint32_t top = tau_l;
                if (nm <= 32) top = warp_sort_desc_u32(lane < nm ? s_vm[warp][lane] : 0u);
                __syncwarp();
                if (lane < K) s_vm[warp][lane] = top;
            }
            __syncthreads();
            // tau: the K-th largest of the warps' lists (each warp, redundantly),
            // a bound on the chunk's K-th largest value
            {
                int ptr = 0;
                uint32_t head = lane < kWarps ? s_vm[lane][0] : 0u;
                for (int r = 0; r < K; ++r) {
                    tau = __reduce_max_sync(0xffffffffu, head);
                    const unsigned holders = __ballot_sync(0xffffffffu, head == tau);
                    if (lane == __ffs(holders) - 1) {
                        ++ptr;
                        head = ptr < K ? s_vm[lane][ptr] : 0u;
                    }
                }
            }
            gather((tau == 0u) ? -INFINITY : float_from_ord(tau));
            __syncthreads();
            cnt = s_cnt;
            if (cnt > kChunkCand) {
                cta_exact_top_k<Chunk>(vec, c0, V, K, s_red, out);  // degenerate ties
            } else {
                tau_run = max(tau_run, tau);  // (uniform: every warp computed tau)
            }
        }
        if (tid == 0) {
            if (cnt <= kChunkCand) {
                out->count = cnt;
                out->tau = tau;
            }
            float m = s_wms[0].x, sm = s_wms[0].y;
#pragma unroll
            for (int i = 1; i < kWarps; ++i) ms_combine(m, sm, s_wms[i].x, s_wms[i].y, kLog2e);
            out->m = m;
            out->s = sm;
        }
        __syncthreads();  // the stage and the shared counters are free again
    }
}

// One CTA per row merges the row's chunk outputs.  Every chunk holds >= K
// elements >= its tau, so the row's K best keys are >= tau2 = max over chunks
// of tau; the kept keys >= tau2 are gathered and each is ranked by counting
// the larger ones (the K of rank < K are the answer, in order).  The
// logsumexp combines the chunks' (max, sum) pairs.  Each thread issues a batch
// of kMergeLoads key loads before using any.
constexpr int kMergeThreads = 256;
constexpr int kMergeLoads = 8;
__global__ void __launch_bounds__(kMergeThreads)
topk_merge_kernel(const ChunkOut* __restrict__ outs, int nchunks, int K,
                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_logp,
                  float* __restrict__ lse) {
    __shared__ __align__(16) uint64_t s_c[kMergeCand];
    __shared__ uint64_t s_sel[DDTREE_MAX_K];
    __shared__ int s_n[kMaxChunks];
    __shared__ uint32_t s_tau[kMergeThreads / 32];
    __shared__ float2 s_ms[kMergeThreads / 32];
    __shared__ int s_cnt;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.x;
    if (tid == 0) s_cnt = 0;
    if (tid < K) s_sel[tid] = 0ull;
    pdl_wait();
    const ChunkOut* ro = outs + (size_t)row * nchunks;
    // the first batch of key slots is loaded with the chunk headers (one round
    // trip); slots past a chunk's count are dropped once the counts are known
    const int nslots = nchunks * kChunkCand;
    uint64_t kv0[kMergeLoads];
#pragma unroll
    for (int u = 0; u < kMergeLoads; ++u) {
        const int i = u * kMergeThreads + tid;
        kv0[u] = i < nslots ? __ldcg((const unsigned long long*)&ro[i / kChunkCand].keys[i % kChunkCand])
                            : 0ull;
    }
    uint32_t tau2 = 0u;
    float mt = -INFINITY, st = 0.f;
    for (int c = tid; c < nchunks; c += kMergeThreads) {
        tau2 = max(tau2, __ldcg(&ro[c].tau));
        ms_combine(mt, st, __ldcg(&ro[c].m), __ldcg(&ro[c].s), kLog2e);
        s_n[c] = min(__ldcg(&ro[c].count), kChunkCand);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        tau2 = max(tau2, __shfl_xor_sync(0xffffffffu, tau2, o));
        const float mo = __shfl_xor_sync(0xffffffffu, mt, o);
        const float so = __shfl_xor_sync(0xffffffffu, st, o);
        ms_combine(mt, st, mo, so, kLog2e);
    }
    if (lane == 0) {
        s_tau[warp] = tau2;
        s_ms[warp] = make_float2(mt, st);
    }
    __syncthreads();
    tau2 = s_tau[0];
    mt = s_ms[0].x;
    st = s_ms[0].y;
#pragma unroll
    for (int i = 1; i < kMergeThreads / 32; ++i) {
        tau2 = max(tau2, s_tau[i]);
        ms_combine(mt, st, s_ms[i].x, s_ms[i].y, kLog2e);
    }
    pdl_trigger();
    // gather the kept keys >= tau2 (slot k of chunk c is index c * kChunkCand + k)
    for (int b0 = 0; b0 < nslots; b0 += kMergeLoads * kMergeThreads) {
        uint64_t kv[kMergeLoads];
#pragma unroll
        for (int u = 0; u < kMergeLoads; ++u) {
            const int i = b0 + u * kMergeThreads + tid;
            const int c = i / kChunkCand, k = i - c * kChunkCand;
            if (b0 == 0) kv[u] = (i < nslots && k < s_n[c]) ? kv0[u] : 0ull;
            else kv[u] = (i < nslots && k < s_n[c])
                             ? __ldcg((const unsigned long long*)&ro[c].keys[k]) : 0ull;
        }
#pragma unroll
        for (int u = 0; u < kMergeLoads; ++u) {
            if (kv[u] != 0ull && (uint32_t)(kv[u] >> 32) >= tau2) {
                const int at = atomicAdd(&s_cnt, 1);
                if (at < kMergeCand) s_c[at] = kv[u];
            }
        }
    }
    __syncthreads();
    const int cnt = s_cnt;
    if (cnt <= kMergeCand) {
        for (int i = tid; i < cnt; i += kMergeThreads) {
            const uint64_t key = s_c[i];
            const int rank = count_larger(s_c, cnt, key);
            if (rank < K) s_sel[rank] = key;
        }
    } else {
        // Degenerate ties: K rounds of a CTA maximum below the previous one over
        // every kept key (correctness only).
        uint64_t prev = ~0ull;
        for (int r = 0; r < K; ++r) {
            uint64_t tb = 0ull;
            for (int i = tid; i < nslots; i += kMergeThreads) {
                const int c = i / kChunkCand, k = i - c * kChunkCand;
                if (k < s_n[c]) {
                    const uint64_t key = __ldcg((const unsigned long long*)&ro[c].keys[k]);
                    if (key < prev && key > tb) tb = key;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tb = umax64(tb, shfl_xor_u64(tb, o));
            __syncthreads();
            if (lane == 0) s_c[warp] = tb;
            __syncthreads();
            tb = s_c[0];
            for (int i = 1; i < kMergeThreads / 32; ++i) tb = umax64(tb, s_c[i]);
            if (tid == 0) s_sel[r] = tb;
            prev = tb;
        }
    }
    __syncthreads();
    if (warp != 0) return;
    const float M = (mt == -INFINITY) ? 0.f : mt;
    const float logS = logf(st);
    if (lane < K) {
        const uint64_t key = s_sel[lane];
        topk_idx[(size_t)row * K + lane] = (int32_t)key_index(key);
        topk_logp[(size_t)row * K + lane] = (key_value(key) - M) - logS;
    }
    if (lane == 0 && lse) lse[row] = M + logS;
}

int chunks_at(int V, int dtype, int bytes) {
    const int size = bytes / (dtype == DDTREE_BF16 ? 2 : 4);
    return (V + size - 1) / size;
}

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

// Chunks per row: small ones when even those fit in one wave of CTAs.
struct ChunkPlan {
    bool small;
    int nch;
};
ChunkPlan chunk_plan(int rows, int V, int dtype) {
    const long slots = (long)num_sms_topk() * kCtasPerSm;
    const bool small = (long)chunks_at(V, dtype, kChunkSmall) * rows <= slots;
    return {small, chunks_at(V, dtype, small ? kChunkSmall : kChunkBig)};
}

// Workspace: one ChunkOut per (row, chunk).
size_t topk_layout_bytes(int rows, int V, int dtype) {
    return (size_t)rows * chunk_plan(rows, V, dtype).nch * sizeof(ChunkOut);
}

}  // namespace

bool topk_supported(int V, int dtype, int K) {
    return topk_chunks(V, dtype) <= kMaxChunks && K >= 1 && K <= DDTREE_MAX_K;
}

int topk_chunks(int V, int dtype) { return chunks_at(V, dtype, kChunkSmall); }

size_t topk_workspace_bytes(int rows, int V, int dtype, int K) {
    (void)K;
    return topk_layout_bytes(rows, V, dtype);
}

template <bool BF16, int BYTES>
cudaError_t launch_partials(const TopkArgs& a, int nch, bool aligned, int total, int per,
                            ChunkOut* outs, cudaStream_t s) {
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t ring = (size_t)kStages * BYTES;
    std::call_once(once[dev & 63], [&] {
        attr_err[dev & 63] = cudaFuncSetAttribute(
            topk_kernel<BF16, BYTES>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ring);
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    const int grid = (total + per - 1) / per;
    return launch_pdl(topk_kernel<BF16, BYTES>, dim3(grid), dim3(kThreads), ring, s, a.logits,
                      a.V, a.row_stride, a.K, nch, aligned, total, per, outs, a.err);
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s) {
    const int es = a.dtype == DDTREE_BF16 ? 2 : 4;
    const bool aligned = ((uintptr_t)a.logits % 16 == 0) && ((a.row_stride * es) % 16 == 0);
    ChunkOut* outs = (ChunkOut*)a.ws;
    // one wave of persistent CTAs, each streaming a contiguous run of chunks
    const long slots = (long)num_sms_topk() * kCtasPerSm;
    const ChunkPlan cp = chunk_plan(a.rows, a.V, a.dtype);
    const int nch = cp.nch;
    const long total = (long)nch * a.rows;
    const int per = (int)((total + slots - 1) / slots);
    cudaError_t e;
    if (a.dtype == DDTREE_BF16)
        e = cp.small ? launch_partials<true, kChunkSmall>(a, nch, aligned, (int)total, per, outs, s)
                     : launch_partials<true, kChunkBig>(a, nch, aligned, (int)total, per, outs, s);
    else
        e = cp.small ? launch_partials<false, kChunkSmall>(a, nch, aligned, (int)total, per, outs, s)
                     : launch_partials<false, kChunkBig>(a, nch, aligned, (int)total, per, outs, s);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_merge_kernel, dim3(a.rows), dim3(kMergeThreads), 0, s,
                      (const ChunkOut*)outs, nch, a.K, a.topk_idx, a.topk_logp, a.lse);
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
    // (every partial the merge reads is written by the same call: no clearing)
    if (need) {
        const cudaError_t e = noalloc_scratch(&scratch);
        if (e != cudaSuccess) return (ddtree_status)ddt::launch_status(e);
    }
    ddt::TopkArgs a{draft_logits, dtype, rows, V, row_stride, K, topk_idx, topk_logp, lse,
                    scratch, ddt::error_word()};
    return (ddtree_status)ddt::launch_status(ddt::launch_topk(a, (cudaStream_t)stream));
}
