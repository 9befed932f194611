// topk.cu -- step 1 of a DDTree round: per-position log-softmax and top-K of
// the draft logits ("Accelerating Speculative Decoding with Block Diffusion
// Draft Trees", §3 marginals q_i; §4.3 log-probabilities; App. A restricted
// prefix set).
//
// One row = one (sequence, draft position), V logits, split into chunks of
// 32 KB (16384 bf16 or 8192 fp32 logits).  A persistent wave of CTAs streams
// the (row, chunk) list, each CTA a contiguous run of chunks through a ring of
// shared-memory stages filled by bulk copies a few chunks ahead, so HBM is
// read once and stays busy.  Each warp of a CTA owns one eighth of a chunk and
// needs no CTA-wide step: one pass over its vectors in shared memory gives
// every vector's maximum and each lane's online (max, sum of exponentials);
// the warp combines them into its (m, s) and selects its K best (value,
// index) keys without per-element insertion: tau_w, the K-th largest of its
// 32 lane maxima, bounds its K-th largest value from below, so only elements
// >= tau_w (usually about 2K) are gathered and sorted (one warp bitonic sort;
// ranked by counting when more than 32).  Every warp writes one sorted K-list
// with its (m, s).  A second, PDL-chained kernel (one warp per row) merges a
// row's lists the same way -- the keys at or above the largest list-K-th key,
// sorted -- and forms the logsumexp.
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
constexpr int kWarpCand = 64;    // candidates a warp gathers before its slow path
constexpr int kMergeCand = 1024; // candidates the merge gathers before its slow path

// Warp-wide bitonic sort of one uint64 per lane, descending (lane 0 largest).
DDT_DEV uint64_t warp_sort_desc_u64(uint64_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const uint64_t o = __shfl_xor_sync(0xffffffffu, v, j);
            const bool keep_max = (((lane & k) == 0) == ((lane & j) == 0));
            v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
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

// The K largest of up to kWarpCand (or any number, on the slow path) candidate
// keys: lanes < K return them in descending order, the others 0.
// `count` keys are in buf (when count <= cap).
DDT_DEV uint64_t warp_top_k(uint64_t* buf, int count, int cap, int K, uint64_t* sel) {
    const int lane = threadIdx.x & 31;
    if (count <= 32) {
        const uint64_t key = warp_sort_desc_u64(lane < count ? buf[lane] : 0ull);
        return lane < K ? key : 0ull;
    }
    (void)cap;
    if (lane < K) sel[lane] = 0ull;
    __syncwarp();
    for (int i = lane; i < count; i += 32) {
        const uint64_t key = buf[i];
        const int rank = count_larger(buf, count, key);
        if (rank < K) sel[rank] = key;
    }
    __syncwarp();
    const uint64_t key = lane < K ? sel[lane] : 0ull;
    __syncwarp();
    return key;
}

// Persistent: CTA i handles chunks [i per, (i+1) per) of the flattened
// (row, chunk) list, streaming them through a ring of kStages shared-memory
// stages (bulk copies issued kStages-1 chunks ahead).  Every warp selects the
// K best keys and the (m, s) of its eighth of the chunk; warp 0 merges the
// eight into the chunk's list (row, chunk): K keys to keys[list * K], (m, s)
// to ms[list].
template <bool BF16, int CHUNK_BYTES>
__global__ void __launch_bounds__(kThreads)
topk_kernel(const void* __restrict__ logits, int V, int64_t row_stride, int K, int nchunks,
            bool aligned, int total, int per, float2* __restrict__ ms,
            uint64_t* __restrict__ keys, uint32_t* err) {
    using Chunk = SmemChunk<BF16, CHUNK_BYTES / (BF16 ? 2 : 4)>;
    constexpr int VEC = Chunk::VEC;
    constexpr int VPW = Chunk::NVEC / kWarps;  // vectors per warp
    constexpr int PL = VPW / 32;               // vectors per lane
    extern __shared__ __align__(128) uint8_t s_ring[];  // kStages x Chunk::BYTES
    __shared__ __align__(8) uint64_t s_bar[kStages];
    __shared__ __align__(16) uint64_t s_wc[kWarps][kWarpCand];
    __shared__ uint64_t s_wsel[kWarps][DDTREE_MAX_K];
    __shared__ __align__(16) uint64_t s_cc[kWarps * DDTREE_MAX_K];
    __shared__ float2 s_wms[kWarps];

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
    for (int j = 0; j < nmine; ++j) {
        if (j + kStages - 1 < nmine) issue(j + kStages - 1);  // into the stage freed last step
        if (j == nmine - 1) pdl_trigger();
        const int w = w0 + j;
        const int c0 = (w % nchunks) * Chunk::SIZE;
        if (!Chunk::wait_ring(&s_bar[j % kStages], (uint32_t)((j / kStages) & 1))) {
            if (tid == 0) record_error(err, ERR_TOPK | ERR_WAIT_TIMEOUT);
            return;  // a copy never landed
        }
        const uint4* vw = reinterpret_cast<const uint4*>(s_ring + (j % kStages) * Chunk::BYTES) +
                          warp * VPW;
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
        // tau_w: the warp has >= K elements >= it (K lanes' maxima)
        const uint32_t tau_w = warp_kth_largest(e_lane < V ? ord_from_float(mt) : 0u, K);
        const float tv = (tau_w == 0u) ? -INFINITY : float_from_ord(tau_w);
        float m_w = mt, s_w = a0 + a1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, m_w, o);
            const float so = __shfl_xor_sync(0xffffffffu, s_w, o);
            ms_combine(m_w, s_w, mo, so, kLog2e);
        }

        // ---- candidates: elements >= tau_w of the vectors whose maximum reaches it ----
        int mine = 0;
#pragma unroll
        for (int i = 0; i < PL; ++i) {
            if (vmx[i] >= tv) {
                float x[VEC];
                Chunk::unpack(vw[lane + 32 * i], x);
                const int e = e_lane + 32 * i * VEC;
#pragma unroll
                for (int k = 0; k < VEC; ++k) mine += (x[k] >= tv && e + k < V) ? 1 : 0;
            }
        }
        int incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        const int count = __shfl_sync(0xffffffffu, incl, 31);
        uint64_t sel;
        if (count <= kWarpCand) {
            int pos = incl - mine;
#pragma unroll
            for (int i = 0; i < PL; ++i) {
                if (mine && vmx[i] >= tv) {
                    float x[VEC];
                    Chunk::unpack(vw[lane + 32 * i], x);
                    const int e = e_lane + 32 * i * VEC;
#pragma unroll
                    for (int k = 0; k < VEC; ++k)
                        if (x[k] >= tv && e + k < V)
                            s_wc[warp][pos++] = value_index_key(x[k], (uint32_t)(e + k));
                }
            }
            __syncwarp();
            sel = warp_top_k(s_wc[warp], count, kWarpCand, K, s_wsel[warp]);
        } else {
            // Degenerate ties: exact selection, K rounds of a warp maximum below
            // the previous one (rare path; correctness only).
            uint64_t prev = ~0ull;
            sel = 0ull;
            for (int r = 0; r < K; ++r) {
                uint64_t tb = 0ull;
                for (int i = 0; i < PL; ++i) {
                    float x[VEC];
                    Chunk::unpack(vw[lane + 32 * i], x);
                    const int e = e_lane + 32 * i * VEC;
                    for (int k = 0; k < VEC; ++k) {
                        if (e + k < V) {
                            const uint64_t key = value_index_key(x[k], (uint32_t)(e + k));
                            if (key < prev && key > tb) tb = key;
                        }
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) tb = umax64(tb, shfl_xor_u64(tb, o));
                if (lane == r) sel = tb;
                prev = tb;
            }
        }
        if (lane < K) s_wsel[warp][lane] = sel;
        if (lane == 0) s_wms[warp] = make_float2(m_w, s_w);
        __syncthreads();
        if (warp == 0) {
            // the chunk's list: the K best of the warps' lists, keys >= the
            // largest warp-K-th key (that warp alone holds K keys >= it)
            uint64_t tau = lane < kWarps ? s_wsel[lane][K - 1] : 0ull;
            float2 p = lane < kWarps ? s_wms[lane] : make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                tau = umax64(tau, shfl_xor_u64(tau, o));
                const float mo = __shfl_xor_sync(0xffffffffu, p.x, o);
                const float so = __shfl_xor_sync(0xffffffffu, p.y, o);
                ms_combine(p.x, p.y, mo, so, kLog2e);
            }
            int cnt = 0;
            for (int t0 = 0; t0 < kWarps * K; t0 += 32) {
                const int t = t0 + lane, wv = t / K;
                const uint64_t key = t < kWarps * K ? s_wsel[wv][t - wv * K] : 0ull;
                const bool in = key >= tau && key != 0ull;
                const unsigned bal = __ballot_sync(0xffffffffu, in);
                if (in) s_cc[cnt + __popc(bal & ((1u << lane) - 1u))] = key;
                cnt += __popc(bal);
            }
            __syncwarp();
            const uint64_t best = warp_top_k(s_cc, cnt, kWarps * DDTREE_MAX_K, K, s_wsel[0]);
            if (lane < K) keys[(size_t)w * K + lane] = best;
            if (lane == 0) ms[w] = p;
        }
        __syncthreads();  // the stage and the candidate buffers are free again
    }
}

// One warp per row merges the row's nchunks lists.  The row's K best keys are
// >= tau2 = the largest K-th key of any list (that list alone holds K keys >=
// tau2), so only the keys >= tau2 -- usually K to 2K of them -- are gathered
// and sorted (bitonic, or ranked by counting when more than 32).  The
// logsumexp combines the lists' (max, sum) pairs.  Each lane issues its loads
// in batches before using any.
constexpr int kMergeThreads = 32;
constexpr int kMergeLoads = 8;
__global__ void __launch_bounds__(kMergeThreads)
topk_merge_kernel(const float2* __restrict__ ms, const uint64_t* __restrict__ keys, int nlists,
                  int K, int32_t* __restrict__ topk_idx, float* __restrict__ topk_logp,
                  float* __restrict__ lse) {
    __shared__ __align__(16) uint64_t s_c[kMergeCand];
    __shared__ uint64_t s_sel[DDTREE_MAX_K];
    const int lane = threadIdx.x;
    const int row = blockIdx.x;
    pdl_wait();
    const float2* rms = ms + (size_t)row * nlists;
    const uint64_t* rk = keys + (size_t)row * nlists * K;
    const int nk = nlists * K;
    uint64_t kv[kMergeLoads];
#pragma unroll
    for (int u = 0; u < kMergeLoads; ++u) {
        const int t = lane + 32 * u;
        kv[u] = t < nk ? __ldcg((const unsigned long long*)&rk[t]) : 0ull;
    }
    uint64_t tau2 = 0ull;
    float mt = -INFINITY, st = 0.f;
    for (int l = lane; l < nlists; l += 32) {
        tau2 = umax64(tau2, __ldcg((const unsigned long long*)&rk[(size_t)l * K + K - 1]));
        const float2 p = __ldcg(&rms[l]);
        ms_combine(mt, st, p.x, p.y, kLog2e);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        tau2 = umax64(tau2, shfl_xor_u64(tau2, o));
        const float mo = __shfl_xor_sync(0xffffffffu, mt, o);
        const float so = __shfl_xor_sync(0xffffffffu, st, o);
        ms_combine(mt, st, mo, so, kLog2e);
    }
    pdl_trigger();
    int cnt = 0;
    for (int t0 = 0; t0 < nk; t0 += 32 * kMergeLoads) {
        if (t0 > 0) {
#pragma unroll
            for (int u = 0; u < kMergeLoads; ++u) {
                const int t = t0 + lane + 32 * u;
                kv[u] = t < nk ? __ldcg((const unsigned long long*)&rk[t]) : 0ull;
            }
        }
#pragma unroll
        for (int u = 0; u < kMergeLoads; ++u) {
            const bool in = kv[u] >= tau2 && kv[u] != 0ull;
            const unsigned bal = __ballot_sync(0xffffffffu, in);
            const int at = cnt + __popc(bal & ((1u << lane) - 1u));
            if (in && at < kMergeCand) s_c[at] = kv[u];
            cnt += __popc(bal);
        }
    }
    __syncwarp();
    uint64_t sel;
    if (cnt <= kMergeCand) {
        sel = warp_top_k(s_c, cnt, kMergeCand, K, s_sel);
    } else {
        // Degenerate ties: K rounds of a warp maximum below the previous one.
        uint64_t prev = ~0ull;
        sel = 0ull;
        for (int r = 0; r < K; ++r) {
            uint64_t tb = 0ull;
            for (int t = lane; t < nk; t += 32) {
                const uint64_t key = __ldcg((const unsigned long long*)&rk[t]);
                if (key < prev && key > tb) tb = key;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tb = umax64(tb, shfl_xor_u64(tb, o));
            if (lane == r) sel = tb;
            prev = tb;
        }
    }
    const float M = (mt == -INFINITY) ? 0.f : mt;
    const float logS = logf(st);
    if (lane < K) {
        topk_idx[(size_t)row * K + lane] = (int32_t)key_index(sel);
        topk_logp[(size_t)row * K + lane] = (key_value(sel) - M) - logS;
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

struct TopkWs {
    size_t ms, keys, total;
};
// Workspace: (m, s) of every list, then its K keys (K <= 0: room for any K).
TopkWs topk_layout(int rows, int V, int dtype, int K) {
    const size_t lists = (size_t)rows * chunk_plan(rows, V, dtype).nch;
    const size_t kk = (K > 0 && K <= DDTREE_MAX_K) ? (size_t)K : (size_t)DDTREE_MAX_K;
    TopkWs w;
    w.ms = 0;
    w.keys = align_up(lists * sizeof(float2), 256);
    w.total = w.keys + lists * kk * sizeof(uint64_t);
    return w;
}

}  // namespace

bool topk_supported(int V, int dtype, int K) {
    return topk_chunks(V, dtype) <= kMaxChunks && K >= 1 && K <= DDTREE_MAX_K;
}

int topk_chunks(int V, int dtype) { return chunks_at(V, dtype, kChunkSmall); }

size_t topk_workspace_bytes(int rows, int V, int dtype, int K) {
    return topk_layout(rows, V, dtype, K).total;
}

template <bool BF16, int BYTES>
cudaError_t launch_partials(const TopkArgs& a, int nch, bool aligned, int total, int per,
                            float2* ms, uint64_t* keys, cudaStream_t s) {
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
                      a.V, a.row_stride, a.K, nch, aligned, total, per, ms, keys, a.err);
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s) {
    const int es = a.dtype == DDTREE_BF16 ? 2 : 4;
    const bool aligned = ((uintptr_t)a.logits % 16 == 0) && ((a.row_stride * es) % 16 == 0);
    const TopkWs wl = topk_layout(a.rows, a.V, a.dtype, a.K);
    float2* ms = (float2*)((char*)a.ws + wl.ms);
    uint64_t* keys = (uint64_t*)((char*)a.ws + wl.keys);
    // one wave of persistent CTAs, each streaming a contiguous run of chunks
    const long slots = (long)num_sms_topk() * kCtasPerSm;
    const ChunkPlan cp = chunk_plan(a.rows, a.V, a.dtype);
    const bool small = cp.small;
    const int nch = cp.nch;
    const long total = (long)nch * a.rows;
    const int per = (int)((total + slots - 1) / slots);
    cudaError_t e;
    if (a.dtype == DDTREE_BF16)
        e = small ? launch_partials<true, kChunkSmall>(a, nch, aligned, (int)total, per, ms, keys, s)
                  : launch_partials<true, kChunkBig>(a, nch, aligned, (int)total, per, ms, keys, s);
    else
        e = small ? launch_partials<false, kChunkSmall>(a, nch, aligned, (int)total, per, ms, keys, s)
                  : launch_partials<false, kChunkBig>(a, nch, aligned, (int)total, per, ms, keys, s);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_merge_kernel, dim3(a.rows), dim3(kMergeThreads), 0, s,
                      (const float2*)ms, (const uint64_t*)keys, nch, a.K, a.topk_idx,
                      a.topk_logp, a.lse);
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
    const size_t need = ddt::topk_workspace_bytes(rows, V, dtype, K);
    if (need > DDTREE_NOALLOC_SCRATCH_BYTES) return DDTREE_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    // (every partial the merge reads is written by the same call: no clearing)
    if (need && noalloc_scratch(&scratch) != cudaSuccess) return DDTREE_ERR_CUDA;
    ddt::TopkArgs a{draft_logits, dtype, rows, V, row_stride, K, topk_idx, topk_logp, lse,
                    scratch, nullptr};
    return ddt::launch_topk(a, (cudaStream_t)stream) == cudaSuccess ? DDTREE_OK : DDTREE_ERR_CUDA;
}
