// topk.cu -- step 1 of a DDTree round: per-position log-softmax and top-K of
// the draft logits ("Accelerating Speculative Decoding with Block Diffusion
// Draft Trees", §3 marginals q_i; §4.3 log-probabilities; App. A restricted
// prefix set).
//
// One row = one (sequence, draft position), V logits, split into chunks of
// 32 KB (16384 bf16 or 8192 fp32 logits).  A persistent wave of CTAs streams
// the (row, chunk) list, each CTA a contiguous run of chunks through a ring of
// shared-memory stages filled by bulk copies a few chunks ahead, so HBM is
// read once and stays busy.  Per chunk, one pass over shared memory gives
// every vector's maximum and each thread's online (max, sum of exponentials);
// from those come the chunk's m_c = max, s_c = sum exp(x - m_c), and its K
// best (value, index) keys.  Top-K selection avoids per-element insertion:
// every warp finds tau_w, the K-th largest of its 32 lane maxima, the CTA takes
// tau = max_w tau_w -- a lower bound on the chunk's K-th largest value -- and
// only elements >= tau (typically ~2K) are appended to a shared buffer (one
// shared atomic per warp), then sorted by one warp (or ranked by counting when
// there are more than 32).  A second, PDL-chained kernel (one warp per row)
// merges each row's chunk partials the same way -- the keys at or above the
// largest chunk-K-th key, sorted -- and forms the logsumexp.
#include <mutex>

#include "chunk.cuh"
#include "internal.h"

#include "../../include/ddtree.h"

namespace ddt {

namespace {

constexpr int kThreads = 256;
constexpr int kChunkBytes = 32768;
constexpr int kCandCap = 1024;
constexpr int kMaxChunks = 128;
constexpr int kStages = 3;       // chunks in flight per CTA
constexpr int kCtasPerSm = 2;

struct TopkPartial {
    float m;   // chunk max
    float s;   // sum exp(x - m) over the chunk
    uint64_t keys[DDTREE_MAX_K];
};

// Rank of every key of cand[0..cnt) (keys are distinct) by counting the larger
// ones; keys of rank < K land in sel[rank].  Whole CTA; sel must be zeroed.
DDT_DEV void cta_rank_select(const uint64_t* cand, int cnt, int K, uint64_t* sel) {
    for (int i = threadIdx.x; i < cnt; i += kThreads) {
        const uint64_t ki = cand[i];
        const int rank = count_larger(cand, cnt, ki);
        if (rank < K) sel[rank] = ki;
    }
}

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

// Persistent: CTA i handles chunks [i per, (i+1) per) of the flattened
// (row, chunk) list, streaming them through a ring of kStages shared-memory
// stages (bulk copies issued kStages-1 chunks ahead).
template <bool BF16>
__global__ void __launch_bounds__(kThreads)
topk_kernel(const void* __restrict__ logits, int V, int64_t row_stride, int K, int nchunks,
            bool aligned, int total, int per, int32_t* __restrict__ topk_idx,
            float* __restrict__ topk_logp, float* __restrict__ lse,
            TopkPartial* __restrict__ parts, uint32_t* err) {
    using Chunk = SmemChunk<BF16, kChunkBytes / (BF16 ? 2 : 4)>;
    constexpr int VEC = Chunk::VEC;
    constexpr int PER = Chunk::NVEC / kThreads;  // vectors per thread
    extern __shared__ __align__(128) uint8_t s_ring[];  // kStages x Chunk::BYTES
    __shared__ __align__(8) uint64_t s_bar[kStages];
    __shared__ __align__(16) uint64_t s_cand[kCandCap];
    __shared__ uint64_t s_sel[DDTREE_MAX_K];
    __shared__ float s_wmax[kThreads / 32], s_wsum[kThreads / 32];
    __shared__ uint32_t s_wtau[kThreads / 32];
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
    for (int j = 0; j < nmine; ++j) {
        if (j + kStages - 1 < nmine) issue(j + kStages - 1);  // into the stage freed last step
        if (j == nmine - 1) pdl_trigger();
        const int w = w0 + j, row = w / nchunks, chunk = w - row * nchunks;
        const int c0 = chunk * Chunk::SIZE;
        if (tid == 0) s_cnt = 0;
        if (tid < K) s_sel[tid] = 0ull;
        if (!Chunk::wait_ring(&s_bar[j % kStages], (uint32_t)((j / kStages) & 1))) {
            if (tid == 0) record_error(err, ERR_TOPK | ERR_WAIT_TIMEOUT);
            return;  // a copy never landed
        }
        const uint4* vec = reinterpret_cast<const uint4*>(s_ring + (j % kStages) * Chunk::BYTES);

        // ---- one pass over the chunk: every vector's maximum, and per thread an
        // online (max, sum of exponentials), rescaled when its maximum grows ----
        float vmx[PER];
        float mt = -INFINITY;
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const uint4 w = vec[tid + i * kThreads];
            const float vm = Chunk::vmax(w);
            vmx[i] = vm;
            if (vm > mt) {
                const float f = fast_exp2((mt - vm) * kLog2e);  // 0 while mt = -inf
                acc.x *= f;
                acc.y *= f;
                mt = vm;
            }
            if (mt != -INFINITY) Chunk::exp_sum(w, kLog2e, -mt * kLog2e, acc);
        }
        float st = acc.x + acc.y;
        // tau_w = the K-th largest lane maximum of the warp: the chunk has >= K
        // elements >= it, so its top K are among the elements >= tau = max_w tau_w.
        const bool has = c0 + tid * VEC < V;
        const uint32_t tau_w = warp_kth_largest(has ? ord_from_float(mt) : 0u, K);
        // the warp's (max, sum), each lane's sum rescaled to the warp maximum
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, mt, o);
            const float so = __shfl_xor_sync(0xffffffffu, st, o);
            const float mx = fmaxf(mt, mo);
            st = (mt == -INFINITY ? 0.f : st * fast_exp2((mt - mx) * kLog2e)) +
                 (mo == -INFINITY ? 0.f : so * fast_exp2((mo - mx) * kLog2e));
            mt = mx;
        }
        if (lane == 0) {
            s_wmax[warp] = mt;
            s_wsum[warp] = st;
            s_wtau[warp] = tau_w;
        }
        __syncthreads();
        float m = s_wmax[0];
        uint32_t tau = s_wtau[0];
#pragma unroll
        for (int i = 1; i < kThreads / 32; ++i) {
            m = fmaxf(m, s_wmax[i]);
            tau = max(tau, s_wtau[i]);
        }
        const float ref = (m == -INFINITY) ? 0.f : m;
        float S = 0.f;
#pragma unroll
        for (int i = 0; i < kThreads / 32; ++i)
            S += s_wmax[i] == -INFINITY ? 0.f : s_wsum[i] * fast_exp2((s_wmax[i] - ref) * kLog2e);

        // ---- candidates: elements >= tau, from the vectors whose maximum reaches it ----
        const float tv = (tau == 0u) ? -INFINITY : float_from_ord(tau);
        int mine = 0;  // this thread's candidates
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            if (vmx[i] >= tv) {
                const int v = tid + i * kThreads;
                float x[VEC];
                Chunk::unpack(vec[v], x);
#pragma unroll
                for (int k = 0; k < VEC; ++k) mine += (x[k] >= tv && c0 + v * VEC + k < V) ? 1 : 0;
            }
        }
        // one shared atomic per warp reserves the warp's slots
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
            for (int i = 0; i < PER; ++i) {
                const int v = tid + i * kThreads;
                if (vmx[i] >= tv) {
                    float x[VEC];
                    Chunk::unpack(vec[v], x);
#pragma unroll
                    for (int k = 0; k < VEC; ++k) {
                        const int e = c0 + v * VEC + k;
                        if (x[k] >= tv && e < V) {
                            if (pos < kCandCap) s_cand[pos] = value_index_key(x[k], (uint32_t)e);
                            ++pos;
                        }
                    }
                }
            }
        }
        __syncthreads();
        const int cnt = s_cnt;

        if (cnt <= 32) {
            if (warp == 0) {
                const uint64_t key = warp_sort_desc_u64(lane < cnt ? s_cand[lane] : 0ull);
                if (lane < K) s_sel[lane] = key;
            }
        } else if (cnt <= kCandCap) {
            cta_rank_select(s_cand, cnt, K, s_sel);
        } else {
            // Degenerate ties overflowed the buffer: exact K-round selection
            // (rare path; correctness only).
            uint64_t prev = ~0ull;
            for (int r = 0; r < K; ++r) {
                uint64_t tb = 0ull;
                for (int i = 0; i < PER; ++i) {
                    const int v = tid + i * kThreads;
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
                if (lane == 0) s_cand[warp] = tb;
                __syncthreads();
                uint64_t cb = s_cand[0];
                for (int i = 1; i < kThreads / 32; ++i) cb = umax64(cb, s_cand[i]);
                if (tid == 0) s_sel[r] = cb;
                prev = cb;
                __syncthreads();
            }
        }
        __syncthreads();

        const float M = ref;

        if (nchunks > 1) {  // the merge kernel finishes the row
            if (warp == 0) {
                TopkPartial* p = parts + (size_t)row * nchunks + chunk;
                if (lane < K) p->keys[lane] = s_sel[lane];
                if (lane == 0) {
                    p->m = m;
                    p->s = S;
                }
            }
        } else if (warp == 0) {
            const float logS = logf(S);
            if (lane < K) {
                const uint64_t key = s_sel[lane];
                topk_idx[(size_t)row * K + lane] = (int32_t)key_index(key);
                topk_logp[(size_t)row * K + lane] = (key_value(key) - M) - logS;
            }
            if (lane == 0 && lse) lse[row] = M + logS;
        }
        __syncthreads();  // the stage, the candidates and the selection are free again
    }
}

// One warp per row merges its chunk partials.  The row's K best keys are >=
// tau2 = the largest K-th key of any chunk (that chunk alone holds K keys >=
// tau2), so only the keys >= tau2 -- usually K to 2K of them -- are sorted
// (one warp bitonic sort, or ranked by counting when more than 32).  The
// logsumexp combines the chunks' (max, sum) pairs.
constexpr int kMergeThreads = 32;
__global__ void __launch_bounds__(kMergeThreads)
topk_merge_kernel(const TopkPartial* __restrict__ parts, int nchunks, int K,
                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_logp,
                  float* __restrict__ lse) {
    __shared__ __align__(16) uint64_t s_keys[kCandCap];
    __shared__ __align__(16) uint64_t s_c[kCandCap];
    __shared__ uint64_t s_sel[DDTREE_MAX_K];
    const int lane = threadIdx.x;
    const int row = blockIdx.x;
    pdl_wait();
    const TopkPartial* rp = parts + (size_t)row * nchunks;
    const int nk = nchunks * K;
    // every load of the row in one round trip
    constexpr int kPerLane = kMaxChunks / 32;
    uint64_t tau2 = 0ull;
    float cm[kPerLane], cs[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int c = lane + 32 * i;
        cm[i] = -INFINITY;
        cs[i] = 0.f;
        if (c < nchunks) {
            tau2 = umax64(tau2, __ldcg((const unsigned long long*)&rp[c].keys[K - 1]));
            cm[i] = __ldcg(&rp[c].m);
            cs[i] = __ldcg(&rp[c].s);
        }
    }
    for (int t = lane; t < nk; t += 32) {
        const int c = t / K, k = t - c * K;
        s_keys[t] = __ldcg((const unsigned long long*)&rp[c].keys[k]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tau2 = umax64(tau2, shfl_xor_u64(tau2, o));
    float mm = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) mm = fmaxf(mm, cm[i]);
    mm = warp_max(mm);
    const float M = (mm == -INFINITY) ? 0.f : mm;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i)
        ss += (cm[i] == -INFINITY) ? 0.f : cs[i] * fast_exp2((cm[i] - M) * kLog2e);
    ss = warp_sum(ss);
    __syncwarp();
    pdl_trigger();
    // keys >= tau2, compacted in list order
    int cnt = 0;
    for (int t0 = 0; t0 < nk; t0 += 32) {
        const int t = t0 + lane;
        const uint64_t key = t < nk ? s_keys[t] : 0ull;
        const bool in = key >= tau2 && key != 0ull;
        const unsigned bal = __ballot_sync(0xffffffffu, in);
        if (in) s_c[cnt + __popc(bal & ((1u << lane) - 1u))] = key;
        cnt += __popc(bal);
    }
    __syncwarp();
    if (cnt <= 32) {
        const uint64_t key = warp_sort_desc_u64(lane < cnt ? s_c[lane] : 0ull);
        if (lane < K) s_sel[lane] = key;
    } else {
        if (lane < K) s_sel[lane] = 0ull;
        __syncwarp();
        for (int i = lane; i < cnt; i += 32) {
            const uint64_t key = s_c[i];
            const int rank = count_larger(s_c, cnt, key);
            if (rank < K) s_sel[rank] = key;
        }
    }
    __syncwarp();
    const float logS = logf(ss);
    if (lane < K) {
        const uint64_t key = s_sel[lane];
        topk_idx[(size_t)row * K + lane] = (int32_t)key_index(key);
        topk_logp[(size_t)row * K + lane] = (key_value(key) - M) - logS;
    }
    if (lane == 0 && lse) lse[row] = M + logS;
}

int chunk_elems(int dtype) { return kChunkBytes / (dtype == DDTREE_BF16 ? 2 : 4); }

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

}  // namespace

bool topk_supported(int V, int dtype, int K) {
    const int nch = topk_chunks(V, dtype);
    return nch <= kMaxChunks && nch * K <= kCandCap;
}

int topk_chunks(int V, int dtype) {
    const int size = chunk_elems(dtype);
    return (V + size - 1) / size;
}

size_t topk_workspace_bytes(int rows, int V, int dtype) {
    const int nch = topk_chunks(V, dtype);
    if (nch <= 1) return 0;
    return (size_t)rows * nch * sizeof(TopkPartial);
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s) {
    const int nch = topk_chunks(a.V, a.dtype);
    const int es = a.dtype == DDTREE_BF16 ? 2 : 4;
    const bool aligned = ((uintptr_t)a.logits % 16 == 0) && ((a.row_stride * es) % 16 == 0);
    TopkPartial* parts = nch > 1 ? (TopkPartial*)a.ws : nullptr;
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t ring = (size_t)kStages * kChunkBytes;
    std::call_once(once[dev & 63], [&] {
        cudaError_t e = cudaFuncSetAttribute(topk_kernel<true>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ring);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(topk_kernel<false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ring);
        attr_err[dev & 63] = e;
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    // one wave of persistent CTAs, each streaming a contiguous run of chunks
    const long total = (long)nch * a.rows;
    const long slots = (long)num_sms_topk() * kCtasPerSm;
    const int per = (int)((total + slots - 1) / slots);
    const int grid = (int)((total + per - 1) / per);
    auto kern = (a.dtype == DDTREE_BF16) ? topk_kernel<true> : topk_kernel<false>;
    cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kThreads), ring, s, a.logits, a.V,
                               a.row_stride, a.K, nch, aligned, (int)total, per, a.topk_idx,
                               a.topk_logp, a.lse, parts, a.err);
    if (e != cudaSuccess || nch <= 1) return e;
    return launch_pdl(topk_merge_kernel, dim3(a.rows), dim3(kMergeThreads), 0, s,
                      (const TopkPartial*)parts, nch, a.K, a.topk_idx, a.topk_logp, a.lse);
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
    const size_t need = ddt::topk_workspace_bytes(rows, V, dtype);
    if (need > DDTREE_NOALLOC_SCRATCH_BYTES) return DDTREE_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    // (every partial the merge reads is written by the same call: no clearing)
    if (need && noalloc_scratch(&scratch) != cudaSuccess) return DDTREE_ERR_CUDA;
    ddt::TopkArgs a{draft_logits, dtype, rows, V, row_stride, K, topk_idx, topk_logp, lse,
                    scratch, nullptr};
    return ddt::launch_topk(a, (cudaStream_t)stream) == cudaSuccess ? DDTREE_OK : DDTREE_ERR_CUDA;
}
