// accept_path.cu -- the acceptance walk reading only the rows on the accepted
// path ("Accelerating Speculative Decoding with Block Diffusion Draft Trees",
// §4.1: the walk follows the target's decoding rule from the root; a node's
// target token decides which child, if any, is accepted next).
//
// The full-tree accept resolves the target's token at every node; the walk
// only ever needs it at the root and at the accepted nodes, at most L + 1 of
// the N + 1 rows.  Here one CTA per sequence walks level by level: it streams
// the current node's logit row through a ring of shared-memory stages filled
// by bulk copies, resolves that row's token (greedy argmax, or the same
// inverse-CDF sample with the same Philox uniform as the full-tree kernel),
// looks up the child carrying that token and moves to it.  HBM traffic per
// sequence: (accept_len + 1) x V x elem instead of (n + 1) x V x elem; the
// price is a dependent chain of rows, so it pays when N is much larger than
// the accepted length.  Outputs are those of ddtree_accept; target_token is
// filled on the path only (-1 elsewhere).
#include <mutex>

#include "chunk.cuh"
#include "internal.h"
#include "sampling.cuh"

#include "../../include/ddtree.h"

namespace ddt {

namespace {

constexpr int kThreads = kSampleThreads;
constexpr int kChunkBytes = 32768;
constexpr int kStages = 3;
constexpr int kMaxChunks = 128;

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
accept_path_kernel(const void* __restrict__ logits, int V, int64_t row_stride, int nchunks,
                   bool aligned, const int32_t* __restrict__ parent,
                   const int32_t* __restrict__ token, const int32_t* __restrict__ n_nodes, int L,
                   int N, float temperature, float c_exp, uint64_t seed, uint64_t step,
                   int32_t* __restrict__ target_token, int32_t* __restrict__ accept_len,
                   int32_t* __restrict__ accepted_nodes, int32_t* __restrict__ out_tokens,
                   int32_t* __restrict__ next_bonus, uint32_t* err) {
    using Chunk = SmemChunk<BF16, kChunkBytes / (BF16 ? 2 : 4)>;
    constexpr int VEC = Chunk::VEC;
    constexpr int PER = Chunk::NVEC / kThreads;  // vectors per thread per chunk
    extern __shared__ __align__(128) uint8_t s_ring[];  // kStages x Chunk::BYTES
    __shared__ __align__(8) uint64_t s_bar[kStages];
    __shared__ float2 s_part[kMaxChunks];
    __shared__ float s_red[2 * (kThreads / 32)];
    __shared__ unsigned long long s_key[kThreads / 32];
    __shared__ int s_next, s_pick, s_cstar, s_first, s_lastnz;
    __shared__ float s_tloc;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x, R = N + 1;
    const bool sample = temperature > 0.f;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) sm100::mbar_init(&s_bar[s], 1);
        sm100::mbar_init_fence();
    }
    __syncthreads();
    pdl_wait();
    const int n = n_nodes[b];
    if (n < 0 || n > N) {
        if (tid == 0) record_error(err, ERR_ACCEPT | ERR_BAD_N_NODES);
        return;
    }
    if (target_token)
        for (int u = tid; u < R; u += kThreads) target_token[(size_t)b * R + u] = -1;
    const int32_t* par = parent + (size_t)b * R;
    const int32_t* tk = token + (size_t)b * R;

    int jg = 0;  // chunks issued so far through the ring (stage = jg % kStages)
    int cur = 0, len = 0, bonus = 0;
    for (;;) {
        const char* rowp = (const char*)logits + ((size_t)b * R + cur) * (size_t)row_stride * Chunk::ES;
        auto issue = [&](int c, int j) {
            Chunk::issue_ring(s_ring + (j % kStages) * Chunk::BYTES, &s_bar[j % kStages], rowp,
                              c * Chunk::SIZE, V, aligned);
        };
        for (int c = 0; c < kStages - 1 && c < nchunks; ++c) issue(c, jg + c);
        unsigned long long best = 0ull;  // greedy: (value, lowest index) key
        for (int c = 0; c < nchunks; ++c) {
            const int j = jg + c;
            if (c + kStages - 1 < nchunks) issue(c + kStages - 1, j + kStages - 1);
            if (!Chunk::wait_ring(&s_bar[j % kStages], (uint32_t)((j / kStages) & 1))) {
                if (tid == 0) record_error(err, ERR_ACCEPT | ERR_WAIT_TIMEOUT);
                return;
            }
            const uint4* vec = reinterpret_cast<const uint4*>(s_ring + (j % kStages) * Chunk::BYTES);
            const int c0 = c * Chunk::SIZE;
            if (!sample) {
                // the thread's first maximum in token order: a vector is unpacked
                // only when its maximum beats the best so far
                float bv = best ? key_value(best) : -INFINITY;
#pragma unroll
                for (int i = 0; i < PER; ++i) {
                    const int v = tid + i * kThreads;
                    const float vm = Chunk::vmax(vec[v]);
                    if (vm > bv) {
                        float x[VEC];
                        Chunk::unpack(vec[v], x);
                        int e = -1;
#pragma unroll
                        for (int k = VEC - 1; k >= 0; --k)
                            if (x[k] == vm && c0 + v * VEC + k < V) e = c0 + v * VEC + k;
                        if (e >= 0) {
                            best = value_index_key(vm, (uint32_t)e);
                            bv = vm;
                        }
                    }
                }
            } else {
                // chunk maximum m_c and s_c = sum 2^((x - m_c) c), as in the full-tree kernel
                float tmax = -INFINITY;
#pragma unroll
                for (int i = 0; i < PER; ++i) tmax = fmaxf(tmax, Chunk::vmax(vec[tid + i * kThreads]));
                const float wmax = warp_max(tmax);
                if (lane == 0) s_red[warp] = wmax;
                __syncthreads();
                float cmax = s_red[0];
#pragma unroll
                for (int i = 1; i < kThreads / 32; ++i) cmax = fmaxf(cmax, s_red[i]);
                const float ref = (cmax == -INFINITY) ? 0.f : cmax;
                const float off = -ref * c_exp;
                float ts = 0.f;
#pragma unroll
                for (int i = 0; i < PER; ++i) {
                    float x[VEC];
                    Chunk::unpack(vec[tid + i * kThreads], x);
#pragma unroll
                    for (int k = 0; k < VEC; ++k) ts += fast_exp2(fmaf(x[k], c_exp, off));
                }
                const float wsum = warp_sum(ts);
                if (lane == 0) s_red[kThreads / 32 + warp] = wsum;
                __syncthreads();
                if (tid == 0) {
                    float csum = 0.f;
                    for (int i = 0; i < kThreads / 32; ++i) csum += s_red[kThreads / 32 + i];
                    s_part[c] = make_float2(cmax, csum);
                }
            }
            __syncthreads();  // the stage (and the reduction scratch) are free again
        }
        jg += nchunks;

        // ---- the row's token ----
        int t;
        if (!sample) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) best = umax64(best, shfl_xor_u64(best, o));
            if (lane == 0) s_key[warp] = best;
            __syncthreads();
            unsigned long long k = s_key[0];
#pragma unroll
            for (int i = 1; i < kThreads / 32; ++i) k = umax64(k, s_key[i]);
            t = (int)key_index(k);
        } else {
            if (tid == 0) {
                // the chunk sums combined in fp64; the chunk where U Z is crossed
                float M = -INFINITY;
                for (int c = 0; c < nchunks; ++c) M = fmaxf(M, s_part[c].x);
                double Z = 0.0;
                for (int c = 0; c < nchunks; ++c)
                    Z += (double)s_part[c].y * (double)fast_exp2((s_part[c].x - M) * c_exp);
                const double target = (double)node_uniform(seed, step, (uint64_t)b, (uint64_t)cur) * Z;
                double cum = 0.0;
                int cs = nchunks - 1;
                float tloc = 0.f;
                for (int c = 0; c < nchunks; ++c) {
                    const double scale = (double)fast_exp2((s_part[c].x - M) * c_exp);
                    const double contrib = (double)s_part[c].y * scale;
                    if (cum + contrib > target || c == nchunks - 1) {
                        cs = c;
                        tloc = (scale > 0.0) ? (float)((target - cum) / scale) : 0.f;
                        break;
                    }
                    cum += contrib;
                }
                s_cstar = cs;
                s_tloc = tloc;
                s_first = 0x7fffffff;
                s_lastnz = -1;
            }
            __syncthreads();
            const int cs = s_cstar;
            const float tloc = s_tloc;
            const float mref = fmaxf(s_part[cs].x, -3.0e38f);
            // rescan chunk cs (from L2) with a contiguous segment per thread
            constexpr int SEG = Chunk::SIZE / kThreads;
            const int e0 = cs * Chunk::SIZE + tid * SEG;
            auto weight = [&](int e) {
                float v = -INFINITY;
                if (e < V) {
                    if (BF16) v = bf16lo((uint32_t)__ldcg((const unsigned short*)rowp + e));
                    else v = __ldcg((const float*)rowp + e);
                }
                return fast_exp2((v - mref) * c_exp);
            };
            float tsum = 0.f;
#pragma unroll 8
            for (int i = 0; i < SEG; ++i) tsum += weight(e0 + i);
            float total;
            const float before = block_exclusive_scan(tsum, s_red, total);
            if (tsum > 0.f) {
                if (tloc < before + tsum) atomicMin(&s_first, tid);
                atomicMax(&s_lastnz, tid);
            }
            __syncthreads();
            const int owner = (s_first != 0x7fffffff) ? s_first : s_lastnz;
            if (tid == owner) {
                float acc = before;
                int p = -1, lastnz = -1;
                for (int i = 0; i < SEG; ++i) {
                    const float wt = weight(e0 + i);
                    acc += wt;
                    if (p < 0 && acc > tloc) p = e0 + i;
                    if (wt > 0.f) lastnz = e0 + i;
                }
                s_pick = (p >= 0) ? p : lastnz;
            }
            if (owner < 0 && tid == 0) s_pick = cs * Chunk::SIZE;
            __syncthreads();
            t = s_pick;
        }
        if (tid == 0) {
            if (target_token) target_token[(size_t)b * R + cur] = t;
            s_next = 0x7fffffff;
        }
        __syncthreads();
        // ---- the child of cur carrying token t (children have distinct tokens) ----
        for (int c = 1 + tid; c <= n; c += kThreads)
            if (par[c] == cur && tk[c] == t) atomicMin(&s_next, c);
        __syncthreads();
        const int next = s_next;
        if (next == 0x7fffffff || len >= L) {
            bonus = t;
            break;
        }
        if (tid == 0) {
            accepted_nodes[(size_t)b * L + len] = next;
            out_tokens[(size_t)b * (L + 1) + len] = tk[next];
        }
        ++len;
        cur = next;
        __syncthreads();
    }
    if (tid == 0) {
        for (int i = len; i < L; ++i) accepted_nodes[(size_t)b * L + i] = -1;
        out_tokens[(size_t)b * (L + 1) + len] = bonus;
        for (int i = len + 1; i <= L; ++i) out_tokens[(size_t)b * (L + 1) + i] = -1;
        accept_len[b] = len;
        next_bonus[b] = bonus;
    }
    pdl_trigger();
}

int path_chunks(int V, int dtype) {
    const int size = kChunkBytes / (dtype == DDTREE_BF16 ? 2 : 4);
    return (V + size - 1) / size;
}

template <bool BF16>
cudaError_t launch_path(const AcceptArgs& a, int nch, bool aligned, float c_exp, cudaStream_t s) {
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t ring = (size_t)kStages * kChunkBytes;
    std::call_once(once[dev & 63], [&] {
        attr_err[dev & 63] = cudaFuncSetAttribute(
            accept_path_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ring);
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    return launch_pdl(accept_path_kernel<BF16>, dim3(a.B), dim3(kThreads), ring, s, a.logits, a.V,
                      a.row_stride, nch, aligned, a.parent, a.token, a.n_nodes, a.L, a.N,
                      a.temperature, c_exp, a.seed, a.step, a.target_token, a.accept_len,
                      a.accepted_nodes, a.out_tokens, a.next_bonus, a.err);
}

}  // namespace

bool accept_path_supported(int V, int dtype) { return path_chunks(V, dtype) <= kMaxChunks; }

cudaError_t launch_accept_path(const AcceptArgs& a, cudaStream_t s) {
    const int nch = path_chunks(a.V, a.dtype);
    const int es = a.dtype == DDTREE_BF16 ? 2 : 4;
    const bool aligned = ((uintptr_t)a.logits % 16 == 0) && ((a.row_stride * es) % 16 == 0);
    const float c_exp = a.temperature > 0.f ? kLog2e / a.temperature : 0.f;
    return a.dtype == DDTREE_BF16 ? launch_path<true>(a, nch, aligned, c_exp, s)
                                  : launch_path<false>(a, nch, aligned, c_exp, s);
}

}  // namespace ddt
