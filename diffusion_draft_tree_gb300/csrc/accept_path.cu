// accept_path.cu -- the acceptance walk reading only the rows on the accepted
// path ("Accelerating Speculative Decoding with Block Diffusion Draft Trees",
// §4.1: the walk follows the target's decoding rule from the root; a node's
// target token decides which child, if any, is accepted next).
//
// The full-tree accept resolves the target's token at every node; the walk
// only ever needs it at the root and at the accepted nodes, at most L + 1 of
// the N + 1 rows.  Here the walk goes level by level: the current node's logit
// row is resolved (greedy argmax, or the same inverse-CDF sample with the same
// Philox uniform as the full-tree kernel), the child carrying that token is
// looked up, and the walk moves to it.  HBM traffic per sequence is
// (accept_len + 1) x V x elem instead of (n + 1) x V x elem; the price is a
// dependent chain of rows, so each level must be cheap in latency.
//
// A sequence is given a cluster of S CTAs.  CTA r loads chunks r, r + S, ...
// of the row (32 KB each, the full-tree kernel's partition) straight into
// registers, reduces them to its partial (the greedy key, or each chunk's
// (m_c, s_c)) and stores that partial into every CTA's shared memory; after
// one cluster barrier each CTA holds all partials locally and takes the same
// decision.  The gathered partials are double-buffered by level parity, so
// that one barrier per level suffices.  The tree's parents and tokens are
// staged once in shared memory as child lists.  Outputs are those of
// ddtree_accept; target_token is filled on the path only (-1 elsewhere).
#include <algorithm>
#include <mutex>

#include "chunk.cuh"
#include "internal.h"
#include "sampling.cuh"

#include "../../include/ddtree.h"

namespace ddt {

namespace {

constexpr int kThreads = kSampleThreads;
constexpr int kChunkBytes = 32768;
constexpr int kMaxChunks = 128;
constexpr int kMaxCluster = 16;
constexpr int kMaxRows = DDTREE_MAX_N + 1;

// Stores v at the address of `local` in the shared memory of cluster CTA `rank`.
DDT_DEV void st_peer_u64(void* local, int rank, unsigned long long v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(
                     sm100::mapa_shared(sm100::smem_u32(local), (uint32_t)rank)),
                 "l"(v)
                 : "memory");
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 2)
accept_path_kernel(const void* __restrict__ logits, int V, int64_t row_stride, int nchunks,
                   int S, bool aligned, const int32_t* __restrict__ parent,
                   const int32_t* __restrict__ token, const int32_t* __restrict__ n_nodes, int L,
                   int N, float temperature, float c_exp, uint64_t seed, uint64_t step,
                   int32_t* __restrict__ target_token, int32_t* __restrict__ accept_len,
                   int32_t* __restrict__ accepted_nodes, int32_t* __restrict__ out_tokens,
                   int32_t* __restrict__ next_bonus, uint32_t* err) {
    using Chunk = SmemChunk<BF16, kChunkBytes / (BF16 ? 2 : 4)>;
    constexpr int VEC = Chunk::VEC, ES = Chunk::ES, SIZE = Chunk::SIZE;
    constexpr int PER = Chunk::NVEC / kThreads;  // vectors per thread per chunk
    __shared__ int s_par[kMaxRows];               // the tree, staged once
    __shared__ int s_tok[kMaxRows];
    __shared__ unsigned long long s_gkey[2][kMaxCluster];  // gathered greedy keys, by parity
    __shared__ float2 s_gpart[2][kMaxChunks];     // gathered chunk partials, by parity
    __shared__ float2 s_own[kMaxChunks];          // this CTA's chunk partials of the level
    __shared__ float s_red[2 * (kThreads / 32)];
    __shared__ unsigned long long s_key[kThreads / 32];
    __shared__ int s_next, s_pick, s_cstar, s_first, s_lastnz;
    __shared__ float s_tloc, s_u;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the cluster of S CTAs of sequence b; CTA r owns chunks r, r + S, ...
    const int b = blockIdx.x / S, r = blockIdx.x % S, R = N + 1;
    const int nloc = (nchunks - r + S - 1) / S;
    const bool sample = temperature > 0.f;
    pdl_wait();
    const int n = n_nodes[b];
    if (n < 0 || n > N) {  // the same n in every CTA of the cluster: all leave here
        if (tid == 0 && r == 0) record_error(err, ERR_ACCEPT | ERR_BAD_N_NODES);
        return;
    }
    const char* base = (const char*)logits + (size_t)b * R * (size_t)row_stride * ES;
    // the 16-byte vector of the row at rowp starting at element e (past V: -inf)
    auto load_vec = [&](const char* rowp, int e) -> uint4 {
        if (aligned && e + VEC <= V) return ld_stream_v4(rowp + (size_t)e * ES);
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (BF16) {
                const int e0 = e + 2 * q;
                const uint32_t lo = e0 < V ? __ldg((const unsigned short*)rowp + e0) : 0xff80u;
                const uint32_t hi = e0 + 1 < V ? __ldg((const unsigned short*)rowp + e0 + 1) : 0xff80u;
                w[q] = lo | (hi << 16);
            } else {
                w[q] = e + q < V ? __ldg((const unsigned int*)rowp + e + q) : 0xff800000u;
            }
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    };
    // this thread's vectors of chunk c (strided by the CTA, so that loads coalesce)
    auto load = [&](const char* rowp, int c, uint4 (&d)[PER]) {
#pragma unroll
        for (int i = 0; i < PER; ++i) d[i] = load_vec(rowp, c * SIZE + (tid + i * kThreads) * VEC);
    };
    // the root row's first chunk is in flight while the tree is staged
    uint4 cur_v[PER], nxt_v[PER];
    load(base, r, cur_v);

    for (int u = tid; u <= n; u += kThreads) {
        s_par[u] = parent[(size_t)b * R + u];
        s_tok[u] = token[(size_t)b * R + u];
    }
    if (target_token && r == 0)
        for (int u = tid; u < R; u += kThreads) target_token[(size_t)b * R + u] = -1;
    // the tree is staged, and every CTA of the cluster has started before any
    // stores into its shared memory
    if (S > 1) sm100::cluster_sync();
    else __syncthreads();

    int cur = 0, len = 0, bonus = 0;
    for (int level = 0;; ++level) {
        const int slot = level & 1;
        const char* rowp = base + (size_t)cur * (size_t)row_stride * ES;
        if (level > 0) load(rowp, r, cur_v);
        // the node's uniform, while the loads are in flight (read after the exchange)
        if (sample && tid == kThreads - 32) s_u = node_uniform(seed, step, (uint64_t)b, (uint64_t)cur);
        unsigned long long best = 0ull;  // greedy: (value, lowest index) key
        for (int lc = 0; lc < nloc; ++lc) {
            const int c = r + lc * S, c0 = c * SIZE;
            if (lc + 1 < nloc) load(rowp, c + S, nxt_v);
            if (!sample) {
                // the thread's first maximum in token order: a vector is unpacked
                // only when its maximum beats the best so far
                float bv = best ? key_value(best) : -INFINITY;
#pragma unroll
                for (int i = 0; i < PER; ++i) {
                    const float vm = Chunk::vmax(cur_v[i]);
                    if (vm > bv) {
                        const int e0 = c0 + (tid + i * kThreads) * VEC;
                        float x[VEC];
                        Chunk::unpack(cur_v[i], x);
                        int e = -1;
#pragma unroll
                        for (int k = VEC - 1; k >= 0; --k)
                            if (x[k] == vm && e0 + k < V) e = e0 + k;
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
                for (int i = 0; i < PER; ++i) tmax = fmaxf(tmax, Chunk::vmax(cur_v[i]));
                const float wmax = warp_max(tmax);
                if (lane == 0) s_red[warp] = wmax;
                __syncthreads();
                float cmax = s_red[0];
#pragma unroll
                for (int q = 1; q < kThreads / 32; ++q) cmax = fmaxf(cmax, s_red[q]);
                const float ref = (cmax == -INFINITY) ? 0.f : cmax;
                const float off = -ref * c_exp;
                float ts = 0.f;
#pragma unroll
                for (int i = 0; i < PER; ++i) {
                    float x[VEC];
                    Chunk::unpack(cur_v[i], x);
#pragma unroll
                    for (int k = 0; k < VEC; ++k) ts += fast_exp2(fmaf(x[k], c_exp, off));
                }
                const float wsum = warp_sum(ts);
                if (lane == 0) s_red[kThreads / 32 + warp] = wsum;
                __syncthreads();
                if (tid == 0) {
                    float csum = 0.f;
                    for (int q = 0; q < kThreads / 32; ++q) csum += s_red[kThreads / 32 + q];
                    s_own[lc] = make_float2(cmax, csum);
                }
            }
            if (lc + 1 < nloc) {
#pragma unroll
                for (int i = 0; i < PER; ++i) cur_v[i] = nxt_v[i];
            }
        }

        // ---- publish this CTA's partial in every CTA of the cluster ----
        if (!sample) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) best = umax64(best, shfl_xor_u64(best, o));
            if (lane == 0) s_key[warp] = best;
            __syncthreads();
            if (warp == 0) {
                // every lane ends with the CTA's key: lane q stores it into CTA q
                unsigned long long k = lane < kThreads / 32 ? s_key[lane] : 0ull;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) k = umax64(k, shfl_xor_u64(k, o));
                if (lane < S) {
                    if (lane == r) s_gkey[slot][r] = k;
                    else st_peer_u64(&s_gkey[slot][r], lane, k);
                }
            }
        } else {
            __syncthreads();  // s_own complete
            for (int q = lane; q < S * nloc; q += 32) {
                if (warp != 0) break;
                const int dst = q % S, lc = q / S, c = r + lc * S;
                const float2 v = s_own[lc];
                const unsigned long long bits =
                    (unsigned long long)__float_as_uint(v.x) |
                    ((unsigned long long)__float_as_uint(v.y) << 32);
                if (dst == r) s_gpart[slot][c] = v;
                else st_peer_u64(&s_gpart[slot][c], dst, bits);
            }
        }
        if (S > 1) sm100::cluster_sync();  // release our stores, acquire the peers'
        else __syncthreads();

        // ---- the row's token and the child carrying it ----
        // (one warp; the lowest-index child of cur with token t, as a warp min)
        auto find_child = [&](int t) {
            int nx = 0x7fffffff;
            for (int c = 1 + lane; c <= n; c += 32)
                if (s_par[c] == cur && s_tok[c] == t) nx = min(nx, c);
            return __reduce_min_sync(0xffffffffu, nx);
        };
        if (!sample) {
            if (warp == 0) {
                unsigned long long k = lane < S ? s_gkey[slot][lane] : 0ull;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) k = umax64(k, shfl_xor_u64(k, o));
                const int t = (int)key_index(k);
                const int nx = find_child(t);
                if (lane == 0) {
                    s_pick = t;
                    s_next = nx;
                }
            }
        } else {
            if (warp == 0) {
                // the chunk sums combined across the warp; the chunk where U Z is
                // crossed, from an inclusive scan in chunk order (fp32: the chunk
                // sums themselves are fp32, so this adds no more than they hold)
                const float2* part = s_gpart[slot];
                float M = -INFINITY;
                for (int c = lane; c < nchunks; c += 32) M = fmaxf(M, part[c].x);
                M = warp_max(M);
                float z = 0.f;
                for (int c = lane; c < nchunks; c += 32)
                    z += part[c].y * fast_exp2((part[c].x - M) * c_exp);
                const float target = s_u * warp_sum(z);
                float carry = 0.f;
                for (int g = 0; g < nchunks; g += 32) {
                    const int c = g + lane;
                    float scale = 0.f, contrib = 0.f;
                    if (c < nchunks) {
                        scale = fast_exp2((part[c].x - M) * c_exp);
                        contrib = part[c].y * scale;
                    }
                    float incl = contrib;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float up = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += up;
                    }
                    const bool cross = c < nchunks && (carry + incl > target || c == nchunks - 1);
                    const unsigned m = __ballot_sync(0xffffffffu, cross);
                    if (m) {
                        if (lane == __ffs(m) - 1) {
                            s_cstar = c;
                            s_tloc = (scale > 0.f) ? (target - (carry + incl - contrib)) / scale : 0.f;
                        }
                        break;
                    }
                    carry += __shfl_sync(0xffffffffu, incl, 31);
                }
                if (lane == 0) {
                    s_first = 0x7fffffff;
                    s_lastnz = -1;
                }
            }
            __syncthreads();
            const int cs = s_cstar;
            const float tloc = s_tloc;
            const float mref = fmaxf(s_gpart[slot][cs].x, -3.0e38f);
            // rescan chunk cs (from L2; every CTA of the cluster alike).  Warp w
            // takes the w-th eighth of the chunk in lane-strided vectors, so that
            // each load reads 512 contiguous bytes; the element order is
            // (warp, i, lane).  The crossing vector is the first whose running
            // sum passes tloc.
            constexpr int WV = PER * 32;  // vectors per warp
            const int vb = warp * WV, ebase = cs * SIZE;
#pragma unroll
            for (int i = 0; i < PER; ++i) cur_v[i] = load_vec(rowp, ebase + (vb + i * 32 + lane) * VEC);
            float vsum[PER], excl[PER], run = 0.f;
            int lastnz = -1;
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                float x[VEC];
                Chunk::unpack(cur_v[i], x);
                float vs = 0.f;
#pragma unroll
                for (int k = 0; k < VEC; ++k) vs += fast_exp2((x[k] - mref) * c_exp);
                vsum[i] = vs;
                float incl = vs;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float up = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += up;
                }
                excl[i] = run + incl - vs;
                run += __shfl_sync(0xffffffffu, incl, 31);
                const unsigned m = __ballot_sync(0xffffffffu, vs > 0.f);
                if (m) lastnz = vb + i * 32 + 31 - __clz(m);
            }
            if (lane == 0) s_red[warp] = run;
            __syncthreads();
            float wbefore = 0.f;
            for (int q = 0; q < warp; ++q) wbefore += s_red[q];
            int cand = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const unsigned m = __ballot_sync(0xffffffffu,
                                                 vsum[i] > 0.f && tloc < wbefore + excl[i] + vsum[i]);
                if (m && cand == 0x7fffffff) cand = vb + i * 32 + __ffs(m) - 1;
            }
            if (lane == 0) {
                if (cand != 0x7fffffff) atomicMin(&s_first, cand);
                if (lastnz >= 0) atomicMax(&s_lastnz, lastnz);
            }
            __syncthreads();
            // the vector's lane (or lane 0 of warp 0 when every weight is zero)
            // resolves the token; its warp looks up the child
            const bool crossing = s_first != 0x7fffffff;
            const int own = crossing ? s_first : s_lastnz;
            const int ov = own >= 0 ? own : 0;
            if (warp == ov / WV) {
                const int oi = (ov % WV) / 32, ol = ov % 32;
                int t = ebase;
                if (own >= 0 && lane == ol) {
                    uint4 wv = cur_v[0];
                    float acc = excl[0];
#pragma unroll
                    for (int i = 1; i < PER; ++i)
                        if (i == oi) {
                            wv = cur_v[i];
                            acc = excl[i];
                        }
                    acc += wbefore;
                    float x[VEC];
                    Chunk::unpack(wv, x);
                    int p = -1, klast = 0;
#pragma unroll
                    for (int k = 0; k < VEC; ++k) {
                        const float wt = fast_exp2((x[k] - mref) * c_exp);
                        acc += wt;
                        if (p < 0 && wt > 0.f && acc > tloc) p = k;
                        if (wt > 0.f) klast = k;
                    }
                    t = ebase + ov * VEC + ((crossing && p >= 0) ? p : klast);
                }
                t = __shfl_sync(0xffffffffu, t, ol);
                const int nx = find_child(t);
                if (lane == ol) {
                    s_pick = t;
                    s_next = nx;
                }
            }
        }
        __syncthreads();
        const int t = s_pick, next = s_next;
        if (tid == 0 && r == 0) {
            if (target_token) target_token[(size_t)b * R + cur] = t;
            if (next != 0x7fffffff && len < L) {
                accepted_nodes[(size_t)b * L + len] = next;
                out_tokens[(size_t)b * (L + 1) + len] = s_tok[next];
            }
        }
        if (next == 0x7fffffff || len >= L) {
            bonus = t;
            break;
        }
        ++len;
        cur = next;
    }
    if (tid == 0 && r == 0) {
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

// Clusters of `size` CTAs of this kernel that fit on the GPU at once (0 when
// the size cannot be launched).
template <bool BF16>
int path_active_clusters(int dev, int size) {
    static int cached[64][kMaxCluster + 1];
    static bool done[64][kMaxCluster + 1];
    if (!done[dev & 63][size]) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)size);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = 0;
        cudaLaunchAttribute at;
        at.id = cudaLaunchAttributeClusterDimension;
        at.val.clusterDim.x = (unsigned)size;
        at.val.clusterDim.y = 1;
        at.val.clusterDim.z = 1;
        cfg.attrs = &at;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, accept_path_kernel<BF16>, &cfg) != cudaSuccess) {
            n = 0;
            (void)cudaGetLastError();  // a refused size is not an error of the call
        }
        cached[dev & 63][size] = n;
        done[dev & 63][size] = true;
    }
    return cached[dev & 63][size];
}

// CTAs per sequence: the row's chunks spread evenly over up to kMaxCluster
// CTAs, while B x S stays within two CTAs per SM.
template <bool BF16>
int path_cluster(int dev, int B, int nch) {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int smax = std::max(1, std::min({kMaxCluster, nch, 2 * sms / std::max(B, 1)}));
    const int per = (nch + smax - 1) / smax;  // chunks per CTA
    int S = (nch + per - 1) / per;
    while (S > 1 && path_active_clusters<BF16>(dev, S) < 1) --S;
    return S;
}

template <bool BF16>
cudaError_t launch_path(const AcceptArgs& a, int nch, bool aligned, float c_exp, cudaStream_t s) {
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaGetDevice(&dev);
    std::call_once(once[dev & 63], [&] {
        attr_err[dev & 63] = cudaFuncSetAttribute(
            accept_path_kernel<BF16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    const int S = path_cluster<BF16>(dev, a.B, nch);
    return launch_pdl_cluster(accept_path_kernel<BF16>, dim3((unsigned)(a.B * S)), dim3(kThreads),
                              0, s, (unsigned)S, a.logits, a.V, a.row_stride, nch, S, aligned,
                              a.parent, a.token, a.n_nodes, a.L, a.N, a.temperature, c_exp,
                              a.seed, a.step, a.target_token, a.accept_len, a.accepted_nodes,
                              a.out_tokens, a.next_bonus, a.err);
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
