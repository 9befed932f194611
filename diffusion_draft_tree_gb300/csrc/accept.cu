// accept.cu -- step 4 of a DDTree round: the target's decoding rule at every
// tree node, then the acceptance walk ("Accelerating Speculative Decoding with
// Block Diffusion Draft Trees", §4.1: walk the tree with the target's decoding
// rule, accept the matched path, the first unmatched target token becomes the
// next bonus; §5 / App. B: temperatures 0 and 1).
//
// One persistent wave streams every live node row once from HBM.  The rows
// are cut into 8 KB segments and the flattened (sequence, node, segment) list
// is split into contiguous runs, one per warp; a warp loads a whole segment
// straight into registers (16-byte loads, every load of the segment in
// flight at once) and reduces it without any CTA barrier:
//   T = 0: the segment's (max, lowest index), folded into the row's 64-bit
//          slot with one atomicMax;
//   T > 0: the segment's max m_s and s_s = sum 2^((x - m_s) c), c = log2(e)/T;
//          the warp that completes a row (atomic count of its segments)
//          resolves the row's inverse-CDF sample: the segment in which the
//          running sum crosses U * Z, then that segment rescanned (from L2) in
//          token order.
// The last CTA to finish (atomic ticket over the grid) runs the walk of every
// sequence, one warp per sequence, with the tree's target tokens and chosen
// children in shared memory.
#include <mutex>

#include "chunk.cuh"
#include "internal.h"
#include "sampling.cuh"

#include "../../include/ddtree.h"

namespace ddt {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSegBytes = 8192;                 // one warp's unit of work
constexpr int kVpl = kSegBytes / 16 / 32;       // 16-byte vectors per lane per segment
constexpr int kMaxSegs = 512;                   // per row
constexpr int kCtasPerSm = 3;

struct AcceptWs {
    unsigned int* row_cnt;        // [B][N+1] segments done (sampling)
    unsigned int* done;           // CTAs done
    float2* parts;                // [B][N+1][nseg]: (m_s, s_s) (sampling)
    int32_t* tok;                 // [B][N+1] sampled target tokens
    unsigned long long* row_best; // [B][N+1] greedy: max (value, lowest index) key
};

template <bool BF16>
struct Seg {
    static constexpr int ES = BF16 ? 2 : 4;
    static constexpr int VEC = 16 / ES;              // elements per vector
    static constexpr int SIZE = kSegBytes / ES;      // elements per segment
    static constexpr uint32_t NEG_INF = BF16 ? 0xff80u : 0xff800000u;

    // element k of a vector (k a compile-time constant in every caller)
    DDT_DEV static float elem(const uint4& w, int k) {
        const uint32_t a[4] = {w.x, w.y, w.z, w.w};
        if (BF16) return (k & 1) ? bf16hi(a[k >> 1]) : bf16lo(a[k >> 1]);
        return __uint_as_float(a[k]);
    }
    DDT_DEV static float vmax(const uint4& w) {
        if (BF16) {
            const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&w.x);
            const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w.y);
            const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&w.z);
            const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&w.w);
            const __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
            return fmaxf(__low2float(m), __high2float(m));
        }
        return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)),
                     fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
    }
    // a0 + a1 += 2^(x c + off) over the vector's elements
    DDT_DEV static void exp_sum(const uint4& w, float c, float off, float& a0, float& a1) {
        const uint32_t a[4] = {w.x, w.y, w.z, w.w};
        if (BF16) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                a0 += fast_exp2(fmaf(bf16lo(a[p]), c, off));
                a1 += fast_exp2(fmaf(bf16hi(a[p]), c, off));
            }
        } else {
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                a0 += fast_exp2(fmaf(__uint_as_float(a[2 * p]), c, off));
                a1 += fast_exp2(fmaf(__uint_as_float(a[2 * p + 1]), c, off));
            }
        }
    }
    // Vector `e` (element index of its first element, a multiple of VEC) of
    // the row; elements at or past V read -inf.  Aligned rows: one 16-byte
    // streaming load; otherwise element by element.
    DDT_DEV static uint4 load(const char* rowp, int e, int V, bool aligned) {
        if (aligned && e + VEC <= V) return ld_stream_v4(rowp + (size_t)e * ES);
        uint32_t w[4];
        if (BF16) {
            const unsigned short* p = reinterpret_cast<const unsigned short*>(rowp);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t lo = e + 2 * i < V ? (uint32_t)__ldg(p + e + 2 * i) : NEG_INF;
                const uint32_t hi = e + 2 * i + 1 < V ? (uint32_t)__ldg(p + e + 2 * i + 1) : NEG_INF;
                w[i] = lo | (hi << 16);
            }
        } else {
            const unsigned int* p = reinterpret_cast<const unsigned int*>(rowp);
#pragma unroll
            for (int i = 0; i < 4; ++i) w[i] = e + i < V ? __ldg(p + e + i) : NEG_INF;
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    // Element e of the row from L2 (coherent), -inf past V.
    DDT_DEV static float at(const char* rowp, int e, int V) {
        if (e >= V) return -INFINITY;
        if (BF16) return bf16lo((uint32_t)__ldcg(reinterpret_cast<const unsigned short*>(rowp) + e));
        return __ldcg(reinterpret_cast<const float*>(rowp) + e);
    }
};

// Merges (m, s) pairs: s2 rescaled to the larger maximum (exp base 2^(x c)).
DDT_DEV void ms_merge(float& m, float& s, float m2, float s2, float c) {
    const float mx = fmaxf(m, m2);
    s = (m == -INFINITY ? 0.f : s * fast_exp2((m - mx) * c)) +
        (m2 == -INFINITY ? 0.f : s2 * fast_exp2((m2 - mx) * c));
    m = mx;
}

DDT_DEV double shfl_up_f64(double v, int o) {
    return __longlong_as_double(
        (long long)__shfl_up_sync(0xffffffffu, (unsigned long long)__double_as_longlong(v), o));
}

// The inverse-CDF sample of one row (one warp): Z = sum_s s_s 2^((m_s - M) c)
// over the row's segment partials; the segment in which the running sum
// crosses U * Z; that segment rescanned in token order (a lane owns 1/32 of
// it, contiguous).  Returns the token, in every lane.
template <bool BF16>
DDT_DEV int resolve_row(const char* rowp, const float2* parts, int nseg, int V, float c_exp,
                        float u) {
    using S = Seg<BF16>;
    const int lane = threadIdx.x & 31;
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
    const double target = (double)u * Z;
    // running sum over segments, 32 at a time, until it passes the target
    int cs = nseg - 1;
    float tloc = 0.f;
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
    // rescan segment cs: weights relative to its own maximum
    const float mref = fmaxf(__ldcg(&parts[cs]).x, -3.0e38f);
    constexpr int PER = S::SIZE / 32;
    const int e0 = cs * S::SIZE + lane * PER;
    float sum = 0.f;
#pragma unroll 8
    for (int i = 0; i < PER; ++i) sum += fast_exp2((S::at(rowp, e0 + i, V) - mref) * c_exp);
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
    if (owner >= 0 && lane == owner) {
        float acc = before;
        int p = -1, lastnz = -1;
        for (int i = 0; i < PER; ++i) {
            const float w = fast_exp2((S::at(rowp, e0 + i, V) - mref) * c_exp);
            acc += w;
            if (p < 0 && acc > tloc) p = e0 + i;
            if (w > 0.f) lastnz = e0 + i;
        }
        pick = p >= 0 ? p : lastnz;
    }
    return owner >= 0 ? __shfl_sync(0xffffffffu, pick, owner) : pick;
}

template <bool BF16, bool SAMPLE>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
accept_kernel(const void* __restrict__ logits, int V, int64_t row_stride, int nseg, bool aligned,
              int B, int per, const int32_t* __restrict__ parent,
              const int32_t* __restrict__ token, const int32_t* __restrict__ n_nodes, int L,
              int N, float c_exp, uint64_t seed, uint64_t step,
              int32_t* __restrict__ target_token, int32_t* __restrict__ accept_len,
              int32_t* __restrict__ accepted_nodes, int32_t* __restrict__ out_tokens,
              int32_t* __restrict__ next_bonus, AcceptWs ws, uint32_t* err) {
    using S = Seg<BF16>;
    constexpr int VEC = S::VEC;
    extern __shared__ int s_walk[];  // kWarps x [tok(N+1) | chosen(N+1)] (last CTA only)
    __shared__ bool s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int R = N + 1;
    const long total = (long)B * R * nseg;
    const long i0 = ((long)blockIdx.x * kWarps + warp) * per;
    const long i1 = min(total, i0 + per);
    pdl_wait();

    int cur_b = -1, n = -1;
    for (long it = i0; it < i1; ++it) {
        const int row = (int)(it / nseg), seg = (int)(it - (long)row * nseg);
        const int b = row / R, u = row - b * R;
        if (b != cur_b) {
            cur_b = b;
            n = __ldg(&n_nodes[b]);
            if ((n < 0 || n > N) && lane == 0 && u == 0 && seg == 0)
                record_error(err, ERR_ACCEPT | ERR_BAD_N_NODES);
        }
        if (n < 0 || n > N || u > n) continue;  // a bad tree, or a row past it
        const char* rowp = (const char*)logits + (size_t)row * (size_t)row_stride * S::ES;
        const int e0 = seg * S::SIZE;
        uint4 v[kVpl];
#pragma unroll
        for (int k = 0; k < kVpl; ++k) v[k] = S::load(rowp, e0 + (lane + 32 * k) * VEC, V, aligned);
        if (!SAMPLE) {
            // the segment's maximum and its lowest index
            float best = -INFINITY;
            uint4 bv = make_uint4(0, 0, 0, 0);
            int bk = -1;
#pragma unroll
            for (int k = 0; k < kVpl; ++k) {
                const float vm = S::vmax(v[k]);
                if (vm > best) {
                    best = vm;
                    bv = v[k];
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
            if (lane == 0 && first != 0x7fffffff)
                atomicMax(&ws.row_best[row], value_index_key(wmax, (uint32_t)first));
        } else {
            // the segment's (max, sum of exponentials), online per lane
            float m = -INFINITY, a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int k = 0; k < kVpl; ++k) {
                const float vm = S::vmax(v[k]);
                if (vm > m) {
                    const float f = fast_exp2((m - vm) * c_exp);  // 0 while m = -inf
                    a0 *= f;
                    a1 *= f;
                    m = vm;
                }
                if (m != -INFINITY) S::exp_sum(v[k], c_exp, -m * c_exp, a0, a1);
            }
            float s = a0 + a1;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float mo = __shfl_xor_sync(0xffffffffu, m, o);
                const float so = __shfl_xor_sync(0xffffffffu, s, o);
                ms_merge(m, s, mo, so, c_exp);
            }
            unsigned int prev = 0;
            if (lane == 0) {
                ws.parts[(size_t)row * nseg + seg] = make_float2(m, s);
                __threadfence();
                prev = atomicAdd(&ws.row_cnt[row], 1u);
            }
            prev = __shfl_sync(0xffffffffu, prev, 0);
            if (prev + 1u == (unsigned)nseg) {  // this warp completed the row
                __threadfence();
                const float uu = node_uniform(seed, step, (uint64_t)b, (uint64_t)u);
                const int pick = resolve_row<BF16>(rowp, ws.parts + (size_t)row * nseg, nseg, V,
                                                   c_exp, uu);
                if (lane == 0) {
                    ws.row_cnt[row] = 0u;  // ready for the next call
                    ws.tok[row] = pick;
                    __threadfence();
                }
            }
        }
    }
    pdl_trigger();

    // ---- the last CTA to finish walks every sequence --------------------------
    __syncthreads();
    if (tid == 0) s_last = ticket_is_last(ws.done, gridDim.x);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    int* s_tok = s_walk + warp * 2 * R;
    int* s_ch = s_tok + R;
    for (int b = warp; b < B; b += kWarps) {
        const int nb = __ldcg(&n_nodes[b]);
        if (nb < 0 || nb > N) continue;  // recorded above; outputs left untouched
        for (int i = lane; i <= nb; i += 32) {
            const size_t r = (size_t)b * R + i;
            int t;
            if (!SAMPLE) {
                const unsigned long long k = __ldcg(&ws.row_best[r]);
                t = (int)key_index(k);
                ws.row_best[r] = 0ull;  // ready for the next call
            } else {
                t = __ldcg(&ws.tok[r]);
            }
            s_tok[i] = t;
            s_ch[i] = -1;
            if (target_token) target_token[r] = t;
        }
        if (target_token)
            for (int i = nb + 1 + lane; i < R; i += 32) target_token[(size_t)b * R + i] = -1;
        __syncwarp();
        // chosen[p] = the child c of p whose token equals the target's token at p
        for (int c = 1 + lane; c <= nb; c += 32) {
            const int p = __ldg(&parent[(size_t)b * R + c]);
            if (p < 0 || p >= c) {
                record_error(err, ERR_ACCEPT | ERR_BAD_TREE);
                continue;
            }
            if (__ldg(&token[(size_t)b * R + c]) == s_tok[p]) s_ch[p] = c;
        }
        __syncwarp();
        if (lane == 0) {
            int cur = 0, len = 0;
            int32_t* acc = accepted_nodes + (size_t)b * L;
            int32_t* ot = out_tokens + (size_t)b * (L + 1);
            while (len < L && s_ch[cur] >= 0) {
                ot[len] = s_tok[cur];  // the accepted child's token is the target's at cur
                cur = s_ch[cur];
                acc[len] = cur;
                ++len;
            }
            for (int i = len; i < L; ++i) acc[i] = -1;
            const int bonus = s_tok[cur];
            ot[len] = bonus;
            for (int i = len + 1; i <= L; ++i) ot[i] = -1;
            accept_len[b] = len;
            next_bonus[b] = bonus;
        }
        __syncwarp();
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
    l.parts = align_up(l.done + 4, 256);
    l.tok = align_up(l.parts + (size_t)B * R * nseg * sizeof(float2), 256);
    l.row_best = align_up(l.tok + (size_t)B * R * 4, 256);
    l.total = align_up(l.row_best + (size_t)B * R * 8, 256);
    return l;
}

template <bool BF16, bool SAMPLE>
cudaError_t launch_one(const AcceptArgs& a, int nseg, bool aligned, float c_exp, AcceptWs ws,
                       cudaStream_t s) {
    auto kern = accept_kernel<BF16, SAMPLE>;
    const size_t smem = (size_t)kWarps * 2 * (a.N + 1) * sizeof(int);
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaGetDevice(&dev);
    std::call_once(once[dev & 63], [&] {  // the largest walk area any tree needs
        attr_err[dev & 63] = cudaFuncSetAttribute(
            kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
            (int)(kWarps * 2 * (DDTREE_MAX_N + 1) * sizeof(int)));
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    // one wave: every warp takes a contiguous run of segments
    const long total = (long)a.B * (a.N + 1) * nseg;
    const long warps = (long)num_sms_accept() * kCtasPerSm * kWarps;
    const int per = (int)((total + warps - 1) / warps);
    const int grid = (int)((total + (long)per * kWarps - 1) / ((long)per * kWarps));
    return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, a.logits, a.V, a.row_stride,
                      nseg, aligned, a.B, per, a.parent, a.token, a.n_nodes, a.L, a.N, c_exp,
                      a.seed, a.step, a.target_token, a.accept_len, a.accepted_nodes,
                      a.out_tokens, a.next_bonus, ws, a.err);
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
