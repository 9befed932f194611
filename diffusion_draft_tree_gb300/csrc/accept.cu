// accept.cu -- step 4 of a DDTree round: the target's decoding rule at every
// tree node, then the acceptance walk ("Accelerating Speculative Decoding with
// Block Diffusion Draft Trees", §4.1: walk the tree with the target's decoding
// rule, accept the matched path, the first unmatched target token becomes the
// next bonus; §5 / App. B: temperatures 0 and 1).
//
// Grid = (vocabulary chunk, node, sequence): every live node row is streamed
// once from HBM, split over enough CTAs to fill the GPU.
//   T = 0: each CTA finds its chunk's (max, lowest index);
//   T > 0: each CTA finds its chunk's max m_c and s_c = sum 2^((x - m_c) c),
//          c = log2(e) / T.
// Greedy: each CTA folds its (value, lowest index) key into the row's 64-bit
// slot with one atomicMax, and the last CTA of the sequence (atomic ticket over
// all its rows and chunks, no spinning) walks the tree.  Sampling: the last
// CTA of a row resolves its inverse-CDF sample -- it locates the chunk in which
// the running sum crosses U * Z and rescans only that chunk (from L2) -- and
// the last row of a sequence to resolve runs the walk.
#include "chunk.cuh"
#include "internal.h"
#include "sampling.cuh"

#include "../../include/ddtree.h"

namespace ddt {

namespace {

constexpr int kThreads = 256;
static_assert(kThreads == kSampleThreads, "the block scan assumes this CTA size");
constexpr int kChunkBytes = 32768;
constexpr int kMaxChunks = 128;

struct AcceptWs {
    unsigned int* row_tickets;    // [B][N+1] (sampling)
    unsigned int* seq_tickets;    // [B]
    float2* parts;                // [B][N+1][nchunks]: (m_c, s_c) (sampling)
    int32_t* tok;                 // [B][N+1] sampled target tokens
    unsigned long long* row_best; // [B][N+1] greedy: max (value, lowest index) key
};

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 5)
accept_kernel(const void* __restrict__ logits, int V, int64_t row_stride, int nchunks,
              bool aligned, const int32_t* __restrict__ parent, const int32_t* __restrict__ token,
              const int32_t* __restrict__ n_nodes, int L, int N, float temperature, float c_exp,
              uint64_t seed, uint64_t step, int32_t* __restrict__ target_token,
              int32_t* __restrict__ accept_len, int32_t* __restrict__ accepted_nodes,
              int32_t* __restrict__ out_tokens, int32_t* __restrict__ next_bonus, AcceptWs ws,
              uint32_t* err) {
    using Chunk = SmemChunk<BF16, kChunkBytes / (BF16 ? 2 : 4)>;
    constexpr int VEC = Chunk::VEC;
    constexpr int PER = Chunk::NVEC / kThreads;  // vectors per thread
    __shared__ __align__(128) uint8_t s_buf[Chunk::BYTES];
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ float s_red[2 * (kThreads / 32)];
    __shared__ int s_ired[kThreads / 32];
    __shared__ bool s_flag;
    __shared__ int s_pick;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int chunk = blockIdx.x, u = blockIdx.y, b = blockIdx.z;
    const int R = N + 1;
    const size_t row = (size_t)b * R + u;
    const char* rowp = (const char*)logits + row * (size_t)row_stride * Chunk::ES;
    const int c0 = chunk * Chunk::SIZE;
    pdl_wait();
    // Start the row's bulk copy before the tree size arrives; rows past the
    // tree wait for their copy and leave.
    Chunk::issue(s_buf, &s_bar, rowp, c0, V, aligned);
    const int n = n_nodes[b];
    const bool ok = Chunk::wait(&s_bar);
    if (n < 0 || n > N) {
        if (tid == 0 && chunk == 0 && u == 0) record_error(err, ERR_ACCEPT | ERR_BAD_N_NODES);
        return;
    }
    if (u > n) return;
    if (!ok) {
        if (tid == 0) record_error(err, ERR_ACCEPT | ERR_WAIT_TIMEOUT);
        return;
    }
    const uint4* vec = reinterpret_cast<const uint4*>(s_buf);

    // ---- per-chunk partial ----------------------------------------------------
    float tmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < PER; ++i) tmax = fmaxf(tmax, Chunk::vmax(vec[tid + i * kThreads]));
    const float wmax = warp_max(tmax);
    if (lane == 0) s_red[warp] = wmax;
    __syncthreads();
    float cmax = s_red[0];
#pragma unroll
    for (int i = 1; i < kThreads / 32; ++i) cmax = fmaxf(cmax, s_red[i]);
    const bool sample = temperature > 0.f;
    float csum = 0.f;
    int cidx = -1;
    if (!sample) {
        // lowest index holding the chunk maximum: only threads that hold it scan
        int first = 0x7fffffff;
        if (tmax == cmax) {
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int v = tid + i * kThreads;
                const uint4 w = vec[v];
                if (first == 0x7fffffff && Chunk::vmax(w) == cmax) {
                    float x[VEC];
                    Chunk::unpack(w, x);
#pragma unroll
                    for (int k = 0; k < VEC; ++k) {
                        const int e = c0 + v * VEC + k;
                        if (x[k] == cmax && e < V && e < first) first = e;
                    }
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
        if (lane == 0) s_ired[warp] = first;
        __syncthreads();
        first = s_ired[0];
#pragma unroll
        for (int i = 1; i < kThreads / 32; ++i) first = min(first, s_ired[i]);
        cidx = (first == 0x7fffffff) ? -1 : first;
    } else {
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
        const float w = warp_sum(ts);
        if (lane == 0) s_red[kThreads / 32 + warp] = w;
        __syncthreads();
        for (int i = 0; i < kThreads / 32; ++i) csum += s_red[kThreads / 32 + i];
    }

    __shared__ int s_tok[DDTREE_MAX_N + 1];
    // the walk's tree lives in the chunk buffer, free once the chunk is reduced
    int* s_par = reinterpret_cast<int*>(s_buf);
    int* s_tk = s_par + (DDTREE_MAX_N + 1);
    int* s_chosen = s_tk + (DDTREE_MAX_N + 1);
    static_assert(3 * (DDTREE_MAX_N + 1) * 4 <= Chunk::BYTES, "walk arrays fit the chunk buffer");
    pdl_trigger();
    if (!sample) {
        // greedy: one 64-bit atomicMax per CTA resolves the row; the last CTA of
        // the whole sequence (all rows, all chunks) walks the tree.
        if (tid == 0) {
            if (cidx >= 0) atomicMax(&ws.row_best[row], value_index_key(cmax, (uint32_t)cidx));
            s_flag = ticket_is_last(&ws.seq_tickets[b], (unsigned)((n + 1) * nchunks));
        }
        __syncthreads();
        if (!s_flag) return;
        for (int i = tid; i <= n; i += kThreads) {
            unsigned long long* rb = &ws.row_best[(size_t)b * R + i];
            const unsigned long long k = __ldcg(rb);
            s_par[i] = parent[(size_t)b * R + i];  // the tree, in the same round trip
            s_tk[i] = token[(size_t)b * R + i];
            s_chosen[i] = -1;
            s_tok[i] = (int)key_index(k);
            *rb = 0ull;  // ready for the next call
            if (target_token) target_token[(size_t)b * R + i] = (int)key_index(k);
        }
        __syncthreads();
    } else {
    float2* rparts = ws.parts + row * nchunks;
    if (tid == 0) {
        rparts[chunk] = make_float2(cmax, csum);
        s_flag = ticket_is_last(&ws.row_tickets[row], (unsigned)nchunks);
    }
    __syncthreads();
    if (!s_flag) return;

    // ---- last CTA of this row: resolve the row's token ---------------------------
    __shared__ float2 s_part[kMaxChunks];
    for (int c = tid; c < nchunks; c += kThreads) s_part[c] = __ldcg(&rparts[c]);
    __syncthreads();
    int pick = -1;
    {
        // Z = sum_c s_c 2^((m_c - M) c); target = U * Z; find the crossing chunk.
        __shared__ int s_cstar;
        __shared__ float s_tloc;
        if (tid == 0) {
            // the few chunk sums are combined in fp64
            float M = -INFINITY;
            for (int c = 0; c < nchunks; ++c) M = fmaxf(M, s_part[c].x);
            double Z = 0.0;
            for (int c = 0; c < nchunks; ++c)
                Z += (double)s_part[c].y * (double)fast_exp2((s_part[c].x - M) * c_exp);
            const double target = (double)node_uniform(seed, step, (uint64_t)b, (uint64_t)u) * Z;
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
        }
        __syncthreads();
        const int cs = s_cstar;
        const float tloc = s_tloc;
        const float mref = fmaxf(s_part[cs].x, -3.0e38f);
        // Rescan chunk cs with a contiguous segment per thread, in token order.
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
        // The owner is the first thread whose running sum passes tloc; if
        // rounding leaves none (tloc at the chunk's very end), the last thread
        // with nonzero weight.
        __shared__ int s_first, s_lastnz;
        if (tid == 0) { s_first = 0x7fffffff; s_lastnz = -1; }
        __syncthreads();
        if (tsum > 0.f) {
            if (tloc < before + tsum) atomicMin(&s_first, tid);
            atomicMax(&s_lastnz, tid);
        }
        __syncthreads();
        const int owner = (s_first != 0x7fffffff) ? s_first : s_lastnz;
        if (tid == owner) {  // walks its segment again, in token order
            float acc = before;
            int p = -1, lastnz = -1;
            for (int i = 0; i < SEG; ++i) {
                const float w = weight(e0 + i);
                acc += w;
                if (p < 0 && acc > tloc) p = e0 + i;
                if (w > 0.f) lastnz = e0 + i;
            }
            s_pick = (p >= 0) ? p : lastnz;
        }
        if (owner < 0 && tid == 0) s_pick = cs * Chunk::SIZE;
        __syncthreads();
        pick = s_pick;
    }
    if (tid == 0) {
        ws.tok[row] = pick;
        if (target_token) target_token[row] = pick;
        s_flag = ticket_is_last(&ws.seq_tickets[b], (unsigned)(n + 1));
    }
    __syncthreads();
    if (!s_flag) return;
    for (int i = tid; i <= n; i += kThreads) {
        s_tok[i] = __ldcg(&ws.tok[(size_t)b * R + i]);
        s_par[i] = parent[(size_t)b * R + i];  // the tree, in the same round trip
        s_tk[i] = token[(size_t)b * R + i];
        s_chosen[i] = -1;
    }
    __syncthreads();
    }  // sampling

    // ---- last row of the sequence: the walk ---------------------------------------
    // chosen[p] = the child c of p whose token equals the target's token at p.
    for (int c = 1 + tid; c <= n; c += kThreads) {
        const int p = s_par[c];
        if (p < 0 || p >= c) {
            record_error(err, ERR_ACCEPT | ERR_BAD_TREE);
            continue;
        }
        if (s_tk[c] == s_tok[p]) s_chosen[p] = c;  // children have distinct tokens
    }
    __syncthreads();
    if (tid == 0) {
        int cur = 0, len = 0;
        int32_t* acc = accepted_nodes + (size_t)b * L;
        int32_t* ot = out_tokens + (size_t)b * (L + 1);
        while (len < L && s_chosen[cur] >= 0) {
            cur = s_chosen[cur];
            acc[len] = cur;
            ot[len] = s_tk[cur];
            ++len;
        }
        for (int i = len; i < L; ++i) acc[i] = -1;
        const int bonus = s_tok[cur];
        ot[len] = bonus;
        for (int i = len + 1; i <= L; ++i) ot[i] = -1;
        accept_len[b] = len;
        next_bonus[b] = bonus;
    }
    if (target_token) {
        for (int i = n + 1 + tid; i < R; i += kThreads) target_token[(size_t)b * R + i] = -1;
    }
}

struct WsLayout {
    size_t row_tickets, seq_tickets, parts, tok, row_best, total;
};

WsLayout accept_layout(int B, int N, int nch) {
    WsLayout l;
    const size_t R = (size_t)N + 1;
    l.row_tickets = 0;
    l.seq_tickets = align_up(l.row_tickets + (size_t)B * R * 4, 256);
    l.parts = align_up(l.seq_tickets + (size_t)B * 4, 256);
    l.tok = align_up(l.parts + (size_t)B * R * nch * sizeof(float2), 256);
    l.row_best = align_up(l.tok + (size_t)B * R * 4, 256);
    l.total = align_up(l.row_best + (size_t)B * R * 8, 256);
    return l;
}

}  // namespace

bool accept_supported(int V, int dtype) {
    const int size = kChunkBytes / (dtype == DDTREE_BF16 ? 2 : 4);
    return (V + size - 1) / size <= kMaxChunks;
}

namespace {

int accept_chunks(int V, int dtype) {
    const int size = kChunkBytes / (dtype == DDTREE_BF16 ? 2 : 4);
    return (V + size - 1) / size;
}

}  // namespace

size_t accept_workspace_bytes(int B, int N, int V, int dtype) {
    return accept_layout(B, N, accept_chunks(V, dtype)).total;
}

cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s) {
    const int nch = accept_chunks(a.V, a.dtype);
    const WsLayout l = accept_layout(a.B, a.N, nch);
    char* base = (char*)a.ws;
    AcceptWs ws{(unsigned int*)(base + l.row_tickets), (unsigned int*)(base + l.seq_tickets),
                (float2*)(base + l.parts), (int32_t*)(base + l.tok),
                (unsigned long long*)(base + l.row_best)};
    const int es = a.dtype == DDTREE_BF16 ? 2 : 4;
    const bool aligned = ((uintptr_t)a.logits % 16 == 0) && ((a.row_stride * es) % 16 == 0);
    const float c_exp = a.temperature > 0.f ? kLog2e / a.temperature : 0.f;
    dim3 grid(nch, a.N + 1, a.B);
    auto kern = (a.dtype == DDTREE_BF16) ? accept_kernel<true> : accept_kernel<false>;
    return launch_pdl(kern, grid, dim3(kThreads), 0, s, a.logits, a.V, a.row_stride, nch, aligned,
                      a.parent, a.token, a.n_nodes, a.L, a.N, a.temperature, c_exp, a.seed,
                      a.step, a.target_token, a.accept_len, a.accepted_nodes, a.out_tokens,
                      a.next_bonus, ws, a.err);
}

}  // namespace ddt
