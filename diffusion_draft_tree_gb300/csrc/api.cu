// api.cu -- the C ABI (include/ddtree.h): host-side validation, the per-device
// error word, and dispatch to the kernel launchers.  No allocation, no
// synchronisation except in ddtree_device_check().
#include <initializer_list>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

#include "../../include/ddtree.h"

namespace {

constexpr int kMaxDevices = 64;
uint32_t* g_err_ptr[kMaxDevices];
std::mutex g_err_mu;

}  // namespace

// One error word per device; kernels record the first inconsistency they meet.
static __device__ uint32_t g_ddtree_error_word;

namespace ddt {

// Device address of this device's error word (looked up once per device).
uint32_t* error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> g(g_err_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ddtree_error_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = (uint32_t*)p;
    }
    return g_err_ptr[dev];
}

}  // namespace ddt

namespace {

using ddt::error_word;

inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }
// Every pointer of 4-byte elements (int32, uint32, float) on its grid; null
// entries (optional outputs) pass.
inline bool aligned4(std::initializer_list<const void*> ps) {
    for (const void* p : ps)
        if (p && !aligned(p, 4)) return false;
    return true;
}

thread_local const char* t_last_cuda_error = "no error";

ddtree_status launched(cudaError_t e) {
    if (e == cudaSuccess) return DDTREE_OK;
    t_last_cuda_error = cudaGetErrorName(e);
    return DDTREE_ERR_CUDA;
}

}  // namespace

namespace ddt {
int launch_status(cudaError_t e) { return (int)launched(e); }
}  // namespace ddt

extern "C" {

const char* ddtree_last_cuda_error(void) { return t_last_cuda_error; }

const char* ddtree_status_str(ddtree_status s) {
    switch (s) {
        case DDTREE_OK: return "ok";
        case DDTREE_ERR_INVALID_ARG: return "invalid argument";
        case DDTREE_ERR_UNSUPPORTED: return "unsupported shape";
        case DDTREE_ERR_CUDA: return "CUDA error";
        case DDTREE_ERR_DEVICE: return "kernel recorded bad device data or a timeout";
    }
    return "unknown status";
}

size_t ddtree_workspace_size(ddtree_op op, int B, int L, int N, int V, int K, int dtype, int Hq,
                             int Hkv, int D, int64_t cache_cap) {
    switch (op) {
        case DDTREE_OP_TOPK:
            if (B <= 0 || V <= 0 || (dtype != DDTREE_BF16 && dtype != DDTREE_FP32)) return 0;
            return ddt::topk_workspace_bytes(B * (L > 0 ? L : 1), V, dtype, K);
        case DDTREE_OP_TREE_ATTN:
            if (B <= 0 || N < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || cache_cap < 0) return 0;
            return ddt::attn_workspace_bytes(B, N, Hq, Hkv, D, cache_cap);
        case DDTREE_OP_ACCEPT:
            if (B <= 0 || N < 0 || V <= 0 || (dtype != DDTREE_BF16 && dtype != DDTREE_FP32))
                return 0;
            return ddt::accept_workspace_bytes(B, N, V, dtype);
    }
    return 0;
}

ddtree_status ddtree_topk(const void* draft_logits, int dtype, int rows, int V,
                          int64_t row_stride, int K, int32_t* topk_idx, float* topk_logp,
                          float* lse, void* workspace, size_t ws_bytes, void* stream) {
    if (!draft_logits || !topk_idx || !topk_logp) return DDTREE_ERR_INVALID_ARG;
    if (dtype != DDTREE_BF16 && dtype != DDTREE_FP32) return DDTREE_ERR_INVALID_ARG;
    if (rows <= 0 || rows > 65535 || V <= 0 || row_stride < V || K < 1 || K > V)
        return DDTREE_ERR_INVALID_ARG;
    if (K > DDTREE_MAX_K || !ddt::topk_supported(V, dtype, K)) return DDTREE_ERR_UNSUPPORTED;
    if (!aligned(draft_logits, dtype == DDTREE_BF16 ? 2 : 4)) return DDTREE_ERR_INVALID_ARG;
    if (!aligned4({topk_idx, topk_logp, lse})) return DDTREE_ERR_INVALID_ARG;
    const size_t need = ddt::topk_workspace_bytes(rows, V, dtype, K);
    if (need && (!workspace || ws_bytes < need || !aligned(workspace, 256)))
        return DDTREE_ERR_INVALID_ARG;
    ddt::TopkArgs a{draft_logits, dtype, rows, V, row_stride, K, topk_idx, topk_logp, lse,
                    workspace, error_word()};
    return launched(ddt::launch_topk(a, (cudaStream_t)stream));
}

namespace {
ddtree_status build_common(bool heap, const float* topk_logp, const int32_t* topk_idx,
                           const int32_t* bonus, const int32_t* prefix_len, int B, int L, int K,
                           int N, int32_t* parent, int32_t* depth, int32_t* rank, int32_t* token,
                           int32_t* pos_id, float* score, int32_t* child_count,
                           uint32_t* anc_mask, int32_t* n_nodes, void* stream) {
    if (!topk_logp || !topk_idx || !bonus || !prefix_len || !parent || !depth || !rank ||
        !token || !pos_id || !score || !child_count || !anc_mask || !n_nodes)
        return DDTREE_ERR_INVALID_ARG;
    if (B <= 0 || B > 65535 || L <= 0 || K <= 0 || N < 0) return DDTREE_ERR_INVALID_ARG;
    if (!aligned4({topk_logp, topk_idx, bonus, prefix_len, parent, depth, rank, token, pos_id,
                   score, child_count, anc_mask, n_nodes}))
        return DDTREE_ERR_INVALID_ARG;
    if (L > DDTREE_MAX_L || K > DDTREE_MAX_K || N > DDTREE_MAX_N) return DDTREE_ERR_UNSUPPORTED;
    ddt::BuildArgs a{topk_logp, topk_idx, bonus, prefix_len, B, L, K, N, parent, depth, rank,
                     token, pos_id, score, child_count, anc_mask, n_nodes, error_word()};
    return launched(heap ? ddt::launch_build(a, (cudaStream_t)stream)
                         : ddt::launch_build_level(a, (cudaStream_t)stream));
}
}  // namespace

ddtree_status ddtree_build(const float* topk_logp, const int32_t* topk_idx, const int32_t* bonus,
                           const int32_t* prefix_len, int B, int L, int K, int N,
                           int32_t* parent, int32_t* depth, int32_t* rank, int32_t* token,
                           int32_t* pos_id, float* score, int32_t* child_count,
                           uint32_t* anc_mask, int32_t* n_nodes, void* stream) {
    return build_common(false, topk_logp, topk_idx, bonus, prefix_len, B, L, K, N, parent, depth,
                        rank, token, pos_id, score, child_count, anc_mask, n_nodes, stream);
}

ddtree_status ddtree_build_heap(const float* topk_logp, const int32_t* topk_idx,
                                const int32_t* bonus, const int32_t* prefix_len, int B, int L,
                                int K, int N, int32_t* parent, int32_t* depth, int32_t* rank,
                                int32_t* token, int32_t* pos_id, float* score,
                                int32_t* child_count, uint32_t* anc_mask, int32_t* n_nodes,
                                void* stream) {
    return build_common(true, topk_logp, topk_idx, bonus, prefix_len, B, L, K, N, parent, depth,
                        rank, token, pos_id, score, child_count, anc_mask, n_nodes, stream);
}

ddtree_status ddtree_tree_attn(const void* q, const void* k_cache, const void* v_cache,
                               int64_t cache_cap, const void* k_tree, const void* v_tree,
                               const int32_t* prefix_len, const int32_t* n_nodes,
                               const uint32_t* anc_mask, int B, int N, int Hq, int Hkv, int D,
                               float scale, void* out, float* lse, void* workspace,
                               size_t ws_bytes, void* stream) {
    if (!q || !k_cache || !v_cache || !k_tree || !v_tree || !prefix_len || !n_nodes ||
        !anc_mask || !out)
        return DDTREE_ERR_INVALID_ARG;
    if (B <= 0 || N < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || cache_cap < 0 || !(scale > 0.f))
        return DDTREE_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    if (N > DDTREE_MAX_N || (D != 64 && D != 128) || (G & (G - 1)) || G > 128)
        return DDTREE_ERR_UNSUPPORTED;
    for (const void* p : {q, k_cache, v_cache, k_tree, v_tree, (const void*)out})
        if (!aligned(p, 16)) return DDTREE_ERR_INVALID_ARG;
    if (!aligned4({prefix_len, n_nodes, anc_mask, lse})) return DDTREE_ERR_INVALID_ARG;
    const size_t need = ddt::attn_workspace_bytes(B, N, Hq, Hkv, D, cache_cap);
    if (need && (!workspace || ws_bytes < need || !aligned(workspace, 256)))
        return DDTREE_ERR_INVALID_ARG;
    ddt::AttnArgs a{q, k_cache, v_cache, cache_cap, k_tree, v_tree, prefix_len, n_nodes, anc_mask,
                    B, N, Hq, Hkv, D, scale, out, lse, workspace, error_word()};
    return launched(ddt::launch_tree_attn(a, (cudaStream_t)stream));
}

ddtree_status ddtree_accept(const void* target_logits, int dtype, int64_t row_stride,
                            const int32_t* parent, const int32_t* token, const int32_t* n_nodes,
                            int B, int L, int N, int V, float temperature, uint64_t seed,
                            uint64_t step, int32_t* target_token, int32_t* accept_len,
                            int32_t* accepted_nodes, int32_t* out_tokens, int32_t* next_bonus,
                            void* workspace, size_t ws_bytes, void* stream) {
    if (!target_logits || !parent || !token || !n_nodes || !accept_len || !accepted_nodes ||
        !out_tokens || !next_bonus)
        return DDTREE_ERR_INVALID_ARG;
    if (dtype != DDTREE_BF16 && dtype != DDTREE_FP32) return DDTREE_ERR_INVALID_ARG;
    if (B <= 0 || B > 65535 || L <= 0 || N < 0 || V <= 0 || row_stride < V ||
        !(temperature >= 0.f) || temperature > 1e30f)
        return DDTREE_ERR_INVALID_ARG;
    if (N > DDTREE_MAX_N || L > DDTREE_MAX_L || !ddt::accept_supported(V, dtype))
        return DDTREE_ERR_UNSUPPORTED;
    if (!aligned(target_logits, dtype == DDTREE_BF16 ? 2 : 4)) return DDTREE_ERR_INVALID_ARG;
    if (!aligned4({parent, token, n_nodes, target_token, accept_len, accepted_nodes, out_tokens,
                   next_bonus}))
        return DDTREE_ERR_INVALID_ARG;
    const size_t need = ddt::accept_workspace_bytes(B, N, V, dtype);
    if (!workspace || ws_bytes < need || !aligned(workspace, 256)) return DDTREE_ERR_INVALID_ARG;
    ddt::AcceptArgs a{target_logits, dtype, row_stride, parent, token, n_nodes, B, L, N, V,
                      temperature, seed, step, target_token, accept_len, accepted_nodes,
                      out_tokens, next_bonus, workspace, error_word()};
    return launched(ddt::launch_accept(a, (cudaStream_t)stream));
}

ddtree_status ddtree_accept_path(const void* target_logits, int dtype, int64_t row_stride,
                                 const int32_t* parent, const int32_t* token,
                                 const int32_t* n_nodes, int B, int L, int N, int V,
                                 float temperature, uint64_t seed, uint64_t step,
                                 int32_t* target_token, int32_t* accept_len,
                                 int32_t* accepted_nodes, int32_t* out_tokens,
                                 int32_t* next_bonus, void* stream) {
    if (!target_logits || !parent || !token || !n_nodes || !accept_len || !accepted_nodes ||
        !out_tokens || !next_bonus)
        return DDTREE_ERR_INVALID_ARG;
    if (dtype != DDTREE_BF16 && dtype != DDTREE_FP32) return DDTREE_ERR_INVALID_ARG;
    if (B <= 0 || B > 65535 || L <= 0 || N < 0 || V <= 0 || row_stride < V ||
        !(temperature >= 0.f) || temperature > 1e30f)
        return DDTREE_ERR_INVALID_ARG;
    if (N > DDTREE_MAX_N || L > DDTREE_MAX_L || !ddt::accept_path_supported(V, dtype))
        return DDTREE_ERR_UNSUPPORTED;
    if (!aligned(target_logits, dtype == DDTREE_BF16 ? 2 : 4)) return DDTREE_ERR_INVALID_ARG;
    if (!aligned4({parent, token, n_nodes, target_token, accept_len, accepted_nodes, out_tokens,
                   next_bonus}))
        return DDTREE_ERR_INVALID_ARG;
    ddt::AcceptArgs a{target_logits, dtype, row_stride, parent, token, n_nodes, B, L, N, V,
                      temperature, seed, step, target_token, accept_len, accepted_nodes,
                      out_tokens, next_bonus, nullptr, error_word()};
    return launched(ddt::launch_accept_path(a, (cudaStream_t)stream));
}

ddtree_status ddtree_commit(void* k_cache, void* v_cache, int64_t cache_cap, const void* k_tree,
                            const void* v_tree, const int32_t* accept_len,
                            const int32_t* accepted_nodes, int32_t* prefix_len, int B, int L,
                            int N, int Hkv, int D, void* stream) {
    if (!k_cache || !v_cache || !k_tree || !v_tree || !accept_len || !accepted_nodes ||
        !prefix_len)
        return DDTREE_ERR_INVALID_ARG;
    if (B <= 0 || B > 65535 || L <= 0 || N < 0 || Hkv <= 0 || D <= 0 || cache_cap <= 0)
        return DDTREE_ERR_INVALID_ARG;
    if (L > DDTREE_MAX_L || N > DDTREE_MAX_N || D % 8 != 0) return DDTREE_ERR_UNSUPPORTED;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_tree, 16) ||
        !aligned(v_tree, 16) || !aligned(accept_len, 4) || !aligned(accepted_nodes, 4) ||
        !aligned(prefix_len, 4))
        return DDTREE_ERR_INVALID_ARG;
    ddt::CommitArgs a{k_cache, v_cache, cache_cap, k_tree, v_tree, accept_len, accepted_nodes,
                      prefix_len, B, L, N, Hkv, D, error_word()};
    return launched(ddt::launch_commit(a, (cudaStream_t)stream));
}

namespace {

// One warp waits, through the bounded wait every kernel of the library uses, on
// an mbarrier that nothing arrives on; when the bound passes it records the
// timeout in the error word and returns, as a kernel whose copy never landed
// does.
__global__ void selftest_wait_kernel(uint64_t limit_ns, uint32_t* err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        ddt::sm100::mbar_init(&bar, 1);
        ddt::sm100::mbar_init_fence();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !ddt::sm100::mbar_wait(&bar, 0, nullptr, limit_ns))
        ddt::record_error(err, ddt::ERR_SELFTEST | ddt::ERR_WAIT_TIMEOUT);
}

}  // namespace

ddtree_status ddtree_selftest_wait(uint32_t limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 1000000) return DDTREE_ERR_INVALID_ARG;
    uint32_t* err = error_word();
    if (!err) return DDTREE_ERR_CUDA;
    selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint64_t)limit_us * 1000ull, err);
    return launched(cudaGetLastError());
}

ddtree_status ddtree_device_check(void* stream, uint32_t* detail) {
    uint32_t* p = error_word();
    if (!p) return DDTREE_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t v = 0, zero = 0;
    if (cudaMemcpyAsync(&v, p, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return DDTREE_ERR_CUDA;
    if (cudaMemcpyAsync(p, &zero, sizeof zero, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return DDTREE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DDTREE_ERR_CUDA;
    if (detail) *detail = v;
    return v ? DDTREE_ERR_DEVICE : DDTREE_OK;
}

}  // extern "C"
