// internal.h -- launchers behind the C ABI (host side).  Every launcher
// assumes its arguments were validated by api.cu and only enqueues work.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ddt {

// ---- step 1: log-softmax + top-K ------------------------------------------
struct TopkArgs {
    const void* logits;
    int dtype;  // 0 bf16, 1 fp32
    int rows, V;
    int64_t row_stride;
    int K;
    int32_t* topk_idx;
    float* topk_logp;
    float* lse;
    void* ws;
    uint32_t* err;
};
bool topk_supported(int V, int dtype, int K);
size_t topk_workspace_bytes(int rows, int V, int dtype, int K);  // K <= 0: any K
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s);

// ---- step 2: heap tree build -----------------------------------------------
struct BuildArgs {
    const float* topk_logp;
    const int32_t* topk_idx;
    const int32_t* bonus;
    const int32_t* prefix_len;
    int B, L, K, N;
    int32_t *parent, *depth, *rank, *token, *pos_id;
    float* score;
    int32_t* child_count;
    uint32_t* anc_mask;
    int32_t* n_nodes;
    uint32_t* err;
};
cudaError_t launch_build(const BuildArgs& a, cudaStream_t s);        // warp heap
cudaError_t launch_build_level(const BuildArgs& a, cudaStream_t s);  // level-synchronous

// ---- step 3: tree attention --------------------------------------------------
struct AttnArgs {
    const void *q, *k_cache, *v_cache;
    int64_t cache_cap;
    const void *k_tree, *v_tree;
    const int32_t* prefix_len;
    const int32_t* n_nodes;
    const uint32_t* anc_mask;
    int B, N, Hq, Hkv, D;
    float scale;
    void* out;
    float* lse;
    void* ws;
    uint32_t* err;
};
size_t attn_workspace_bytes(int B, int N, int Hq, int Hkv, int D, int64_t cache_cap);
cudaError_t launch_tree_attn(const AttnArgs& a, cudaStream_t s);

// ---- step 4: decoding rule + walk -------------------------------------------
struct AcceptArgs {
    const void* logits;
    int dtype;
    int64_t row_stride;
    const int32_t *parent, *token, *n_nodes;
    int B, L, N, V;
    float temperature;
    uint64_t seed, step;
    int32_t *target_token, *accept_len, *accepted_nodes, *out_tokens, *next_bonus;
    void* ws;
    uint32_t* err;
};
size_t accept_workspace_bytes(int B, int N, int V, int dtype);
bool accept_supported(int V, int dtype);
cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s);
// The walk reading only the rows on the accepted path (no workspace).
bool accept_path_supported(int V, int dtype);
cudaError_t launch_accept_path(const AcceptArgs& a, cudaStream_t s);

// ---- after the walk: commit the accepted path to the KV cache -----------------
struct CommitArgs {
    void *k_cache, *v_cache;
    int64_t cache_cap;
    const void *k_tree, *v_tree;
    const int32_t *accept_len, *accepted_nodes;
    int32_t* prefix_len;
    int B, L, N, Hkv, D;
    uint32_t* err;
};
cudaError_t launch_commit(const CommitArgs& a, cudaStream_t s);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---- shared by the entry points (api.cu) --------------------------------------
// Device address of the current device's error word (nullptr if the lookup
// fails); kernels record the first inconsistency or timeout they meet there.
uint32_t* error_word();
// The ddtree_status for a CUDA result; a failure is remembered for
// ddtree_last_cuda_error().
int launch_status(cudaError_t e);

}  // namespace ddt
