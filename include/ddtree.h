/*
 * ddtree.h -- C ABI of the DDTree per-round hot path on one GB300 (sm_103a).
 *
 * One decoding round of DDTree ("Accelerating Speculative Decoding with Block
 * Diffusion Draft Trees", Ringel & Romano; summary at paperlayer.ai) is four
 * calls, issued in this order on one CUDA stream:
 *
 *   ddtree_topk       per-position log-softmax + top-K of the draft logits
 *   ddtree_build      best-first heap: the N most probable prefixes as a tree
 *   ddtree_tree_attn  one target layer's attention over the tree, ancestor-only
 *   ddtree_accept     the target's decoding rule per node, then the walk
 *
 * Conventions shared by every call:
 *   - Every pointer argument is DEVICE memory owned by the caller, except where
 *     a parameter says otherwise.  The library never allocates, frees or
 *     synchronises; all work is enqueued on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and runs asynchronously.
 *   - Arrays are dense, row-major (C order), with the shapes written as
 *     [d0][d1]...; "bf16" means IEEE bfloat16 bit patterns.
 *   - Arguments are validated on the host before any launch; a bad argument
 *     returns DDTREE_ERR_INVALID_ARG (or DDTREE_ERR_UNSUPPORTED for a legal but
 *     unimplemented shape) and enqueues nothing.  Every int32 / uint32 / float
 *     array must be aligned to its element size (4 bytes); bf16 logits to 2
 *     bytes; the stricter rules of individual calls are stated with them.  A launch failure returns
 *     DDTREE_ERR_CUDA.  Inconsistent device-side data (an index out of range,
 *     a prefix longer than the cache) is skipped by the kernels, never
 *     dereferenced, and recorded in a per-device error word that
 *     ddtree_device_check() reads.
 *   - Floating-point inputs must be finite (no NaN); padding regions that a
 *     call documents as unread may hold anything.
 *   - Calls that take a workspace use it for cross-CTA partial results and
 *     completion counters.  Its size comes from ddtree_workspace_size(); it
 *     must be 256-byte aligned and zero-filled before its first use (e.g. one
 *     cudaMemsetAsync when it is allocated).  Each call leaves its counters at
 *     zero again, so a workspace can be reused call after call by the SAME
 *     operation with the same sizes (a top-K call leaves all of the workspace
 *     it used at zero, so top-K may also change sizes); two calls that may run
 *     concurrently need separate workspaces.
 *
 * Symbols used below: B sequences, L draft positions per block, V vocabulary,
 * K tokens kept per position, N node budget (drafted nodes; the root is extra,
 * so a tree has up to N+1 rows), P_b prefix length of sequence b, Hq / Hkv
 * query / key-value heads, G = Hq / Hkv, D head dimension, W = ceil((N+1)/32).
 */
#ifndef DDTREE_H
#define DDTREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DDTREE_OK = 0,
    DDTREE_ERR_INVALID_ARG = 1, /* null pointer, out-of-range size, misalignment */
    DDTREE_ERR_UNSUPPORTED = 2, /* legal but not implemented (e.g. D not 64/128) */
    DDTREE_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed */
    DDTREE_ERR_DEVICE = 4       /* a kernel recorded bad device-side data or a timeout */
} ddtree_status;

typedef enum { DDTREE_BF16 = 0, DDTREE_FP32 = 1 } ddtree_dtype;

/* Operation ids for ddtree_workspace_size. */
typedef enum { DDTREE_OP_TOPK = 0, DDTREE_OP_TREE_ATTN = 2, DDTREE_OP_ACCEPT = 3 } ddtree_op;

/* Upper limits of this implementation. */
#define DDTREE_MAX_K 32
#define DDTREE_MAX_L 16
#define DDTREE_MAX_N 1024

/* Bytes of workspace that `op` needs for the given sizes (0 if it needs none,
 * or on an invalid combination).  Arguments an op does not use are ignored:
 *   TOPK:      rows = B*L, V, K, dtype
 *   TREE_ATTN: B, N, Hq, Hkv, D, cache_cap
 *   ACCEPT:    B, N, V, dtype */
size_t ddtree_workspace_size(ddtree_op op, int B, int L, int N, int V, int K, int dtype, int Hq,
                             int Hkv, int D, int64_t cache_cap);

/* Step 1 -- per-position log-softmax and top-K.
 * Pages: §3 (the drafter gives one marginal q_i per position), §4.3 (the heap
 * works on log-probabilities; each position's tokens ranked best first),
 * App. A (the "restricted prefix set": K tokens kept per position).
 *   draft_logits  [rows][row_stride] of `dtype` (bf16 or fp32); row r holds the
 *                 V logits of one (sequence, position), rows = B*L.  Row starts
 *                 need not be 16-byte aligned (an aligned layout is faster).
 *   K             1..min(V, DDTREE_MAX_K).
 * Outputs (device):
 *   topk_idx  int32 [rows][K]: token ids ordered by logit descending, lower id
 *             first among equal logits (-0.0 equals +0.0);
 *   topk_logp fp32  [rows][K]: x - logsumexp(row);
 *   lse       fp32  [rows] (nullable): logsumexp of the row.
 * Workspace: ddtree_workspace_size(DDTREE_OP_TOPK, ...). */
ddtree_status ddtree_topk(const void* draft_logits, int dtype, int rows, int V,
                          int64_t row_stride, int K, int32_t* topk_idx, float* topk_logp,
                          float* lse, void* workspace, size_t ws_bytes, void* stream);

/* Bytes of device scratch built into the library for ddtree_topk_noalloc. */
#define DDTREE_NOALLOC_SCRATCH_BYTES (1u << 20)

/* ddtree_topk without a workspace argument.  The paper has no counterpart:
 * this exists for callers that may not allocate device memory themselves --
 * code that runs inside a host framework whose memory pool it does not own,
 * or a latency-critical path where cudaMalloc's implicit synchronisation is
 * not allowed -- and so cannot hand in a workspace.
 * Arguments, outputs and results are those of ddtree_topk.  The cross-CTA
 * partials use one array of DDTREE_NOALLOC_SCRATCH_BYTES inside the library
 * (a static device array: every GPU that loads the library holds it until the
 * process exits); the call allocates nothing.  It needs
 * ddtree_workspace_size(DDTREE_OP_TOPK, ...) bytes of it; a larger problem is
 * rejected with DDTREE_ERR_UNSUPPORTED before anything is enqueued (for
 * V = 151936 bf16 that is 10286 rows at K = 8, 1348 rows at K = 32).
 * The first call made on a device looks up the array's device address on that
 * device (make it with the device current, before any stream capture).  The
 * array starts zeroed and every call leaves all of it that it used at zero
 * again, so calls of any sizes follow one another with nothing cleared in
 * between; a kernel whose copy
 * never landed (a bounded wait that timed out) records that in the device
 * error word, which ddtree_device_check() reports.
 * All calls share the one array: calls whose kernels can overlap on the GPU
 * (other streams, other threads) race and give wrong results; serialise them. */
ddtree_status ddtree_topk_noalloc(const void* draft_logits, int dtype, int rows, int V,
                                  int64_t row_stride, int K, int32_t* topk_idx,
                                  float* topk_logp, float* lse, void* stream);

/* Step 2 -- the tree of the N most probable prefixes (Algorithm 1's result).
 * Pages: §4.1 (the bonus token is the root), §4.2 (the best valid tree under
 * the surrogate is the set of the N most probable prefixes), §4.3 / App. A
 * (pop N times; after each pop offer the prefix's next sibling and best child).
 * A prefix's score is the fp32 sum of its tokens' log-probs, formed as parent
 * score + log-prob.  Priority: higher score, then smaller depth, then earlier
 * parent, then lower rank -- a strict total order, so node ids are canonical.
 *   topk_logp fp32 [B][L][K] (each row sorted descending), topk_idx int32
 *   [B][L][K], bonus int32 [B], prefix_len int32 [B]; L <= DDTREE_MAX_L,
 *   K <= DDTREE_MAX_K, 0 <= N <= DDTREE_MAX_N.
 * Outputs, node 0 = root, nodes 1..n in pop order (n = n_nodes[b] <= N):
 *   parent, depth, rank, token, pos_id, child_count  int32 [B][N+1]
 *   score fp32 [B][N+1]  (log prefix probability; root 0)
 *   anc_mask uint32 [B][N+1][W]: bit a%32 of word a/32 in row u is set iff node
 *            a is u itself or an ancestor of u (the ancestor-only mask)
 *   n_nodes int32 [B]
 * pos_id = prefix_len + depth.  Rows past n: ints -1, child_count 0,
 * score -inf, mask 0.  No workspace.
 * This call builds the tree level by level (depth 1, 2, ...: the top N of all
 * prefixes up to depth d are the top N of those up to depth d-1 plus the
 * children of their depth-(d-1) nodes), one CTA per sequence, in L parallel
 * steps; ddtree_build_heap below runs the heap itself.  Both return the same
 * arrays bit for bit. */
ddtree_status ddtree_build(const float* topk_logp, const int32_t* topk_idx, const int32_t* bonus,
                           const int32_t* prefix_len, int B, int L, int K, int N,
                           int32_t* parent, int32_t* depth, int32_t* rank, int32_t* token,
                           int32_t* pos_id, float* score, int32_t* child_count,
                           uint32_t* anc_mask, int32_t* n_nodes, void* stream);

/* Algorithm 1 as the pages state it: a best-first heap (§4.3, App. A) that pops
 * N times, after each pop offering the popped prefix's next sibling and best
 * child; one warp per sequence keeps the frontier in registers.  Same
 * arguments, outputs and results as ddtree_build; its N pops are sequential,
 * so it is slower for large N. */
ddtree_status ddtree_build_heap(const float* topk_logp, const int32_t* topk_idx,
                                const int32_t* bonus, const int32_t* prefix_len, int B, int L,
                                int K, int N, int32_t* parent, int32_t* depth, int32_t* rank,
                                int32_t* token, int32_t* pos_id, float* score,
                                int32_t* child_count, uint32_t* anc_mask, int32_t* n_nodes,
                                void* stream);

/* Step 3 -- tree attention of one target layer.
 * Pages: §4.1 and the abstract (all drafted nodes are verified in one target
 * forward pass with an ancestor-only attention mask), App. B (the pages' own
 * runs used a dense masked attention because FlashAttention-2 lacks the
 * pattern).  For node u <= n_nodes[b] and query head h (KV head g = h / G):
 *   out[b][u][h] = softmax_j(scale * q . k_j) v_j over j in
 *                  {prefix 0..P_b-1} U {tree nodes a with bit a set in row u}.
 *   q        bf16 [B][N+1][Hq][D] (positions already encoded by the caller)
 *   k_cache, v_cache  bf16 [B][Hkv][cache_cap][D]; rows >= P_b are not used
 *   k_tree, v_tree    bf16 [B][N+1][Hkv][D]; rows of nodes > n_nodes[b] unused
 *   prefix_len int32 [B] (0..cache_cap), n_nodes int32 [B], anc_mask as above
 *   D in {64, 128}; G a power of two <= 128; 0 <= N <= DDTREE_MAX_N;
 *   every device pointer 16-byte aligned.
 * Outputs: out bf16 [B][N+1][Hq][D] (rows past n_nodes are zero);
 *          lse fp32 [B][N+1][Hq] (nullable; natural-log sum of exps, -inf past n).
 * Workspace: ddtree_workspace_size(DDTREE_OP_TREE_ATTN, ...), which is 0 (and
 * `workspace` may be NULL) when the problem has fewer (sequence, KV head,
 * query-tile pair) units than the GPU has SMs: the KV splits of a unit then run
 * as one thread-block cluster and merge in on-chip shared memory.  Larger
 * batches merge their splits through the workspace. */
ddtree_status ddtree_tree_attn(const void* q, const void* k_cache, const void* v_cache,
                               int64_t cache_cap, const void* k_tree, const void* v_tree,
                               const int32_t* prefix_len, const int32_t* n_nodes,
                               const uint32_t* anc_mask, int B, int N, int Hq, int Hkv, int D,
                               float scale, void* out, float* lse, void* workspace,
                               size_t ws_bytes, void* stream);

/* Step 4 -- the target's decoding rule and the acceptance walk.
 * Pages: §4.1 (walk the tree with the target's decoding rule; the matched path
 * is accepted and the first unmatched target token becomes the next bonus),
 * §5 / App. B (temperatures 0 and 1).
 *   target_logits [B][N+1][row_stride] of `dtype`: the target's next-token
 *                 logits at every node; rows past n_nodes[b] are not read.
 *   parent, token int32 [B][N+1] and n_nodes [B] from ddtree_build.
 *   temperature   0 -> greedy: t[u] = argmax (lowest id on ties);
 *                 > 0 -> t[u] = smallest v with C_v > U*Z where
 *                 C_v = sum_{w<=v} exp((x_w - max)/T), Z = C_{V-1} and U is a
 *                 Philox4x64-10 uniform: key (seed, step), counter
 *                 (b, u, 0, 0), U = (x0 >> 40) * 2^-24.
 * Outputs: target_token int32 [B][N+1] (nullable; -1 past n), accept_len int32
 * [B] (0..L), accepted_nodes int32 [B][L] (-1 padded), out_tokens int32
 * [B][L+1] (the accepted tokens, then the bonus; -1 padded), next_bonus [B].
 * Workspace: ddtree_workspace_size(DDTREE_OP_ACCEPT, ...). */
ddtree_status ddtree_accept(const void* target_logits, int dtype, int64_t row_stride,
                            const int32_t* parent, const int32_t* token, const int32_t* n_nodes,
                            int B, int L, int N, int V, float temperature, uint64_t seed,
                            uint64_t step, int32_t* target_token, int32_t* accept_len,
                            int32_t* accepted_nodes, int32_t* out_tokens, int32_t* next_bonus,
                            void* workspace, size_t ws_bytes, void* stream);

/* Step 4, reading only the accepted path.  Same arguments and results as
 * ddtree_accept (accept_len, accepted_nodes, out_tokens, next_bonus are
 * identical; the same Philox uniform per node), except that target_token is
 * written only for the nodes the walk visits (the root and the accepted
 * nodes; -1 elsewhere) and no workspace is needed.  The pages' walk needs the
 * target's token only on that path (§4.1), so HBM traffic is
 * (accept_len + 1) x V x elem per sequence instead of (n + 1) x V x elem; the
 * rows are resolved one after another, so it pays when N >> accept_len.  Each
 * sequence runs on a thread-block cluster of up to 16 CTAs that split every
 * row (V <= 128 x 32 KB of logits per row).  A greedy result is identical to
 * ddtree_accept's; a sampled token can differ from it only when U·Z lies
 * within the fp32 rounding of a CDF boundary (the chunk sums are combined in
 * fp32 here, in fp64 there). */
ddtree_status ddtree_accept_path(const void* target_logits, int dtype, int64_t row_stride,
                                 const int32_t* parent, const int32_t* token,
                                 const int32_t* n_nodes, int B, int L, int N, int V,
                                 float temperature, uint64_t seed, uint64_t step,
                                 int32_t* target_token, int32_t* accept_len,
                                 int32_t* accepted_nodes, int32_t* out_tokens,
                                 int32_t* next_bonus, void* stream);

/* After the walk -- commit the accepted path to the KV cache.
 * Pages: §3 (the bonus token is not yet in the cache when the round starts),
 * §4.1 (the root is the bonus token; the matched path is accepted): the
 * verified tokens join the prefix the next round attends to.
 *   k_cache, v_cache bf16 [B][Hkv][cache_cap][D], written in place.
 *   k_tree, v_tree   bf16 [B][N+1][Hkv][D]: the tree K/V given to
 *                    ddtree_tree_attn (keys computed at position P_b + depth).
 *   accept_len [B], accepted_nodes [B][L] from ddtree_accept.
 *   prefix_len [B]: read, then advanced in place to P_b + accept_len[b] + 1.
 * For each sequence the path rows -- node 0 (this round's bonus) followed by
 * the accepted nodes -- are copied, for every KV head, to cache positions
 * P_b .. P_b + accept_len[b] (path index = depth = position offset).  D must be
 * a multiple of 8 and every K/V pointer 16-byte aligned.  A sequence whose
 * path does not fit (P_b + accept_len + 1 > cache_cap) or names a node outside
 * [1, N] is left unchanged and recorded in the device error word.
 * No workspace. */
ddtree_status ddtree_commit(void* k_cache, void* v_cache, int64_t cache_cap, const void* k_tree,
                            const void* v_tree, const int32_t* accept_len,
                            const int32_t* accepted_nodes, int32_t* prefix_len, int B, int L,
                            int N, int Hkv, int D, void* stream);

/* Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns DDTREE_OK, DDTREE_ERR_DEVICE (and the recorded code in
 * *detail when non-null: which kernel and what was wrong), or DDTREE_ERR_CUDA.
 * Code: high byte = kernel (1 top-K, 2 build, 3 tree attention, 4 accept,
 * 5 commit, 15 ddtree_selftest_wait), low byte = reason (1 bad prefix length,
 * 2 bad node count, 3 bad tree or path, 4 a bounded wait timed out, 5 bad
 * input, 6 internal plan). */
ddtree_status ddtree_device_check(void* stream, uint32_t* detail);

/* Failure-reporting self-test (diagnostics; the paper has no counterpart).
 * Every wait inside the library's kernels (for a bulk copy to land, for the
 * tensor core, for another warp's results) is bounded in wall time: when the
 * bound passes, the kernel records "a bounded wait timed out" in the device
 * error word and unwinds, leaving the CUDA context usable.  This call enqueues
 * one warp that waits, through that same bounded wait, on a barrier that
 * nothing ever signals, with the bound shortened to limit_us microseconds
 * (1 .. 1000000).  A later ddtree_device_check() returns DDTREE_ERR_DEVICE
 * with detail 0x0F000004; nothing faults and the wait always ends.
 * Returns DDTREE_ERR_INVALID_ARG for a limit out of range. */
ddtree_status ddtree_selftest_wait(uint32_t limit_us, void* stream);

/* Name of the CUDA error behind the calling thread's most recent
 * DDTREE_ERR_CUDA (e.g. "cudaErrorInvalidValue"), or "no error". */
const char* ddtree_last_cuda_error(void);

/* Static description of a status code. */
const char* ddtree_status_str(ddtree_status s);

#ifdef __cplusplus
}
#endif
#endif /* DDTREE_H */
