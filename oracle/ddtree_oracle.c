/*
 * ddtree_oracle.c -- plain, slow CPU oracle for one DDTree round.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the bench's CPU-baseline
 * leg use it.  It shares no code, header, table or constant generator with the
 * CUDA library; it has its own enums and its own Philox.
 *
 * Source: "Accelerating Speculative Decoding with Block Diffusion Draft Trees"
 * (Ringel & Romano), as summarised on paperlayer.ai/abs/2604.12989v1:
 *   - §3: the drafter emits one marginal distribution q_i per draft position;
 *   - §4.1: the bonus token is the tree root, all drafted nodes are verified in
 *     one target pass with an ancestor-only mask, and the walk follows the
 *     target's decoding rule, accepting the matched path; the first unmatched
 *     target token becomes the next bonus;
 *   - §4.2: the surrogate (expected accepted length under the factorised draft
 *     distribution) is a sum of prefix probabilities, so the best valid tree of
 *     at most B nodes is the set of the B most probable prefixes;
 *   - §4.3 / App. A: a best-first heap that, after each pop, offers the popped
 *     prefix's next sibling and best child returns exactly those prefixes;
 *     log-probabilities are used for numerical stability.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - the "restricted prefix set" keeps the K most probable tokens per position;
 *   - draft probabilities are softmax of the raw draft logits (temperature 1);
 *   - equal logits are ordered by lower token index first;
 *   - the node budget N counts drafted nodes; the root is extra (N+1 rows);
 *   - a prefix's score is the fp32 sum of its path's log-probs, formed as
 *     parent score + log-prob, in path order;
 *   - heap priority: higher score, then smaller depth, then earlier-popped
 *     parent, then lower rank (a strict total order on prefixes);
 *   - tree keys/values of all N+1 tree tokens (root included) are separate
 *     inputs from the prefix cache; query head h reads KV head h / (Hq/Hkv);
 *   - temperature-T sampling is inverse-CDF in token order with one Philox4x64-10
 *     uniform per node, key (seed, step), counter (seq, node, 0, 0),
 *     u = (x0 >> 40) * 2^-24.
 *
 * Floating point is fp64 except where the method's own arithmetic is pinned to
 * fp32 (the heap's path sums).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_BF16 = 0, ORC_FP32 = 1 };

static double orc_load(const void* base, int dtype, int64_t i)
{
    if (dtype == ORC_FP32) return (double)((const float*)base)[i];
    uint32_t u = (uint32_t)((const uint16_t*)base)[i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* Step 1: per-position log-softmax and top-K (§3 marginals; §4.3 logs).     */
/* ------------------------------------------------------------------------ */

/* For every row r < rows of `logits` (row r starts at r*row_stride):
 *   lse[r]          = m + log(sum_v exp(x_v - m)),  m = max_v x_v   (fp64)
 *   topk_idx[r][k]  = the k-th token in the order (x descending, index ascending)
 *   topk_logp64     = x - lse (fp64), topk_logp32 = the same rounded to fp32.
 * Returns 0, or -1 on bad arguments. */
int ddo_topk(const void* logits, int dtype, int rows, int V, int64_t row_stride, int K,
             int32_t* topk_idx, double* topk_logp64, float* topk_logp32, double* lse)
{
    if (!logits || rows < 0 || V <= 0 || K <= 0 || K > V || row_stride < V) return -1;
    for (int r = 0; r < rows; ++r) {
        const int64_t base = (int64_t)r * row_stride;
        double m = -INFINITY;
        for (int v = 0; v < V; ++v) {
            double x = orc_load(logits, dtype, base + v);
            if (x > m) m = x;
        }
        double s = 0.0;
        for (int v = 0; v < V; ++v) s += exp(orc_load(logits, dtype, base + v) - m);
        const double l = m + log(s);
        if (lse) lse[r] = l;
        /* K selection passes: each takes the best element strictly after the
         * previous pick in the (value desc, index asc) order. */
        double prev_x = INFINITY;
        int prev_i = -1;
        for (int k = 0; k < K; ++k) {
            double best_x = -INFINITY;
            int best_i = -1;
            for (int v = 0; v < V; ++v) {
                double x = orc_load(logits, dtype, base + v);
                int after_prev = (x < prev_x) || (x == prev_x && v > prev_i);
                if (!after_prev) continue;
                if (best_i < 0 || x > best_x) { best_x = x; best_i = v; }
            }
            topk_idx[(int64_t)r * K + k] = best_i;
            if (topk_logp64) topk_logp64[(int64_t)r * K + k] = best_x - l;
            if (topk_logp32) topk_logp32[(int64_t)r * K + k] = (float)(best_x - l);
            prev_x = best_x;
            prev_i = best_i;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 2: best-first heap tree build (§4.2-§4.3, App. A).                   */
/* ------------------------------------------------------------------------ */

typedef struct {
    float score; /* fp32 log prefix probability */
    int depth;   /* 1..L */
    int parent;  /* node id of the parent prefix (0 = root) */
    int rank;    /* rank of the last token among its position's top-K */
} orc_cand;

/* a comes before b in the heap's priority order */
static int orc_before(const orc_cand* a, const orc_cand* b)
{
    if (a->score != b->score) return a->score > b->score;
    if (a->depth != b->depth) return a->depth < b->depth;
    if (a->parent != b->parent) return a->parent < b->parent;
    return a->rank < b->rank;
}

static void orc_heap_push(orc_cand* h, int* n, orc_cand c)
{
    int i = (*n)++;
    h[i] = c;
    while (i > 0) {
        int p = (i - 1) / 2;
        if (!orc_before(&h[i], &h[p])) break;
        orc_cand t = h[p]; h[p] = h[i]; h[i] = t;
        i = p;
    }
}

static orc_cand orc_heap_pop(orc_cand* h, int* n)
{
    orc_cand top = h[0];
    h[0] = h[--(*n)];
    int i = 0;
    for (;;) {
        int l = 2 * i + 1, r = l + 1, best = i;
        if (l < *n && orc_before(&h[l], &h[best])) best = l;
        if (r < *n && orc_before(&h[r], &h[best])) best = r;
        if (best == i) break;
        orc_cand t = h[best]; h[best] = h[i]; h[i] = t;
        i = best;
    }
    return top;
}

/* Builds the tree of every sequence b < B.
 * Inputs: logp[B][L][K] (fp32, rows sorted descending), tok[B][L][K], bonus[B],
 * prefix_len[B].  Outputs, node 0 = root, nodes 1..n in pop order, rows past
 * n are padding (ints -1, child_count 0, score -inf, mask 0):
 *   parent, depth, rank, token, pos_id, child_count: int32 [B][N+1]
 *   score: fp32 [B][N+1];  anc_mask: uint32 [B][N+1][W], W = ceil((N+1)/32),
 *   bit a of row u set iff node a is u or one of u's ancestors;  n_nodes[B]. */
int ddo_build(const float* logp, const int32_t* tok, const int32_t* bonus,
              const int32_t* prefix_len, int B, int L, int K, int N,
              int32_t* parent, int32_t* depth, int32_t* rank, int32_t* token,
              int32_t* pos_id, float* score, int32_t* child_count, uint32_t* anc_mask,
              int32_t* n_nodes)
{
    if (B < 0 || L <= 0 || K <= 0 || N < 0) return -1;
    const int R = N + 1, W = (N + 1 + 31) / 32;
    orc_cand* heap = (orc_cand*)malloc(sizeof(orc_cand) * (size_t)(2 * N + 2));
    if (!heap) return -1;
    for (int b = 0; b < B; ++b) {
        const float* lp = logp + (int64_t)b * L * K;
        const int32_t* tk = tok + (int64_t)b * L * K;
        int32_t* par = parent + (int64_t)b * R;
        int32_t* dep = depth + (int64_t)b * R;
        int32_t* rk = rank + (int64_t)b * R;
        int32_t* tkn = token + (int64_t)b * R;
        int32_t* pos = pos_id + (int64_t)b * R;
        float* sc = score + (int64_t)b * R;
        int32_t* cc = child_count + (int64_t)b * R;
        uint32_t* am = anc_mask + (int64_t)b * R * W;
        for (int u = 0; u < R; ++u) {
            par[u] = -1; dep[u] = -1; rk[u] = -1; tkn[u] = -1; pos[u] = -1;
            sc[u] = -INFINITY; cc[u] = 0;
        }
        memset(am, 0, sizeof(uint32_t) * (size_t)R * W);
        /* root = the bonus token, the empty draft prefix, probability 1 */
        dep[0] = 0; tkn[0] = bonus[b]; pos[0] = prefix_len[b]; sc[0] = 0.0f;
        int hn = 0, n = 0;
        if (N > 0) {
            orc_cand c0 = { sc[0] + lp[0], 1, 0, 0 }; /* root score + log-prob */
            orc_heap_push(heap, &hn, c0);
        }
        while (n < N && hn > 0) {
            orc_cand c = orc_heap_pop(heap, &hn);
            const int id = ++n;
            par[id] = c.parent;
            dep[id] = c.depth;
            rk[id] = c.rank;
            tkn[id] = tk[(c.depth - 1) * K + c.rank];
            pos[id] = prefix_len[b] + c.depth;
            sc[id] = c.score;
            cc[c.parent] += 1;
            if (c.rank + 1 < K) { /* next sibling: same parent, next rank */
                orc_cand s = { sc[c.parent] + lp[(c.depth - 1) * K + c.rank + 1], c.depth,
                               c.parent, c.rank + 1 };
                orc_heap_push(heap, &hn, s);
            }
            if (c.depth < L) { /* best child: this prefix extended by rank 0 */
                orc_cand ch = { c.score + lp[c.depth * K + 0], c.depth + 1, id, 0 };
                orc_heap_push(heap, &hn, ch);
            }
        }
        n_nodes[b] = n;
        /* ancestor-only mask: follow parents from each node up to the root */
        for (int u = 0; u <= n; ++u)
            for (int a = u; a >= 0; a = par[a]) am[(int64_t)u * W + a / 32] |= 1u << (a % 32);
    }
    free(heap);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 3: tree attention of one target layer (§4.1 ancestor-only mask).     */
/* ------------------------------------------------------------------------ */

/* One (sequence b, KV head g) unit: every node u in [u_lo, u_hi) and every query
 * head h with h / G == g.  Layouts (bf16 bits):
 *   q [B][N+1][Hq][D], k_cache/v_cache [B][Hkv][cache_cap][D],
 *   k_tree/v_tree [B][N+1][Hkv][D];  out fp64 [B][N+1][Hq][D], lse fp64 [B][N+1][Hq].
 * Key set of node u: prefix positions 0..P_b-1, then tree nodes a whose bit is
 * set in u's ancestor row.  Rows past n_nodes get out = 0 and lse = -inf. */
int ddo_tree_attn_unit(int b, int g, int u_lo, int u_hi, const uint16_t* q, const uint16_t* k_cache,
                       const uint16_t* v_cache, int64_t cache_cap, const uint16_t* k_tree,
                       const uint16_t* v_tree, const int32_t* prefix_len,
                       const int32_t* n_nodes, const uint32_t* anc_mask, int B, int N, int Hq,
                       int Hkv, int D, double scale, double* out, double* lse)
{
    if (b < 0 || b >= B || g < 0 || g >= Hkv || Hq % Hkv) return -1;
    const int G = Hq / Hkv, R = N + 1, W = (N + 1 + 31) / 32;
    const int P = prefix_len[b], n = n_nodes[b];
    if (P < 0 || P > cache_cap || n < 0 || n > N) return -1;
    const int nkeys = P + R;
    double* s = (double*)malloc(sizeof(double) * (size_t)nkeys);
    char* use = (char*)malloc((size_t)nkeys);
    if (!s || !use) { free(s); free(use); return -1; }
    const uint16_t* kc = k_cache + ((int64_t)b * Hkv + g) * cache_cap * D;
    const uint16_t* vc = v_cache + ((int64_t)b * Hkv + g) * cache_cap * D;
    if (u_lo < 0) u_lo = 0;
    if (u_hi > R) u_hi = R;
    for (int u = u_lo; u < u_hi; ++u) {
        for (int h = g * G; h < (g + 1) * G; ++h) {
            double* o = out + (((int64_t)b * R + u) * Hq + h) * D;
            double* l_out = lse ? lse + ((int64_t)b * R + u) * Hq + h : NULL;
            if (u > n) {
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                if (l_out) *l_out = -INFINITY;
                continue;
            }
            const uint16_t* qr = q + (((int64_t)b * R + u) * Hq + h) * D;
            const uint32_t* anc = anc_mask + ((int64_t)b * R + u) * W;
            double m = -INFINITY;
            for (int j = 0; j < nkeys; ++j) {
                const uint16_t* kr;
                if (j < P) {
                    kr = kc + (int64_t)j * D;
                    use[j] = 1;
                } else {
                    const int a = j - P;
                    use[j] = (char)((anc[a / 32] >> (a % 32)) & 1u);
                    kr = k_tree + (((int64_t)b * R + a) * Hkv + g) * D;
                }
                if (!use[j]) continue;
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += orc_load(qr, ORC_BF16, d) * orc_load(kr, ORC_BF16, d);
                s[j] = dot * scale;
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            for (int j = 0; j < nkeys; ++j)
                if (use[j]) { s[j] = exp(s[j] - m); l += s[j]; }
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            for (int j = 0; j < nkeys; ++j) {
                if (!use[j]) continue;
                const uint16_t* vr = (j < P) ? vc + (int64_t)j * D
                                             : v_tree + (((int64_t)b * R + (j - P)) * Hkv + g) * D;
                const double p = s[j] / l;
                for (int d = 0; d < D; ++d) o[d] += p * orc_load(vr, ORC_BF16, d);
            }
            if (l_out) *l_out = m + log(l);
        }
    }
    free(s);
    free(use);
    return 0;
}

int ddo_tree_attn(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                  int64_t cache_cap, const uint16_t* k_tree, const uint16_t* v_tree,
                  const int32_t* prefix_len, const int32_t* n_nodes, const uint32_t* anc_mask,
                  int B, int N, int Hq, int Hkv, int D, double scale, double* out, double* lse)
{
    for (int b = 0; b < B; ++b)
        for (int g = 0; g < Hkv; ++g) {
            int rc = ddo_tree_attn_unit(b, g, 0, N + 1, q, k_cache, v_cache, cache_cap, k_tree, v_tree,
                                        prefix_len, n_nodes, anc_mask, B, N, Hq, Hkv, D, scale,
                                        out, lse);
            if (rc) return rc;
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Counter-based RNG: Philox4x64 with 10 rounds (Salmon, Moraes, Dror, Shaw, */
/* "Parallel random numbers: as easy as 1, 2, 3", SC'11).                    */
/* ------------------------------------------------------------------------ */

void ddo_philox4x64_10(const uint64_t ctr_in[4], const uint64_t key_in[2], uint64_t out[4])
{
    uint64_t x0 = ctr_in[0], x1 = ctr_in[1], x2 = ctr_in[2], x3 = ctr_in[3];
    uint64_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        const unsigned __int128 p0 = (unsigned __int128)0xD2E7470EE14C6C93ULL * x0;
        const unsigned __int128 p1 = (unsigned __int128)0xCA5A826395121157ULL * x2;
        const uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
        const uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
        x0 = hi1 ^ x1 ^ k0;
        x1 = lo1;
        x2 = hi0 ^ x3 ^ k1;
        x3 = lo0;
        k0 += 0x9E3779B97F4A7C15ULL; /* Weyl key schedule */
        k1 += 0xBB67AE8584CAA73BULL;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* uniform in [0,1) for node `node` of sequence `seq`: 24 top bits of x0 */
double ddo_uniform(uint64_t seed, uint64_t step, uint64_t seq, uint64_t node)
{
    const uint64_t ctr[4] = { seq, node, 0, 0 }, key[2] = { seed, step };
    uint64_t o[4];
    ddo_philox4x64_10(ctr, key, o);
    return (double)(o[0] >> 40) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------------ */
/* Step 4: acceptance walk with the target's decoding rule (§4.1).          */
/* ------------------------------------------------------------------------ */

/* Per live node u of sequence b the target's token t[u] is
 *   T == 0: argmax_v logits[b][u][v] (lower index on ties);
 *   T  > 0: the smallest v with C_v > U*Z, C_v = sum_{w<=v} exp((x_w - max)/T),
 *           Z = C_{V-1}, U = ddo_uniform(seed, step, b, u);
 *           margin[b][u] = distance from U*Z to the nearest C boundary, over Z.
 * Walk: from the root, move to the child whose token equals t[current] while
 * one exists; every move accepts that child.  The bonus is t[last].
 * Outputs: target_token [B][N+1] (-1 past n), accept_len [B],
 * accepted_nodes [B][L] (-1 padded), out_tokens [B][L+1] (accepted tokens then
 * the bonus, -1 padded), next_bonus [B], margin [B][N+1] (nullable; +inf when
 * T == 0 or past n). */
int ddo_accept(const void* logits, int dtype, int64_t row_stride, const int32_t* parent,
               const int32_t* token, const int32_t* n_nodes, int B, int L, int N, int V,
               double temperature, uint64_t seed, uint64_t step, int32_t* target_token,
               int32_t* accept_len, int32_t* accepted_nodes, int32_t* out_tokens,
               int32_t* next_bonus, double* margin)
{
    if (B < 0 || L <= 0 || N < 0 || V <= 0 || row_stride < V || temperature < 0) return -1;
    const int R = N + 1;
    for (int b = 0; b < B; ++b) {
        const int n = n_nodes[b];
        if (n < 0 || n > N) return -1;
        int32_t* t = target_token + (int64_t)b * R;
        for (int u = 0; u < R; ++u) {
            t[u] = -1;
            if (margin) margin[(int64_t)b * R + u] = INFINITY;
        }
        for (int u = 0; u <= n; ++u) {
            const int64_t base = ((int64_t)b * R + u) * row_stride;
            double m = -INFINITY;
            int am = 0;
            for (int v = 0; v < V; ++v) {
                double x = orc_load(logits, dtype, base + v);
                if (x > m) { m = x; am = v; }
            }
            if (temperature == 0.0) { t[u] = am; continue; }
            double z = 0.0;
            for (int v = 0; v < V; ++v) z += exp((orc_load(logits, dtype, base + v) - m) / temperature);
            const double target = ddo_uniform(seed, step, (uint64_t)b, (uint64_t)u) * z;
            double c = 0.0, prev = 0.0;
            int pick = V - 1;
            for (int v = 0; v < V; ++v) {
                prev = c;
                c += exp((orc_load(logits, dtype, base + v) - m) / temperature);
                if (c > target) { pick = v; break; }
            }
            t[u] = pick;
            if (margin) {
                double d0 = target - prev, d1 = c - target;
                margin[(int64_t)b * R + u] = (d0 < d1 ? d0 : d1) / z;
            }
        }
        const int32_t* par = parent + (int64_t)b * R;
        const int32_t* tk = token + (int64_t)b * R;
        int32_t* acc = accepted_nodes + (int64_t)b * L;
        int32_t* ot = out_tokens + (int64_t)b * (L + 1);
        for (int i = 0; i < L; ++i) acc[i] = -1;
        for (int i = 0; i <= L; ++i) ot[i] = -1;
        int cur = 0, len = 0;
        for (;;) {
            int next = -1;
            for (int c = 1; c <= n; ++c)
                if (par[c] == cur && tk[c] == t[cur]) { next = c; break; }
            if (next < 0 || len >= L) break;
            acc[len] = next;
            ot[len] = tk[next];
            ++len;
            cur = next;
        }
        ot[len] = t[cur];
        accept_len[b] = len;
        next_bonus[b] = t[cur];
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* After the walk: commit the accepted path to the KV cache (§3 / §4.1: the  */
/* bonus token and the accepted tokens become part of the verified prefix).  */
/* ------------------------------------------------------------------------ */

/* For every sequence b with P = prefix_len[b] and a = accept_len[b], the path
 * rows are node 0 (the root: this round's bonus token) followed by
 * accepted_nodes[b][0..a).  Row i of that path (i = 0..a) is copied, for every
 * KV head g, from k_tree/v_tree[b][node_i][g][:] to k_cache/v_cache[b][g][P+i][:]
 * (bf16 bytes, unchanged), and prefix_len[b] becomes P + a + 1.  The tree
 * rows' keys and values were computed with position id P + depth, and the
 * node at path index i has depth i, so the copied rows sit at their own
 * positions.  Returns 0, or -1 on invalid arguments (a outside [0, L], an
 * accepted node outside [1, N], or P + a + 1 > cache_cap), changing nothing
 * for that sequence and later ones. */
int ddo_commit(uint16_t* k_cache, uint16_t* v_cache, int64_t cache_cap, const uint16_t* k_tree,
               const uint16_t* v_tree, const int32_t* accept_len, const int32_t* accepted_nodes,
               int32_t* prefix_len, int B, int L, int N, int Hkv, int D)
{
    if (B < 0 || L <= 0 || N < 0 || Hkv <= 0 || D <= 0 || cache_cap < 0) return -1;
    const int R = N + 1;
    for (int b = 0; b < B; ++b) {
        const int64_t P = prefix_len[b];
        const int a = accept_len[b];
        if (a < 0 || a > L || P < 0 || P + a + 1 > cache_cap) return -1;
        for (int i = 0; i < a; ++i) {
            const int u = accepted_nodes[(int64_t)b * L + i];
            if (u < 1 || u > N) return -1;
        }
        for (int i = 0; i <= a; ++i) {
            const int u = (i == 0) ? 0 : accepted_nodes[(int64_t)b * L + i - 1];
            for (int g = 0; g < Hkv; ++g) {
                const int64_t src = (((int64_t)b * R + u) * Hkv + g) * D;
                const int64_t dst = (((int64_t)b * Hkv + g) * cache_cap + P + i) * D;
                for (int d = 0; d < D; ++d) {
                    k_cache[dst + d] = k_tree[src + d];
                    v_cache[dst + d] = v_tree[src + d];
                }
            }
        }
        prefix_len[b] = (int32_t)(P + a + 1);
    }
    return 0;
}
