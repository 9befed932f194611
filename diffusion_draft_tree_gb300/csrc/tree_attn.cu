// tree_attn.cu -- step 3 of a DDTree round: one target layer's attention over
// the draft tree ("Accelerating Speculative Decoding with Block Diffusion Draft
// Trees", abstract and §4.1: every drafted node is verified in one target pass
// with an ancestor-only attention mask; App. B: the pages' runs used a dense
// masked attention because FlashAttention-2 cannot express the pattern).
//
// Work unit = (sequence b, KV head g, pair of query tiles, KV split).  A query
// tile holds 128 rows: 128/G tree nodes x the G query heads that share KV head
// g, so the GQA group turns the tree's (N+1) rows into a real dense
// contraction.  The unit streams its KV range in 128-key tiles: prefix tiles
// from the cache, then (last split only) the tree tiles, where the ancestor
// bitmask is applied.
//
// Per CTA: warp 0 issues TMA loads (Q tiles, K and V tiles, 128-byte swizzled)
// into a 2-3 stage K/V ring; warp 1 owns TMEM and issues tcgen05.mma; two
// groups of four warps (one thread per query row) run the online softmax of
// the two query tiles in the log2 domain, with lazy rescaling (O is rescaled
// only when the row max grows by more than 2^8).  P goes back into TMEM as
// bf16 over the S columns it came from and feeds the P V product directly, so
// shared memory holds only Q, K and V.  The two groups alternate on the tensor
// core: while one exponentiates, the other's products run.  When a unit's
// prefix is split, the splits run as one thread-block cluster: each keeps its
// unnormalised O and (m, l) in its own shared memory, and after a cluster
// barrier every CTA merges a slice of the head dimension for all rows, reading
// its peers' partials through distributed shared memory.  Every mbarrier wait
// is bounded in wall time; a timeout records an error and the CTA unwinds.
#include <mutex>
#include <functional>
#include <algorithm>
#include <vector>
#include <tuple>
#include <queue>
#include <map>

#include <cudaTypedefs.h>

#include "internal.h"
#include "sm100.cuh"

#include "../../include/ddtree.h"

namespace ddt {

namespace {

using namespace sm100;

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per KV tile
constexpr int kThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 softmax
constexpr int kHalfBytes = 128 * 128;  // [128 rows][64 bf16], one 128B-swizzled slab
constexpr float kRescaleLog2 = 8.f;
// Column of S_k's TMEM region that holds the bf16 P pairs of keys
// [16 kk, 16 kk + 16): keys 0-95 over the first 48 columns in order, keys
// 96-127 over columns 96-111 (the softmax writes that quarter first, from the
// registers its maximum pass left it in, over its own scores).
DDT_DEV uint32_t p_col(int kk) { return kk < 6 ? (uint32_t)(kk * 8) : (uint32_t)(96 + (kk - 6) * 8); }
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxSplits = 16;  // KV splits of one unit = CTAs of one cluster
constexpr int kLptMaxItems = 128;  // (sequence, split) items ranked in each CTA, at most
// How the KV splits of a unit combine: a single split stores directly; few
// units run each unit's splits as one cluster and merge on chip; many units
// (clusters would fragment the schedule) merge through a global workspace.
constexpr int kMergeNone = 0, kMergeCluster = 1, kMergeGlobal = 2;

template <int D>
struct Cfg {
    static constexpr int NH = D / 64;
    static constexpr int QT_BYTES = NH * kHalfBytes;  // one 128-row query tile
    static constexpr int KV_BYTES = NH * kHalfBytes;  // one K (or V) tile
    static constexpr int NS = (D == 128) ? 2 : 3;
    static constexpr int SMEM = 1024 + 2 * QT_BYTES + NS * 2 * KV_BYTES;
    // Cluster merge: a split's partial O / l (bf16, both tiles) fills the Q
    // region; its (m, l) rows take the last ML_BYTES of the K/V region, the rest
    // of which receives the peers' slices.
    static constexpr int ML_BYTES = 2 * BM * 8;
    static constexpr int RECV_BYTES = NS * 2 * KV_BYTES - ML_BYTES;
    static_assert(D * 2 * 2 * BM == 2 * QT_BYTES, "partial O fills the Q region");
    // Whether a unit of S splits can receive its slices ...
    static constexpr bool recv_fits(int S) {
        return S * (((D / 8 + S - 1) / S) * 2 * BM * 16 + ML_BYTES) <= RECV_BYTES;
    }
    // ... and every unit of a cluster of S (a short sequence uses fewer splits).
    static constexpr bool recv_fits_upto(int S) {
        for (int s = 2; s <= S; ++s)
            if (!recv_fits(s)) return false;
        return true;
    }
};

struct Params {
    const int32_t* prefix_len;
    const int32_t* n_nodes;
    const uint32_t* anc_mask;
    uint16_t* out;
    float* lse;
    uint32_t* part_o;       // global merge: [B*Hkv*mtiles][smax][D/2][128] bf16 pairs of O / l
    float* part_ml;         // global merge: [B*Hkv*mtiles][smax][2][128]
    unsigned int* tickets;  // global merge: [B*Hkv*mpairs]
    int B, N, Hq, Hkv, G, W, mtiles, mpairs, tps, smax;
    int merge;              // how the KV splits of a unit combine: kMerge*
    int lpt;                // non-cluster plans: CTAs ordered longest split first
    int64_t cache_cap;
    float scale_log2;
    uint32_t* err;
};

// Named barrier over the 256 softmax threads (both query tiles).
DDT_DEV void softmax_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// ... and the AND of `v` over them.
DDT_DEV bool softmax_bar_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// One CTA = one (sequence b, KV head g, pair of 128-row query tiles, KV split).
// Warp 0: TMA producer.  Warp 1: TMEM owner and MMA issuer.  Warps 2-5: softmax
// of query tile 0; warps 6-9: softmax of query tile 1.  Per KV tile j the
// tensor core runs S_k = Q_k K_j^T into TMEM columns [128k, 128k+128); softmax
// group k reads S_k, writes P_k (bf16) over the first 64 of those columns, and
// the tensor core runs O_k += P_k V_j with P_k read straight from TMEM.  While
// one group exponentiates, the tensor core works on the other group's tile.
// A unit's key tiles are its prefix tiles followed by its tree tiles; split s
// takes tiles [s tps, (s+1) tps) of that list.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
tree_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                 const __grid_constant__ CUtensorMap tm_vc,
                 const __grid_constant__ CUtensorMap tm_kt,
                 const __grid_constant__ CUtensorMap tm_vt, const Params p) {
    using C = Cfg<D>;
    constexpr int NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_q, bar_full[NS], bar_empty[NS], bar_sfull[2],
        bar_pfull[2], bar_odone[2], bar_recv;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ bool s_last;
    __shared__ float2 s_ml1[BM];  // lone tile: (m, l) of the second group's key halves

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- set-up that reads no global memory (overlaps the previous kernel) -------
    if (tid == 0) {
        mbar_init(&bar_q, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&bar_sfull[k], 1);
            mbar_init(&bar_pfull[k], 128);
            mbar_init(&bar_odone[k], 1);
        }
        mbar_init(&bar_recv, 1);
        s_abort = 0;
        mbar_init_fence();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_kc);
        tma_prefetch_desc(&tm_vc);
        tma_prefetch_desc(&tm_kt);
        tma_prefetch_desc(&tm_vt);
    }
    if (warp == 1) tmem_alloc(&s_tmem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    // S_k / P_k at columns 128k; O_k at 256 + D*k
    auto free_tmem = [&]() {  // only on exits where no tcgen05 operation was issued
        if (warp == 1) tmem_dealloc(tmem, kTmemCols);
    };

    // ---- decode the unit.  Cluster plans: a unit's KV splits are consecutive
    // CTAs (one cluster; split == rank in it).  Otherwise the tile pairs that
    // read the same KV range are consecutive CTAs, so they run at the same time
    // and the range comes from DRAM once for all of them.
    // Longest first (p.lpt): the (sequence, split) items are ranked by their key
    // tiles, descending (ties by item), and CTA r * Hkv * mpairs + ... takes the
    // item of rank r, so a ragged batch's long splits start in the first wave
    // and the short ones fill the tail.
    int idx = blockIdx.x;
    int split = 0, mpair, g, b = 0;
    if (p.merge == kMergeCluster) {
        split = idx % p.smax;
        idx /= p.smax;
        mpair = idx % p.mpairs;
        idx /= p.mpairs;
        g = idx % p.Hkv;
        b = idx / p.Hkv;
    } else if (p.lpt) {
        mpair = idx % p.mpairs;
        idx /= p.mpairs;
        g = idx % p.Hkv;  // (idx / Hkv: the item's rank, resolved below)
    } else {
        mpair = idx % p.mpairs;
        idx /= p.mpairs;
        split = idx % p.smax;
        idx /= p.smax;
        g = idx % p.Hkv;
        b = idx / p.Hkv;
    }
    const int R = p.N + 1, G = p.G;
    pdl_wait();
    if (p.merge != kMergeCluster && p.lpt) {
        // (dynamic shared memory is free until the first copy below is issued)
        int* s_w = reinterpret_cast<int*>(smem_raw);  // [kLptMaxItems] key tiles
        int* s_perm = s_w + kLptMaxItems;              // [kLptMaxItems] item of rank r
        const int items = p.B * p.smax;
        for (int i = tid; i < items; i += kThreads) {
            const int bb = i / p.smax, ss = i - bb * p.smax;
            const int pb = p.prefix_len[bb], nb = p.n_nodes[bb];
            int w = 0;
            if (pb >= 0 && pb <= p.cache_cap && nb >= 0 && nb <= p.N) {
                const int tot = (pb + BN - 1) / BN + (nb + 1 + BN - 1) / BN;
                w = max(0, min(tot, (ss + 1) * p.tps) - ss * p.tps);
            }
            s_w[i] = w;
        }
        __syncthreads();
        for (int i = tid; i < items; i += kThreads) {
            const int wi = s_w[i];
            int rk = 0;
            for (int j = 0; j < items; ++j) {
                const int wj = s_w[j];
                rk += (wj > wi || (wj == wi && j < i)) ? 1 : 0;
            }
            s_perm[rk] = i;
        }
        __syncthreads();
        const int item = s_perm[idx / p.Hkv];
        b = item / p.smax;
        split = item - b * p.smax;
        __syncthreads();  // (the scratch is read before any copy lands there)
    }
    const int P = p.prefix_len[b];
    const int n = p.n_nodes[b];
    if (P < 0 || P > p.cache_cap || n < 0 || n > p.N) {  // (the whole cluster exits here)
        if (tid == 0 && split == 0 && mpair == 0 && g == 0)
            record_error(p.err, ERR_ATTN | (n < 0 || n > p.N ? ERR_BAD_N_NODES : ERR_BAD_PREFIX_LEN));
        free_tmem();
        return;
    }
    const int npt = (P + BN - 1) / BN;      // prefix tiles
    const int ntt = (n + 1 + BN - 1) / BN;  // tree tiles
    const int splits = (npt + ntt + p.tps - 1) / p.tps;
    const int nodes_per_tile = BM / G;
    const int mt0 = 2 * mpair, mt1 = mt0 + 1;
    const int u00 = mt0 * nodes_per_tile, u01 = mt1 * nodes_per_tile;
    const bool tile1 = mt1 < p.mtiles;          // the second tile exists
    const bool has1 = tile1 && (u01 <= n);      // ... and holds a live node
    // The last query tile of an odd count (R G = 128 m + G r, e.g. N + 1 nodes with
    // N a power of two) is alone: both softmax groups then work on it, each on
    // one 64-key half of every key tile, and merge their (m, l, O) at the end.
    const bool dual = !tile1;
    const bool two = has1 || dual;              // two S / P / O groups in flight
    if (u00 > n) {  // every query row of both tiles is padding: zeros, once
        if (split == 0) {
            for (int r = tid; r < 2 * BM; r += kThreads) {
                const int u = u00 + r / G, h = g * G + r % G;
                if (u >= R || (r >= BM && !tile1)) continue;
                uint4* o = (uint4*)(p.out + (((size_t)b * R + u) * p.Hq + h) * D);
#pragma unroll
                for (int i = 0; i < D / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
                if (p.lse) p.lse[((size_t)b * R + u) * p.Hq + h] = -INFINITY;
            }
        }
        free_tmem();
        return;  // (the whole cluster takes this exit: it depends on b and mpair only)
    }
    if (split >= splits) {  // no KV tiles here: only keep the cluster's barrier count
        if (p.merge == kMergeCluster) {
            cluster_sync_relaxed();
            cluster_sync_relaxed();
        }
        free_tmem();
        return;
    }
    const int t_begin = split * p.tps;
    const int t_end = min(npt + ntt, t_begin + p.tps);
    const int nprefix = max(0, min(npt, t_end) - t_begin);
    const int tree_first = max(t_begin, npt) - npt;  // first tree tile of this split
    const int nt = t_end - t_begin;                  // >= 1; tiles >= nprefix are tree tiles

    // ---- shared memory carve-up (1024-byte aligned for the 128B swizzle) ----------
    const uint32_t base_u32 = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_u32 - smem_u32(smem_raw));
    uint8_t* sq = base;                          // two query tiles
    uint8_t* sk = sq + 2 * C::QT_BYTES;          // NS stages of K
    uint8_t* sv = sk + NS * C::KV_BYTES;         // NS stages of V

    auto fail = [&]() {
        record_error(p.err, ERR_ATTN | ERR_WAIT_TIMEOUT);
        s_abort = 1;
    };

    if (warp == 0) {
        // =========================== TMA producer ===========================
        if (lane == 0) {
            mbar_arrive_expect_tx(&bar_q, (has1 ? 2 : 1) * C::QT_BYTES);
            for (int h = 0; h < C::NH; ++h) {
                tma_load_3d(sq + h * kHalfBytes, &tm_q, &bar_q, 64 * h, g * G, b * R + u00);
                if (has1)
                    tma_load_3d(sq + C::QT_BYTES + h * kHalfBytes, &tm_q, &bar_q, 64 * h, g * G,
                                b * R + u01);
            }
            for (int j = 0; j < nt; ++j) {
                const int s = j % NS;
                if (!mbar_wait(&bar_empty[s], ((j / NS) & 1) ^ 1, &s_abort)) { fail(); break; }
                mbar_arrive_expect_tx(&bar_full[s], 2 * C::KV_BYTES);
                uint8_t* dk = sk + s * C::KV_BYTES;
                uint8_t* dv = sv + s * C::KV_BYTES;
                if (j < nprefix) {
                    const int p0 = (t_begin + j) * BN;
                    for (int h = 0; h < C::NH; ++h) {
                        tma_load_3d(dk + h * kHalfBytes, &tm_kc, &bar_full[s], 64 * h, p0, b * p.Hkv + g);
                        tma_load_3d(dv + h * kHalfBytes, &tm_vc, &bar_full[s], 64 * h, p0, b * p.Hkv + g);
                    }
                } else {
                    const int a0 = (tree_first + j - nprefix) * BN;
                    for (int h = 0; h < C::NH; ++h) {
                        tma_load_3d(dk + h * kHalfBytes, &tm_kt, &bar_full[s], 64 * h, g, b * R + a0);
                        tma_load_3d(dv + h * kHalfBytes, &tm_vt, &bar_full[s], 64 * h, g, b * R + a0);
                    }
                }
            }
        }
    } else if (warp == 1) {
        // =========================== MMA issuer =============================
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, 0, 0);
            constexpr uint32_t idesc_qk_half = idesc_bf16_f32(BM, BN / 2, 0, 0);
            constexpr uint32_t kHalfRows = (BN / 2) * 128;  // bytes of 64 key rows in a slab
            constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, 0, 1);
            const uint32_t q_addr = smem_u32(sq);
            auto qk = [&](int j, int k) {
                // dual: query tile 0 against keys [64k, 64k + 64) of the tile
                const uint32_t k_addr = smem_u32(sk + (j % NS) * C::KV_BYTES) + (dual ? k * kHalfRows : 0u);
                const uint32_t qa = q_addr + (dual ? 0u : k * C::QT_BYTES);
                const uint32_t idesc = dual ? idesc_qk_half : idesc_qk;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                    mma_bf16_ss(tmem + k * BN, smem_desc_sw128(qa + off, 16, 1024),
                                smem_desc_sw128(k_addr + off, 16, 1024), idesc, kk > 0);
                }
                mma_commit(&bar_sfull[k]);
            };
            auto pv = [&](int j, int k) {
                const uint32_t v_addr = smem_u32(sv + (j % NS) * C::KV_BYTES) + (dual ? k * kHalfRows : 0u);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    if (dual && kk >= BN / 32) break;  // 64 keys: P columns [0, 32)
                    mma_bf16_ts(tmem + 256 + k * D, tmem + k * BN + p_col(kk),
                                smem_desc_sw128(v_addr + kk * 2048, kHalfBytes, 1024), idesc_pv,
                                (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&bar_odone[k]);
            };
            bool ok = mbar_wait(&bar_q, 0, &s_abort) && mbar_wait(&bar_full[0], 0, &s_abort);
            if (!ok) fail();
            if (ok) {
                tc_fence_after();
                qk(0, 0);
                if (two) qk(0, 1);
            }
            for (int j = 0; ok && j < nt; ++j) {
                if (!mbar_wait(&bar_pfull[0], j & 1, &s_abort)) { fail(); break; }
                tc_fence_after();
                pv(j, 0);
                if (j + 1 < nt) {
                    if (!mbar_wait(&bar_full[(j + 1) % NS], ((j + 1) / NS) & 1, &s_abort)) { fail(); break; }
                    tc_fence_after();
                    qk(j + 1, 0);  // issued after pv(j, 0): reuses S_0/P_0 in order
                }
                if (two) {
                    if (!mbar_wait(&bar_pfull[1], j & 1, &s_abort)) { fail(); break; }
                    tc_fence_after();
                    pv(j, 1);
                }
                mma_commit(&bar_empty[j % NS]);
                if (two && j + 1 < nt) qk(j + 1, 1);
            }
        }
    } else {
        // ==================== softmax / epilogue, one thread per query row ====================
        const int k = (warp - 2) >> 2;            // query tile of this group
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;         // query row == TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tm_s = tmem + lane_off + k * BN;
        const uint32_t tm_o = tmem + lane_off + 256 + k * D;
        const bool mine = (k == 0) || has1;        // this group owns a query tile
        const bool work = mine || dual;            // ... or half of tile 0's keys
        const int key0 = dual ? k * (BN / 2) : 0;  // first key of the group's columns
        const int ncol = dual ? BN / 2 : BN;       // keys per tile of the group
        const int u = (k == 0 || dual ? u00 : u01) + r / G;
        const int hh = g * G + r % G;
        const bool row_valid = work && (u <= n);
        const float sl2 = p.scale_log2;
        // ancestor words of this row for the next tree tile, fetched one tile ahead
        uint32_t am[4] = {0u, 0u, 0u, 0u};
        auto fetch_mask = [&](int tt) {
            const uint32_t* mrow = p.anc_mask + ((size_t)b * R + u) * p.W;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int wi = tt * (BN / 32) + c;
                am[c] = (row_valid && wi < p.W) ? __ldg(&mrow[wi]) : 0u;
            }
        };
        if (nprefix < nt) fetch_mask(tree_first);
        // O_k *= factor (the running maximum grew by more than 2^8)
        auto rescale_o = [&](float factor) {
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t t[32];
                tmem_ld32(tm_o + c * 32, t);
                tmem_ld_wait();
                tmem_ld_fence(t);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    t[i] = __float_as_uint(__uint_as_float(t[i]) * factor);
                tmem_st32(tm_o + c * 32, t);
            }
        };
        float m_run = -INFINITY, l = 0.f;          // running max (scaled, log2), sum
        bool ok = true;
        for (int j = 0; work && j < nt; ++j) {
            const int s = j % NS;
            if (!mbar_wait(&bar_sfull[k], j & 1, &s_abort)) { fail(); ok = false; break; }
            tc_fence_after();
            // ---- validity of the tile's keys: one 32-bit mask per 32 columns ----
            // (a whole prefix tile needs none; the last, partial prefix tile keys
            // below the prefix length; a tree tile the row's ancestor bits)
            const bool is_tree = (j >= nprefix);
            const int a0 = (tree_first + j - nprefix) * BN;
            const int lim_t = is_tree ? (n + 1 - a0) : (P - (t_begin + j) * BN);
            const bool key_r_valid = r < lim_t;
            const int lim = lim_t - key0;  // valid keys among the group's columns
            const bool full = !is_tree && lim >= ncol;
            uint32_t vm[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int rem = lim - 32 * c;
                vm[c] = rem >= 32 ? ~0u : (rem <= 0 ? 0u : ((1u << rem) - 1u));
            }
            if (is_tree) {
                const bool hi = dual && k == 1;  // keys 64-127: ancestor words 2, 3
#pragma unroll
                for (int c = 0; c < 4; ++c) vm[c] &= (c < 2 && hi) ? am[c + 2] : am[c];
                if (j + 1 < nt) fetch_mask(tree_first + j + 1 - nprefix);
            }
            float sum = 0.f;
            if (full) {
                // ---- a whole prefix tile: both passes read S_k in 32-column
                // quarters, the next quarter's TMEM load in flight while the
                // current one is used ----
                uint32_t qa[32], qb[32];
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                auto qmax = [&](const uint32_t (&q)[32]) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) mx[i & 3] = fmaxf(mx[i & 3], __uint_as_float(q[i]));
                };
                tmem_ld32(tm_s, qa);
                tmem_ld_wait();
                tmem_ld_fence(qa);
                tmem_ld32(tm_s + 32, qb);
                qmax(qa);
                tmem_ld_wait();
                tmem_ld_fence(qb);
                if (!dual) {
                    tmem_ld32(tm_s + 64, qa);
                    qmax(qb);
                    tmem_ld_wait();
                    tmem_ld_fence(qa);
                    tmem_ld32(tm_s + 96, qb);
                    qmax(qa);
                    tmem_ld_wait();
                    tmem_ld_fence(qb);
                }
                qmax(qb);
                const float mt_raw = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                const float m_new = fmaxf(m_run, mt_raw * sl2);
                const bool resc = m_new > m_run + kRescaleLog2;
                const float m_use = resc ? m_new : m_run;
                const float factor = resc ? fast_exp2(m_run - m_new) : 1.f;
                // O_k is stable here: the commit that signalled S_k covers the
                // previous tile's P_k V product.
                if (j >= 1 && __any_sync(0xffffffffu, factor != 1.f)) rescale_o(factor);
                l *= factor;
                m_run = m_use;
                // P = 2^(s*scale*log2e - m) as bf16 pairs: quarter c's 32 weights
                // go to columns p_col(2c) .. +16 of S_k, whose scores are read
                // before (the row sum takes the fp32 weights: their bf16 rounding
                // averages out over a whole tile)
                const float neg = (m_use == -INFINITY) ? 0.f : -m_use;
                float2 acc = make_float2(0.f, 0.f);
                auto qexp = [&](const uint32_t (&q)[32], int c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float2 y = ffma2(make_float2(__uint_as_float(q[2 * i]), __uint_as_float(q[2 * i + 1])), sl2, neg);
                        const float2 e = make_float2(fast_exp2(y.x), fast_exp2(y.y));
                        pk[i] = pack_bf16x2(e.x, e.y);
                        acc = fadd2(acc, e);
                    }
                    tmem_st16(tm_s + p_col(2 * c), pk);
                };
                if (dual) {  // both quarters are still in registers
                    qexp(qb, 1);
                    qexp(qa, 0);
                } else {
                // the last quarter is still in qb: first, while quarter 0 loads
                tmem_ld32(tm_s, qa);
                qexp(qb, 3);
                tmem_ld_wait();
                tmem_ld_fence(qa);
                tmem_ld32(tm_s + 32, qb);
                qexp(qa, 0);
                tmem_ld_wait();
                tmem_ld_fence(qb);
                tmem_ld32(tm_s + 64, qa);
                qexp(qb, 1);
                tmem_ld_wait();
                tmem_ld_fence(qa);
                qexp(qa, 2);
                }
                sum = acc.x + acc.y;
            } else {
            // ---- pass 1: row max, 64 columns per TMEM wait, four independent chains ----
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c0 = 0; c0 < 4; c0 += 2) {
                uint32_t t[32], t2[32];
                tmem_ld32(tm_s + 32 * c0, t);
                tmem_ld32(tm_s + 32 * c0 + 32, t2);
                tmem_ld_wait();
                {
                    const uint32_t m = vm[c0], m2 = vm[c0 + 1];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        mx[i & 3] = fmaxf(mx[i & 3], ((m >> i) & 1u) ? __uint_as_float(t[i]) : -INFINITY);
                        mx[i & 3] = fmaxf(mx[i & 3], ((m2 >> i) & 1u) ? __uint_as_float(t2[i]) : -INFINITY);
                    }
                }
            }
            const float mt_raw = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            const float m_new = fmaxf(m_run, mt_raw * sl2);
            const bool resc = m_new > m_run + kRescaleLog2;
            const float m_use = resc ? m_new : m_run;
            const float factor = resc ? fast_exp2(m_run - m_new) : 1.f;
            // O_k is stable here: the commit that signalled S_k covers the
            // previous tile's P_k V product.
            if (j >= 1 && __any_sync(0xffffffffu, factor != 1.f)) rescale_o(factor);
            l *= factor;
            m_run = m_use;

            // ---- pass 2: P = 2^(s*scale*log2e - m) as bf16 pairs, 64 columns at a
            // time, written at the P columns of those keys (p_col), whose scores
            // are all read before they are written
            const float neg = (m_use == -INFINITY) ? 0.f : -m_use;
#pragma unroll 1
            for (int half = 0; half < (dual ? 1 : 2); ++half) {
                uint32_t t0[32], t1[32], pk[32];
                tmem_ld32(tm_s + half * 64, t0);
                tmem_ld32(tm_s + half * 64 + 32, t1);
                tmem_ld_wait();
                // few keys (partial or tree tile): the row sum takes exactly the
                // bf16 weights the P V product sees
                const uint32_t m0 = half ? vm[2] : vm[0], m1 = half ? vm[3] : vm[1];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float a = ((m0 >> (2 * i)) & 1u) ? fast_exp2(fmaf(__uint_as_float(t0[2 * i]), sl2, neg)) : 0.f;
                    const float bq = ((m0 >> (2 * i + 1)) & 1u) ? fast_exp2(fmaf(__uint_as_float(t0[2 * i + 1]), sl2, neg)) : 0.f;
                    const float c = ((m1 >> (2 * i)) & 1u) ? fast_exp2(fmaf(__uint_as_float(t1[2 * i]), sl2, neg)) : 0.f;
                    const float d = ((m1 >> (2 * i + 1)) & 1u) ? fast_exp2(fmaf(__uint_as_float(t1[2 * i + 1]), sl2, neg)) : 0.f;
                    pk[i] = pack_bf16x2(a, bq);
                    pk[16 + i] = pack_bf16x2(c, d);
                    sum += (__uint_as_float(pk[i] << 16) + __uint_as_float(pk[i] & 0xffff0000u)) +
                           (__uint_as_float(pk[16 + i] << 16) + __uint_as_float(pk[16 + i] & 0xffff0000u));
                }
                if (half == 0) {
                    tmem_st32(tm_s, pk);
                } else {  // keys 64-95 and 96-127 at their P columns
                    uint32_t lo[16], hi[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        lo[i] = pk[i];
                        hi[i] = pk[16 + i];
                    }
                    tmem_st16(tm_s + p_col(4), lo);
                    tmem_st16(tm_s + p_col(6), hi);
                }
            }
            }
            tmem_st_wait();
            l += sum;
            if (k == 0 && !key_r_valid) {
                // key r of this tile is past the sequence: zero its V row so that
                // uninitialised cache memory (possibly NaN) cannot reach O.
                if (!mbar_wait(&bar_full[s], (j / NS) & 1, &s_abort)) { fail(); ok = false; break; }
                uint8_t* vrow = sv + s * C::KV_BYTES + r * 128;
#pragma unroll
                for (int h = 0; h < C::NH; ++h)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *(uint4*)(vrow + h * kHalfBytes + i * 16) = make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();
            }
            tc_fence_before();
            mbar_arrive(&bar_pfull[k]);
        }

        // ---- epilogue (every softmax thread runs the same barrier sequence) ----
        if (work && ok && !mbar_wait(&bar_odone[k], (nt - 1) & 1, &s_abort)) { fail(); ok = false; }
        if (dual && k == 1) s_ml1[r] = make_float2(m_run, l);
        const bool all_ok = softmax_bar_and(ok);
        const bool have = all_ok && mine;          // warp-uniform
        tc_fence_after();
        if (dual && have) {
            // fold the second group's keys into O_0: O = w0 O_0 + w1 O_1,
            // l = w0 l_0 + w1 l_1, w_k = 2^(m_k - M), 0 for a group without keys
            // (both 0 for a row without keys).  No per-row branch: the TMEM loads
            // and stores are warp-collective.
            const float2 ml1 = s_ml1[r];
            const float M = fmaxf(m_run, ml1.x);
            const float w0 = m_run == -INFINITY ? 0.f : fast_exp2(m_run - M);
            const float w1 = ml1.x == -INFINITY ? 0.f : fast_exp2(ml1.x - M);
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t t0[32], t1[32];
                tmem_ld32(tm_o + c * 32, t0);
                tmem_ld32(tm_o + D + c * 32, t1);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    t0[i] = __float_as_uint(w0 * __uint_as_float(t0[i]) + w1 * __uint_as_float(t1[i]));
                tmem_st32(tm_o + c * 32, t0);
            }
            tmem_st_wait();
            l = w0 * l + w1 * ml1.y;
            m_run = M;
        }
        const bool row_out = (k == 0 || tile1) && u < R;
        uint4* dst = (uint4*)(p.out + (((size_t)b * R + u) * p.Hq + hh) * D);
        // writes 32 output columns of this row, scaled by inv
        auto store32 = [&](int c, const float (&v)[32], float inv) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                dst[c * 4 + i] =
                    make_uint4(pack_bf16x2(v[8 * i] * inv, v[8 * i + 1] * inv),
                               pack_bf16x2(v[8 * i + 2] * inv, v[8 * i + 3] * inv),
                               pack_bf16x2(v[8 * i + 4] * inv, v[8 * i + 5] * inv),
                               pack_bf16x2(v[8 * i + 6] * inv, v[8 * i + 7] * inv));
        };
        auto store_lse = [&](bool live, float M, float Ls) {
            if (p.lse)
                p.lse[((size_t)b * R + u) * p.Hq + hh] =
                    live ? (M + __log2f(Ls)) * 0.6931471805599453f : -INFINITY;
        };
        auto store_zero = [&]() {
            float z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) store32(c, z, 0.f);
            store_lse(false, 0.f, 0.f);
        };
        if (splits == 1) {
            if (have) {
                const bool live = row_valid && l > 0.f;
                const float inv = live ? 1.f / l : 0.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t t[32];
                    tmem_ld32(tm_o + c * 32, t);
                    tmem_ld_wait();
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = live ? __uint_as_float(t[i]) : 0.f;
                    if (row_out) store32(c, v, inv);
                }
                if (row_out) store_lse(live, m_run, l);
            } else if (all_ok && row_out) {  // a tile of padding rows
                store_zero();
            }
        } else if (p.merge == kMergeCluster) {
            if (have) {
                // This split's partial into its own shared memory (Q and K/V stages
                // are free: every MMA has completed): O / l as bf16, 8 columns per
                // 16-byte group, [D/8][256 rows]; then (m, l) as float2 [256 rows].
                uint4* part = reinterpret_cast<uint4*>(base);
                const int row2 = k * BM + r;
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t t[32];
                    tmem_ld32(tm_o + c * 32, t);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        part[(c * 4 + i) * 2 * BM + row2] = make_uint4(
                            pack_bf16x2(__uint_as_float(t[8 * i]) * inv, __uint_as_float(t[8 * i + 1]) * inv),
                            pack_bf16x2(__uint_as_float(t[8 * i + 2]) * inv, __uint_as_float(t[8 * i + 3]) * inv),
                            pack_bf16x2(__uint_as_float(t[8 * i + 4]) * inv, __uint_as_float(t[8 * i + 5]) * inv),
                            pack_bf16x2(__uint_as_float(t[8 * i + 6]) * inv, __uint_as_float(t[8 * i + 7]) * inv));
                }
                reinterpret_cast<float2*>(sk + C::RECV_BYTES)[row2] = make_float2(m_run, l);
            }
            fence_proxy_async_smem();  // the partial leaves by bulk copy (async proxy)
        } else {
            // Global merge: partial O / l as bf16 pairs [D/2][128] plus (m, l) in
            // fp32; the last split of the unit (atomic ticket) merges them.
            const size_t tslot = ((size_t)(b * p.Hkv + g) * p.mtiles + mt0 + k) * p.smax;
            if (have) {
                uint32_t* po = p.part_o + (tslot + split) * (D / 2) * BM;
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t t[32];
                    tmem_ld32(tm_o + c * 32, t);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        po[(c * 16 + i) * BM + r] = pack_bf16x2(__uint_as_float(t[2 * i]) * inv,
                                                                __uint_as_float(t[2 * i + 1]) * inv);
                }
                p.part_ml[(tslot + split) * 2 * BM + r] = m_run;
                p.part_ml[(tslot + split) * 2 * BM + BM + r] = l;
                __threadfence();
            }
            softmax_bar();
            if (tid == 64) {
                // every split takes its ticket, also after a timeout, so that the
                // counter returns to zero for the next call
                const bool last = ticket_is_last(&p.tickets[(b * p.Hkv + g) * p.mpairs + mpair],
                                                 (unsigned)splits);
                s_last = all_ok && last;
            }
            softmax_bar();
            if (s_last && mine) {
                // out = sum_s w_s o_s / sum_s w_s, w_s = l_s 2^(m_s - M)
                float M = -INFINITY;
                for (int s2 = 0; s2 < splits; ++s2)
                    M = fmaxf(M, __ldcg(&p.part_ml[(tslot + s2) * 2 * BM + r]));
                const float mref = (M == -INFINITY) ? 0.f : M;
                float Ls = 0.f;
                for (int s2 = 0; s2 < splits; ++s2)
                    Ls += __ldcg(&p.part_ml[(tslot + s2) * 2 * BM + BM + r]) *
                          fast_exp2(__ldcg(&p.part_ml[(tslot + s2) * 2 * BM + r]) - mref);
                const bool live = row_valid && Ls > 0.f;
                const float inv = live ? 1.f / Ls : 0.f;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0.f;
#pragma unroll 2
                    for (int s2 = 0; live && s2 < splits; ++s2) {
                        const size_t sl = tslot + s2;
                        const float w = __ldcg(&p.part_ml[sl * 2 * BM + BM + r]) *
                                        fast_exp2(__ldcg(&p.part_ml[sl * 2 * BM + r]) - mref);
                        const uint32_t* q = p.part_o + sl * (D / 2) * BM + (size_t)(c * 16) * BM + r;
                        uint32_t x[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) x[i] = __ldcg(&q[i * BM]);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            v[2 * i] += w * __uint_as_float(x[i] << 16);
                            v[2 * i + 1] += w * __uint_as_float(x[i] & 0xffff0000u);
                        }
                    }
                    if (row_out) store32(c, v, inv);
                }
                if (row_out) store_lse(live, M, Ls);
            }
            if (all_ok && !mine && row_out && split == 0) store_zero();  // padding tile
        }
        tc_fence_before();
    }

    // ---- teardown: every thread arrives here (all waits are bounded) -------------
    tc_fence_before();
    __syncthreads();
    pdl_trigger();
    if (p.merge == kMergeCluster) {
        // Execution order is all that is needed: every split's partial is written
        // and read only by its own copy engine; every K/V stage is idle.
        cluster_sync_relaxed();
        if (splits > 1 && !C::recv_fits(splits)) {  // the plan rules this out
            if (tid == 0 && split == 0) record_error(p.err, ERR_ATTN | ERR_PLAN);
        } else if (splits > 1) {
            // Split o owns head-dimension columns [8 lo(o), 8 hi(o)).  Each CTA's
            // copy engine sends every owner its slice of this CTA's partial and its
            // (m, l) rows, into the owner's (now idle) K/V stages, completing on the
            // owner's bar_recv; the owner then merges from its own shared memory:
            // out = sum_s w_s o_s / sum_s w_s, o_s = O_s / l_s, w_s = l_s 2^(m_s - M).
            constexpr int nch = D / 8;             // 8-column chunks of 256 rows x 16 B
            constexpr uint32_t kChunk = 2 * BM * 16;
            constexpr uint32_t kMl = 2 * BM * 8;
            const int c_lo = split * nch / splits, c_hi = (split + 1) * nch / splits;
            const uint32_t slot = (uint32_t)((nch + splits - 1) / splits) * kChunk;
            const uint32_t part_s = smem_u32(base);
            const uint32_t ml_s = smem_u32(sk + C::RECV_BYTES);
            const uint32_t recv_s = smem_u32(sk);
            const uint32_t recv_ml_s = recv_s + (uint32_t)splits * slot;
            if (tid == 0) {
                mbar_arrive_expect_tx(&bar_recv, (uint32_t)(splits - 1) *
                                                     ((uint32_t)(c_hi - c_lo) * kChunk + kMl));
                for (int i = 1; i < splits; ++i) {
                    const uint32_t o = (uint32_t)((split + i) % splits);
                    const int lo = (int)o * nch / splits, hi = ((int)o + 1) * nch / splits;
                    const uint32_t rbar = mapa_shared(smem_u32(&bar_recv), o);
                    bulk_copy_s2s(mapa_shared(recv_s + (uint32_t)split * slot, o),
                                  part_s + (uint32_t)lo * kChunk, (uint32_t)(hi - lo) * kChunk, rbar);
                    bulk_copy_s2s(mapa_shared(recv_ml_s + (uint32_t)split * kMl, o), ml_s, kMl, rbar);
                }
            }
            if (warp >= 2) {
                const int k = (warp - 2) >> 2;
                const int r = (warp & 3) * 32 + lane;
                const int row2 = k * BM + r;
                const int u = (k == 0 ? u00 : u01) + r / G;
                const int hh = g * G + r % G;
                const bool mine = (k == 0) || has1;
                const bool row_out = (k == 0 || tile1) && u < R;
                const bool row_valid = mine && u <= n;
                if (!mbar_wait(&bar_recv, 0, nullptr) && lane == 0)
                    record_error(p.err, ERR_ATTN | ERR_WAIT_TIMEOUT);
                const float2* mls[kMaxSplits];
                const uint4* prt[kMaxSplits];  // chunk c_lo of each split's slice
#pragma unroll
                for (int s2 = 0; s2 < kMaxSplits; ++s2) {
                    const bool self = s2 == split;
                    mls[s2] = reinterpret_cast<const float2*>(
                        self ? sk + C::RECV_BYTES : sk + splits * slot + s2 * kMl);
                    prt[s2] = reinterpret_cast<const uint4*>(self ? base + c_lo * kChunk
                                                                  : sk + s2 * slot);
                }
                float M = -INFINITY, Ls = 0.f;
                float w[kMaxSplits];
                if (row_valid) {
                    float2 ml[kMaxSplits];
#pragma unroll
                    for (int s2 = 0; s2 < kMaxSplits; ++s2) {
                        ml[s2] = s2 < splits ? mls[s2][row2] : make_float2(-INFINITY, 0.f);
                        M = fmaxf(M, ml[s2].x);
                    }
                    const float mref = (M == -INFINITY) ? 0.f : M;
#pragma unroll
                    for (int s2 = 0; s2 < kMaxSplits; ++s2) {
                        w[s2] = s2 < splits ? ml[s2].y * fast_exp2(ml[s2].x - mref) : 0.f;
                        Ls += w[s2];
                    }
                }
                const bool live = row_valid && Ls > 0.f;
                const float inv = live ? 1.f / Ls : 0.f;
                if (row_out) {
                    uint4* dst = (uint4*)(p.out + (((size_t)b * R + u) * p.Hq + hh) * D);
#pragma unroll 1
                    for (int c = c_lo; c < c_hi; ++c) {
                        float acc[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
                        if (live) {
#pragma unroll
                            for (int s2 = 0; s2 < kMaxSplits; ++s2) {
                                if (s2 < splits) {
                                    const uint4 x = prt[s2][(c - c_lo) * 2 * BM + row2];
                                    const uint32_t q[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        acc[2 * e] = fmaf(w[s2], __uint_as_float(q[e] << 16), acc[2 * e]);
                                        acc[2 * e + 1] = fmaf(w[s2], __uint_as_float(q[e] & 0xffff0000u), acc[2 * e + 1]);
                                    }
                                }
                            }
                        }
                        dst[c] = make_uint4(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                            pack_bf16x2(acc[2] * inv, acc[3] * inv),
                                            pack_bf16x2(acc[4] * inv, acc[5] * inv),
                                            pack_bf16x2(acc[6] * inv, acc[7] * inv));
                    }
                    if (split == 0 && p.lse)
                        p.lse[((size_t)b * R + u) * p.Hq + hh] =
                            live ? (M + __log2f(Ls)) * 0.6931471805599453f : -INFINITY;
                }
            }
        }
        cluster_sync_relaxed();  // every copy out of this CTA's shared memory has landed
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------- host side ---------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
    });
    return fn;
}

bool make_map(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {d0, d1 ? d1 : 1, d2 ? d2 : 1};
    cuuint64_t strides[2] = {s1_bytes, s2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Plan {
    int mtiles, mpairs, tps, smax, merge;
};

// Streaming multiprocessors of the current device (148 if the query fails).
int num_sms() {
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

// Per-unit tile counts bounding a plan: the longest prefix and the largest tree.
struct Tiles {
    int prefix, tree;
};
Tiles max_tiles(int N, int64_t cache_cap) {
    return {(int)((cache_cap + BN - 1) / BN), (N + 1 + BN - 1) / BN};
}

Plan plan_base(int N, int Hq, int Hkv) {
    Plan pl{};
    const int G = Hq / Hkv;
    pl.mtiles = ((N + 1) * G + BM - 1) / BM;
    pl.mpairs = (pl.mtiles + 1) / 2;
    return pl;
}

long plan_units(const Plan& pl, int B, int Hkv) { return (long)B * Hkv * pl.mpairs; }

// Predicted span of `units` units of T key tiles, each cut into splits of tps
// tiles (the last one shorter), every split a CTA per query-tile pair, the CTAs
// started longest first on `sms` SMs, each costing tiles + 2 (set-up, merge).
long lpt_span(long units, int T, int tps, int sms) {
    std::vector<long> sizes;
    for (int s0 = 0; s0 < T; s0 += tps) sizes.push_back(std::min(T, s0 + tps) - s0 + 2);
    std::sort(sizes.begin(), sizes.end(), std::greater<long>());
    std::priority_queue<long, std::vector<long>, std::greater<long>> sm;
    for (int i = 0; i < sms; ++i) sm.push(0);
    long span = 0;
    for (const long z : sizes)
        for (long u = 0; u < units; ++u) {
            const long e = sm.top() + z;
            sm.pop();
            sm.push(e);
            span = std::max(span, e);
        }
    return span;
}

// Many units fill the GPU without clusters: split only long tile lists, into
// four pieces merged through the workspace.  The pieces are a quarter of the
// longest list each, unless a longer first three and a short last one pack the
// SMs' waves better: with the CTAs ordered longest first the short ones fill
// the last wave (1152 equal CTAs on 152 SMs leave it 40 % empty).  Every size
// up to just under a third is scored by lpt_span, and the best is taken when
// it beats the quarter by at least 2 %.  The choice assumes every unit as long
// as the longest; it is cached per shape.
Plan plan_many(const Plan& base, Tiles t, long units, int sms) {
    Plan pl = base;
    const int T = t.prefix + t.tree;
    pl.tps = T > 64 ? std::max(32, (T + 3) / 4) : T;
    if (T > 64 && pl.tps > 32) {
        static std::mutex mu;
        static std::map<std::tuple<int, long, int>, int> cache;
        std::lock_guard<std::mutex> lock(mu);
        const auto key = std::make_tuple(T, units, sms);
        const auto it = cache.find(key);
        if (it != cache.end()) {
            pl.tps = it->second;
        } else {
            const long quarter = lpt_span(units, T, pl.tps, sms);
            long best = quarter;
            int best_tps = pl.tps;
            for (int tps = pl.tps + 1; (T + tps - 1) / tps == 4; ++tps) {
                const long span = lpt_span(units, T, tps, sms);
                if (span < best) {
                    best = span;
                    best_tps = tps;
                }
            }
            if (best * 100 < quarter * 98) pl.tps = best_tps;  // a clear gain only
            cache[key] = pl.tps;
        }
    }
    pl.smax = (T + pl.tps - 1) / pl.tps;
    pl.merge = pl.smax > 1 ? kMergeGlobal : kMergeNone;
    return pl;
}

// Few units: split each unit's tiles over a cluster of S CTAs, with the fewest
// tiles per split (at least 2) for which every unit's cluster is resident at
// once: units x S CTAs within one wave, and the device able to co-schedule that
// many clusters of S (active(S) reports how many it can).
template <typename Active>
Plan plan_few(const Plan& base, Tiles t, long units, int sms, Active active) {
    Plan pl = base;
    const int T = t.prefix + t.tree;
    pl.tps = T;
    for (int tps = 2; tps < T; ++tps) {
        const int S = (T + tps - 1) / tps;
        if (S > kMaxSplits || units * S > sms) continue;
        if (active(S) < units) continue;
        pl.tps = tps;
        break;
    }
    pl.smax = (T + pl.tps - 1) / pl.tps;
    pl.merge = pl.smax > 1 ? kMergeCluster : kMergeNone;
    return pl;
}

struct WsLayout {
    size_t tickets, part_o, part_ml, total;
};

// Workspace of the global merge (empty for the other plans).
WsLayout attn_layout(const Plan& pl, int B, int Hkv, int D) {
    WsLayout w{};
    if (pl.merge != kMergeGlobal) return w;
    const size_t tiles = (size_t)B * Hkv * pl.mtiles;  // partials per query tile
    w.tickets = 0;  // one counter per (sequence, KV head, tile pair)
    w.part_o = align_up((size_t)B * Hkv * pl.mpairs * 4, 256);
    w.part_ml = align_up(w.part_o + tiles * pl.smax * (size_t)D * BM * 2, 256);
    w.total = align_up(w.part_ml + tiles * pl.smax * 2 * BM * 4, 256);
    return w;
}

// Co-resident clusters of `size` CTAs of tree_attn_kernel<D> on device `dev`
// (0 if that size cannot launch).  Needs the kernel's attributes set first.
template <int D>
int active_clusters(int dev, int size) {
    static int cached[64][kMaxSplits + 1];
    static bool done[64][kMaxSplits + 1];
    if (size < 1 || size > kMaxSplits) return 0;
    if (!done[dev & 63][size]) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)size);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = Cfg<D>::SMEM;
        cudaLaunchAttribute at;
        at.id = cudaLaunchAttributeClusterDimension;
        at.val.clusterDim.x = (unsigned)size;
        at.val.clusterDim.y = 1;
        at.val.clusterDim.z = 1;
        cfg.attrs = &at;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, tree_attn_kernel<D>, &cfg) != cudaSuccess) {
            n = 0;
            (void)cudaGetLastError();  // a refused size is not an error of the call
        }
        cached[dev & 63][size] = n;
        done[dev & 63][size] = true;
    }
    return cached[dev & 63][size];
}

template <int D>
cudaError_t launch_d(const AttnArgs& a, cudaStream_t s) {
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaGetDevice(&dev);
    std::call_once(once[dev & 63], [&] {
        cudaError_t e = cudaFuncSetAttribute(tree_attn_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tree_attn_kernel<D>,
                                     cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        attr_err[dev & 63] = e;
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    const Plan base = plan_base(a.N, a.Hq, a.Hkv);
    const Tiles t = max_tiles(a.N, a.cache_cap);
    const long units = plan_units(base, a.B, a.Hkv);
    const int sms = num_sms();
    const Plan pl = units >= sms ? plan_many(base, t, units, sms)
                                 : plan_few(base, t, units, sms,
                                            [&](int S) {
                                                return Cfg<D>::recv_fits_upto(S) ? active_clusters<D>(dev, S) : 0;
                                            });
    const WsLayout wl = attn_layout(pl, a.B, a.Hkv, D);
    const int G = a.Hq / a.Hkv, R = a.N + 1;
    CUtensorMap mq, mkc, mvc, mkt, mvt;
    const uint64_t rowb = (uint64_t)D * 2;
    bool ok = make_map(&mq, a.q, D, a.Hq, (uint64_t)a.B * R, rowb, rowb * a.Hq, 64, G, BM / G);
    ok = ok && make_map(&mkc, a.k_cache, D, a.cache_cap, (uint64_t)a.B * a.Hkv, rowb,
                        rowb * (a.cache_cap ? a.cache_cap : 1), 64, BN, 1);
    ok = ok && make_map(&mvc, a.v_cache, D, a.cache_cap, (uint64_t)a.B * a.Hkv, rowb,
                        rowb * (a.cache_cap ? a.cache_cap : 1), 64, BN, 1);
    ok = ok && make_map(&mkt, a.k_tree, D, a.Hkv, (uint64_t)a.B * R, rowb, rowb * a.Hkv, 64, 1, BN);
    ok = ok && make_map(&mvt, a.v_tree, D, a.Hkv, (uint64_t)a.B * R, rowb, rowb * a.Hkv, 64, 1, BN);
    if (!ok) return cudaErrorInvalidValue;
    Params p;
    p.prefix_len = a.prefix_len;
    p.n_nodes = a.n_nodes;
    p.anc_mask = a.anc_mask;
    p.out = (uint16_t*)a.out;
    p.lse = a.lse;
    char* ws = (char*)a.ws;
    const bool glob = pl.merge == kMergeGlobal;
    p.tickets = glob ? (unsigned int*)(ws + wl.tickets) : nullptr;
    p.part_o = glob ? (uint32_t*)(ws + wl.part_o) : nullptr;
    p.part_ml = glob ? (float*)(ws + wl.part_ml) : nullptr;
    p.B = a.B; p.N = a.N; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = G; p.W = (a.N + 1 + 31) / 32;
    p.mtiles = pl.mtiles; p.mpairs = pl.mpairs; p.tps = pl.tps; p.smax = pl.smax;
    p.merge = pl.merge;
    p.lpt = (pl.merge != kMergeCluster && (long)a.B * pl.smax <= kLptMaxItems) ? 1 : 0;
    p.cache_cap = a.cache_cap;
    p.scale_log2 = a.scale * kLog2e;
    p.err = a.err;
    const long grid = units * pl.smax;
    return launch_pdl_cluster(tree_attn_kernel<D>, dim3((unsigned)grid), dim3(kThreads),
                              (size_t)Cfg<D>::SMEM, s,
                              pl.merge == kMergeCluster ? (unsigned)pl.smax : 1u, mq, mkc, mvc,
                              mkt, mvt, p);
}

}  // namespace

// Only plans for many units (no clusters) merge their KV splits in a workspace.
size_t attn_workspace_bytes(int B, int N, int Hq, int Hkv, int D, int64_t cache_cap) {
    const Plan base = plan_base(N, Hq, Hkv);
    if (plan_units(base, B, Hkv) < num_sms()) return 0;
    return attn_layout(plan_many(base, max_tiles(N, cache_cap), plan_units(base, B, Hkv), num_sms()),
                       B, Hkv, D).total;
}

cudaError_t launch_tree_attn(const AttnArgs& a, cudaStream_t s) {
    if (a.D == 128) return launch_d<128>(a, s);
    return launch_d<64>(a, s);
}

}  // namespace ddt
