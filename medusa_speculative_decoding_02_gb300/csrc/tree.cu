// tree.cu -- budgeted candidate tree, one CTA per sequence.
//
// "Medusa 深读" §6.2 builds the tree greedily: starting from the children of
// the root, repeatedly move the frontier node of largest path weight into the
// tree and add its children to the frontier, until the budget of n nodes is
// spent.  The path weight is a product of per-level weights; here the levels
// are the heads' own top-s probabilities, so a node's score is the sum of its
// path's log-probabilities, accumulated from depth 1 down in fp64.
//
// Because every log-probability is <= 0, a child never outscores its parent,
// and with ties broken towards the smaller depth an ancestor always precedes
// its descendants.  The greedy picks are therefore exactly the first n nodes
// of the whole Cartesian tree in the order (score desc, depth asc, rank path
// asc).  The kernel finds them level by level without a serial frontier:
//   level 1 candidates are the s_1 root children; level D candidates are the
//   children of the level D-1 survivors; a level keeps its best n candidates
//   (no node outside a level's best n can be among the global first n);
//   finally the survivors of all levels are ranked together and the first n
//   kept.  Ranks come from counting how many candidates precede each one,
//   which is deterministic and needs no sort.  Full trees of at most 512
//   nodes skip the level cut and rank all their nodes at once.
// Node identity is (depth, rank path) with the rank path packed four bits per
// level, level 1 in the top nibble, so equal-depth paths compare
// lexicographically as integers.
//
// Outputs follow the canonical order (root, then depth, then rank path) and
// "Medusa 深读" §6.1: parent index, depth, position id = P_b + depth (nodes of
// one depth share one position), ancestor bitmask rows (self and ancestors
// set), and the root-to-leaf node lists of every leaf.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace medusa {

namespace {

constexpr int kTreeThreads = 1024;

__device__ __forceinline__ int nib_shift(int depth) { return 28 - 4 * (depth - 1); }

// Order-preserving integer image of an fp64 score (no NaN; -0 folded into
// +0), so every comparison below is integer work: GB300's fp64 rate is a
// small fraction of its integer rate.
__device__ __forceinline__ uint64_t score_key(double s) {
    const uint64_t u = static_cast<uint64_t>(__double_as_longlong(s + 0.0));
    return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}

// node a is taken before node b: larger score, then smaller depth, then the
// smaller rank path; lo = depth << 32 | path
__device__ __forceinline__ bool precedes(uint64_t ka, uint64_t la, uint64_t kb, uint64_t lb) {
    return ka > kb || (ka == kb && la < lb);
}

// Full Cartesian trees up to this many nodes are ranked in one pass over all
// their nodes; larger ones go level by level.
constexpr int kDirectMax = 512;

struct TreeSmem {
    double *cand_score;
    uint64_t *cand_key;
    uint64_t *cand_lo;     // depth << 32 | rank path
    double *kept_score;
    uint64_t *kept_key;
    uint64_t *kept_lo;
    uint64_t *sel_lo;      // the n picks, any order
    uint64_t *c_lo;        // canonical order: c_lo[0] = root, ascending
    int *c_parent;
    int *has_child;
    int *leaf_of;
};

__host__ __device__ inline size_t take_bytes(size_t &o, size_t bytes, size_t align) {
    o = (o + align - 1) / align * align;
    const size_t at = o;
    o += bytes;
    return at;
}

__host__ __device__ inline int tree_cand_cap(int S, int n, long long full) {
    if (full <= kDirectMax) return (int)full;
    return n * S > S ? n * S : S;
}

__host__ __device__ inline size_t tree_smem_layout(int K, int S, int n, long long full, TreeSmem *p,
                                                   char *base) {
    const int cand_cap = tree_cand_cap(S, n, full);
    const int kept_cap = full <= kDirectMax ? 1 : K * n;
    const int R = n + 1;
    size_t o = 0;
    const size_t a0 = take_bytes(o, sizeof(double) * cand_cap, 8);
    const size_t a1 = take_bytes(o, sizeof(uint64_t) * cand_cap, 8);
    const size_t a2 = take_bytes(o, sizeof(uint64_t) * cand_cap, 8);
    const size_t a3 = take_bytes(o, sizeof(double) * kept_cap, 8);
    const size_t a4 = take_bytes(o, sizeof(uint64_t) * kept_cap, 8);
    const size_t a5 = take_bytes(o, sizeof(uint64_t) * kept_cap, 8);
    const size_t a6 = take_bytes(o, sizeof(uint64_t) * n, 8);
    const size_t a7 = take_bytes(o, sizeof(uint64_t) * R, 8);
    const size_t a8 = take_bytes(o, sizeof(int) * R, 4);
    const size_t a9 = take_bytes(o, sizeof(int) * R, 4);
    const size_t a10 = take_bytes(o, sizeof(int) * R, 4);
    if (p) {
        p->cand_score = reinterpret_cast<double *>(base + a0);
        p->cand_key = reinterpret_cast<uint64_t *>(base + a1);
        p->cand_lo = reinterpret_cast<uint64_t *>(base + a2);
        p->kept_score = reinterpret_cast<double *>(base + a3);
        p->kept_key = reinterpret_cast<uint64_t *>(base + a4);
        p->kept_lo = reinterpret_cast<uint64_t *>(base + a5);
        p->sel_lo = reinterpret_cast<uint64_t *>(base + a6);
        p->c_lo = reinterpret_cast<uint64_t *>(base + a7);
        p->c_parent = reinterpret_cast<int *>(base + a8);
        p->has_child = reinterpret_cast<int *>(base + a9);
        p->leaf_of = reinterpret_cast<int *>(base + a10);
    }
    return (o + 15) / 16 * 16;
}

struct TreeArgs {
    const int32_t *root;
    const int32_t *ids;
    const float *logp;
    long long logp_bstride;  // elements between sequences' tables (0: one shared table)
    int K, S, n;
    long long full;  // nodes of the full Cartesian tree (capped)
    int s[MEDUSA_MAX_HEADS];
    // full trees of at most kDirectMax nodes: level D (1-based) holds node
    // indices [lvl_base[D-1], lvl_base[D]), and mdiv[j] = ceil(2^16 / s[j])
    // divides by s[j] exactly for dividends below 4096
    int lvl_base[MEDUSA_MAX_HEADS + 1];
    uint32_t mdiv[MEDUSA_MAX_HEADS];
    const int32_t *prefix_len;
    int32_t *tokens, *parent, *depth, *pos_id;
    uint64_t *anc_mask;
    int32_t *paths, *n_leaf;
    int *status;
};

__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Number of entries of (key, lo)[0..c) that are taken before (ki, li):
// computed by one warp, lanes splitting the entries.
__device__ __forceinline__ int count_before(const uint64_t *key, const uint64_t *lo, int c,
                                            uint64_t ki, uint64_t li, int lane) {
    int cnt = 0;
#pragma unroll 4
    for (int j = lane; j < c; j += kWarp) cnt += precedes(key[j], lo[j], ki, li);
    return warp_sum_int(cnt);
}

// Rank every item i < c of (key, lo)[0..c) -- the number of entries taken
// before it -- with four threads per item, each counting a quarter of the
// entries (threads of an item read the same words: shared-memory
// broadcasts), combined by two shuffles; the entry of rank r < n goes to
// out[r].  All threads of the CTA call it (the shuffles need full warps).
__device__ __forceinline__ void rank_quad(const uint64_t *key, const uint64_t *lo, int c, int n,
                                          uint64_t *out, int tid, int nt) {
    for (int base = 0; base < c; base += nt / 4) {
        const int i = base + (tid >> 2), q = tid & 3;
        int cnt = 0;
        if (i < c) {
            const uint64_t ki = key[i], li = lo[i];
#pragma unroll 4
            for (int j = q; j < c; j += 4) cnt += precedes(key[j], lo[j], ki, li);
        }
        cnt += __shfl_xor_sync(0xffffffffu, cnt, 1);
        cnt += __shfl_xor_sync(0xffffffffu, cnt, 2);
        if (i < c && q == 0 && cnt < n) out[cnt] = lo[i];
    }
}

// The level-wise passes of large trees give one warp per item and split the
// comparisons over its lanes, so the longest dependent chain is ~c/32 shared
// loads plus a five-step shuffle.
__global__ void __launch_bounds__(kTreeThreads) build_tree_kernel(TreeArgs a) {
    pdl_enter();
    extern __shared__ __align__(16) char tsm[];
    __shared__ double lp[MEDUSA_MAX_HEADS][MEDUSA_MAX_TOP_S];
    __shared__ int tid_tok[MEDUSA_MAX_HEADS][MEDUSA_MAX_TOP_S];
    __shared__ int warp_leaves[kTreeThreads / kWarp];
    TreeSmem sm;
    tree_smem_layout(a.K, a.S, a.n, a.full, &sm, tsm);
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nt = blockDim.x, nw = nt >> 5;
    const int K = a.K, S = a.S, n = a.n, R = n + 1;
    const int W = (R + 63) / 64;

    // the scalars the last phase needs, loaded with the tables
    __shared__ int s_root, s_prefix;
    if (tid == 0) {
        s_root = a.root[b];
        s_prefix = a.prefix_len ? a.prefix_len[b] : 0;
    }
    for (int i = tid; i < R; i += nt) sm.has_child[i] = 0;
    for (int i = tid; i < K * S; i += nt) {
        const int k = i / S, r = i - k * S;
        const float v = a.logp[(size_t)b * a.logp_bstride + (size_t)k * S + r];
        if (r < a.s[k] && (v > 0.f || v != v)) set_status(a.status, MEDUSA_DEV_BAD_SCORE);
        lp[k][r] = (double)v;
        tid_tok[k][r] = a.ids[((size_t)b * K + k) * S + r];
    }
    __syncthreads();

    if (a.full <= kDirectMax) {
        // ---- small tree: every node of the full tree.  Node t of level D
        // has local index l = t - lvl_base[D-1], whose mixed-radix digits
        // (level 1 most significant) are its rank path; the score is summed
        // from depth 1 down in fp64, as the frontier does.
        const int full = (int)a.full;
        for (int t = tid; t < full; t += nt) {
            int D = 1;
            while (t >= a.lvl_base[D]) ++D;
            uint32_t l = (uint32_t)(t - a.lvl_base[D - 1]);
            uint32_t path = 0;
            for (int j = D - 1; j >= 0; --j) {
                const uint32_t q = (l * a.mdiv[j]) >> 16;  // l / s[j]
                path |= (l - q * (uint32_t)a.s[j]) << nib_shift(j + 1);
                l = q;
            }
            double sc = 0.0;
            for (int j = 0; j < D; ++j) {
                const double v = lp[j][(path >> nib_shift(j + 1)) & 0xFu];
                sc = (j == 0) ? v : sc + v;
            }
            sm.cand_key[t] = score_key(sc);
            sm.cand_lo[t] = ((uint64_t)D << 32) | path;
        }
        __syncthreads();
        rank_quad(sm.cand_key, sm.cand_lo, full, n, sm.sel_lo, tid, nt);
    } else {
        // ---- large tree: level D keeps its best n candidates (a node
        // outside them cannot be among the first n overall)
        int prev_count = 0, prev_off = 0;
        for (int D = 1; D <= K; ++D) {
            const int sD = a.s[D - 1];
            const int c = (D == 1) ? sD : prev_count * sD;
            const int sh = nib_shift(D);
            for (int i = tid; i < c; i += nt) {
                double sc;
                uint32_t pa;
                if (D == 1) {
                    sc = lp[0][i];
                    pa = (uint32_t)i << sh;
                } else {
                    const int p = i / sD, r = i - p * sD;
                    sc = sm.kept_score[prev_off + p] + lp[D - 1][r];
                    pa = (uint32_t)sm.kept_lo[prev_off + p] | ((uint32_t)r << sh);
                }
                sm.cand_score[i] = sc;
                sm.cand_key[i] = score_key(sc);
                sm.cand_lo[i] = ((uint64_t)D << 32) | pa;
            }
            __syncthreads();
            const int off = (D == 1) ? 0 : prev_off + prev_count;
            for (int i = warp; i < c; i += nw) {
                const int cnt = count_before(sm.cand_key, sm.cand_lo, c, sm.cand_key[i],
                                             sm.cand_lo[i], lane);
                if (lane == 0 && cnt < n) {
                    sm.kept_score[off + cnt] = sm.cand_score[i];
                    sm.kept_key[off + cnt] = sm.cand_key[i];
                    sm.kept_lo[off + cnt] = sm.cand_lo[i];
                }
            }
            prev_off = off;
            prev_count = c < n ? c : n;
            __syncthreads();
        }
        const int total = prev_off + prev_count;
        for (int i = warp; i < total; i += nw) {
            const int cnt = count_before(sm.kept_key, sm.kept_lo, total, sm.kept_key[i],
                                         sm.kept_lo[i], lane);
            if (lane == 0 && cnt < n) sm.sel_lo[cnt] = sm.kept_lo[i];
        }
    }
    __syncthreads();

    // ---- canonical order (root, then (depth, rank path) ascending; the lo
    // words are distinct) and parents in one pass, four threads per node: a
    // node's place is 1 + the number of picks below its lo word, and its
    // parent -- the node one level up with the same rank path minus the last
    // rank, always a pick too (a child never precedes its parent) -- sits at
    // 1 + the number of picks below the parent's lo word
    for (int base = 0; base < n; base += nt / 4) {
        const int i = base + (tid >> 2), q = tid & 3;
        int cnt = 0, pcnt = 0, D = 0;
        uint64_t li = 0;
        if (i < n) {
            li = sm.sel_lo[i];
            D = (int)(li >> 32);
            const uint32_t ppath = (uint32_t)li & ~((uint32_t)0xF << nib_shift(D));
            const uint64_t want = D > 1 ? ((uint64_t)(D - 1) << 32) | ppath : 0;
#pragma unroll 4
            for (int j = q; j < n; j += 4) {
                const uint64_t lj = sm.sel_lo[j];
                cnt += lj < li;
                pcnt += lj < want;
            }
        }
        cnt += __shfl_xor_sync(0xffffffffu, cnt, 1);
        cnt += __shfl_xor_sync(0xffffffffu, cnt, 2);
        pcnt += __shfl_xor_sync(0xffffffffu, pcnt, 1);
        pcnt += __shfl_xor_sync(0xffffffffu, pcnt, 2);
        if (i < n && q == 0) {
            const int p = D > 1 ? 1 + pcnt : 0;
            sm.c_lo[1 + cnt] = li;
            sm.c_parent[1 + cnt] = p;
            sm.has_child[p] = 1;
        }
    }
    if (tid == 0) {
        sm.c_lo[0] = 0;
        sm.c_parent[0] = -1;
    }
    __syncthreads();

    // ---- per-node outputs; leaves numbered by a ballot scan
    const int P = s_prefix;
    const bool leaf = tid < R && !sm.has_child[tid];
    const unsigned bal = __ballot_sync(0xffffffffu, leaf);
    if (lane == 0) warp_leaves[warp] = __popc(bal);
    __syncthreads();
    // leaves before this warp and in total: one shuffle scan of the per-warp
    // counts (nw <= 32)
    int incl = lane < nw ? warp_leaves[lane] : 0;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const int nl = __shfl_sync(0xffffffffu, incl, kWarp - 1);
    const int before = warp > 0 ? __shfl_sync(0xffffffffu, incl, warp - 1) : 0;
    if (leaf) sm.leaf_of[before + __popc(bal & ((1u << lane) - 1u))] = tid;
    if (tid < R) {
        const int i = tid;
        const uint64_t li = sm.c_lo[i];
        const int D = (int)(li >> 32);
        const size_t o = (size_t)b * R + i;
        int tok;
        if (i == 0) {
            tok = s_root;
        } else {
            const int r = (int)(((uint32_t)li >> nib_shift(D)) & 0xF);
            tok = tid_tok[D - 1][r];
        }
        a.tokens[o] = tok;
        a.parent[o] = sm.c_parent[i];
        a.depth[o] = D;
        a.pos_id[o] = P + D;
        // one walk up the ancestors sets the bits of every mask word
        uint64_t mw[4] = {0, 0, 0, 0};  // W <= 4 (R <= 256)
        for (int x = i; x >= 0; x = sm.c_parent[x]) {
            const uint64_t bit = (uint64_t)1 << (x & 63);
            const int w = x >> 6;
            mw[0] |= w == 0 ? bit : 0;
            mw[1] |= w == 1 ? bit : 0;
            mw[2] |= w == 2 ? bit : 0;
            mw[3] |= w == 3 ? bit : 0;
        }
        for (int w = 0; w < W; ++w)
            a.anc_mask[o * W + w] = w == 0 ? mw[0] : w == 1 ? mw[1] : w == 2 ? mw[2] : mw[3];
    }
    __syncthreads();
    if (tid == 0) a.n_leaf[b] = nl;
    const int cols = K + 1;
    for (int e = tid; e < n * cols; e += nt) {
        const int li = e / cols, q = e - li * cols;
        int v = -1;
        if (li < nl) {
            int x = sm.leaf_of[li];
            const int D = (int)(sm.c_lo[x] >> 32);
            if (q <= D) {
                for (int up = D - q; up > 0; --up) x = sm.c_parent[x];
                v = x;
            }
        }
        a.paths[(size_t)b * n * cols + e] = v;
    }
}

}  // namespace

size_t tree_workspace_bytes(int B, int K, int S, int n) {
    (void)B; (void)K; (void)S; (void)n;
    return MEDUSA_WS_HEADER;
}

cudaError_t launch_build_tree(const int32_t *root, const int32_t *ids, const float *logp,
                              bool shared_table, int B, int K, const int32_t *s_host, int S,
                              int n, const int32_t *prefix_len, int32_t *tokens, int32_t *parent,
                              int32_t *depth, int32_t *pos_id, uint64_t *anc_mask, int32_t *paths,
                              int32_t *n_leaf, void *ws, cudaStream_t stream) {
    TreeArgs a;
    a.root = root;
    a.ids = ids;
    a.logp = logp;
    a.logp_bstride = shared_table ? 0 : (long long)K * S;
    a.K = K;
    {
        long long full = 0, level = 1;
        for (int k = 0; k < K; ++k) {
            level *= s_host[k];
            full += level;
            if (full > (1 << 20)) break;
        }
        a.full = full;
    }
    a.S = S;
    a.n = n;
    for (int k = 0; k < MEDUSA_MAX_HEADS; ++k) a.s[k] = k < K ? s_host[k] : 0;
    {
        long long base = 0, level = 1;
        a.lvl_base[0] = 0;
        for (int k = 0; k < MEDUSA_MAX_HEADS; ++k) {
            if (k < K && a.full <= kDirectMax) {
                level *= s_host[k];
                base += level;
            }
            a.lvl_base[k + 1] = (int)std::min<long long>(base, 1 << 20);
            a.mdiv[k] = k < K ? (65536u + (uint32_t)s_host[k] - 1u) / (uint32_t)s_host[k] : 0u;
        }
    }
    a.prefix_len = prefix_len;
    a.tokens = tokens;
    a.parent = parent;
    a.depth = depth;
    a.pos_id = pos_id;
    a.anc_mask = anc_mask;
    a.paths = paths;
    a.n_leaf = n_leaf;
    a.status = static_cast<int *>(ws);
    const size_t smem = tree_smem_layout(K, S, n, a.full, nullptr, nullptr);
    cudaError_t e = cudaFuncSetAttribute(build_tree_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e) return e;
    e = launch_pdl(build_tree_kernel, dim3(B), dim3(kTreeThreads), smem, stream, a);
    note_launch();
    return e;
}

}  // namespace medusa
