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
//   which is deterministic and needs no sort.
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

constexpr int kTreeThreads = 256;

__device__ __forceinline__ int nib_shift(int depth) { return 28 - 4 * (depth - 1); }

__device__ __forceinline__ bool precedes(double sa, int da, uint32_t pa, double sb, int db,
                                         uint32_t pb) {
    if (sa != sb) return sa > sb;
    if (da != db) return da < db;
    return pa < pb;
}

struct TreeSmem {
    double *cand_score;
    uint32_t *cand_path;
    double *kept_score;
    uint32_t *kept_path;
    unsigned char *kept_depth;
    int *sel_depth;
    uint32_t *sel_path;
    int *c_depth;
    uint32_t *c_path;
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

__host__ __device__ inline size_t tree_smem_layout(int K, int S, int n, TreeSmem *p, char *base) {
    const int cand_cap = n * S > S ? n * S : S;
    const int kept_cap = K * n;
    const int R = n + 1;
    size_t o = 0;
    const size_t a0 = take_bytes(o, sizeof(double) * cand_cap, 8);
    const size_t a1 = take_bytes(o, sizeof(double) * kept_cap, 8);
    const size_t a2 = take_bytes(o, sizeof(uint32_t) * cand_cap, 4);
    const size_t a3 = take_bytes(o, sizeof(uint32_t) * kept_cap, 4);
    const size_t a4 = take_bytes(o, sizeof(int) * n, 4);
    const size_t a5 = take_bytes(o, sizeof(uint32_t) * n, 4);
    const size_t a6 = take_bytes(o, sizeof(int) * R, 4);
    const size_t a7 = take_bytes(o, sizeof(uint32_t) * R, 4);
    const size_t a8 = take_bytes(o, sizeof(int) * R, 4);
    const size_t a9 = take_bytes(o, sizeof(int) * R, 4);
    const size_t a10 = take_bytes(o, sizeof(int) * n, 4);
    const size_t a11 = take_bytes(o, kept_cap, 1);
    if (p) {
        p->cand_score = reinterpret_cast<double *>(base + a0);
        p->kept_score = reinterpret_cast<double *>(base + a1);
        p->cand_path = reinterpret_cast<uint32_t *>(base + a2);
        p->kept_path = reinterpret_cast<uint32_t *>(base + a3);
        p->sel_depth = reinterpret_cast<int *>(base + a4);
        p->sel_path = reinterpret_cast<uint32_t *>(base + a5);
        p->c_depth = reinterpret_cast<int *>(base + a6);
        p->c_path = reinterpret_cast<uint32_t *>(base + a7);
        p->c_parent = reinterpret_cast<int *>(base + a8);
        p->has_child = reinterpret_cast<int *>(base + a9);
        p->leaf_of = reinterpret_cast<int *>(base + a10);
        p->kept_depth = reinterpret_cast<unsigned char *>(base + a11);
    }
    return (o + 15) / 16 * 16;
}

struct TreeArgs {
    const int32_t *root;
    const int32_t *ids;
    const float *logp;
    int K, S, n;
    int s[MEDUSA_MAX_HEADS];
    const int32_t *prefix_len;
    int32_t *tokens, *parent, *depth, *pos_id;
    uint64_t *anc_mask;
    int32_t *paths, *n_leaf;
    int *status;
};

__global__ void __launch_bounds__(kTreeThreads) build_tree_kernel(TreeArgs a) {
    extern __shared__ __align__(16) char tsm[];
    __shared__ double lp[MEDUSA_MAX_HEADS][MEDUSA_MAX_TOP_S];
    __shared__ int tid_tok[MEDUSA_MAX_HEADS][MEDUSA_MAX_TOP_S];
    __shared__ int level_off[MEDUSA_MAX_HEADS + 1];
    __shared__ int n_leaf_s;
    TreeSmem sm;
    tree_smem_layout(a.K, a.S, a.n, &sm, tsm);
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int K = a.K, S = a.S, n = a.n, R = n + 1;
    const int W = (R + 63) / 64;

    for (int i = tid; i < K * S; i += nt) {
        const int k = i / S, r = i - k * S;
        const float v = a.logp[((size_t)b * K + k) * S + r];
        if (r < a.s[k] && (v > 0.f || v != v)) set_status(a.status, MEDUSA_DEV_BAD_SCORE);
        lp[k][r] = (double)v;
        tid_tok[k][r] = a.ids[((size_t)b * K + k) * S + r];
    }
    if (tid == 0) {
        level_off[0] = 0;
        n_leaf_s = 0;
    }
    __syncthreads();

    // ---- level-wise survivors
    int prev_count = 0, prev_off = 0;
    for (int D = 1; D <= K; ++D) {
        const int sD = a.s[D - 1];
        const int c = (D == 1) ? sD : prev_count * sD;
        const int sh = nib_shift(D);
        for (int i = tid; i < c; i += nt) {
            if (D == 1) {
                sm.cand_score[i] = lp[0][i];
                sm.cand_path[i] = (uint32_t)i << sh;
            } else {
                const int p = i / sD, r = i - p * sD;
                sm.cand_score[i] = sm.kept_score[prev_off + p] + lp[D - 1][r];
                sm.cand_path[i] = sm.kept_path[prev_off + p] | ((uint32_t)r << sh);
            }
        }
        __syncthreads();
        const int off = (D == 1) ? 0 : prev_off + prev_count;
        for (int i = tid; i < c; i += nt) {
            const double si = sm.cand_score[i];
            const uint32_t pi = sm.cand_path[i];
            int rank = 0;
            for (int j = 0; j < c; ++j) {
                const double sj = sm.cand_score[j];
                rank += (sj > si) || (sj == si && sm.cand_path[j] < pi);
            }
            if (rank < n) {
                sm.kept_score[off + rank] = si;
                sm.kept_path[off + rank] = pi;
                sm.kept_depth[off + rank] = (unsigned char)D;
            }
        }
        prev_off = off;
        prev_count = c < n ? c : n;
        if (tid == 0) level_off[D] = off + prev_count;
        __syncthreads();
    }
    const int total = level_off[K];

    // ---- global first n among all survivors
    for (int i = tid; i < total; i += nt) {
        const double si = sm.kept_score[i];
        const int di = sm.kept_depth[i];
        const uint32_t pi = sm.kept_path[i];
        int rank = 0;
        for (int j = 0; j < total; ++j)
            rank += precedes(sm.kept_score[j], sm.kept_depth[j], sm.kept_path[j], si, di, pi);
        if (rank < n) {
            sm.sel_depth[rank] = di;
            sm.sel_path[rank] = pi;
        }
    }
    __syncthreads();

    // ---- canonical order: root, then (depth, rank path)
    if (tid == 0) {
        sm.c_depth[0] = 0;
        sm.c_path[0] = 0;
        sm.c_parent[0] = -1;
    }
    for (int i = tid; i < n; i += nt) {
        const int di = sm.sel_depth[i];
        const uint32_t pi = sm.sel_path[i];
        int ci = 1;
        for (int j = 0; j < n; ++j) {
            const int dj = sm.sel_depth[j];
            ci += (dj < di) || (dj == di && sm.sel_path[j] < pi);
        }
        sm.c_depth[ci] = di;
        sm.c_path[ci] = pi;
    }
    for (int i = tid; i < R; i += nt) sm.has_child[i] = 0;
    __syncthreads();
    for (int i = 1 + tid; i < R; i += nt) {
        const int D = sm.c_depth[i];
        int p = 0;
        if (D > 1) {
            const uint32_t pp = sm.c_path[i] & ~((uint32_t)0xF << nib_shift(D));
            p = -1;
            for (int j = 1; j < i; ++j)
                if (sm.c_depth[j] == D - 1 && sm.c_path[j] == pp) {
                    p = j;
                    break;
                }
        }
        sm.c_parent[i] = p;
        if (p >= 0) sm.has_child[p] = 1;
    }
    __syncthreads();

    // ---- per-node outputs
    const int P = a.prefix_len ? a.prefix_len[b] : 0;
    for (int i = tid; i < R; i += nt) {
        const int D = sm.c_depth[i];
        const size_t o = (size_t)b * R + i;
        int tok;
        if (i == 0) {
            tok = a.root[b];
        } else {
            const int r = (int)((sm.c_path[i] >> nib_shift(D)) & 0xF);
            tok = tid_tok[D - 1][r];
        }
        a.tokens[o] = tok;
        a.parent[o] = sm.c_parent[i];
        a.depth[o] = D;
        a.pos_id[o] = P + D;
        uint64_t m[4] = {0, 0, 0, 0};
        for (int x = i; x >= 0; x = sm.c_parent[x]) m[x >> 6] |= (uint64_t)1 << (x & 63);
        for (int w = 0; w < W; ++w) a.anc_mask[o * W + w] = m[w];
        if (!sm.has_child[i]) {
            int li = 0;
            for (int j = 0; j < i; ++j) li += !sm.has_child[j];
            sm.leaf_of[li] = i;
            atomicAdd(&n_leaf_s, 1);
        }
    }
    __syncthreads();
    const int nl = n_leaf_s;
    if (tid == 0) a.n_leaf[b] = nl;
    const int cols = K + 1;
    for (int e = tid; e < n * cols; e += nt) {
        const int li = e / cols, q = e - li * cols;
        int v = -1;
        if (li < nl) {
            int x = sm.leaf_of[li];
            const int D = sm.c_depth[x];
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

cudaError_t launch_build_tree(const int32_t *root, const int32_t *ids, const float *logp, int B,
                              int K, const int32_t *s_host, int S, int n,
                              const int32_t *prefix_len, int32_t *tokens, int32_t *parent,
                              int32_t *depth, int32_t *pos_id, uint64_t *anc_mask, int32_t *paths,
                              int32_t *n_leaf, void *ws, cudaStream_t stream) {
    TreeArgs a;
    a.root = root;
    a.ids = ids;
    a.logp = logp;
    a.K = K;
    a.S = S;
    a.n = n;
    for (int k = 0; k < MEDUSA_MAX_HEADS; ++k) a.s[k] = k < K ? s_host[k] : 0;
    a.prefix_len = prefix_len;
    a.tokens = tokens;
    a.parent = parent;
    a.depth = depth;
    a.pos_id = pos_id;
    a.anc_mask = anc_mask;
    a.paths = paths;
    a.n_leaf = n_leaf;
    a.status = static_cast<int *>(ws);
    const size_t smem = tree_smem_layout(K, S, n, nullptr, nullptr);
    cudaError_t e = cudaFuncSetAttribute(build_tree_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e) return e;
    build_tree_kernel<<<B, kTreeThreads, smem, stream>>>(a);
    note_launch();
    return cudaGetLastError();
}

}  // namespace medusa
