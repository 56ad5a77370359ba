// posterior.cu -- acceptance and the longest accepted path.
//
// A tree node's token is judged by the verification logits of its parent's
// row (that row is the target model's distribution for the next position).
//   greedy  ("Medusa Part I" Part 2): accept iff the token is the row argmax.
//   typical ("Medusa 深读" §5): accept iff p(x) > min(eps, delta*exp(-H(p))),
//           p = softmax(logits / T), H in nats.
// The root is accepted unconditionally ("Medusa 深读" §5); a node counts only
// if its whole branch is accepted ("Medusa Part I" Part 2: a rejection ends
// the prefix); the deepest counted node wins and its row's argmax is the next
// token.
//
// Two kernels:
//   posterior_rows_kernel    each logits row split over a few CTAs (enough for
//                            every SM): one streaming pass with 16-byte loads
//                            computes the slice's argmax and, for typical
//                            acceptance, the shifted sums S = sum 2^(y-m),
//                            A = sum 2^(y-m) (y-m) in the log2 domain
//                            (y = logit * log2(e) / T).  Slices go to scratch;
//                            merged, they give H = ln S - ln2 * A / S.
//   posterior_select_kernel  one CTA per sequence, one thread per node:
//                            per-node decision, prefix-AND down the tree
//                            level by level, longest path, next token (and,
//                            for a step executor, a completion word raised
//                            in page-locked memory once all is written).
#include <algorithm>
#include <climits>

#include "commit.cuh"
#include "common.cuh"
#include "launch.h"

namespace medusa {

namespace {

constexpr int kRowThreads = 256;
constexpr int kMaxSplits = 8;
constexpr int kSelectThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Statistics of one slice of a logits row (a row is split over several CTAs).
struct RowPart {
    float amax;   // largest logit of the slice
    int arg;      // its token id (smallest id among equal values)
    float m2;     // max of y = logit * log2(e) / T over the slice
    float S;      // sum 2^(y - m2)
    float A;      // sum 2^(y - m2) (y - m2)
};

// (m, S, A) triple of shifted sums in the log2 domain
struct Moments {
    float m, S, A;
    __device__ __forceinline__ void merge(float m2, float S2, float A2) {
        if (S2 == 0.f) return;
        if (S == 0.f) {
            m = m2; S = S2; A = A2;
            return;
        }
        const float mn = fmaxf(m, m2);
        const float f1 = exp2f(m - mn), f2 = exp2f(m2 - mn);
        A = f1 * (A + S * (m - mn)) + f2 * (A2 + S2 * (m2 - mn));
        S = S * f1 + S2 * f2;
        m = mn;
    }
};

template <typename T, bool TYPICAL>
__global__ void __launch_bounds__(kRowThreads)
posterior_rows_kernel(const T *__restrict__ logits, int R, int V, int splits, float y_scale,
                      RowPart *__restrict__ parts) {
    constexpr int VN = Vec16<T>::N;
    constexpr int U = 4;
    __shared__ float s_val[kRowThreads / kWarp];
    __shared__ int s_id[kRowThreads / kWarp];
    __shared__ float s_m[kRowThreads / kWarp], s_S[kRowThreads / kWarp], s_A[kRowThreads / kWarp];
    const int sp = blockIdx.x, row = blockIdx.y, b = blockIdx.z;
    const uint4 *x = reinterpret_cast<const uint4 *>(logits + ((size_t)b * R + row) * V);
    const int nvec = V / VN;
    const int v_lo = (int)(((long long)sp * nvec) / splits);
    const int v_hi = (int)(((long long)(sp + 1) * nvec) / splits);
    // This CTA's slice of the logits is pulled into L2 while the previous
    // kernel finishes: a prefetch stays inside the logits tensor and reads
    // nothing into the kernel, and L2 stays coherent with any writer, so it
    // may precede the wait.  Four threads split the slice.
    if (threadIdx.x < 4) {
        const int n = v_hi - v_lo;
        const int q0 = v_lo + (int)((long long)threadIdx.x * n / 4);
        const int q1 = v_lo + (int)((long long)(threadIdx.x + 1) * n / 4);
        if (q1 > q0) prefetch_l2_bulk(x + q0, (unsigned)(q1 - q0) * 16u);
    }
    pdl_enter();
    // argmax by 16-byte group: the running best group (its max, index and
    // raw words) moves only on a strictly larger group max, so the earliest
    // group holding the thread's max wins; its first element equal to that
    // max is the smallest id (a group of all -inf or NaN still enters first)
    float gbest = -INFINITY;
    int gidx = -1;
    uint4 graw = make_uint4(0u, 0u, 0u, 0u);
    Moments mo{-INFINITY, 0.f, 0.f};
    // two register buffers: the next batch's loads are in flight while this
    // batch is reduced
    uint4 cur[U], nxt[U];
    int base = v_lo + threadIdx.x;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int idx = base + u * kRowThreads;
        if (idx < v_hi) cur[u] = ld_stream16(x + idx);
    }
    for (; base < v_hi; base += kRowThreads * U) {
        const int nb = base + kRowThreads * U;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int idx = nb + u * kRowThreads;
            if (idx < v_hi) nxt[u] = ld_stream16(x + idx);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int idx = base + u * kRowThreads;
            if (idx < v_hi) {
                float f[VN];
                Vec16<T>::widen(cur[u], f);
                float vm = f[0];
#pragma unroll
                for (int e = 1; e < VN; ++e) vm = fmaxf(vm, f[e]);
                if (vm > gbest || gidx < 0) {
                    gbest = vm;
                    gidx = idx;
                    graw = cur[u];
                }
                if (TYPICAL) {
                    const float m_new = fmaxf(mo.m, vm * y_scale);
                    if (m_new > mo.m) {
                        if (mo.S != 0.f) {
                            const float f1 = exp2f(mo.m - m_new);
                            mo.A = f1 * (mo.A + mo.S * (mo.m - m_new));
                            mo.S *= f1;
                        }
                        mo.m = m_new;
                    }
#pragma unroll
                    for (int e = 0; e < VN; ++e) {
                        // clamped: a -inf logit adds 0 to both sums (0 * -inf
                        // would make A NaN); 2^-127 flushes to 0 all the same
                        const float t = fmaxf(fmaf(f[e], y_scale, -mo.m), -127.f);
                        const float p = ex2_approx(t);
                        mo.S += p;
                        mo.A = fmaf(p, t, mo.A);
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) cur[u] = nxt[u];
    }
    float bv = -INFINITY;
    int bi = INT_MAX;
    if (gidx >= 0) {
        float f[VN];
        Vec16<T>::widen(graw, f);
        int e0 = 0;  // no element equals a NaN group max: its first element
#pragma unroll
        for (int e = VN - 1; e >= 0; --e)
            if (f[e] == gbest) e0 = e;
        bv = f[e0];
        bi = gidx * VN + e0;
    }
    // warp reductions
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) {
            bv = ov;
            bi = oi;
        }
        if (TYPICAL) {
            const float om = __shfl_xor_sync(0xffffffffu, mo.m, o);
            const float oS = __shfl_xor_sync(0xffffffffu, mo.S, o);
            const float oA = __shfl_xor_sync(0xffffffffu, mo.A, o);
            mo.merge(om, oS, oA);
        }
    }
    if (lane == 0) {
        s_val[warp] = bv;
        s_id[warp] = bi;
        s_m[warp] = mo.m;
        s_S[warp] = mo.S;
        s_A[warp] = mo.A;
    }
    __syncthreads();
    if (warp == 0) {
        // the warps' states, merged by the first warp in three shuffle rounds
        constexpr int NW = kRowThreads / kWarp;
        static_assert(NW == 8, "merge rounds assume eight warps");
        const bool have = lane < NW;
        bv = have ? s_val[lane] : -INFINITY;
        bi = have ? s_id[lane] : INT_MAX;
        mo = Moments{have ? s_m[lane] : -INFINITY, have ? s_S[lane] : 0.f,
                     have ? s_A[lane] : 0.f};
#pragma unroll
        for (int o = NW / 2; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (better(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
            if (TYPICAL) {
                const float om = __shfl_xor_sync(0xffffffffu, mo.m, o);
                const float oS = __shfl_xor_sync(0xffffffffu, mo.S, o);
                const float oA = __shfl_xor_sync(0xffffffffu, mo.A, o);
                mo.merge(om, oS, oA);
            }
        }
    }
    if (threadIdx.x == 0) {
        RowPart pt;
        pt.amax = bv;
        pt.arg = bi;
        pt.m2 = mo.m;
        pt.S = mo.S;
        pt.A = mo.A;
        parts[((size_t)b * R + row) * splits + sp] = pt;
    }
}

// A row's slices, all loaded in one round (independent loads: the merge
// below would otherwise wait on each in turn).
struct RowSlices {
    RowPart p[kMaxSplits];
    __device__ __forceinline__ void load(const RowPart *__restrict__ parts, int splits) {
#pragma unroll
        for (int k = 0; k < kMaxSplits; ++k)
            if (k < splits) p[k] = parts[k];
    }
};

// Merge the slices of one row: argmax, and log2 S, H (nats) when typical.
__device__ __forceinline__ void row_stats(const RowSlices &rs, int splits, bool typical, int &arg,
                                          float &m2, float &log2s, float &H) {
    float bv = -INFINITY;
    int bi = INT_MAX;
    Moments mo{-INFINITY, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kMaxSplits; ++k) {
        if (k >= splits) break;
        const RowPart pt = rs.p[k];
        if (better(pt.amax, pt.arg, bv, bi)) {
            bv = pt.amax;
            bi = pt.arg;
        }
        if (typical) mo.merge(pt.m2, pt.S, pt.A);
    }
    arg = bi;
    m2 = mo.m;
    log2s = typical ? log2f(mo.S) : 0.f;
    H = typical ? logf(mo.S) - kLn2 * mo.A / mo.S : 0.f;
}

template <typename T>
__global__ void __launch_bounds__(kSelectThreads)
posterior_select_kernel(const T *__restrict__ logits, const int32_t *__restrict__ tokens,
                        const int32_t *__restrict__ parent, const int32_t *__restrict__ depth,
                        const RowPart *__restrict__ parts, int splits, int R, int V, int K,
                        int typical,
                        float y_scale, float log2_eps, float log2_delta,
                        int32_t *__restrict__ accept_len, int32_t *__restrict__ path,
                        int32_t *__restrict__ path_tokens, int32_t *__restrict__ next_token,
                        int32_t *__restrict__ accept_out, CommitArgs ca, int *status,
                        uint32_t *done) {
    const int b = blockIdx.x;
    const int i = threadIdx.x;
    // Completion word of this sequence (page-locked host memory of a step
    // executor, or null): each run of the step adds one once every result
    // of the CTA is written.  Its previous value was written by the previous
    // run's copy of this kernel, long complete, so it is read before the
    // launch wait.
    uint32_t seq = 0;
    if (done && i == 0) seq = *reinterpret_cast<volatile uint32_t *>(done + b) + 1u;
    // The one predecessor of this kernel that can still be running is the
    // rows kernel, and it writes only the row slices: the tree arrays and the
    // logits were complete before it passed its own launch wait, so they are
    // read before ours (the node's entries and, for typical acceptance, its
    // token's logit in its parent's row); the slices are read after it.
    int par = -1, dep = 0, tk = 0;
    float y_tok = 0.f;
    // the commit's cache pointers and prefix length (caller inputs as well)
    void *kc = nullptr, *vc = nullptr;
    int P = 0;
    if (ca.k_cache) {
        kc = ca.k_cache[b];
        vc = ca.v_cache[b];
        P = ca.prefix_len[b];
    }
    if (i < R) {
        const size_t o = (size_t)b * R + i;
        par = parent[o];
        dep = depth[o];
        tk = tokens[o];
        if (typical && i > 0 && par >= 0 && par < i && tk >= 0 && tk < V)
            y_tok = Vec16<T>::load1(logits + ((size_t)b * R + par) * V + tk);
    }
    pdl_enter();
    __shared__ int s_acc[MEDUSA_MAX_TREE_ROWS];
    __shared__ int s_chain[MEDUSA_MAX_TREE_ROWS];
    __shared__ int s_par[MEDUSA_MAX_TREE_ROWS];
    __shared__ int s_dep[MEDUSA_MAX_TREE_ROWS];
    __shared__ int s_tok[MEDUSA_MAX_TREE_ROWS];
    __shared__ int s_arg[MEDUSA_MAX_TREE_ROWS];  // argmax of each node's own row
    __shared__ int s_L, s_best;
    __shared__ int s_path[MEDUSA_MAX_HEADS + 1];
    __shared__ int s_code;
    if (i == 0) {
        s_L = 0;
        s_best = INT_MAX;
    }
    if (i < R) {
        s_par[i] = par;
        s_dep[i] = dep;
        s_tok[i] = tk;
        s_chain[i] = (i == 0);
        if (i == 0 && (dep != 0 || par != -1)) {
            set_status(status, MEDUSA_DEV_BAD_DEPTH);
            s_dep[0] = 0;
            s_par[0] = -1;
        }
    }
    // this node's own row (the next token if the path ends here) and its
    // parent's row: every slice of both in one round of loads
    RowSlices own, up;
    if (i < R) {
        own.load(parts + ((size_t)b * R + i) * splits, splits);
        if (i > 0 && par >= 0 && par < i) up.load(parts + ((size_t)b * R + par) * splits, splits);
    }
    __syncthreads();
    if (i < R) {
        {
            int arg;
            float m2, log2s, H;
            row_stats(own, splits, false, arg, m2, log2s, H);
            s_arg[i] = arg;
        }
        int acc = 1;
        if (i > 0) {
            const int p = s_par[i], tok = s_tok[i], D = s_dep[i];
            bool ok = true;
            if (p < 0 || p >= i) {
                set_status(status, MEDUSA_DEV_BAD_PARENT);
                ok = false;
            } else if (D < 1 || D > K || D != s_dep[p] + 1) {
                set_status(status, MEDUSA_DEV_BAD_DEPTH);
                ok = false;
            } else if (tok < 0 || tok >= V) {
                set_status(status, MEDUSA_DEV_BAD_TOKEN);
                ok = false;
            }
            if (!ok) {
                acc = 0;
            } else {
                int arg;
                float m2, log2s, H;
                row_stats(up, splits, typical, arg, m2, log2s, H);  // p == par here
                if (!typical) {
                    acc = (tok == arg);
                } else {
                    const float y = y_tok * y_scale;  // loaded before the launch wait
                    const float lp2 = y - m2 - log2s;
                    const float thr2 = fminf(log2_eps, log2_delta - H * kLog2e);
                    acc = lp2 > thr2;
                }
            }
        }
        s_acc[i] = acc;
        if (accept_out) accept_out[(size_t)b * R + i] = acc;
    }
    __syncthreads();
    for (int D = 1; D <= K; ++D) {
        if (i < R && i > 0 && s_dep[i] == D && s_acc[i]) {
            const int p = s_par[i];
            if (p >= 0 && p < i) s_chain[i] = s_chain[p];
        }
        __syncthreads();
    }
    if (i < R && s_chain[i]) atomicMax(&s_L, s_dep[i]);
    __syncthreads();
    if (i < R && s_chain[i] && s_dep[i] == s_L) atomicMin(&s_best, i);
    if (i <= K) {
        path[(size_t)b * (K + 1) + i] = -1;
        path_tokens[(size_t)b * (K + 1) + i] = -1;
        s_path[i] = -1;
    }
    __syncthreads();
    if (i == 0) {
        const int best = s_best < R ? s_best : 0;
        const int L = s_best < R ? s_L : 0;
        for (int x = best, q = L; x >= 0 && q >= 0; x = s_par[x], --q) {
            path[(size_t)b * (K + 1) + q] = x;
            path_tokens[(size_t)b * (K + 1) + q] = s_tok[x];
            s_path[q] = x;
            if (x == 0) break;
        }
        s_L = L;
        accept_len[b] = L;
        next_token[b] = s_arg[best];
    }
    if (ca.k_cache) {  // uniform over the CTA
        // commit of the accepted path into the KV cache (medusa_commit_kv)
        __syncthreads();
        if (i == 0) {
            s_code = commit_check(kc, vc, P, s_path, s_L, K, R);
            if (s_code != MEDUSA_DEV_OK) set_status(status, s_code);
            ca.new_prefix_len[b] = s_code == MEDUSA_DEV_OK ? P + s_L + 1 : P;
        }
        __syncthreads();
        if (s_code == MEDUSA_DEV_OK)
            commit_columns(kc, vc, P, s_path, s_L, ca.row_vecs, i, blockDim.x);
    }
    if (done) {  // uniform over the CTA
        // every thread's writes reach the system before the completion word
        __threadfence_system();
        __syncthreads();
        if (i == 0) *reinterpret_cast<volatile uint32_t *>(done + b) = seq;
    }
}

// Slices per logits row: enough CTAs for two per SM on 152 SMs, at most 8.
int row_splits(int B, int R) {
    const int rows = B * R;
    return std::max(1, std::min(kMaxSplits, (2 * 152 + rows - 1) / rows));
}

template <typename T>
cudaError_t run_posterior(const void *logits, const int32_t *tokens, const int32_t *parent,
                          const int32_t *depth, int B, int R, int V, int K, bool typical,
                          float eps, float delta, float temperature, int32_t *accept_len,
                          int32_t *path, int32_t *path_tokens, int32_t *next_token,
                          int32_t *accept, const CommitArgs &commit, void *ws,
                          cudaStream_t stream, uint32_t *done) {
    int *status = static_cast<int *>(ws);
    RowPart *parts = reinterpret_cast<RowPart *>(static_cast<char *>(ws) + MEDUSA_WS_HEADER);
    const T *lg = static_cast<const T *>(logits);
    const float y_scale = kLog2e / temperature;
    const int splits = row_splits(B, R);
    cudaError_t e = launch_pdl(typical ? posterior_rows_kernel<T, true> : posterior_rows_kernel<T, false>,
                               dim3(splits, R, B), dim3(kRowThreads), 0, stream, lg, R, V, splits,
                               y_scale, parts);
    note_launch();
    if (e) return e;
    e = launch_pdl(posterior_select_kernel<T>, dim3(B), dim3(kSelectThreads), 0, stream, lg, tokens,
                   parent, depth, static_cast<const RowPart *>(parts), splits, R, V, K,
                   typical ? 1 : 0, y_scale, log2f(eps), log2f(delta), accept_len, path,
                   path_tokens, next_token, accept, commit, status, done);
    note_launch();
    return e;
}

}  // namespace

size_t posterior_workspace_bytes(int B, int R) {
    return MEDUSA_WS_HEADER + (size_t)B * R * kMaxSplits * sizeof(RowPart);
}

cudaError_t launch_posterior(medusa_dtype dtype, const void *logits, const int32_t *tokens,
                             const int32_t *parent, const int32_t *depth, int B, int R, int V,
                             int K, medusa_accept_mode mode, float eps, float delta,
                             float temperature, int32_t *accept_len, int32_t *path,
                             int32_t *path_tokens, int32_t *next_token, int32_t *accept,
                             void *const *k_cache, void *const *v_cache,
                             const int32_t *prefix_len, int H, int dh, int32_t *new_prefix_len,
                             void *ws, cudaStream_t stream, uint32_t *done) {
    const bool typical = mode == MEDUSA_TYPICAL;
    const size_t elt = dtype == MEDUSA_BF16 ? 2 : 4;
    CommitArgs commit;
    commit.k_cache = k_cache;  // nullptr: no commit
    commit.v_cache = v_cache;
    commit.prefix_len = prefix_len;
    commit.new_prefix_len = new_prefix_len;
    commit.row_vecs = k_cache ? (int)((size_t)H * dh * elt / 16) : 0;
    if (dtype == MEDUSA_BF16)
        return run_posterior<bf16>(logits, tokens, parent, depth, B, R, V, K, typical, eps, delta,
                                   temperature, accept_len, path, path_tokens, next_token, accept,
                                   commit, ws, stream, done);
    return run_posterior<float>(logits, tokens, parent, depth, B, R, V, K, typical, eps, delta,
                                temperature, accept_len, path, path_tokens, next_token, accept,
                                commit, ws, stream, done);
}

}  // namespace medusa
