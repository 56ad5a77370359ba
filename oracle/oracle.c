/*
 * oracle.c -- plain, slow, float64 CPU oracle for one Medusa decoding step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; the two are compared element by element on the same seeded
 * inputs.
 *
 * Every function states the passage it follows.  Pages cited:
 *   [P1] "Medusa: Faster LLM text generation" (nazmi.tech): sections
 *        "Inference / Proposals and a tree", "Tree attention",
 *        "Acceptance rules".
 *   [P2] "Medusa 深读" (jokeuncle.pages.dev): §3.1 (Medusa head, eq. for
 *        p_t^(k), initialisation), §5 (typical acceptance rule and the
 *        unconditional first token), §6.1 (Cartesian tree, node count, tree
 *        mask, shared position index), §6.2 (greedy sparse tree under a
 *        budget, worked example).
 *        Also [P1] "Acceptance rules" (exact speculative decoding) and
 *        [P2] §3's remark on recovering the target distribution.
 *   [P3] "Medusa Part I" (sudhirpol522.github.io): Part 2 (greedy
 *        verification stops at the first mismatch; progress guarantee),
 *        Part 3 (ResidualBlock: hidden + SiLU(Linear(hidden)), vocab
 *        projection without bias).
 *
 * Arithmetic is IEEE double throughout.  Inputs are float32 arrays or bf16
 * bit patterns (uint16); each element is widened on read, never copied out
 * as a whole.  Build with -ffp-contract=off so that x86 and Arm give the same
 * bits.
 *
 * The file is compiled twice.  liboracle.so is the serial build every parity
 * test uses.  liboracle_omp.so is the same source with -fopenmp, used only to
 * time the CPU baseline on all host cores: the `omp parallel for` pragmas
 * below spread independent output elements (heads' rows, attention heads,
 * posterior nodes) over threads, and each element is still computed by the
 * same sequential loop, so both builds give the same bits.  Without -fopenmp
 * the pragmas are ignored.
 *
 * Parity status of each function (pins live in tests/test_oracle_pins.py):
 *   oracle_heads              pinned (identity-initialised heads reproduce
 *                             the LM-head softmax; numpy float64 matmul +
 *                             closed-form softmax on tiny sizes)
 *   oracle_lm_head            pinned (equals oracle_heads with W1 = 0, b1 = 0,
 *                             W2 = W_lm; hand-built one-hot rows give
 *                             closed-form logits and log Z)
 *   oracle_build_tree         pinned (worked example of [P2] §6.2; node-count
 *                             closed form of [P2] §6.1; brute-force optimality)
 *   oracle_tree_attention     pinned (per-path causal attention via torch
 *                             float64 scaled_dot_product_attention; chain tree)
 *   oracle_posterior          pinned (first-mismatch stop, progress guarantee,
 *                             closed-form typical thresholds, uniform-row
 *                             entropy = ln V)
 *   oracle_softmax_entropy    pinned (uniform row, two-point distribution)
 *   oracle_commit_kv          pinned (hand-built gathers in the tests)
 *   oracle_philox4x64         pinned (numpy's Philox4x64-10 bit generator)
 *   oracle_draft_sample       pinned (Gumbel-max frequencies against the
 *                             closed-form softmax, chi-square)
 *   oracle_speculative_posterior pinned (emitted-token frequencies equal p;
 *                             acceptance rate = sum_v min(p, q); q = p
 *                             accepts every draft)
 * The choice among exactly tied alternatives (equal logits, equal path
 * scores) is fixed by a stated convention, not by the pages.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads the parallel loops use (1 in the serial build). */
int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_GREEDY = 0, ORC_TYPICAL = 1 };

#define ORC_MAX_DEPTH 8

/* Read element i of an array stored as float32 or as bf16 bits, as double.
 * bf16 is the upper half of an IEEE binary32, so widening is a shift. */
static double rd(int dtype, const void *p, size_t i)
{
    if (dtype == ORC_F32)
        return (double)((const float *)p)[i];
    uint32_t bits = ((uint32_t)((const uint16_t *)p)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* O1. Medusa heads.                                                          */
/*                                                                            */
/* [P2] §3.1: p^(k) = softmax(W2^(k) (SiLU(W1^(k) h) + h)), W1 in R^{d x d},  */
/* W2 in R^{V x d}.  [P3] Part 3 ResidualBlock adds a bias b1 inside SiLU and */
/* the vocab projection has no bias.  SiLU(u) = u * sigmoid(u).               */
/* Each head keeps its top-s tokens ([P2] §6.1).  Ranking: larger logit      */
/* first; equal logits -> smaller token id first (convention).               */
/*                                                                            */
/* h [B][d], W1 [K][d][d] (row = output unit), b1 [K][d] or NULL,            */
/* W2 [K][V][d].  Outputs topk_ids/topk_logp [B][K][s]; optional             */
/* logits_out [B][K][V] and logz_out [B][K] for gap checks.                  */
/* ------------------------------------------------------------------------ */
int oracle_heads(int dtype, const void *h, const void *W1, const void *b1,
                 const void *W2, int B, int d, int V, int K, int s,
                 int32_t *topk_ids, double *topk_logp, double *logits_out,
                 double *logz_out)
{
    if (B < 1 || d < 1 || V < 1 || K < 1 || s < 1 || s > V)
        return 1;
    double *z = (double *)malloc((size_t)d * sizeof(double));
    double *lg = (double *)malloc((size_t)V * sizeof(double));
    char *taken = (char *)malloc((size_t)V);
    if (!z || !lg || !taken) {
        free(z); free(lg); free(taken);
        return 2;
    }
    for (int b = 0; b < B; ++b) {
        for (int k = 0; k < K; ++k) {
            /* residual block: z = h + SiLU(W1 h + b1) */
#pragma omp parallel for schedule(static)
            for (int j = 0; j < d; ++j) {
                double u = 0.0;
                for (int c = 0; c < d; ++c)
                    u += rd(dtype, W1, ((size_t)k * d + j) * d + c) *
                         rd(dtype, h, (size_t)b * d + c);
                if (b1)
                    u += rd(dtype, b1, (size_t)k * d + j);
                double silu = u / (1.0 + exp(-u));
                z[j] = rd(dtype, h, (size_t)b * d + j) + silu;
            }
            /* vocabulary projection: logits = W2 z */
#pragma omp parallel for schedule(static)
            for (int v = 0; v < V; ++v) {
                double acc = 0.0;
                for (int c = 0; c < d; ++c)
                    acc += rd(dtype, W2, ((size_t)k * V + v) * d + c) * z[c];
                lg[v] = acc;
            }
            /* log of the softmax normaliser: log sum_v exp(logit_v) */
            double m = lg[0];
            for (int v = 1; v < V; ++v)
                if (lg[v] > m) m = lg[v];
            double S = 0.0;
            for (int v = 0; v < V; ++v)
                S += exp(lg[v] - m);
            double logz = m + log(S);
            /* top-s by repeated selection of the best remaining token */
            memset(taken, 0, (size_t)V);
            for (int r = 0; r < s; ++r) {
                int best = -1;
                for (int v = 0; v < V; ++v) {
                    if (taken[v]) continue;
                    if (best < 0 || lg[v] > lg[best]) best = v;
                }
                taken[best] = 1;
                size_t o = ((size_t)b * K + k) * s + r;
                topk_ids[o] = best;
                topk_logp[o] = lg[best] - logz;
            }
            if (logits_out)
                memcpy(logits_out + ((size_t)b * K + k) * V, lg,
                       (size_t)V * sizeof(double));
            if (logz_out)
                logz_out[(size_t)b * K + k] = logz;
        }
    }
    free(z); free(lg); free(taken);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* O1'. The base model's LM head on the same hidden state.                   */
/*                                                                            */
/* [P1] Introduction and [P3] (the heads and the LM head read one final      */
/* hidden state h): logits = W_lm h, no residual block, no bias.  [P2] §5:   */
/* the LM head's greedy token is the root of the candidate tree, accepted    */
/* unconditionally.  Outputs, per sequence: the top-s tokens (larger logit   */
/* first, equal logits -> smaller id first), their log-probabilities under   */
/* softmax(logits); entry 0 is the greedy root token.                        */
/*                                                                            */
/* h [B][d], W_lm [V][d].  topk_ids/topk_logp [B][s]; optional logits_out    */
/* [B][V] and logz_out [B].                                                  */
/* ------------------------------------------------------------------------ */
int oracle_lm_head(int dtype, const void *h, const void *W_lm, int B, int d,
                   int V, int s, int32_t *topk_ids, double *topk_logp,
                   double *logits_out, double *logz_out)
{
    if (B < 1 || d < 1 || V < 1 || s < 1 || s > V)
        return 1;
    double *lg = (double *)malloc((size_t)V * sizeof(double));
    char *taken = (char *)malloc((size_t)V);
    if (!lg || !taken) {
        free(lg); free(taken);
        return 2;
    }
    for (int b = 0; b < B; ++b) {
#pragma omp parallel for schedule(static)
        for (int v = 0; v < V; ++v) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += rd(dtype, W_lm, (size_t)v * d + c) * rd(dtype, h, (size_t)b * d + c);
            lg[v] = acc;
        }
        double m = lg[0];
        for (int v = 1; v < V; ++v)
            if (lg[v] > m) m = lg[v];
        double S = 0.0;
        for (int v = 0; v < V; ++v)
            S += exp(lg[v] - m);
        double logz = m + log(S);
        memset(taken, 0, (size_t)V);
        for (int r = 0; r < s; ++r) {
            int best = -1;
            for (int v = 0; v < V; ++v) {
                if (taken[v]) continue;
                if (best < 0 || lg[v] > lg[best]) best = v;
            }
            taken[best] = 1;
            topk_ids[(size_t)b * s + r] = best;
            topk_logp[(size_t)b * s + r] = lg[best] - logz;
        }
        if (logits_out)
            memcpy(logits_out + (size_t)b * V, lg, (size_t)V * sizeof(double));
        if (logz_out)
            logz_out[b] = logz;
    }
    free(lg); free(taken);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* O2. Candidate tree, built greedily under a node budget.                   */
/*                                                                            */
/* [P2] §6.2: a node is a rank path (i_1..i_k); its weight is the product of */
/* per-level weights; starting from the children of the root, repeatedly     */
/* take the frontier node of largest weight into the tree and add its        */
/* children to the frontier, n times.  Here the per-level weights are the    */
/* heads' own probabilities, passed as log-probabilities, so the path score  */
/* is the sum of the log-probabilities along the path, summed from depth 1   */
/* downward.  [P2] §6.1: a node sees the root and its own ancestors; all     */
/* nodes of one depth share one position index.                             */
/*                                                                            */
/* Conventions (the pages are silent): score ties go to the smaller depth,   */
/* then to the lexicographically smaller rank path.  Output order is         */
/* canonical: root first, then by depth, then by rank path (so parent index  */
/* < child index and every depth is one contiguous block).                   */
/*                                                                            */
/* logp[b][k][r] with row stride s_stride, r < s[k].  Outputs per sequence:  */
/* R = n + 1 rows: tokens, parent (-1 at root), depth, pos_id = P_b + depth, */
/* anc_mask [R][W] (W = ceil(R/64)), paths [n][K+1] (-1 padded), n_leaf,     */
/* and cut_gap = (score of the n-th pick) - (best score left in the          */
/* frontier), +inf when the frontier is empty.                               */
/* ------------------------------------------------------------------------ */
typedef struct {
    int depth;
    int rank[ORC_MAX_DEPTH];
    double score;
} orc_node;

/* 1 if a is taken before b */
static int orc_before(const orc_node *a, const orc_node *b)
{
    if (a->score != b->score) return a->score > b->score;
    if (a->depth != b->depth) return a->depth < b->depth;
    for (int j = 0; j < a->depth; ++j)
        if (a->rank[j] != b->rank[j]) return a->rank[j] < b->rank[j];
    return 0;
}

/* canonical order: depth, then rank path */
static int orc_canon_less(const orc_node *a, const orc_node *b)
{
    if (a->depth != b->depth) return a->depth < b->depth;
    for (int j = 0; j < a->depth; ++j)
        if (a->rank[j] != b->rank[j]) return a->rank[j] < b->rank[j];
    return 0;
}

int oracle_build_tree(const int32_t *root, const int32_t *topk_ids,
                      const double *topk_logp, int B, int K, const int32_t *s,
                      int s_stride, int n, const int32_t *prefix_len,
                      int32_t *tokens, int32_t *parent, int32_t *depth,
                      int32_t *pos_id, uint64_t *anc_mask, int32_t *paths,
                      int32_t *n_leaf, double *cut_gap)
{
    if (B < 1 || K < 1 || K > ORC_MAX_DEPTH || n < 1)
        return 1;
    long total = 0, level = 1;
    for (int k = 0; k < K; ++k) {
        if (s[k] < 1 || s[k] > s_stride) return 1;
        level *= s[k];
        total += level;
        if (total > 1000000) break;
    }
    if (n > total) return 1;
    const int R = n + 1;
    const int W = (R + 63) / 64;
    /* frontier never holds more than every child of every pick plus s_1 */
    const long cap = (long)s[0] + (long)n * s_stride;
    orc_node *front = (orc_node *)malloc((size_t)cap * sizeof(orc_node));
    orc_node *sel = (orc_node *)malloc((size_t)n * sizeof(orc_node));
    int *par = (int *)malloc((size_t)R * sizeof(int));
    char *has_child = (char *)malloc((size_t)R);
    if (!front || !sel || !par || !has_child) {
        free(front); free(sel); free(par); free(has_child);
        return 2;
    }
    for (int b = 0; b < B; ++b) {
        const int32_t *ids_b = topk_ids + (size_t)b * K * s_stride;
        const double *lp_b = topk_logp + (size_t)b * K * s_stride;
        long nf = 0;
        for (int r = 0; r < s[0]; ++r) {
            orc_node c;
            memset(&c, 0, sizeof c);
            c.depth = 1;
            c.rank[0] = r;
            c.score = lp_b[r];
            front[nf++] = c;
        }
        for (int t = 0; t < n; ++t) {
            long best = 0;
            for (long f = 1; f < nf; ++f)
                if (orc_before(&front[f], &front[best])) best = f;
            orc_node pick = front[best];
            front[best] = front[--nf];
            sel[t] = pick;
            if (pick.depth < K) {
                for (int c = 0; c < s[pick.depth]; ++c) {
                    orc_node ch = pick;
                    ch.depth = pick.depth + 1;
                    ch.rank[pick.depth] = c;
                    ch.score = pick.score + lp_b[(size_t)pick.depth * s_stride + c];
                    front[nf++] = ch;
                }
            }
        }
        if (cut_gap) {
            if (nf == 0) {
                cut_gap[b] = INFINITY;
            } else {
                long best = 0;
                for (long f = 1; f < nf; ++f)
                    if (orc_before(&front[f], &front[best])) best = f;
                cut_gap[b] = sel[n - 1].score - front[best].score;
            }
        }
        /* canonical order (insertion sort; n is small) */
        for (int i = 1; i < n; ++i) {
            orc_node x = sel[i];
            int j = i - 1;
            while (j >= 0 && orc_canon_less(&x, &sel[j])) {
                sel[j + 1] = sel[j];
                --j;
            }
            sel[j + 1] = x;
        }
        int32_t *tok = tokens + (size_t)b * R;
        int32_t *pa = parent + (size_t)b * R;
        int32_t *de = depth + (size_t)b * R;
        int32_t *po = pos_id + (size_t)b * R;
        uint64_t *am = anc_mask + (size_t)b * R * W;
        const int P = prefix_len ? prefix_len[b] : 0;
        tok[0] = root[b];
        par[0] = -1;
        de[0] = 0;
        for (int i = 0; i < n; ++i) {
            const orc_node *x = &sel[i];
            tok[i + 1] = ids_b[(size_t)(x->depth - 1) * s_stride + x->rank[x->depth - 1]];
            de[i + 1] = x->depth;
            int p = 0;
            if (x->depth > 1) {
                p = -1;
                for (int j = 0; j < n; ++j) {
                    if (sel[j].depth != x->depth - 1) continue;
                    int same = 1;
                    for (int q = 0; q < x->depth - 1; ++q)
                        if (sel[j].rank[q] != x->rank[q]) { same = 0; break; }
                    if (same) { p = j + 1; break; }
                }
                if (p < 0) {   /* impossible for a greedy frontier tree */
                    free(front); free(sel); free(par); free(has_child);
                    return 3;
                }
            }
            par[i + 1] = p;
        }
        for (int i = 0; i < R; ++i) {
            pa[i] = par[i];
            po[i] = P + de[i];
            for (int w = 0; w < W; ++w)
                am[(size_t)i * W + w] = 0;
            for (int a = i; a >= 0; a = par[a])
                am[(size_t)i * W + a / 64] |= (uint64_t)1 << (a % 64);
        }
        memset(has_child, 0, (size_t)R);
        for (int i = 1; i < R; ++i)
            has_child[par[i]] = 1;
        int32_t *pt = paths + (size_t)b * n * (K + 1);
        for (size_t e = 0; e < (size_t)n * (K + 1); ++e)
            pt[e] = -1;
        int nl = 0;
        for (int i = 0; i < R; ++i) {
            if (has_child[i]) continue;
            int chain[ORC_MAX_DEPTH + 1];
            int len = 0;
            for (int a = i; a >= 0; a = par[a])
                chain[len++] = a;
            for (int q = 0; q < len; ++q)
                pt[(size_t)nl * (K + 1) + q] = chain[len - 1 - q];
            ++nl;
        }
        n_leaf[b] = nl;
    }
    free(front); free(sel); free(par); free(has_child);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* O3. Tree attention, direct definition.                                    */
/*                                                                            */
/* [P1] "Tree attention" and [P2] §6.1: every tree node attends to the whole */
/* prefix and to its own branch ancestors (itself included), never to other */
/* branches.  Cache slots 0..P_b-1 hold the prefix, slots P_b..P_b+R-1 hold  */
/* the tree nodes in canonical order.  Scores are scale * q.k, softmax over  */
/* the visible slots, output = sum of probabilities times values.            */
/*                                                                            */
/* q [B][R][H][dh]; k_cache[b], v_cache[b] each [P_b+R][H][dh]; anc_mask     */
/* [B][R][W]; out [B][R][H][dh] in double.                                   */
/* ------------------------------------------------------------------------ */
int oracle_tree_attention(int dtype, const void *q, const void *const *k_cache,
                          const void *const *v_cache, const int32_t *prefix_len,
                          const uint64_t *anc_mask, int B, int R, int H, int dh,
                          double scale, double *out)
{
    if (B < 1 || R < 1 || H < 1 || dh < 1)
        return 1;
    const int W = (R + 63) / 64;
    int maxslots = 0;
    for (int b = 0; b < B; ++b)
        if (prefix_len[b] + R > maxslots) maxslots = prefix_len[b] + R;
    /* one score row per attention head, so that heads are independent */
    double *sc_all = (double *)malloc((size_t)H * maxslots * sizeof(double));
    char *vis = (char *)malloc((size_t)maxslots);
    if (!sc_all || !vis) { free(sc_all); free(vis); return 2; }
    for (int b = 0; b < B; ++b) {
        const int P = prefix_len[b];
        const int nslot = P + R;
        for (int i = 0; i < R; ++i) {
            const uint64_t *row = anc_mask + ((size_t)b * R + i) * W;
            for (int j = 0; j < nslot; ++j) {
                if (j < P) {
                    vis[j] = 1;
                } else {
                    int t = j - P;
                    vis[j] = (char)((row[t / 64] >> (t % 64)) & 1u);
                }
            }
#pragma omp parallel for schedule(static)
            for (int hh = 0; hh < H; ++hh) {
                double *sc = sc_all + (size_t)hh * maxslots;
                size_t qo = (((size_t)b * R + i) * H + hh) * dh;
                double m = -INFINITY;
                for (int j = 0; j < nslot; ++j) {
                    if (!vis[j]) continue;
                    size_t ko = ((size_t)j * H + hh) * dh;
                    double dot = 0.0;
                    for (int c = 0; c < dh; ++c)
                        dot += rd(dtype, q, qo + c) * rd(dtype, k_cache[b], ko + c);
                    sc[j] = scale * dot;
                    if (sc[j] > m) m = sc[j];
                }
                double L = 0.0;
                for (int j = 0; j < nslot; ++j)
                    if (vis[j]) {
                        sc[j] = exp(sc[j] - m);
                        L += sc[j];
                    }
                for (int c = 0; c < dh; ++c) {
                    double acc = 0.0;
                    for (int j = 0; j < nslot; ++j)
                        if (vis[j])
                            acc += sc[j] * rd(dtype, v_cache[b], ((size_t)j * H + hh) * dh + c);
                    out[qo + c] = acc / L;
                }
            }
        }
    }
    free(sc_all); free(vis);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Entropy of softmax(x / T), natural log: H(p) = -sum_x p(x) log p(x)       */
/* ([P2] §5).  Also used by the tests to set logits temperatures.            */
/* ------------------------------------------------------------------------ */
double oracle_softmax_entropy(const double *x, int V, double T)
{
    double m = -INFINITY;
    for (int v = 0; v < V; ++v)
        if (x[v] / T > m) m = x[v] / T;
    double S = 0.0;
    for (int v = 0; v < V; ++v)
        S += exp(x[v] / T - m);
    double Hn = 0.0;
    for (int v = 0; v < V; ++v) {
        double p = exp(x[v] / T - m) / S;
        if (p > 0.0)
            Hn -= p * log(p);
    }
    return Hn;
}

/* ------------------------------------------------------------------------ */
/* O4. Posterior: acceptance and the longest accepted path.                  */
/*                                                                            */
/* A node's token is judged by the verification logits of its parent row:   */
/* row p holds the target model's distribution for the token after node p.   */
/*   greedy  ([P3] Part 2): accept iff the token is the argmax of the row.   */
/*   typical ([P2] §5): accept iff p(x) > min(eps, delta * exp(-H(p))),      */
/*           p = softmax(logits / T), H natural-log entropy.                 */
/* The root (the LM head's greedy token) is accepted unconditionally         */
/* ([P2] §5).  A node counts only if every ancestor is accepted (a           */
/* rejection ends the prefix, [P3] Part 2).  The committed path is the       */
/* longest such chain ([P2] §5 "longest fully accepted prefix"); among equal */
/* depths the smallest canonical index wins (convention).  next_token is the */
/* argmax of the best node's row (the next greedy token; at least one token  */
/* is always produced, [P3] Part 2).  Argmax ties -> smallest token id.      */
/*                                                                            */
/* logits [B][R][V]; tokens/parent/depth [B][R], parent[i] < i for i > 0.    */
/* Outputs accept_len [B], path/path_tokens [B][K+1] (-1 padded),            */
/* next_token [B]; optional accept [B][R] (per-node decision, root = 1) and  */
/* margin [B][R] (log p - log threshold for typical, +inf otherwise).        */
/* If forced_accept is non-NULL, its per-node decisions replace the computed */
/* ones (used to re-run the path choice on another implementation's flags). */
/* ------------------------------------------------------------------------ */
static int orc_argmax_row(int dtype, const void *logits, size_t off, int V)
{
    int best = 0;
    double bv = rd(dtype, logits, off);
    for (int v = 1; v < V; ++v) {
        double x = rd(dtype, logits, off + v);
        if (x > bv) { bv = x; best = v; }
    }
    return best;
}

int oracle_posterior(int dtype, const void *logits, const int32_t *tokens,
                     const int32_t *parent, const int32_t *depth, int B, int R,
                     int V, int K, int mode, double eps, double delta, double T,
                     const int32_t *forced_accept, int32_t *accept_len,
                     int32_t *path, int32_t *path_tokens, int32_t *next_token,
                     int32_t *accept, double *margin)
{
    if (B < 1 || R < 1 || V < 1 || K < 0 || !(T > 0.0))
        return 1;
    for (size_t i = 0; i < (size_t)B * R; ++i) {
        if (i % R == 0) continue;
        const int p = parent[i];
        if (p < 0 || p >= (int)(i % R) || tokens[i] < 0 || tokens[i] >= V)
            return 3;
    }
    /* one widened row per node, so that nodes are independent */
    double *x_all = (double *)malloc((size_t)R * V * sizeof(double));
    int *acc = (int *)malloc((size_t)R * sizeof(int));
    int *chain = (int *)malloc((size_t)R * sizeof(int));
    if (!x_all || !acc || !chain) { free(x_all); free(acc); free(chain); return 2; }
    for (int b = 0; b < B; ++b) {
        const int32_t *tok = tokens + (size_t)b * R;
        const int32_t *pa = parent + (size_t)b * R;
        const int32_t *de = depth + (size_t)b * R;
        acc[0] = 1;
        if (margin) margin[(size_t)b * R] = INFINITY;
#pragma omp parallel for schedule(dynamic, 1)
        for (int i = 1; i < R; ++i) {
            const int p = pa[i];
            double *x = x_all + (size_t)i * V;
            size_t off = ((size_t)b * R + p) * V;
            double mg = INFINITY;
            if (mode == ORC_GREEDY) {
                acc[i] = (orc_argmax_row(dtype, logits, off, V) == tok[i]);
            } else {
                for (int v = 0; v < V; ++v)
                    x[v] = rd(dtype, logits, off + v);
                double Hn = oracle_softmax_entropy(x, V, T);
                double m = -INFINITY;
                for (int v = 0; v < V; ++v)
                    if (x[v] / T > m) m = x[v] / T;
                double S = 0.0;
                for (int v = 0; v < V; ++v)
                    S += exp(x[v] / T - m);
                double ptok = exp(x[tok[i]] / T - m) / S;
                double e_thr = delta * exp(-Hn);
                double thr = eps < e_thr ? eps : e_thr;
                acc[i] = ptok > thr;
                mg = log(ptok) - log(thr);
            }
            if (forced_accept)
                acc[i] = forced_accept[(size_t)b * R + i] != 0;
            if (margin) margin[(size_t)b * R + i] = mg;
        }
        if (accept)
            for (int i = 0; i < R; ++i)
                accept[(size_t)b * R + i] = acc[i];
        /* prefix-AND along each branch (parent index < child index) */
        chain[0] = 1;
        for (int i = 1; i < R; ++i)
            chain[i] = acc[i] && chain[pa[i]];
        int L = 0, best = 0;
        for (int i = 1; i < R; ++i)
            if (chain[i] && de[i] > L) { L = de[i]; best = i; }
        int32_t *pth = path + (size_t)b * (K + 1);
        int32_t *ptk = path_tokens + (size_t)b * (K + 1);
        for (int q = 0; q <= K; ++q) { pth[q] = -1; ptk[q] = -1; }
        for (int a = best; a >= 0; a = pa[a]) {
            pth[de[a]] = a;
            ptk[de[a]] = tok[a];
        }
        accept_len[b] = L;
        next_token[b] = orc_argmax_row(dtype, logits, ((size_t)b * R + best) * V, V);
    }
    free(x_all); free(acc); free(chain);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Commit of the accepted path into the KV cache.                            */
/*                                                                            */
/* [P1] Introduction: the accepted prefix becomes the next context; [P2] §5: */
/* the longest fully accepted prefix is committed.  The cache of sequence b  */
/* holds the tree nodes in slots P_b .. P_b+R-1 (canonical order).  The      */
/* accepted path root -> best has accept_len+1 nodes; slot P_b + q receives  */
/* the K/V of path node q (q = 0 .. accept_len), and the new prefix length   */
/* is P_b + accept_len + 1.  Rows are copied as raw bytes.                   */
/* cache[b] has rows of row_bytes bytes (H * dh * element size).             */
/* ------------------------------------------------------------------------ */
int oracle_commit_kv(void *const *k_cache, void *const *v_cache,
                     const int32_t *prefix_len, const int32_t *path,
                     const int32_t *accept_len, int B, int K, size_t row_bytes,
                     int32_t *new_prefix_len)
{
    unsigned char *tmp = (unsigned char *)malloc(row_bytes * (size_t)(K + 1) * 2);
    if (!tmp) return 2;
    for (int b = 0; b < B; ++b) {
        const int P = prefix_len[b];
        const int L = accept_len[b];
        const int32_t *pth = path + (size_t)b * (K + 1);
        /* read every source row before writing (sources and targets overlap) */
        for (int q = 0; q <= L; ++q) {
            size_t src = (size_t)(P + pth[q]) * row_bytes;
            memcpy(tmp + (size_t)q * row_bytes, (unsigned char *)k_cache[b] + src, row_bytes);
            memcpy(tmp + (size_t)(K + 1 + q) * row_bytes, (unsigned char *)v_cache[b] + src, row_bytes);
        }
        for (int q = 0; q <= L; ++q) {
            size_t dst = (size_t)(P + q) * row_bytes;
            memcpy((unsigned char *)k_cache[b] + dst, tmp + (size_t)q * row_bytes, row_bytes);
            memcpy((unsigned char *)v_cache[b] + dst, tmp + (size_t)(K + 1 + q) * row_bytes, row_bytes);
        }
        new_prefix_len[b] = P + L + 1;
    }
    free(tmp);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* O5. Exact speculative sampling on a chain of sampled drafts.               */
/*                                                                            */
/* [P1] Acceptance rules and [P2] §3 (the remark on lossless recovery) and   */
/* §5: drafts are sampled from the heads' own normalised distributions q_k;  */
/* each is accepted with probability min(1, p/q) under the verifying model's */
/* p; at the first rejection a replacement is sampled from the normalised    */
/* positive residual max(0, p - q); if every draft is accepted, one more     */
/* token is sampled from p at the last row.  This preserves p exactly.       */
/*                                                                            */
/* Readings (the pages leave these open): q_k = softmax(head logits / T) and */
/* p = softmax(verification logits / T) with one temperature T; the drafts   */
/* form a chain x_1..x_K, x_k from head k independently (the heads do not see */
/* each other's drafts, [P2] §3); the root x_0 is given and accepted.         */
/* Sampling from weights w_v uses the Gumbel-max rule: the token with the    */
/* largest log w_v + G_v, G_v = -log(-log u_v), smaller id on exact ties.   */
/*                                                                            */
/* Random numbers: Philox4x64-10 (Salmon, Moraes, Dror and Shaw, "Parallel   */
/* random numbers: as easy as 1, 2, 3", SC 2011), counter = (v / 4, row, b,  */
/* purpose), key = (seed, step); the uniform for index v is word v % 4 of    */
/* the output, as ((w >> 41) + 0.5) * 2^-23 (24 significant bits, exactly   */
/* representable in float32, never 0 or 1).                                  */
/* ------------------------------------------------------------------------ */
enum { ORC_RNG_DRAFT = 1, ORC_RNG_ACCEPT = 2, ORC_RNG_RESAMPLE = 3 };

/* 64 x 64 -> 128-bit product from 32-bit halves */
static void orc_mulhilo64(uint64_t a, uint64_t b, uint64_t *hi, uint64_t *lo)
{
    uint64_t a0 = a & 0xffffffffu, a1 = a >> 32, b0 = b & 0xffffffffu, b1 = b >> 32;
    uint64_t p00 = a0 * b0, p01 = a0 * b1, p10 = a1 * b0, p11 = a1 * b1;
    uint64_t mid = (p00 >> 32) + (p01 & 0xffffffffu) + (p10 & 0xffffffffu);
    *lo = (mid << 32) | (p00 & 0xffffffffu);
    *hi = p11 + (p01 >> 32) + (p10 >> 32) + (mid >> 32);
}

void oracle_philox4x64(const uint64_t *ctr, const uint64_t *key, uint64_t *out)
{
    uint64_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B97F4A7C15ull;   /* Weyl increments of the key */
            k1 += 0xBB67AE8584CAA73Bull;
        }
        uint64_t hi0, lo0, hi1, lo1;
        orc_mulhilo64(0xD2E7470EE14C6C93ull, x0, &hi0, &lo0);
        orc_mulhilo64(0xCA5A826395121157ull, x2, &hi1, &lo1);
        uint64_t y0 = hi1 ^ x1 ^ k0, y1 = lo1, y2 = hi0 ^ x3 ^ k1, y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

double oracle_uniform(uint64_t seed, uint64_t step, int purpose, int b, int row, int v)
{
    uint64_t ctr[4] = {(uint64_t)v >> 2, (uint64_t)row, (uint64_t)b, (uint64_t)purpose};
    uint64_t key[2] = {seed, step}, out[4];
    oracle_philox4x64(ctr, key, out);
    return ((double)(out[v & 3] >> 41) + 0.5) * (1.0 / 8388608.0);
}

static double orc_gumbel(uint64_t seed, uint64_t step, int purpose, int b, int row, int v)
{
    return -log(-log(oracle_uniform(seed, step, purpose, b, row, v)));
}

/* log of the softmax normaliser of x/T over a row */
static double orc_logz_row(int dtype, const void *x, size_t off, int V, double T)
{
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double t = rd(dtype, x, off + v) / T;
        if (t > m) m = t;
    }
    double S = 0.0;
    for (int v = 0; v < V; ++v)
        S += exp(rd(dtype, x, off + v) / T - m);
    return m + log(S);
}

/* Draft sampling: x_k ~ softmax(logits_k / T) for every (sequence, head) by  */
/* Gumbel-max on the heads' logits (computed by oracle_heads).  Optional     */
/* outputs: the logits [B][K][V] and the Gumbel keys [B][K][V].              */
int oracle_draft_sample(int dtype, const void *h, const void *W1, const void *b1,
                        const void *W2, int B, int d, int V, int K, double T,
                        uint64_t seed, uint64_t step, int32_t *drafts,
                        double *logits_out, double *keys_out)
{
    if (!(T > 0.0)) return 1;
    double *lg = (double *)malloc((size_t)B * K * V * sizeof(double));
    int32_t *ids = (int32_t *)malloc((size_t)B * K * sizeof(int32_t));
    double *lp = (double *)malloc((size_t)B * K * sizeof(double));
    double *lz = (double *)malloc((size_t)B * K * sizeof(double));
    if (!lg || !ids || !lp || !lz) {
        free(lg); free(ids); free(lp); free(lz);
        return 2;
    }
    int rc = oracle_heads(dtype, h, W1, b1, W2, B, d, V, K, 1, ids, lp, lg, lz);
    if (rc == 0) {
        for (int b = 0; b < B; ++b)
            for (int k = 0; k < K; ++k) {
                const double *row = lg + ((size_t)b * K + k) * V;
                int best = -1;
                double bk = -INFINITY;
                for (int v = 0; v < V; ++v) {
                    double key = row[v] / T + orc_gumbel(seed, step, ORC_RNG_DRAFT, b, k, v);
                    if (keys_out) keys_out[((size_t)b * K + k) * V + v] = key;
                    if (best < 0 || key > bk) { best = v; bk = key; }
                }
                drafts[(size_t)b * K + k] = best;
            }
        if (logits_out) memcpy(logits_out, lg, (size_t)B * K * V * sizeof(double));
    }
    free(lg); free(ids); free(lp); free(lz);
    return rc;
}

/* Verification of the chain.  logits [B][K+1][V] (row j: the verifying      */
/* model's distribution of the token after x_j), tokens [B][K+1] (x_0 root,  */
/* x_1..x_K drafts), draft_logits [B][K][V] float32 (head k's logits, the    */
/* numerators of q_k).  Outputs accept_len [B], path_tokens [B][K+1] (x_0..  */
/* x_L, -1 padded), next_token [B] (the replacement, or the bonus token),   */
/* accept [B][K] (1 accepted, 0 rejected, -1 not reached), margin [B][K]     */
/* (log p - log q - log u; accepted iff > 0), sample_row [B] (the row the    */
/* next token was drawn from) and sample_keys [B][V] (its Gumbel keys, -inf  */
/* where the weight is 0).  forced_accept [B][K] (or NULL) replaces the       */
/* decisions and forced_next [B] (or NULL) the sampled token, for comparison  */
/* with a run that took a near-tied decision the other way.                  */
int oracle_speculative_posterior(int dtype, const void *logits, const int32_t *tokens,
                                 const float *draft_logits, int B, int V, int K, double T,
                                 uint64_t seed, uint64_t step, const int32_t *forced_accept,
                                 const int32_t *forced_next, int32_t *accept_len,
                                 int32_t *path_tokens, int32_t *next_token, int32_t *accept,
                                 double *margin, int32_t *sample_row, double *sample_keys)
{
    if (!(T > 0.0) || K < 0 || V < 1) return 1;
    double *pr = (double *)malloc((size_t)V * sizeof(double));
    if (!pr) return 2;
    for (int b = 0; b < B; ++b) {
        const int32_t *tk = tokens + (size_t)b * (K + 1);
        for (int k = 0; k < K; ++k) {
            accept[(size_t)b * K + k] = -1;
            margin[(size_t)b * K + k] = 0.0;
        }
        int L = 0;
        for (int k = 1; k <= K; ++k) {
            const size_t prow = ((size_t)b * (K + 1) + (k - 1)) * V;
            const size_t qrow = ((size_t)b * K + (k - 1)) * V;
            const int x = tk[k];
            if (x < 0 || x >= V) { free(pr); return 3; }
            double logp = rd(dtype, logits, prow + x) / T - orc_logz_row(dtype, logits, prow, V, T);
            double logq = (double)draft_logits[qrow + x] / T - orc_logz_row(ORC_F32, draft_logits, qrow, V, T);
            double u = oracle_uniform(seed, step, ORC_RNG_ACCEPT, b, k, 0);
            double mg = logp - logq - log(u);
            margin[(size_t)b * K + (k - 1)] = mg;
            int acc = forced_accept ? (forced_accept[(size_t)b * K + (k - 1)] != 0) : (mg > 0.0);
            accept[(size_t)b * K + (k - 1)] = acc;
            if (!acc) break;
            L = k;
        }
        /* the next token: residual of row L against q_{L+1}, or p_K */
        const size_t prow = ((size_t)b * (K + 1) + L) * V;
        const double lzp = orc_logz_row(dtype, logits, prow, V, T);
        int use_residual = 0;
        if (L < K) {
            const size_t qrow = ((size_t)b * K + L) * V;
            const double lzq = orc_logz_row(ORC_F32, draft_logits, qrow, V, T);
            for (int v = 0; v < V; ++v) {
                double r = exp(rd(dtype, logits, prow + v) / T - lzp) -
                           exp((double)draft_logits[qrow + v] / T - lzq);
                pr[v] = r > 0.0 ? log(r) : -INFINITY;
                if (r > 0.0) use_residual = 1;
            }
        }
        if (!use_residual)   /* all accepted (or an empty residual): sample p_L */
            for (int v = 0; v < V; ++v)
                pr[v] = rd(dtype, logits, prow + v) / T - lzp;
        int best = -1;
        double bk = -INFINITY;
        for (int v = 0; v < V; ++v) {
            double key = pr[v] == -INFINITY ? -INFINITY
                         : pr[v] + orc_gumbel(seed, step, ORC_RNG_RESAMPLE, b, L, v);
            if (sample_keys) sample_keys[(size_t)b * V + v] = key;
            if (key > bk) { best = v; bk = key; }
        }
        if (best < 0) best = 0;
        accept_len[b] = L;
        next_token[b] = forced_next ? forced_next[b] : best;
        if (sample_row) sample_row[b] = L;
        for (int q = 0; q <= K; ++q)
            path_tokens[(size_t)b * (K + 1) + q] = q <= L ? tk[q] : -1;
    }
    free(pr);
    return 0;
}
