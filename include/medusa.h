/*
 * medusa.h -- C ABI of libmedusa_gb300.so: the data-parallel hot path of one
 * Medusa decoding step on one GB300 GPU (sm_103a).
 *
 * The step, as the pages define it:
 *   1. medusa_heads               K Medusa heads read the last hidden state and
 *                                 keep their top-s tokens (medusa_heads_lm:
 *                                 the LM head's root token in the same pass).
 *   2. medusa_build_tree          the proposals become a budgeted candidate tree
 *                                 (medusa_build_tree_static: its shape from a
 *                                 calibrated table instead).
 *   3. medusa_tree_attention      every tree node attends to the prefix and to
 *                                 its own ancestors.
 *   4. medusa_evaluate_posterior  greedy or typical acceptance; the longest
 *                                 accepted path is returned.
 *   5. medusa_commit_kv           the accepted path's K/V rows move into
 *                                 consecutive cache slots and the prefix
 *                                 grows (also fused into the posterior as
 *                                 medusa_evaluate_posterior_commit).
 *   medusa_step_run               1-4 (and 5) with the step's input copies
 *                                 from page-locked host memory, in one call.
 * Page citations are by title and section:
 *   [P1] "Medusa: Faster LLM text generation" (nazmi.tech)
 *   [P2] "Medusa 深读：解码慢不是算力问题，是搬运问题" (jokeuncle.pages.dev)
 *   [P3] "Medusa Part I: Architecture, Training, and Shifted Loss"
 *        (sudhirpol522.github.io)
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers unless the name ends in _host.
 *     The caller allocates and owns every buffer; the library allocates
 *     nothing and keeps no per-call state between calls, except the step
 *     executor (section 7), which owns a side stream and two events.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = legacy default stream).  No call synchronises the host, except
 *     medusa_read_device_status and medusa_step_run when asked to.
 *   - Arguments are validated on the host before any launch.  A bad argument
 *     returns MEDUSA_ERR_INVALID_ARG (or MEDUSA_ERR_UNSUPPORTED for a legal
 *     but unimplemented shape) and launches nothing; medusa_last_error()
 *     then describes it.  A failed launch returns MEDUSA_ERR_CUDA.
 *   - Problems only the device can see (a token id out of range, a prefix
 *     longer than the stated maximum, a non-log-probability score) set the
 *     device status word that sits in the first bytes of the workspace
 *     (first error wins; it stays set until medusa_clear_device_status).
 *     Read it with medusa_read_device_status.
 *   - Workspace: `ws` is a caller-owned device buffer of at least the bytes
 *     the matching *_workspace_size function returns, 256-byte aligned.  One
 *     buffer sized for the largest call may serve every call on one stream.
 *     Zero it once before first use (the status word must start at 0).
 *   - Row-major layouts; "[A,B,C]" lists dimensions outermost first.  Every
 *     tensor pointer must be 16-byte aligned and every innermost dimension a
 *     multiple of 16 bytes where stated.
 *   - bf16 tensors hold IEEE bfloat16; accumulation is fp32 everywhere.
 */
#ifndef MEDUSA_GB300_H
#define MEDUSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MEDUSA_API __attribute__((visibility("default")))
#else
#define MEDUSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum medusa_status {
    MEDUSA_OK = 0,
    MEDUSA_ERR_INVALID_ARG = 1,   /* bad pointer, size or alignment          */
    MEDUSA_ERR_UNSUPPORTED = 2,   /* legal but not implemented               */
    MEDUSA_ERR_WORKSPACE = 3,     /* workspace missing or too small          */
    MEDUSA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed    */
    MEDUSA_ERR_TIMEOUT = 5,       /* a bounded device wait ran out           */
    MEDUSA_ERR_DEVICE_CHECK = 6   /* the device found invalid data           */
} medusa_status;

typedef enum medusa_dtype {
    MEDUSA_F32 = 0,
    MEDUSA_BF16 = 1
} medusa_dtype;

typedef enum medusa_accept_mode {
    MEDUSA_GREEDY = 0,
    MEDUSA_TYPICAL = 1
} medusa_accept_mode;

/* Device status codes written into the workspace status word. */
enum {
    MEDUSA_DEV_OK = 0,
    MEDUSA_DEV_BAD_TOKEN = 1,      /* a token id outside [0, V)               */
    MEDUSA_DEV_BAD_PARENT = 2,     /* parent[i] not in [0, i)                 */
    MEDUSA_DEV_BAD_PREFIX = 3,     /* prefix_len[b] < 0 or > P_max            */
    MEDUSA_DEV_BAD_SCORE = 4,      /* a tree score > 0 or NaN                 */
    MEDUSA_DEV_BAD_DEPTH = 5,      /* depth[i] > K or depth[i] != depth[parent]+1 */
    MEDUSA_DEV_TIMEOUT = 6,        /* a bounded wait gave up                  */
    MEDUSA_DEV_BAD_PATH = 7,       /* accept_len outside 0..min(K,R-1), or a
                                      path entry outside [0, R)              */
    MEDUSA_DEV_BAD_CACHE = 8,      /* a cache pointer NULL or not 16-byte
                                      aligned                                 */
    MEDUSA_DEV_DRAIN_TIMEOUT = 9   /* after a timeout, the drain of the CTA's
                                      own MMAs also gave up; the tensor memory
                                      was freed with an MMA possibly still in
                                      flight, so this call's outputs and later
                                      tensor-core results on the device are
                                      suspect.  Overrides an earlier code.    */
};

/* Limits. */
#define MEDUSA_MAX_HEADS 8        /* K                                         */
#define MEDUSA_MAX_TOP_S 16       /* s_k, and the top-s kept per head          */
#define MEDUSA_MAX_TREE_ROWS 256  /* R = n + 1                                 */
#define MEDUSA_MAX_BATCH 8        /* B for medusa_heads                        */
#define MEDUSA_WS_HEADER 256      /* bytes of workspace before any scratch     */

typedef void *medusa_stream;      /* cudaStream_t */

/* Human-readable name of a status code (static string). */
MEDUSA_API const char *medusa_status_string(medusa_status s);

/* Message of the last failing call on this host thread ("" if none). */
MEDUSA_API const char *medusa_last_error(void);

/* Number of kernels this library has launched in this process. */
MEDUSA_API uint64_t medusa_launch_count(void);

/* Fault injection for the bounded device waits.  The tensor-core attention
 * waits on mbarriers for its own MMAs; each wait gives up after `polls`
 * polls (each poll blocks for a hardware-defined interval), sets
 * MEDUSA_DEV_TIMEOUT, stops the key loop, drains its MMAs and copies with a
 * fixed limit, frees its tensor memory and publishes an empty key range, so
 * the context stays usable.  Freeing assumes an issued MMA finishes within
 * the drain's limit (2^16 polls, far beyond an MMA's latency); if the drain
 * gives up too, the status reads MEDUSA_DEV_DRAIN_TIMEOUT instead.  Default 65536 polls; the environment variable
 * MEDUSA_FAULT_WAIT_BUDGET sets the value the library starts with.  A budget
 * of 0 makes every such wait fail at once: it exercises the timeout path
 * without a hung GPU.  Process-wide; affects launches made after the call. */
MEDUSA_API uint32_t medusa_wait_budget(void);
MEDUSA_API void medusa_set_wait_budget(uint32_t polls);

/* Copy the workspace status word to *status_host.  Synchronises `stream`. */
MEDUSA_API medusa_status medusa_read_device_status(const void *ws, int32_t *status_host,
                                        medusa_stream stream);

/* Reset the workspace status word to 0 (asynchronous on `stream`). */
MEDUSA_API medusa_status medusa_clear_device_status(void *ws, medusa_stream stream);

/* ------------------------------------------------------------------------
 * 1. Medusa heads.
 *
 * [P2] §3.1 (definition of p_t^(k)) and [P3] Part 3 (ResidualBlock,
 * vocabulary projection without bias): for every sequence b and head k
 *     u = W1[k] h[b] + b1[k],   z = h[b] + SiLU(u),   logits = W2[k] z,
 *     p^(k) = softmax(logits)
 * and each head keeps its `top_s` most probable tokens ([P2] §6.1).  The
 * vocabulary logits are never written to memory.
 *
 *   h      [B,d]      dtype
 *   W1     [K,d,d]    dtype; row j holds the weights of output unit j
 *   b1     [K,d]      dtype, or NULL for no bias
 *   W2     [K,V,d]    dtype; row v holds token v's projection
 *   topk_ids  [B,K,top_s] int32  out: token ids, most probable first;
 *                               equal logits rank the smaller id first
 *   topk_logp [B,K,top_s] fp32   out: log p^(k)(token)
 * Requirements: 1 <= B <= 8, 1 <= K <= 8, d % 8 == 0, 1 <= top_s <= 16,
 * top_s <= V, B'*d*4 <= 160 KiB where B' is B rounded up to 1, 2, 4 or 8.
 * Pointers 16-byte aligned.
 * ---------------------------------------------------------------------- */
MEDUSA_API size_t medusa_heads_workspace_size(int B, int K, int d, int V, int top_s);

MEDUSA_API medusa_status medusa_heads(medusa_dtype dtype, const void *h, const void *W1,
                           const void *b1, const void *W2, int B, int d, int V,
                           int K, int top_s, int32_t *topk_ids,
                           float *topk_logp, void *ws, size_t ws_bytes,
                           medusa_stream stream);

/* ------------------------------------------------------------------------
 * 1a. The LM head and the Medusa heads in one pass.
 *
 * [P1] Introduction and [P3] (the base model's LM head and the Medusa heads
 * read the same final hidden state): the LM head's logits are W_lm h (no
 * residual block).  [P2] §5: its greedy token is the tree's root, accepted
 * unconditionally.  The LM head joins the Medusa heads' weight stream as one
 * more head, so the whole proposal stage is one pass over W_lm, W1 and W2.
 *
 *   W_lm      [V,d]   dtype; row v holds token v's projection
 *   root      [B]     int32 out: argmax_v (W_lm h[b])_v (equal logits -> the
 *                     smaller id)
 *   root_logp [B]     fp32  out: log softmax(W_lm h[b])[root]
 * Other arguments, outputs and requirements as medusa_heads; the workspace
 * is medusa_heads_lm_workspace_size(...).
 * ---------------------------------------------------------------------- */
MEDUSA_API size_t medusa_heads_lm_workspace_size(int B, int K, int d, int V, int top_s);

MEDUSA_API medusa_status medusa_heads_lm(medusa_dtype dtype, const void *h, const void *W_lm,
                                         const void *W1, const void *b1, const void *W2, int B,
                                         int d, int V, int K, int top_s, int32_t *root,
                                         float *root_logp, int32_t *topk_ids, float *topk_logp,
                                         void *ws, size_t ws_bytes, medusa_stream stream);

/* ------------------------------------------------------------------------
 * 1b. Medusa heads with library-held scratch (no workspace argument).
 *
 * The pages have no counterpart: this is a calling convention, not part of
 * the method.  It is for callers that cannot allocate device memory at the
 * time they run the heads -- a serving runtime that gives all free HBM to its
 * KV-cache pool at start-up, or a decode loop that cannot afford the
 * device-wide synchronisation of cudaMalloc/cudaFree.  Same arguments and
 * results as medusa_heads, minus the workspace: the scratch is a 4 MiB
 * device array inside the library, reserved on every GPU that loads the
 * library until the process exits.  Shapes whose scratch
 * (medusa_heads_workspace_size) exceeds 4 MiB return MEDUSA_ERR_UNSUPPORTED
 * and launch nothing.  The call allocates nothing.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture.  All calls
 * share the one array: calls that overlap on the GPU race and must be
 * serialised by the caller.  The looked-up address is kept for the life of
 * the process, so resetting a device (cudaDeviceReset) or otherwise
 * re-creating its primary context after the first call is not supported: the
 * saved address would no longer be valid.
 * ---------------------------------------------------------------------- */
MEDUSA_API medusa_status medusa_heads_noalloc(medusa_dtype dtype, const void *h,
                                              const void *W1, const void *b1,
                                              const void *W2, int B, int d, int V,
                                              int K, int top_s, int32_t *topk_ids,
                                              float *topk_logp,
                                              medusa_stream stream);

/* ------------------------------------------------------------------------
 * 1c. Sampled drafts (for exact speculative sampling, section 6).
 *
 * [P1] Acceptance rules and [P2] §3: for the verification to preserve the
 * verifying model's distribution, each draft must be a sample of its head's
 * own normalised distribution q_k = softmax(logits_k / temperature).  Same
 * pass as medusa_heads; instead of the top-s list, head k of sequence b
 * draws x_k = argmax_v (logits_k[v] / T + G_v) (Gumbel-max, the smaller id
 * on exact ties), G_v = -log(-log u) with u the Philox4x64-10 uniform of
 * stream (purpose 1, row k, sequence b) at index v under key (seed, step)
 * (counter (v/4, k, b, 1), word v%4, u = ((w >> 41) + 0.5) * 2^-23).
 *
 *   drafts       [B,K]    int32 out
 *   draft_logits [B,K,V]  fp32 out: the heads' logits (before 1/T), which
 *                         medusa_speculative_posterior needs for q
 * Requirements as medusa_heads; temperature > 0; workspace
 * medusa_heads_workspace_size(B, K, d, V, 1).
 * ---------------------------------------------------------------------- */
MEDUSA_API medusa_status medusa_heads_sample(medusa_dtype dtype, const void *h, const void *W1,
                                             const void *b1, const void *W2, int B, int d,
                                             int V, int K, float temperature, uint64_t seed,
                                             uint64_t step, int32_t *drafts,
                                             float *draft_logits, void *ws, size_t ws_bytes,
                                             medusa_stream stream);

/* ------------------------------------------------------------------------
 * 2. Candidate tree under a node budget.
 *
 * [P2] §6.2 (greedy construction within a budget: repeatedly take the
 * frontier node of largest path weight, then add its children) with the
 * heads' own probabilities as the per-level weights, so a rank path
 * (i_1..i_k) scores sum_j topk_logp[b][j-1][i_j] (summed from depth 1 down,
 * in fp64).  [P2] §6.1 (tree mask and shared position index).
 * Ties: equal scores go to the smaller depth, then to the lexicographically
 * smaller rank path.  Output order is canonical: root first, then by depth,
 * then by rank path, so parent[i] < i and each depth is contiguous.
 *
 *   root       [B]              int32  the LM head's greedy token per sequence
 *   topk_ids   [B,K,top_s]      int32  from medusa_heads
 *   topk_logp  [B,K,top_s]      fp32   log-probabilities (must be <= 0)
 *   s_host     [K]   HOST       int32  candidates used at depth k+1, 1..top_s
 *   n                                  tree nodes besides the root; R = n+1
 *   prefix_len [B] or NULL      int32  P_b, for pos_id (NULL = 0)
 * Outputs (R = n+1, W = ceil(R/64)):
 *   tokens [B,R], parent [B,R] (-1 at root), depth [B,R], pos_id [B,R] =
 *   P_b + depth, anc_mask [B,R,W] uint64 (bit j of row i set iff node j is
 *   node i or one of its ancestors), paths [B,n,K+1] (node indices root ->
 *   leaf for each leaf in canonical order, -1 padded), n_leaf [B].
 * Requirements: K <= 8, R <= 256, n <= sum_k prod_{j<=k} s_j.
 * ---------------------------------------------------------------------- */
MEDUSA_API size_t medusa_build_tree_workspace_size(int B, int K, int top_s, int n);

MEDUSA_API medusa_status medusa_build_tree(const int32_t *root, const int32_t *topk_ids,
                                const float *topk_logp, int B, int K,
                                const int32_t *s_host, int top_s, int n,
                                const int32_t *prefix_len, int32_t *tokens,
                                int32_t *parent, int32_t *depth,
                                int32_t *pos_id, uint64_t *anc_mask,
                                int32_t *paths, int32_t *n_leaf, void *ws,
                                size_t ws_bytes, medusa_stream stream);

/* ------------------------------------------------------------------------
 * 2b. Candidate tree from a calibrated, static table.
 *
 * [P2] §6.2: the per-level weights a_k^(i) (how often head k's rank-i token
 * is right, measured once on a calibration set) fix the tree's shape; the
 * greedy construction under the budget is the one of medusa_build_tree,
 * with log a_k^(i) as the weight of rank i at depth k for every sequence.
 * The shape is therefore the same for every sequence and every step; the
 * tokens come from each sequence's own top-s lists.  Calibrating the table
 * is not part of the library.
 *
 *   log_a  [K,top_s]  fp32 (device), log a_k^(i) <= 0; entries i >= s[k]
 *                     are ignored
 * Other arguments, outputs and requirements as medusa_build_tree.
 * ---------------------------------------------------------------------- */
MEDUSA_API medusa_status medusa_build_tree_static(const int32_t *root, const int32_t *topk_ids,
                                                  const float *log_a, int B, int K,
                                                  const int32_t *s_host, int top_s, int n,
                                                  const int32_t *prefix_len, int32_t *tokens,
                                                  int32_t *parent, int32_t *depth,
                                                  int32_t *pos_id, uint64_t *anc_mask,
                                                  int32_t *paths, int32_t *n_leaf, void *ws,
                                                  size_t ws_bytes, medusa_stream stream);

/* ------------------------------------------------------------------------
 * 3. Tree attention.
 *
 * [P1] "Tree attention" and [P2] §6.1: node i of sequence b attends to every
 * prefix slot and to the tree slots of its own ancestors (itself included),
 * never to another branch:
 *     out[b,i,h] = softmax_j( scale * q[b,i,h] . K_b[j,h] + M_i(j) ) V_b[j,h]
 * with M_i(j) = 0 for j < P_b or for tree slot j = P_b + t where bit t of
 * anc_mask[b,i] is set, -inf otherwise.
 *
 *   q         [B,R,H,dh]                 dtype (RoPE, if any, already applied)
 *   k_cache   [B] device array of device pointers; sequence b's cache is
 *             [>= P_b+R, H, dh] dtype: prefix in slots 0..P_b-1, the tree
 *             nodes (canonical order) in slots P_b..P_b+R-1
 *   v_cache   same layout as k_cache
 *   prefix_len [B] int32 (device), 0 <= P_b <= P_max
 *   anc_mask  [B,R,W] uint64 from medusa_build_tree
 *   out       [B,R,H,dh] dtype
 * Requirements: dh in {64,128}; R <= 256; bf16: any P_max; f32: P_max + R
 * <= 16384.
 * ---------------------------------------------------------------------- */
MEDUSA_API size_t medusa_tree_attention_workspace_size(medusa_dtype dtype, int B, int R,
                                            int H, int dh, int P_max);

MEDUSA_API medusa_status medusa_tree_attention(medusa_dtype dtype, const void *q,
                                    const void *const *k_cache,
                                    const void *const *v_cache,
                                    const int32_t *prefix_len, int P_max,
                                    const uint64_t *anc_mask, int B, int R,
                                    int H, int dh, float scale, void *out,
                                    void *ws, size_t ws_bytes,
                                    medusa_stream stream);

/* ------------------------------------------------------------------------
 * 4. Posterior: acceptance and the longest accepted path.
 *
 * Node i's token is judged by the verification logits of its parent's row.
 *   MEDUSA_GREEDY  ([P3] Part 2): accept iff the token is that row's argmax.
 *   MEDUSA_TYPICAL ([P2] §5):  accept iff p(x) > min(eps, delta*exp(-H(p))),
 *                  p = softmax(logits / temperature), H in nats.
 * The root (the LM head's greedy token) is accepted unconditionally ([P2] §5);
 * a node counts only if all its ancestors are accepted ([P3] Part 2); the
 * deepest such node wins, the smallest canonical index among equals.
 *
 *   logits [B,R,V] dtype; tokens/parent/depth [B,R] int32 from
 *   medusa_build_tree (parent[i] < i).
 * Outputs:
 *   accept_len [B]         accepted nodes beyond the root, 0..K
 *   path [B,K+1]           node indices root -> best (-1 padded)
 *   path_tokens [B,K+1]    their tokens (-1 padded)
 *   next_token [B]         argmax of the best node's row (ties -> smaller id)
 *   accept [B,R] or NULL   per-node decision (root = 1)
 * The outputs may be device memory or page-locked host memory that the
 * device addresses at the same pointer (cudaHostAlloc, or cudaHostRegister
 * with mapping, under unified addressing): the kernel then writes the
 * results straight to the host, readable once the stream has synchronised,
 * with no copy back.  Pageable host memory is rejected
 * (MEDUSA_ERR_INVALID_ARG).
 * Requirements: R <= 256, K <= 8, V % 8 == 0 (bf16) or V % 4 == 0 (f32),
 * temperature > 0, eps > 0, delta > 0.
 * ---------------------------------------------------------------------- */
MEDUSA_API size_t medusa_posterior_workspace_size(int B, int R);

MEDUSA_API medusa_status medusa_evaluate_posterior(medusa_dtype dtype, const void *logits,
                                        const int32_t *tokens,
                                        const int32_t *parent,
                                        const int32_t *depth, int B, int R,
                                        int V, int K, medusa_accept_mode mode,
                                        float eps, float delta,
                                        float temperature, int32_t *accept_len,
                                        int32_t *path, int32_t *path_tokens,
                                        int32_t *next_token, int32_t *accept,
                                        void *ws, size_t ws_bytes,
                                        medusa_stream stream);

/* ------------------------------------------------------------------------
 * 6. Exact speculative sampling on a chain of sampled drafts.
 *
 * [P1] Acceptance rules; [P2] §3 (drafts from known normalised q_k with
 * p/q acceptance and (p - q)+ correction recover the target distribution)
 * and §5.  The candidate is a chain x_0 (the root, accepted), x_1..x_K
 * (x_k sampled from q_k by medusa_heads_sample).  With p_j = softmax(logits
 * row j / T): draft x_k is accepted iff u_k * q_k(x_k) < p_{k-1}(x_k), u_k
 * the uniform of stream (purpose 2, row k, sequence b) at index 0; the
 * first rejection at k = L+1 ends the chain and the next token is sampled
 * from max(0, p_L - q_{L+1}) normalised (if that residual is empty in fp32,
 * from p_L); with all K accepted it is sampled from p_K.  Samples use the
 * Gumbel-max rule with stream (purpose 3, row L, sequence b).
 *
 *   logits       [B,K+1,V] dtype  verification rows of x_0..x_K
 *   tokens       [B,K+1]   int32  x_0..x_K (a chain: row j judges x_{j+1})
 *   draft_logits [B,K,V]   fp32   from medusa_heads_sample
 * Outputs: accept_len [B] = L; path_tokens [B,K+1] = x_0..x_L, -1 padded;
 * next_token [B]; accept [B,K] or NULL (1 accepted, 0 the rejection, -1
 * not reached).  Requirements: 1 <= K <= 8, V % 8 == 0, temperature > 0.
 * A draft token outside [0, V) counts as rejected and sets
 * MEDUSA_DEV_BAD_TOKEN.
 * ---------------------------------------------------------------------- */
MEDUSA_API size_t medusa_speculative_workspace_size(int B, int K);

MEDUSA_API medusa_status medusa_speculative_posterior(
    medusa_dtype dtype, const void *logits, const int32_t *tokens, const float *draft_logits,
    int B, int V, int K, float temperature, uint64_t seed, uint64_t step, int32_t *accept_len,
    int32_t *path_tokens, int32_t *next_token, int32_t *accept, void *ws, size_t ws_bytes,
    medusa_stream stream);

/* ------------------------------------------------------------------------
 * 5. Commit of the accepted path into the KV cache.
 *
 * [P1] Introduction and [P2] §5: the accepted tokens become part of the
 * context for the next step, so the K/V the verification pass computed for
 * them is kept and the rest of the tree is dropped.  With the tree nodes in
 * cache slots P_b .. P_b+R-1 (canonical order, as medusa_tree_attention
 * reads them) and the accepted path root -> best of accept_len[b]+1 nodes,
 * slot P_b + q receives the K and V rows of node path[b][q] for
 * q = 0 .. accept_len[b], and new_prefix_len[b] = P_b + accept_len[b] + 1.
 * The next step's root is the posterior's next_token.  Rows are copied as
 * raw bytes; every source row is read before any target row is written, so
 * overlapping sources and targets are handled.  Slots past the new prefix
 * keep stale data.
 *
 *   k_cache, v_cache  [B] device arrays of device pointers, each to a
 *                     sequence's [>= P_b+R, H, dh] dtype cache (16-byte
 *                     aligned; checked on the device: MEDUSA_DEV_BAD_CACHE)
 *   prefix_len [B]    int32 P_b >= 0 (device; MEDUSA_DEV_BAD_PREFIX)
 *   path [B,K+1]      int32 node indices from medusa_evaluate_posterior
 *   accept_len [B]    int32 0 .. min(K, R-1) (MEDUSA_DEV_BAD_PATH)
 *   new_prefix_len [B] int32 out; must not alias prefix_len
 * A sequence that fails a device check is left untouched and gets
 * new_prefix_len = prefix_len.  Requirements: K <= 8, R <= 256,
 * H*dh*sizeof(dtype) a multiple of 16.  Needs a workspace of
 * MEDUSA_WS_HEADER bytes (the status word).
 * ---------------------------------------------------------------------- */
MEDUSA_API medusa_status medusa_commit_kv(medusa_dtype dtype, void *const *k_cache,
                                          void *const *v_cache, const int32_t *prefix_len,
                                          const int32_t *path, const int32_t *accept_len,
                                          int B, int K, int R, int H, int dh,
                                          int32_t *new_prefix_len, void *ws, size_t ws_bytes,
                                          medusa_stream stream);

/* ------------------------------------------------------------------------
 * 4+5. Posterior and commit in one call: medusa_evaluate_posterior's
 * results, then the commit of medusa_commit_kv done by the same kernel that
 * picks the path (no extra launch).  `dtype` is that of the logits and of
 * the caches.  Arguments and requirements are the union of the two calls;
 * the workspace is medusa_posterior_workspace_size(B, R).
 * ---------------------------------------------------------------------- */
MEDUSA_API medusa_status medusa_evaluate_posterior_commit(
    medusa_dtype dtype, const void *logits, const int32_t *tokens, const int32_t *parent,
    const int32_t *depth, int B, int R, int V, int K, medusa_accept_mode mode, float eps,
    float delta, float temperature, int32_t *accept_len, int32_t *path, int32_t *path_tokens,
    int32_t *next_token, int32_t *accept, void *const *k_cache, void *const *v_cache,
    const int32_t *prefix_len, int H, int dh, int32_t *new_prefix_len, void *ws,
    size_t ws_bytes, medusa_stream stream);

/* ------------------------------------------------------------------------
 * 7. The decoding step as one call: a step executor.
 *
 * [P1] Introduction and [P2] §3-§6: one Medusa step is heads -> candidate
 * tree -> tree attention -> posterior (and, optionally, the commit).  The
 * executor issues that sequence with the step's input copies in one host
 * call, so that a caller whose inputs sit in page-locked host memory pays
 * no per-call overhead of its own between them:
 *   1. `early` copies on `stream` (the inputs of the heads and the tree:
 *      the hidden state, the root token),
 *   2. medusa_heads,
 *   3. `late` copies on the executor's own side stream, which first waits
 *      for everything issued to `stream` before this run (the inputs of the
 *      attention and the posterior: q, the tree's K/V rows, the
 *      verification logits); they travel during the heads pass,
 *   4. medusa_build_tree, then `stream` waits for the side stream,
 *   5. medusa_tree_attention,
 *   6. medusa_evaluate_posterior, or medusa_evaluate_posterior_commit when
 *      new_prefix_len is not NULL.
 * Every kernel is stream-launched with programmatic dependent launch, as
 * the separate calls are.  The results equal those of the separate calls
 * on the same inputs.
 *
 * The descriptor names every buffer of the step; each field has the meaning
 * it has in the call it is passed to (R = n + 1; the tree's outputs are
 * the attention's and the posterior's inputs).  Copies: `dst` device
 * memory, `src` page-locked host memory or device memory (each copy's
 * direction is resolved at create, which refuses any other memory with
 * MEDUSA_ERR_INVALID_ARG), `bytes` > 0; at most MEDUSA_STEP_MAX_COPIES in
 * each list.  One workspace serves all
 * four calls (at least the largest of their *_workspace_size values).
 *
 * medusa_step_create validates the descriptor's structure (NULL
 * pointers, counts, sizes) before touching CUDA, copies the descriptor, the
 * copy lists and s_host, and creates a non-blocking side stream and two
 * events on the current device (and, in graph mode, a capture stream and
 * the graph; with page-locked results, B completion words of page-locked
 * host memory): the only CUDA objects the library owns.  It allocates no
 * device memory of its own.  The buffers the descriptor names must stay
 * allocated, at the same addresses, while the executor lives; new inputs
 * are written into the same host buffers before each run.
 * With flags = MEDUSA_STEP_GRAPH, create also runs the sequence once under
 * stream capture (on a capture stream of its own; nothing executes) and
 * instantiates it as a CUDA graph, so that each run is one graph launch:
 * the launches keep their programmatic-dependent-launch edges, and the
 * wait budget (medusa_set_wait_budget) in force at create is the one the
 * graph's attention uses.  A call's validation failure then surfaces at
 * create.
 * medusa_step_run issues one step on `stream`; with `synchronize` != 0 it
 * also waits for the step: when the posterior's results are page-locked host
 * memory, until every sequence's results (and the fused commit) are written
 * -- the posterior's last kernel raises a completion word in page-locked
 * memory that the executor owns, and the host polls it (the stream may
 * still be retiring that kernel; work issued later is ordered after it) --
 * and otherwise, or if the word has not come after 20 ms, until the stream
 * is idle.  Runs of one executor go to one stream (or are ordered by the
 * caller).  A call's own validation or launch failure
 * stops the run there and returns that call's status.  One executor serves
 * one host thread at a time.  medusa_step_destroy releases the side stream,
 * events and graph (after the work they carry has completed; freeing the
 * completion words waits for the device); NULL is a no-op.
 * medusa_step_desc_size returns sizeof(medusa_step_desc), so that a binding
 * can check its mirror of the struct.
 * ---------------------------------------------------------------------- */
#define MEDUSA_STEP_MAX_COPIES 64
#define MEDUSA_STEP_GRAPH 1       /* capture the sequence once as a CUDA graph */

typedef struct medusa_copy {
    void *dst;
    const void *src;
    size_t bytes;
} medusa_copy;

typedef struct medusa_step_desc {
    const medusa_copy *early;   /* copies before the heads, on `stream`     */
    int32_t n_early;
    const medusa_copy *late;    /* copies during the heads, on the side     */
    int32_t n_late;
    medusa_dtype dtype;         /* of h, W1, b1, W2, q, caches, logits      */
    /* heads */
    const void *h, *W1, *b1, *W2;
    int32_t B, d, V, K, top_s;
    int32_t *topk_ids;
    float *topk_logp;
    /* tree */
    const int32_t *root;
    const int32_t *s_host;      /* [K] host; copied at create               */
    int32_t n;
    const int32_t *prefix_len;
    int32_t *tokens, *parent, *depth, *pos_id;
    uint64_t *anc_mask;
    int32_t *paths, *n_leaf;
    /* attention */
    const void *q;
    const void *const *k_cache, *const *v_cache;
    int32_t P_max, H, dh;
    float scale;
    void *attn_out;
    /* posterior (and commit) */
    const void *logits;
    medusa_accept_mode mode;
    float eps, delta, temperature;
    int32_t *accept_len, *path, *path_tokens, *next_token, *accept;
    int32_t *new_prefix_len;    /* non-NULL: fused commit into the caches   */
    void *ws;
    size_t ws_bytes;
    int32_t flags;              /* MEDUSA_STEP_GRAPH or 0                   */
} medusa_step_desc;

typedef struct medusa_step_exec medusa_step_exec;

MEDUSA_API size_t medusa_step_desc_size(void);
MEDUSA_API medusa_status medusa_step_create(const medusa_step_desc *desc,
                                            medusa_step_exec **exec_out);
MEDUSA_API medusa_status medusa_step_run(medusa_step_exec *exec, medusa_stream stream,
                                         int synchronize);
/* The wait of medusa_step_run(..., synchronize = 1) on its own: for every run
 * issued so far on `stream` (the host may work between the issue and it). */
MEDUSA_API medusa_status medusa_step_wait(medusa_step_exec *exec, medusa_stream stream);
MEDUSA_API void medusa_step_destroy(medusa_step_exec *exec);

#ifdef __cplusplus
}
#endif

#endif /* MEDUSA_GB300_H */
