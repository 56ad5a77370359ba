// api.cu -- the extern "C" boundary of libmedusa_gb300.so.
//
// Every entry point validates its arguments on the host, launches nothing on
// a bad argument, and maps CUDA failures to MEDUSA_ERR_CUDA.  The message of
// the last failure on the calling thread is kept for medusa_last_error().
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "launch.h"

namespace medusa {

namespace {

thread_local char g_err[512] = "";
std::atomic<uint64_t> g_launches{0};

medusa_status fail(medusa_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

medusa_status cuda_fail(cudaError_t e, const char *where) {
    return fail(MEDUSA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

medusa_status check_ws(const void *ws, size_t have, size_t need, const char *who) {
    if (!ws) return fail(MEDUSA_ERR_WORKSPACE, "%s: workspace is NULL", who);
    if (!aligned256(ws)) return fail(MEDUSA_ERR_WORKSPACE, "%s: workspace not 256-byte aligned", who);
    if (have < need)
        return fail(MEDUSA_ERR_WORKSPACE, "%s: workspace has %zu bytes, needs %zu", who, have, need);
    return MEDUSA_OK;
}

}  // namespace

namespace {

// Poll limit of the bounded device waits; MEDUSA_FAULT_WAIT_BUDGET sets the
// first value (fault injection), medusa_set_wait_budget any later one.
constexpr uint32_t kDefaultWaitPolls = 1u << 16;
std::atomic<uint32_t> g_wait_polls{kDefaultWaitPolls};
std::once_flag g_wait_env_once;

void read_wait_env() {
    const char *v = std::getenv("MEDUSA_FAULT_WAIT_BUDGET");
    if (!v || !*v) return;
    char *end = nullptr;
    const unsigned long n = std::strtoul(v, &end, 10);
    if (end && *end == '\0' && n <= 0xffffffffUL) g_wait_polls.store((uint32_t)n);
}

}  // namespace

uint32_t wait_budget() {
    std::call_once(g_wait_env_once, read_wait_env);
    return g_wait_polls.load(std::memory_order_relaxed);
}

NvtxRange::NvtxRange(const char *name) { nvtxRangePushA(name); }
NvtxRange::~NvtxRange() { nvtxRangePop(); }

int device_sm_count() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        cache[dev] = n;
    }
    return cache[dev];
}

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void set_last_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
}

}  // namespace medusa

using namespace medusa;

extern "C" {

const char *medusa_status_string(medusa_status s) {
    switch (s) {
    case MEDUSA_OK: return "MEDUSA_OK";
    case MEDUSA_ERR_INVALID_ARG: return "MEDUSA_ERR_INVALID_ARG";
    case MEDUSA_ERR_UNSUPPORTED: return "MEDUSA_ERR_UNSUPPORTED";
    case MEDUSA_ERR_WORKSPACE: return "MEDUSA_ERR_WORKSPACE";
    case MEDUSA_ERR_CUDA: return "MEDUSA_ERR_CUDA";
    case MEDUSA_ERR_TIMEOUT: return "MEDUSA_ERR_TIMEOUT";
    case MEDUSA_ERR_DEVICE_CHECK: return "MEDUSA_ERR_DEVICE_CHECK";
    }
    return "MEDUSA_ERR_UNKNOWN";
}

const char *medusa_last_error(void) { return g_err; }

uint64_t medusa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

uint32_t medusa_wait_budget(void) { return wait_budget(); }

void medusa_set_wait_budget(uint32_t polls) {
    std::call_once(g_wait_env_once, read_wait_env);
    g_wait_polls.store(polls, std::memory_order_relaxed);
}

medusa_status medusa_read_device_status(const void *ws, int32_t *status_host, medusa_stream stream) {
    if (!ws || !status_host) return fail(MEDUSA_ERR_INVALID_ARG, "read_device_status: NULL pointer");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(status_host, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (e) return cuda_fail(e, "read_device_status");
    e = cudaStreamSynchronize(st);
    if (e) return cuda_fail(e, "read_device_status");
    return MEDUSA_OK;
}

medusa_status medusa_clear_device_status(void *ws, medusa_stream stream) {
    if (!ws) return fail(MEDUSA_ERR_INVALID_ARG, "clear_device_status: NULL workspace");
    cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream));
    if (e) return cuda_fail(e, "clear_device_status");
    return MEDUSA_OK;
}

// ----------------------------------------------------------------- heads ---

size_t medusa_heads_workspace_size(int B, int K, int d, int V, int top_s) {
    if (B < 1 || K < 1 || d < 1 || V < 1 || top_s < 1) return 0;
    return heads_workspace_bytes(B, K, d, V, top_s);
}

size_t medusa_heads_lm_workspace_size(int B, int K, int d, int V, int top_s) {
    if (B < 1 || K < 1 || d < 1 || V < 1 || top_s < 1) return 0;
    return heads_workspace_bytes(B, K, d, V, top_s, true);
}

}  // extern "C"

namespace {

medusa_status check_heads(const char *who, medusa_dtype dtype, const void *h, const void *W1,
                          const void *b1, const void *W2, int B, int d, int V, int K, int top_s,
                          const int32_t *topk_ids, const float *topk_logp, bool need_logp = true) {
    if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: unknown dtype %d", who, (int)dtype);
    if (!h || !W1 || !W2 || !topk_ids || (need_logp && !topk_logp))
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: NULL tensor pointer", who);
    if (B < 1 || B > MEDUSA_MAX_BATCH)
        return fail(MEDUSA_ERR_UNSUPPORTED, "%s: B=%d outside 1..%d", who, B, MEDUSA_MAX_BATCH);
    if (K < 1 || K > MEDUSA_MAX_HEADS)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: K=%d outside 1..%d", who, K, MEDUSA_MAX_HEADS);
    if (d < 8 || d % 8)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: d=%d must be a positive multiple of 8", who, d);
    if (top_s < 1 || top_s > MEDUSA_MAX_TOP_S || top_s > V)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: top_s=%d outside 1..min(16, V)", who, top_s);
    const int nb = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : 8;  // batch bucket held in smem
    if ((size_t)nb * d * sizeof(float) > 160 * 1024)
        return fail(MEDUSA_ERR_UNSUPPORTED, "%s: %d x d x 4 = %zu bytes exceeds 160 KiB", who, nb,
                    (size_t)nb * d * sizeof(float));
    if (!aligned16(h) || !aligned16(W1) || !aligned16(W2) || (b1 && !aligned16(b1)))
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: tensor pointers must be 16-byte aligned", who);
    return MEDUSA_OK;
}

}  // namespace

extern "C" {

medusa_status medusa_heads(medusa_dtype dtype, const void *h, const void *W1, const void *b1,
                           const void *W2, int B, int d, int V, int K, int top_s,
                           int32_t *topk_ids, float *topk_logp, void *ws, size_t ws_bytes,
                           medusa_stream stream) {
    const NvtxRange range("medusa_heads");
    const char *who = "medusa_heads";
    if (medusa_status s = check_heads(who, dtype, h, W1, b1, W2, B, d, V, K, top_s, topk_ids,
                                      topk_logp))
        return s;
    if (medusa_status s = check_ws(ws, ws_bytes, heads_workspace_bytes(B, K, d, V, top_s), who))
        return s;
    cudaError_t e = launch_heads(dtype, h, nullptr, W1, b1, W2, B, d, V, K, top_s, topk_ids,
                                 topk_logp, nullptr, nullptr, nullptr, ws,
                                 static_cast<cudaStream_t>(stream));
    if (e) return cuda_fail(e, who);
    return MEDUSA_OK;
}

medusa_status medusa_heads_lm(medusa_dtype dtype, const void *h, const void *W_lm, const void *W1,
                              const void *b1, const void *W2, int B, int d, int V, int K,
                              int top_s, int32_t *root, float *root_logp, int32_t *topk_ids,
                              float *topk_logp, void *ws, size_t ws_bytes, medusa_stream stream) {
    const NvtxRange range("medusa_heads_lm");
    const char *who = "medusa_heads_lm";
    if (medusa_status s = check_heads(who, dtype, h, W1, b1, W2, B, d, V, K, top_s, topk_ids,
                                      topk_logp))
        return s;
    if (!W_lm || !root || !root_logp)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: NULL pointer", who);
    if (!aligned16(W_lm))
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: W_lm must be 16-byte aligned", who);
    if (medusa_status s =
            check_ws(ws, ws_bytes, heads_workspace_bytes(B, K, d, V, top_s, true), who))
        return s;
    cudaError_t e = launch_heads(dtype, h, W_lm, W1, b1, W2, B, d, V, K, top_s, topk_ids,
                                 topk_logp, root, root_logp, nullptr, ws,
                                 static_cast<cudaStream_t>(stream));
    if (e) return cuda_fail(e, who);
    return MEDUSA_OK;
}

medusa_status medusa_heads_sample(medusa_dtype dtype, const void *h, const void *W1,
                                  const void *b1, const void *W2, int B, int d, int V, int K,
                                  float temperature, uint64_t seed, uint64_t step,
                                  int32_t *drafts, float *draft_logits, void *ws,
                                  size_t ws_bytes, medusa_stream stream) {
    const NvtxRange range("medusa_heads_sample");
    const char *who = "medusa_heads_sample";
    // drafts is the top-1 list of the perturbed keys; no log-probabilities
    if (medusa_status s =
            check_heads(who, dtype, h, W1, b1, W2, B, d, V, K, 1, drafts, nullptr, false))
        return s;
    if (!draft_logits) return fail(MEDUSA_ERR_INVALID_ARG, "%s: NULL draft_logits", who);
    if (!(temperature > 0.f) || !(temperature < 1e30f))
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: temperature must be positive and finite", who);
    if (medusa_status s = check_ws(ws, ws_bytes, heads_workspace_bytes(B, K, d, V, 1), who))
        return s;
    SampleArgs smp;
    smp.on = 1;
    smp.inv_T = 1.f / temperature;
    smp.seed = seed;
    smp.step = step;
    smp.logits_out = draft_logits;
    cudaError_t e = launch_heads(dtype, h, nullptr, W1, b1, W2, B, d, V, K, 1, drafts, nullptr,
                                 nullptr, nullptr, &smp, ws, static_cast<cudaStream_t>(stream));
    if (e) return cuda_fail(e, who);
    return MEDUSA_OK;
}

// ------------------------------------------------------------------ tree ---

size_t medusa_build_tree_workspace_size(int B, int K, int top_s, int n) {
    return tree_workspace_bytes(B, K, top_s, n);
}

}  // extern "C"

namespace {

medusa_status check_tree(const char *who, const int32_t *root, const int32_t *topk_ids,
                         const float *weights, int B, int K, const int32_t *s_host, int top_s,
                         int n, const int32_t *tokens, const int32_t *parent,
                         const int32_t *depth, const int32_t *pos_id, const uint64_t *anc_mask,
                         const int32_t *paths, const int32_t *n_leaf, const void *ws,
                         size_t ws_bytes) {
    if (!root || !topk_ids || !weights || !s_host || !tokens || !parent || !depth || !pos_id ||
        !anc_mask || !paths || !n_leaf)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: NULL pointer", who);
    if (B < 1) return fail(MEDUSA_ERR_INVALID_ARG, "%s: B=%d", who, B);
    if (K < 1 || K > MEDUSA_MAX_HEADS)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: K=%d outside 1..%d", who, K, MEDUSA_MAX_HEADS);
    if (top_s < 1 || top_s > MEDUSA_MAX_TOP_S)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: top_s=%d outside 1..16", who, top_s);
    long long total = 0, level = 1;
    for (int k = 0; k < K; ++k) {
        if (s_host[k] < 1 || s_host[k] > top_s)
            return fail(MEDUSA_ERR_INVALID_ARG, "%s: s[%d]=%d outside 1..top_s", who, k, s_host[k]);
        level *= s_host[k];
        total += level;
        if (total > (1 << 20)) break;
    }
    if (n < 1 || n + 1 > MEDUSA_MAX_TREE_ROWS)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: n=%d outside 1..%d", who, n,
                    MEDUSA_MAX_TREE_ROWS - 1);
    if (n > total)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: n=%d exceeds the %lld nodes of the full tree",
                    who, n, total);
    return check_ws(ws, ws_bytes, tree_workspace_bytes(B, K, top_s, n), who);
}

}  // namespace

extern "C" {

medusa_status medusa_build_tree(const int32_t *root, const int32_t *topk_ids,
                                const float *topk_logp, int B, int K, const int32_t *s_host,
                                int top_s, int n, const int32_t *prefix_len, int32_t *tokens,
                                int32_t *parent, int32_t *depth, int32_t *pos_id,
                                uint64_t *anc_mask, int32_t *paths, int32_t *n_leaf, void *ws,
                                size_t ws_bytes, medusa_stream stream) {
    const NvtxRange range("medusa_build_tree");
    const char *who = "medusa_build_tree";
    if (medusa_status s = check_tree(who, root, topk_ids, topk_logp, B, K, s_host, top_s, n,
                                     tokens, parent, depth, pos_id, anc_mask, paths, n_leaf, ws,
                                     ws_bytes))
        return s;
    cudaError_t e = launch_build_tree(root, topk_ids, topk_logp, false, B, K, s_host, top_s, n,
                                      prefix_len, tokens, parent, depth, pos_id, anc_mask, paths,
                                      n_leaf, ws, static_cast<cudaStream_t>(stream));
    if (e) return cuda_fail(e, who);
    return MEDUSA_OK;
}

medusa_status medusa_build_tree_static(const int32_t *root, const int32_t *topk_ids,
                                       const float *log_a, int B, int K, const int32_t *s_host,
                                       int top_s, int n, const int32_t *prefix_len,
                                       int32_t *tokens, int32_t *parent, int32_t *depth,
                                       int32_t *pos_id, uint64_t *anc_mask, int32_t *paths,
                                       int32_t *n_leaf, void *ws, size_t ws_bytes,
                                       medusa_stream stream) {
    const NvtxRange range("medusa_build_tree_static");
    const char *who = "medusa_build_tree_static";
    if (medusa_status s = check_tree(who, root, topk_ids, log_a, B, K, s_host, top_s, n, tokens,
                                     parent, depth, pos_id, anc_mask, paths, n_leaf, ws,
                                     ws_bytes))
        return s;
    cudaError_t e = launch_build_tree(root, topk_ids, log_a, true, B, K, s_host, top_s, n,
                                      prefix_len, tokens, parent, depth, pos_id, anc_mask, paths,
                                      n_leaf, ws, static_cast<cudaStream_t>(stream));
    if (e) return cuda_fail(e, who);
    return MEDUSA_OK;
}

// ------------------------------------------------------------- attention ---

size_t medusa_tree_attention_workspace_size(medusa_dtype dtype, int B, int R, int H, int dh,
                                            int P_max) {
    if (B < 1 || R < 1 || H < 1 || dh < 1 || P_max < 0) return 0;
    return attention_workspace_bytes(dtype, B, R, H, dh, P_max);
}

medusa_status medusa_tree_attention(medusa_dtype dtype, const void *q, const void *const *k_cache,
                                    const void *const *v_cache, const int32_t *prefix_len,
                                    int P_max, const uint64_t *anc_mask, int B, int R, int H,
                                    int dh, float scale, void *out, void *ws, size_t ws_bytes,
                                    medusa_stream stream) {
    const NvtxRange range("medusa_tree_attention");
    const char *who = "medusa_tree_attention";
    if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: unknown dtype %d", who, (int)dtype);
    if (!q || !k_cache || !v_cache || !prefix_len || !anc_mask || !out)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: NULL pointer", who);
    if (B < 1 || H < 1) return fail(MEDUSA_ERR_INVALID_ARG, "%s: B=%d H=%d", who, B, H);
    if (R < 1 || R > MEDUSA_MAX_TREE_ROWS)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: R=%d outside 1..%d", who, R, MEDUSA_MAX_TREE_ROWS);
    if (dh != 64 && dh != 128)
        return fail(MEDUSA_ERR_UNSUPPORTED, "%s: dh=%d (supported: 64, 128)", who, dh);
    if (P_max < 0) return fail(MEDUSA_ERR_INVALID_ARG, "%s: P_max=%d", who, P_max);
    if (dtype == MEDUSA_F32 && (long long)P_max + R > 16384)
        return fail(MEDUSA_ERR_UNSUPPORTED, "%s: f32 path needs P_max + R <= 16384", who);
    if (!(scale > 0.f)) return fail(MEDUSA_ERR_INVALID_ARG, "%s: scale must be > 0", who);
    if (!aligned16(q) || !aligned16(out) || !aligned16(anc_mask) || !aligned16(k_cache) ||
        !aligned16(v_cache))
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", who);
    if (medusa_status s = check_ws(ws, ws_bytes, attention_workspace_bytes(dtype, B, R, H, dh, P_max), who))
        return s;
    cudaError_t e = launch_tree_attention(dtype, q, k_cache, v_cache, prefix_len, P_max, anc_mask,
                                          B, R, H, dh, scale, out, ws,
                                          static_cast<cudaStream_t>(stream));
    if (e) return cuda_fail(e, who);
    return MEDUSA_OK;
}

// ------------------------------------------------------------- posterior ---

size_t medusa_posterior_workspace_size(int B, int R) {
    if (B < 1 || R < 1) return 0;
    return posterior_workspace_bytes(B, R);
}

}  // extern "C"

namespace {

// The posterior's results may go to device memory or straight to page-locked
// host memory that the device addresses at the same pointer (cudaHostAlloc,
// or cudaHostRegister with mapping, under unified addressing): the select
// kernel writes them there, and the host reads them after the stream syncs.
// Pageable host memory is refused.  If the runtime cannot answer (no device)
// the check is left to the launch.
medusa_status check_result_pointer(const void *p, const char *who) {
    if (!p) return MEDUSA_OK;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return MEDUSA_OK;
    }
    if (at.type == cudaMemoryTypeUnregistered)
        return fail(MEDUSA_ERR_INVALID_ARG,
                    "%s: a result pointer is pageable host memory (device or pinned host memory)",
                    who);
    if (at.type == cudaMemoryTypeHost && at.devicePointer != p)
        return fail(MEDUSA_ERR_INVALID_ARG,
                    "%s: a pinned host result buffer is not mapped at the same device address",
                    who);
    return MEDUSA_OK;
}

medusa_status check_posterior(const char *who, medusa_dtype dtype, const void *logits,
                              const int32_t *tokens, const int32_t *parent, const int32_t *depth,
                              int B, int R, int V, int K, medusa_accept_mode mode, float eps,
                              float delta, float temperature, const int32_t *accept_len,
                              const int32_t *path, const int32_t *path_tokens,
                              const int32_t *next_token, const void *ws, size_t ws_bytes) {
    if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: unknown dtype %d", who, (int)dtype);
    if (mode != MEDUSA_GREEDY && mode != MEDUSA_TYPICAL)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: unknown mode %d", who, (int)mode);
    if (!logits || !tokens || !parent || !depth || !accept_len || !path || !path_tokens ||
        !next_token)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: NULL pointer", who);
    if (B < 1) return fail(MEDUSA_ERR_INVALID_ARG, "%s: B=%d", who, B);
    if (R < 1 || R > MEDUSA_MAX_TREE_ROWS)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: R=%d outside 1..%d", who, R, MEDUSA_MAX_TREE_ROWS);
    if (K < 0 || K > MEDUSA_MAX_HEADS)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: K=%d outside 0..%d", who, K, MEDUSA_MAX_HEADS);
    const int vn = dtype == MEDUSA_BF16 ? 8 : 4;
    if (V < 1 || V % vn)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: V=%d must be a positive multiple of %d", who, V, vn);
    if (!(temperature > 0.f) || !(eps > 0.f) || !(delta > 0.f))
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: eps, delta and temperature must be > 0", who);
    if (!aligned16(logits))
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: logits must be 16-byte aligned", who);
    if (medusa_status s = check_ws(ws, ws_bytes, posterior_workspace_bytes(B, R), who)) return s;
    const void *outs[4] = {accept_len, path, path_tokens, next_token};
    for (const void *o : outs)
        if (medusa_status s = check_result_pointer(o, who)) return s;
    return MEDUSA_OK;
}

// Host checks of the commit arguments shared by both commit entry points.
medusa_status check_commit(const char *who, medusa_dtype dtype, const void *const *k_cache,
                           const void *const *v_cache, const int32_t *prefix_len,
                           const int32_t *new_prefix_len, int H, int dh) {
    if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: unknown dtype %d", who, (int)dtype);
    if (!k_cache || !v_cache || !prefix_len || !new_prefix_len)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: NULL pointer", who);
    if (static_cast<const void *>(new_prefix_len) == static_cast<const void *>(prefix_len))
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: new_prefix_len must not alias prefix_len", who);
    if (!aligned16(k_cache) || !aligned16(v_cache))
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: cache pointer arrays must be 16-byte aligned", who);
    const size_t elt = dtype == MEDUSA_BF16 ? 2 : 4;
    if (H < 1 || dh < 1 || (long long)H * dh > (1LL << 26))
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: H=%d dh=%d", who, H, dh);
    if (((size_t)H * dh * elt) % 16)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: a cache row (H*dh elements) must be a multiple of 16 bytes",
                    who);
    return MEDUSA_OK;
}

}  // namespace

// The posterior with or without the commit (k_cache non-null) and with an
// optional completion word per sequence (the step executor's).
medusa_status medusa::evaluate_posterior_signalled(
    medusa_dtype dtype, const void *logits, const int32_t *tokens, const int32_t *parent,
    const int32_t *depth, int B, int R, int V, int K, medusa_accept_mode mode, float eps,
    float delta, float temperature, int32_t *accept_len, int32_t *path, int32_t *path_tokens,
    int32_t *next_token, int32_t *accept, void *const *k_cache, void *const *v_cache,
    const int32_t *prefix_len, int H, int dh, int32_t *new_prefix_len, void *ws,
    size_t ws_bytes, cudaStream_t stream, uint32_t *done) {
    const char *who = k_cache ? "medusa_evaluate_posterior_commit" : "medusa_evaluate_posterior";
    if (medusa_status s = check_posterior(who, dtype, logits, tokens, parent, depth, B, R, V, K,
                                          mode, eps, delta, temperature, accept_len, path,
                                          path_tokens, next_token, ws, ws_bytes))
        return s;
    if (medusa_status s = check_result_pointer(accept, who)) return s;
    if (k_cache) {
        if (medusa_status s = check_commit(who, dtype, k_cache, v_cache, prefix_len,
                                           new_prefix_len, H, dh))
            return s;
    }
    cudaError_t e = launch_posterior(dtype, logits, tokens, parent, depth, B, R, V, K, mode, eps,
                                     delta, temperature, accept_len, path, path_tokens, next_token,
                                     accept, k_cache, v_cache, prefix_len, H, dh, new_prefix_len,
                                     ws, stream, done);
    if (e) return cuda_fail(e, who);
    return MEDUSA_OK;
}

extern "C" {

medusa_status medusa_evaluate_posterior(medusa_dtype dtype, const void *logits,
                                        const int32_t *tokens, const int32_t *parent,
                                        const int32_t *depth, int B, int R, int V, int K,
                                        medusa_accept_mode mode, float eps, float delta,
                                        float temperature, int32_t *accept_len, int32_t *path,
                                        int32_t *path_tokens, int32_t *next_token,
                                        int32_t *accept, void *ws, size_t ws_bytes,
                                        medusa_stream stream) {
    const NvtxRange range("medusa_evaluate_posterior");
    return evaluate_posterior_signalled(dtype, logits, tokens, parent, depth, B, R, V, K, mode,
                                        eps, delta, temperature, accept_len, path, path_tokens,
                                        next_token, accept, nullptr, nullptr, nullptr, 0, 0,
                                        nullptr, ws, ws_bytes, static_cast<cudaStream_t>(stream),
                                        nullptr);
}

medusa_status medusa_evaluate_posterior_commit(
    medusa_dtype dtype, const void *logits, const int32_t *tokens, const int32_t *parent,
    const int32_t *depth, int B, int R, int V, int K, medusa_accept_mode mode, float eps,
    float delta, float temperature, int32_t *accept_len, int32_t *path, int32_t *path_tokens,
    int32_t *next_token, int32_t *accept, void *const *k_cache, void *const *v_cache,
    const int32_t *prefix_len, int H, int dh, int32_t *new_prefix_len, void *ws,
    size_t ws_bytes, medusa_stream stream) {
    const NvtxRange range("medusa_evaluate_posterior_commit");
    if (!k_cache)
        return fail(MEDUSA_ERR_INVALID_ARG, "medusa_evaluate_posterior_commit: NULL pointer");
    return evaluate_posterior_signalled(dtype, logits, tokens, parent, depth, B, R, V, K, mode,
                                        eps, delta, temperature, accept_len, path, path_tokens,
                                        next_token, accept, k_cache, v_cache, prefix_len, H, dh,
                                        new_prefix_len, ws, ws_bytes,
                                        static_cast<cudaStream_t>(stream), nullptr);
}

// ----------------------------------------------------------- speculative ---

size_t medusa_speculative_workspace_size(int B, int K) {
    if (B < 1 || K < 1) return 0;
    return speculative_workspace_bytes(B, K);
}

medusa_status medusa_speculative_posterior(medusa_dtype dtype, const void *logits,
                                           const int32_t *tokens, const float *draft_logits,
                                           int B, int V, int K, float temperature, uint64_t seed,
                                           uint64_t step, int32_t *accept_len,
                                           int32_t *path_tokens, int32_t *next_token,
                                           int32_t *accept, void *ws, size_t ws_bytes,
                                           medusa_stream stream) {
    const NvtxRange range("medusa_speculative_posterior");
    const char *who = "medusa_speculative_posterior";
    if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: unknown dtype %d", who, (int)dtype);
    if (!logits || !tokens || !draft_logits || !accept_len || !path_tokens || !next_token)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: NULL pointer", who);
    if (B < 1) return fail(MEDUSA_ERR_INVALID_ARG, "%s: B=%d", who, B);
    if (K < 1 || K > MEDUSA_MAX_HEADS)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: K=%d outside 1..%d", who, K, MEDUSA_MAX_HEADS);
    if (V < 1 || V % 8)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: V=%d must be a positive multiple of 8", who, V);
    if (!(temperature > 0.f) || !(temperature < 1e30f))
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: temperature must be positive and finite", who);
    if (medusa_status s = check_ws(ws, ws_bytes, speculative_workspace_bytes(B, K), who)) return s;
    cudaError_t e = launch_speculative(dtype, logits, tokens, draft_logits, B, V, K, temperature,
                                       seed, step, accept_len, path_tokens, next_token, accept, ws,
                                       static_cast<cudaStream_t>(stream));
    if (e) return cuda_fail(e, who);
    return MEDUSA_OK;
}

// ---------------------------------------------------------------- commit ---

medusa_status medusa_commit_kv(medusa_dtype dtype, void *const *k_cache, void *const *v_cache,
                               const int32_t *prefix_len, const int32_t *path,
                               const int32_t *accept_len, int B, int K, int R, int H, int dh,
                               int32_t *new_prefix_len, void *ws, size_t ws_bytes,
                               medusa_stream stream) {
    const NvtxRange range("medusa_commit_kv");
    const char *who = "medusa_commit_kv";
    if (medusa_status s = check_commit(who, dtype, k_cache, v_cache, prefix_len, new_prefix_len,
                                       H, dh))
        return s;
    if (!path || !accept_len) return fail(MEDUSA_ERR_INVALID_ARG, "%s: NULL pointer", who);
    if (B < 1) return fail(MEDUSA_ERR_INVALID_ARG, "%s: B=%d", who, B);
    if (K < 0 || K > MEDUSA_MAX_HEADS)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: K=%d outside 0..%d", who, K, MEDUSA_MAX_HEADS);
    if (R < 1 || R > MEDUSA_MAX_TREE_ROWS)
        return fail(MEDUSA_ERR_INVALID_ARG, "%s: R=%d outside 1..%d", who, R, MEDUSA_MAX_TREE_ROWS);
    if (medusa_status s = check_ws(ws, ws_bytes, MEDUSA_WS_HEADER, who)) return s;
    cudaError_t e = launch_commit_kv(dtype == MEDUSA_BF16 ? 2 : 4, k_cache, v_cache, prefix_len,
                                     path, accept_len, B, K, R, H, dh, new_prefix_len, ws,
                                     static_cast<cudaStream_t>(stream));
    if (e) return cuda_fail(e, who);
    return MEDUSA_OK;
}

}  // extern "C"
