// launch.h -- internal interface between the C ABI layer (api.cu) and the
// kernel files.  Each launch_* enqueues its kernels on `stream` and returns
// the first CUDA error; arguments were validated by the caller.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "medusa.h"

namespace medusa {

// Launch `kernel` on `stream` with programmatic stream serialization, so that
// its launch may overlap the tail of the previous kernel in the stream (the
// kernel itself calls pdl_enter() before touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// NVTX range around one public call (visible in Nsight timelines; free
// when no tool is attached)
struct NvtxRange {
    explicit NvtxRange(const char *name);
    ~NvtxRange();
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

// poll limit of the bounded device waits inside the main loops (see
// medusa_set_wait_budget); the drain before a kernel frees its resources
// keeps its own fixed limit
uint32_t wait_budget();

int device_sm_count();   // SMs of the current device (cached per device)
void note_launch();      // count one kernel launch
void set_last_error(const char *fmt, ...);  // message for medusa_last_error()

// Sampling mode of the heads pass: each head draws one token from
// softmax(logits * inv_T) by Gumbel-max (random stream: purpose 1, row =
// head, key = (seed, step)); the raw logits go to logits_out [B,K,V] when it
// is not null.
struct SampleArgs {
    int on;
    float inv_T;
    uint64_t seed, step;
    float *logits_out;
};

// Wlm == nullptr: the Medusa heads alone; otherwise the LM head joins the
// pass and writes root / root_logp.  sample == nullptr: top-s mode.
size_t heads_workspace_bytes(int B, int K, int d, int V, int S, bool with_lm_head = false);
cudaError_t launch_heads(medusa_dtype dtype, const void *h, const void *Wlm, const void *W1,
                         const void *b1, const void *W2, int B, int d, int V, int K, int S,
                         int32_t *ids, float *logp, int32_t *root, float *root_logp,
                         const SampleArgs *sample, void *ws, cudaStream_t stream);

size_t tree_workspace_bytes(int B, int K, int S, int n);
// shared_table: logp is one [K, S] table used by every sequence (a calibrated
// tree), otherwise [B, K, S].
cudaError_t launch_build_tree(const int32_t *root, const int32_t *ids, const float *logp,
                              bool shared_table, int B, int K, const int32_t *s_host, int S, int n,
                              const int32_t *prefix_len, int32_t *tokens, int32_t *parent,
                              int32_t *depth, int32_t *pos_id, uint64_t *anc_mask, int32_t *paths,
                              int32_t *n_leaf, void *ws, cudaStream_t stream);

size_t attention_workspace_bytes(medusa_dtype dtype, int B, int R, int H, int dh, int P_max);
cudaError_t launch_tree_attention(medusa_dtype dtype, const void *q, const void *const *k_cache,
                                  const void *const *v_cache, const int32_t *prefix_len,
                                  int P_max, const uint64_t *anc_mask, int B, int R, int H,
                                  int dh, float scale, void *out, void *ws, cudaStream_t stream);

size_t speculative_workspace_bytes(int B, int K);
cudaError_t launch_speculative(medusa_dtype dtype, const void *logits, const int32_t *tokens,
                               const float *draft_logits, int B, int V, int K, float temperature,
                               uint64_t seed, uint64_t step, int32_t *accept_len,
                               int32_t *path_tokens, int32_t *next_token, int32_t *accept,
                               void *ws, cudaStream_t stream);

size_t posterior_workspace_bytes(int B, int R);
cudaError_t launch_posterior(medusa_dtype dtype, const void *logits, const int32_t *tokens,
                             const int32_t *parent, const int32_t *depth, int B, int R, int V,
                             int K, medusa_accept_mode mode, float eps, float delta,
                             float temperature, int32_t *accept_len, int32_t *path,
                             int32_t *path_tokens, int32_t *next_token, int32_t *accept,
                             void *const *k_cache, void *const *v_cache,
                             const int32_t *prefix_len, int H, int dh, int32_t *new_prefix_len,
                             void *ws, cudaStream_t stream, uint32_t *done = nullptr);

// The posterior entry of the step executor: the checks of
// medusa_evaluate_posterior (and, with k_cache, of the commit), then the
// launch with `done` (page-locked host memory, [B] words, or null): each
// sequence's word gains one when its results (and commit) are written.
medusa_status evaluate_posterior_signalled(
    medusa_dtype dtype, const void *logits, const int32_t *tokens, const int32_t *parent,
    const int32_t *depth, int B, int R, int V, int K, medusa_accept_mode mode, float eps,
    float delta, float temperature, int32_t *accept_len, int32_t *path, int32_t *path_tokens,
    int32_t *next_token, int32_t *accept, void *const *k_cache, void *const *v_cache,
    const int32_t *prefix_len, int H, int dh, int32_t *new_prefix_len, void *ws,
    size_t ws_bytes, cudaStream_t stream, uint32_t *done);

// k_cache == nullptr in launch_posterior: no commit.  elt = bytes per element.
cudaError_t launch_commit_kv(size_t elt, void *const *k_cache, void *const *v_cache,
                             const int32_t *prefix_len, const int32_t *path,
                             const int32_t *accept_len, int B, int K, int R, int H, int dh,
                             int32_t *new_prefix_len, void *ws, cudaStream_t stream);

}  // namespace medusa
