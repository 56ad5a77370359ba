// commit.cu -- the standalone KV-cache commit (medusa_commit_kv).
//
// commit_kv_kernel: grid (column blocks, B), 128 threads.  Every CTA of
// sequence b reads the accepted path once into shared memory, applies the
// device checks (each CTA reaches the same decision; the first error code
// wins in the status word), and moves its share of the 16-byte columns with
// commit_columns.  Column block 0 writes new_prefix_len[b].
#include <algorithm>

#include "commit.cuh"
#include "launch.h"

namespace medusa {

namespace {

constexpr int kCommitThreads = 128;

__global__ void __launch_bounds__(kCommitThreads)
commit_kv_kernel(CommitArgs a, const int32_t *__restrict__ path,
                 const int32_t *__restrict__ accept_len, int K, int R, int *status) {
    pdl_enter();
    __shared__ int s_path[MEDUSA_MAX_HEADS + 1];
    __shared__ int s_code;
    const int b = blockIdx.y;
    const int tid = threadIdx.x;
    const int L = accept_len[b];
    const int P = a.prefix_len[b];
    void *kc = a.k_cache[b];
    void *vc = a.v_cache[b];
    if (tid <= K) s_path[tid] = path[(size_t)b * (K + 1) + tid];
    __syncthreads();
    if (tid == 0) {
        s_code = commit_check(kc, vc, P, s_path, L, K, R);
        if (s_code != MEDUSA_DEV_OK) set_status(status, s_code);
        if (blockIdx.x == 0) a.new_prefix_len[b] = s_code == MEDUSA_DEV_OK ? P + L + 1 : P;
    }
    __syncthreads();
    if (s_code != MEDUSA_DEV_OK) return;
    commit_columns(kc, vc, P, s_path, L, a.row_vecs, blockIdx.x * kCommitThreads + tid,
                   gridDim.x * kCommitThreads);
}

}  // namespace

cudaError_t launch_commit_kv(size_t elt, void *const *k_cache, void *const *v_cache,
                             const int32_t *prefix_len, const int32_t *path,
                             const int32_t *accept_len, int B, int K, int R, int H, int dh,
                             int32_t *new_prefix_len, void *ws, cudaStream_t stream) {
    CommitArgs a;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.prefix_len = prefix_len;
    a.new_prefix_len = new_prefix_len;
    a.row_vecs = (int)((size_t)H * dh * elt / 16);
    const int cx = std::max(1, std::min(64, (a.row_vecs + kCommitThreads - 1) / kCommitThreads));
    cudaError_t e = launch_pdl(commit_kv_kernel, dim3(cx, B), dim3(kCommitThreads), 0, stream, a,
                               path, accept_len, K, R, static_cast<int *>(ws));
    note_launch();
    return e;
}

}  // namespace medusa
