// noalloc.cu -- medusa_heads without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they run the heads: a
// serving runtime that hands all free HBM to its KV-cache pool at start-up
// (a later cudaMalloc fails, or takes memory the cache owns), or a decode loop
// that cannot afford cudaMalloc/cudaFree, which synchronise the whole device.
// This entry point gives them the heads with their scratch held in a
// file-scope device array of fixed size instead.
//
// The array is reserved on every GPU that loads the library and stays there
// until the process exits.  All calls share it and it keeps the previous
// call's contents; the heads kernels overwrite every scratch byte before they
// read it, so nothing has to be cleared between calls.  Two calls whose work
// overlaps on the GPU (different streams, or different host threads on one
// device) race on the array: serialise them.
#include <mutex>

#include "launch.h"

namespace medusa {

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB

__device__ __align__(256) unsigned char g_heads_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_heads_scratch on the current device, looked up once per
// device.  In host code the symbol name is only a host-side stand-in, so the
// address must come from cudaGetSymbolAddress.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_heads_scratch);
        if (e) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

}  // namespace medusa

using namespace medusa;

extern "C" medusa_status medusa_heads_noalloc(medusa_dtype dtype, const void *h, const void *W1,
                                              const void *b1, const void *W2, int B, int d, int V,
                                              int K, int top_s, int32_t *topk_ids,
                                              float *topk_logp, medusa_stream stream) {
    const NvtxRange range("medusa_heads_noalloc");
    if (B >= 1 && K >= 1 && d >= 1 && V >= 1 && top_s >= 1) {
        const size_t need = heads_workspace_bytes(B, K, d, V, top_s);
        if (need > kStaticScratchBytes) {
            set_last_error("medusa_heads_noalloc: this shape needs %zu bytes of scratch; the "
                           "static scratch holds %zu bytes (use medusa_heads with a workspace)",
                           need, kStaticScratchBytes);
            return MEDUSA_ERR_UNSUPPORTED;
        }
    }
    void *ws = nullptr;
    cudaError_t e = scratch_address(&ws);
    if (e) {
        set_last_error("medusa_heads_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        return MEDUSA_ERR_CUDA;
    }
    return medusa_heads(dtype, h, W1, b1, W2, B, d, V, K, top_s, topk_ids, topk_logp, ws,
                        kStaticScratchBytes, stream);
}
