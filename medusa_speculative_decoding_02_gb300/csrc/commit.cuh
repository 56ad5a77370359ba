// commit.cuh -- device side of the KV-cache commit, shared by the standalone
// commit kernel (commit.cu) and the posterior's select kernel (posterior.cu).
//
// "Medusa: Faster LLM text generation", Introduction, and "Medusa 深读" §5:
// the accepted prefix becomes the next context.  The tree nodes sit in cache
// slots P .. P+R-1; node path[q] of the accepted path moves to slot P+q.
//
// Each thread owns whole 16-byte column vectors of a cache row.  For each of
// its columns it loads the vector of every accepted path node into registers
// and only then stores them, so no other thread's loads can see a store:
// threads never share a column, and a column's sources are all read before
// any of its targets is written.  No barrier is needed.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace medusa {

struct CommitArgs {
    void *const *k_cache;     // [B] device pointers; nullptr = no commit
    void *const *v_cache;
    const int32_t *prefix_len;
    int32_t *new_prefix_len;
    int row_vecs;             // 16-byte vectors per cache row (H*dh*elt/16)
};

// The checks every commit applies before touching sequence b's cache.
// Returns the device status code (MEDUSA_DEV_OK when the commit may run).
__device__ __forceinline__ int commit_check(const void *kc, const void *vc, int P, const int *pth,
                                            int L, int K, int R) {
    if (!kc || !vc || ((reinterpret_cast<uintptr_t>(kc) | reinterpret_cast<uintptr_t>(vc)) & 15u))
        return MEDUSA_DEV_BAD_CACHE;
    if (P < 0) return MEDUSA_DEV_BAD_PREFIX;
    if (L < 0 || L > K || L > R - 1) return MEDUSA_DEV_BAD_PATH;
    for (int q = 0; q <= L; ++q)
        if (pth[q] < 0 || pth[q] >= R) return MEDUSA_DEV_BAD_PATH;
    return MEDUSA_DEV_OK;
}

// Move rows P+pth[q] -> P+q (q = 0..L) of both caches, for the columns
// c0, c0+stride, ... < row_vecs.  pth[] has been checked (commit_check).
// Rows with pth[q] == q are already in place and are skipped.  The K and V
// loads of a column are all issued before its first store.
__device__ __forceinline__ void commit_columns(void *kc, void *vc, int P, const int *pth, int L,
                                               int row_vecs, int c0, int stride) {
    uint4 *kb = static_cast<uint4 *>(kc);
    uint4 *vb = static_cast<uint4 *>(vc);
    for (int c = c0; c < row_vecs; c += stride) {
        uint4 kbuf[MEDUSA_MAX_HEADS + 1], vbuf[MEDUSA_MAX_HEADS + 1];
#pragma unroll
        for (int q = 0; q <= MEDUSA_MAX_HEADS; ++q)
            if (q <= L && pth[q] != q) {
                const size_t src = (size_t)(P + pth[q]) * row_vecs + c;
                kbuf[q] = kb[src];
                vbuf[q] = vb[src];
            }
#pragma unroll
        for (int q = 0; q <= MEDUSA_MAX_HEADS; ++q)
            if (q <= L && pth[q] != q) {
                const size_t dst = (size_t)(P + q) * row_vecs + c;
                kb[dst] = kbuf[q];
                vb[dst] = vbuf[q];
            }
    }
}

}  // namespace medusa
