// topk.cuh -- warp-level running top-s lists and (max, sum-exp) pairs, used
// by the heads kernels (CUDA-core and tensor-core paths) to keep each head's
// best tokens and its softmax normaliser while the logits stream past.
#pragma once

#include <climits>

#include "common.cuh"

namespace medusa {

// Warp-resident running state for one (head, sequence): online softmax pair
// (identical in every lane) and a top-s list sorted best-first, entry i held
// by lane i (lanes >= S hold nothing).
struct WarpTop {
    float m, s;
    float val;
    int id;
    __device__ __forceinline__ void reset() {
        m = -INFINITY;
        s = 0.f;
        val = -INFINITY;
        id = INT_MAX;
    }
    // fold one logit (value cv of token cid), same in all lanes
    __device__ __forceinline__ void push(float cv, int cid, int S, int lane) {
        if (cv > m) {
            s = s * expf(m - cv) + 1.f;
            m = cv;
        } else {
            s += expf(cv - m);
        }
        insert(cv, cid, S, lane);
    }
    __device__ __forceinline__ void insert(float cv, int cid, int S, int lane) {
        const float wv = __shfl_sync(0xffffffffu, val, S - 1);
        const int wi = __shfl_sync(0xffffffffu, id, S - 1);
        if (!better(cv, cid, wv, wi)) return;  // warp-uniform
        const bool worse = lane < S && better(cv, cid, val, id);
        const unsigned mask = __ballot_sync(0xffffffffu, worse);
        const int pos = __ffs(mask) - 1;
        const float up_v = __shfl_up_sync(0xffffffffu, val, 1);
        const int up_i = __shfl_up_sync(0xffffffffu, id, 1);
        if (lane == pos) {
            val = cv;
            id = cid;
        } else if (lane > pos && lane < S) {
            val = up_v;
            id = up_i;
        }
    }
    // sampling: fold y = logit / T into (m, s), rank by the perturbed key
    __device__ __forceinline__ void push_key(float y, float key, int cid, int S, int lane) {
        if (y > m) {
            s = s * expf(m - y) + 1.f;
            m = y;
        } else {
            s += expf(y - m);
        }
        insert(key, cid, S, lane);
    }
    // merge another (m, s) pair
    __device__ __forceinline__ void merge_ms(float om, float os) {
        if (om == -INFINITY) return;
        if (om > m) {
            s = s * expf(m - om) + os;
            m = om;
        } else {
            s += os * expf(om - m);
        }
    }
};

// Per-warp flushed state in shared memory.
struct TopSlot {
    float m, s;
    float val[MEDUSA_MAX_TOP_S];
    int id[MEDUSA_MAX_TOP_S];
};

__device__ __forceinline__ void flush_slot(TopSlot &slot, const WarpTop &st, int S, int lane) {
    if (lane < S) {
        slot.val[lane] = st.val;
        slot.id[lane] = st.id;
    }
    if (lane == 0) {
        slot.m = st.m;
        slot.s = st.s;
    }
}

// (max, sum-exp) of nslot slots, merged by one warp; valid in every lane.
__device__ __forceinline__ void warp_merge_ms(const TopSlot *slots, int stride, int nslot,
                                              int lane, float &m, float &s) {
    WarpTop t;
    t.reset();
    for (int w = lane; w < nslot; w += kWarp) t.merge_ms(slots[w * stride].m, slots[w * stride].s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, t.m, o);
        const float os = __shfl_xor_sync(0xffffffffu, t.s, o);
        t.merge_ms(om, os);
    }
    m = t.m;
    s = t.s;
}

// compare-exchange so that (va, ia) ends up the better of the two
__device__ __forceinline__ void cx(float &va, int &ia, float &vb, int &ib) {
    if (better(vb, ib, va, ia)) {
        const float tv = va; va = vb; vb = tv;
        const int ti = ia; ia = ib; ib = ti;
    }
}

// Warp top-S selection over up to 32*U candidates plus the warp's running
// list (lanes < S): every lane sorts its own few candidates in registers, then
// S rounds each take the best lane head by a five-step shuffle argmax and pop
// it.  The result is left sorted best-first in lanes 0..S-1 (val, id).
template <int U>
__device__ __forceinline__ void warp_select_top(float (&cv)[U + 1], int (&ci)[U + 1], int S,
                                                int lane, float &val, int &id) {
    // sort the lane's U+1 entries best-first (odd-even transposition)
#pragma unroll
    for (int r = 0; r < U + 1; ++r)
#pragma unroll
        for (int e = (r & 1); e + 1 < U + 1; e += 2) cx(cv[e], ci[e], cv[e + 1], ci[e + 1]);
    float nv = -INFINITY;
    int ni = INT_MAX;
    for (int k = 0; k < S; ++k) {
        float bv = cv[0];
        int bi = ci[0];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (better(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (lane == k) {
            nv = bv;
            ni = bi;
        }
        if (bi != INT_MAX && ci[0] == bi) {  // this lane's head won: pop it
#pragma unroll
            for (int e = 0; e < U; ++e) {
                cv[e] = cv[e + 1];
                ci[e] = ci[e + 1];
            }
            cv[U] = -INFINITY;
            ci[U] = INT_MAX;
        }
    }
    val = nv;
    id = ni;
}

// Top-S of nslot best-first lists (list w at slots[w * stride], S entries
// each, empty entries at the tail) by one warp: groups of 64 candidates (two
// per lane) join the warp's running list in warp_select_top.  The result is
// sorted best-first in lanes 0..S-1.
__device__ __forceinline__ void warp_merge_top(const TopSlot *slots, int stride, int nslot, int S,
                                               int lane, float &val, int &id) {
    constexpr int U = 2;
    const int n = nslot * S;
    val = -INFINITY;
    id = INT_MAX;
    for (int c0 = 0; c0 < n; c0 += kWarp * U) {
        float cv[U + 1];
        int ci[U + 1];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + u * kWarp + lane;
            if (c < n) {
                const int w = c / S, j = c - w * S;
                cv[u] = slots[w * stride].val[j];
                ci[u] = slots[w * stride].id[j];
            } else {
                cv[u] = -INFINITY;
                ci[u] = INT_MAX;
            }
        }
        cv[U] = lane < S ? val : -INFINITY;  // the running list joins the pool
        ci[U] = lane < S ? id : INT_MAX;
        warp_select_top<U>(cv, ci, S, lane, val, id);
    }
}

}  // namespace medusa
