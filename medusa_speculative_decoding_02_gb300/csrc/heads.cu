// heads.cu -- Medusa heads on sm_103a.
//
// Computes, for every sequence b and head k ("Medusa 深读" §3.1, the equation
// for p_t^(k); "Medusa Part I" Part 3, ResidualBlock and the bias-free
// vocabulary projection):
//     u = W1[k] h[b] + b1[k];  z = h[b] + SiLU(u);  logits = W2[k] z
// and keeps the top-s tokens of softmax(logits) ("Medusa 深读" §6.1).
//
// At batch 1 this is a pair of GEMVs: every weight byte is used once, so the
// kernels are HBM-bound and run on CUDA cores.  Design:
//   phase 1  heads_w1_kernel   one warp per output row of W1 (all heads),
//                              16-byte streaming loads, fp32 accumulation,
//                              residual SiLU fused; z kept in fp32 scratch.
//   phase 2  heads_w2_kernel   persistent grid; each CTA streams an equal
//                              slice of every head's W2 rows.  Per row a warp
//                              forms the logit(s), then folds it into a running
//                              (max, sum-exp) pair and a sorted top-s list held
//                              one entry per lane.  The logits never reach HBM:
//                              each CTA writes only its (max, sum, top-s)
//                              partial per (head, sequence).
//   phase 3  heads_reduce_kernel merges the partials of each (head, sequence)
//                              into log Z and the final top-s log-probs.
// z and h sit in shared memory in a split-plane layout (elements 0-3 and 4-7
// of each 8-element vector in separate planes) so that a warp's 16-byte
// shared loads are bank-conflict free.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "launch.h"

namespace medusa {

namespace {

constexpr int kW1Threads = 256;
constexpr int kW2Threads = 512;
constexpr int kW2Warps = kW2Threads / kWarp;
constexpr int kReduceThreads = 256;

// Index (in floats) of element c of vector row b in the split-plane layout.
template <int VN>
__device__ __forceinline__ int plane_index(int b, int c, int nvec) {
    constexpr int NPL = VN / 4;
    const int idx = c / VN;
    const int p = (c % VN) / 4;
    return ((b * NPL + p) * nvec + idx) * 4 + (c & 3);
}

// dot of one 16-byte weight vector with the matching activation elements of
// NB rows stored in split planes.
template <typename T, int NB>
__device__ __forceinline__ void fma_vec(const uint4 &w, const float4 *__restrict__ act, int idx,
                                        int nvec, float (&acc)[NB]) {
    constexpr int VN = Vec16<T>::N;
    constexpr int NPL = VN / 4;
    float f[VN];
    Vec16<T>::widen(w, f);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
#pragma unroll
        for (int p = 0; p < NPL; ++p) {
            const float4 a = act[(b * NPL + p) * nvec + idx];
            acc[b] = fmaf(f[p * 4 + 0], a.x, acc[b]);
            acc[b] = fmaf(f[p * 4 + 1], a.y, acc[b]);
            acc[b] = fmaf(f[p * 4 + 2], a.z, acc[b]);
            acc[b] = fmaf(f[p * 4 + 3], a.w, acc[b]);
        }
    }
}

// Dot products of one weight row (nvec 16-byte vectors) with NB activation
// rows; result replicated in every lane.
template <typename T, int NB, int U>
__device__ __forceinline__ void row_dot(const uint4 *__restrict__ w, const float4 *__restrict__ act,
                                        int nvec, int lane, float (&acc)[NB]) {
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.f;
    for (int base = lane; base < nvec; base += kWarp * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int idx = base + u * kWarp;
            if (idx < nvec) v[u] = ld_stream16(w + idx);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int idx = base + u * kWarp;
            if (idx < nvec) fma_vec<T, NB>(v[u], act, idx, nvec, acc);
        }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = warp_sum(acc[b]);
}

// ------------------------------------------------------------- phase 1 ---

template <typename T, int NB, int U>
__global__ void __launch_bounds__(kW1Threads)
heads_w1_kernel(const T *__restrict__ h, const T *__restrict__ W1, const T *__restrict__ b1,
                float *__restrict__ z, int B, int d, int K) {
    extern __shared__ float4 smem4[];
    float *hs = reinterpret_cast<float *>(smem4);
    constexpr int VN = Vec16<T>::N;
    const int nvec = d / VN;
    for (int i = threadIdx.x; i < NB * d; i += blockDim.x) {
        const int b = i / d, c = i - b * d;
        hs[plane_index<VN>(b, c, nvec)] = (b < B) ? Vec16<T>::load1(h + (size_t)b * d + c) : 0.f;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int rows = K * d;
    for (int row = blockIdx.x * nwarps + warp; row < rows; row += gridDim.x * nwarps) {
        float acc[NB];
        row_dot<T, NB, U>(reinterpret_cast<const uint4 *>(W1 + (size_t)row * d), smem4, nvec, lane,
                          acc);
        if (lane < B) {
            float a = 0.f;
#pragma unroll
            for (int b = 0; b < NB; ++b)
                if (b == lane) a = acc[b];
            const int k = row / d, j = row - k * d;
            const float u = a + (b1 ? Vec16<T>::load1(b1 + row) : 0.f);
            const float silu = u / (1.f + expf(-u));
            z[((size_t)k * B + lane) * d + j] = hs[plane_index<VN>(lane, j, nvec)] + silu;
        }
    }
}

// ------------------------------------------------------------- phase 2 ---

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

// merge a sorted list (best first) into the warp state; stops at the first
// entry that cannot enter
__device__ __forceinline__ void merge_list(WarpTop &st, const float *val, const int *id, int S,
                                           int lane) {
    for (int j = 0; j < S; ++j) {
        const float cv = val[j];
        const int ci = id[j];
        if (ci == INT_MAX) break;
        const float wv = __shfl_sync(0xffffffffu, st.val, S - 1);
        const int wi = __shfl_sync(0xffffffffu, st.id, S - 1);
        if (!better(cv, ci, wv, wi)) break;
        st.insert(cv, ci, S, lane);
    }
}

template <typename T, int NB, int U>
__global__ void __launch_bounds__(kW2Threads, NB <= 1 ? 2 : 1)
heads_w2_kernel(const float *__restrict__ z, const T *__restrict__ W2, int B, int d, int V, int K,
                int S, int hpg, float2 *__restrict__ part_ms, float *__restrict__ part_val,
                int *__restrict__ part_id) {
    extern __shared__ float4 smem4[];
    constexpr int VN = Vec16<T>::N;
    const int nvec = d / VN;
    float4 *zs4 = smem4;                                     // [hpg][NB][planes][nvec]
    float *zs = reinterpret_cast<float *>(smem4);
    TopSlot *slots = reinterpret_cast<TopSlot *>(zs + (size_t)hpg * NB * d);  // [warps][hpg][NB]
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int G = gridDim.x;
    const int g = blockIdx.x;
    const int r0 = (int)(((long long)g * V) / G);
    const int r1 = (int)(((long long)(g + 1) * V) / G);
    const int nrows = r1 - r0;

    for (int k0 = 0; k0 < K; k0 += hpg) {
        const int hk = min(hpg, K - k0);
        // stage z for heads k0 .. k0+hk-1 (zero rows for b >= B)
        for (int i = threadIdx.x; i < hk * NB * d; i += blockDim.x) {
            const int kk = i / (NB * d);
            const int rem = i - kk * NB * d;
            const int b = rem / d, c = rem - b * d;
            zs[(size_t)kk * NB * d + plane_index<VN>(b, c, nvec)] =
                (b < B) ? z[((size_t)(k0 + kk) * B + b) * d + c] : 0.f;
        }
        __syncthreads();

        WarpTop st[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) st[b].reset();
        int cur = 0;
        const int items = hk * nrows;
        for (int it = warp; it < items; it += kW2Warps) {
            const int kk = it / nrows;
            const int v = r0 + (it - kk * nrows);
            while (cur < kk) {
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    flush_slot(slots[(warp * hpg + cur) * NB + b], st[b], S, lane);
                    st[b].reset();
                }
                ++cur;
            }
            float acc[NB];
            const T *wrow = W2 + ((size_t)(k0 + kk) * V + v) * d;
            row_dot<T, NB, U>(reinterpret_cast<const uint4 *>(wrow), zs4 + (size_t)kk * NB * d / 4,
                              nvec, lane, acc);
#pragma unroll
            for (int b = 0; b < NB; ++b)
                if (b < B) st[b].push(acc[b], v, S, lane);
        }
        while (cur < hk) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                flush_slot(slots[(warp * hpg + cur) * NB + b], st[b], S, lane);
                st[b].reset();
            }
            ++cur;
        }
        __syncthreads();

        // merge the warps' states: one warp per (head, sequence)
        for (int pair = warp; pair < hk * B; pair += kW2Warps) {
            const int kk = pair / B, b = pair - kk * B;
            WarpTop acc;
            acc.reset();
            for (int w = 0; w < kW2Warps; ++w) {
                const TopSlot &sl = slots[(w * hpg + kk) * NB + b];
                acc.merge_ms(sl.m, sl.s);
                merge_list(acc, sl.val, sl.id, S, lane);
            }
            const size_t o = ((size_t)(k0 + kk) * B + b) * G + g;
            if (lane == 0) part_ms[o] = make_float2(acc.m, acc.s);
            if (lane < S) {
                part_val[o * S + lane] = acc.val;
                part_id[o * S + lane] = acc.id;
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------- phase 3 ---

__global__ void __launch_bounds__(kReduceThreads)
heads_reduce_kernel(const float2 *__restrict__ part_ms, const float *__restrict__ part_val,
                    const int *__restrict__ part_id, int G, int B, int K, int S,
                    int32_t *__restrict__ topk_ids, float *__restrict__ topk_logp) {
    __shared__ TopSlot slots[kReduceThreads / kWarp];
    const int kb = blockIdx.x;  // k * B + b
    const int k = kb / B, b = kb - k * B;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    WarpTop st;
    st.reset();
    for (int g = warp; g < G; g += nwarps) {
        const size_t o = (size_t)kb * G + g;
        const float2 ms = part_ms[o];
        st.merge_ms(ms.x, ms.y);
        merge_list(st, part_val + o * S, part_id + o * S, S, lane);
    }
    flush_slot(slots[warp], st, S, lane);
    __syncthreads();
    if (warp == 0) {
        WarpTop acc;
        acc.reset();
        for (int w = 0; w < nwarps; ++w) {
            acc.merge_ms(slots[w].m, slots[w].s);
            merge_list(acc, slots[w].val, slots[w].id, S, lane);
        }
        const float logz = acc.m + logf(acc.s);
        if (lane < S) {
            const size_t o = ((size_t)b * K + k) * S + lane;
            topk_ids[o] = acc.id;
            topk_logp[o] = acc.val - logz;
        }
    }
}

// ---------------------------------------------------------------- host ---

constexpr int kMaxW2Ctas = 1024;
constexpr size_t kSmemBudget = 200 * 1024;

int nb_bucket(int B) { return B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : 8; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct HeadsLayout {
    size_t z_off, ms_off, val_off, id_off, total;
};

HeadsLayout heads_layout(int B, int K, int d, int S) {
    HeadsLayout L;
    size_t o = MEDUSA_WS_HEADER;
    L.z_off = o;
    o = align256(o + (size_t)K * B * d * sizeof(float));
    L.ms_off = o;
    o = align256(o + (size_t)K * B * kMaxW2Ctas * sizeof(float2));
    L.val_off = o;
    o = align256(o + (size_t)K * B * kMaxW2Ctas * S * sizeof(float));
    L.id_off = o;
    o = align256(o + (size_t)K * B * kMaxW2Ctas * S * sizeof(int));
    L.total = o;
    return L;
}

template <typename T, int NB>
cudaError_t run_heads(const void *h, const void *W1, const void *b1, const void *W2, int B, int d,
                      int V, int K, int S, int32_t *ids, float *logp, char *ws,
                      cudaStream_t stream) {
    constexpr int U1 = NB <= 4 ? 8 : 4;
    constexpr int U2 = NB <= 4 ? 8 : 4;
    const HeadsLayout L = heads_layout(B, K, d, S);
    float *z = reinterpret_cast<float *>(ws + L.z_off);
    float2 *pms = reinterpret_cast<float2 *>(ws + L.ms_off);
    float *pval = reinterpret_cast<float *>(ws + L.val_off);
    int *pid = reinterpret_cast<int *>(ws + L.id_off);
    const int sms = device_sm_count();
    cudaError_t e;

    // phase 1
    auto k1 = heads_w1_kernel<T, NB, U1>;
    const size_t smem1 = (size_t)NB * d * sizeof(float);
    if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1)))
        return e;
    int occ1 = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ1, k1, kW1Threads, smem1))) return e;
    const int rows1 = K * d;
    const int grid1 = std::max(1, std::min(sms * std::max(occ1, 1), (rows1 + 7) / 8));
    k1<<<grid1, kW1Threads, smem1, stream>>>(static_cast<const T *>(h), static_cast<const T *>(W1),
                                             static_cast<const T *>(b1), z, B, d, K);
    note_launch();
    if ((e = cudaGetLastError())) return e;

    // phase 2
    const size_t per_head = (size_t)NB * d * sizeof(float);
    const size_t slot_per_head = (size_t)kW2Warps * NB * sizeof(TopSlot);
    int hpg = (int)std::min<size_t>(K, std::max<size_t>(1, kSmemBudget / (per_head + slot_per_head)));
    const size_t smem2 = hpg * (per_head + slot_per_head);
    auto k2 = heads_w2_kernel<T, NB, U2>;
    if ((e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2)))
        return e;
    int occ2 = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ2, k2, kW2Threads, smem2))) return e;
    const int G = std::max(1, std::min(kMaxW2Ctas, sms * std::max(occ2, 1)));
    k2<<<G, kW2Threads, smem2, stream>>>(z, static_cast<const T *>(W2), B, d, V, K, S, hpg, pms,
                                         pval, pid);
    note_launch();
    if ((e = cudaGetLastError())) return e;

    // phase 3
    heads_reduce_kernel<<<K * B, kReduceThreads, 0, stream>>>(pms, pval, pid, G, B, K, S, ids, logp);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

size_t heads_workspace_bytes(int B, int K, int d, int V, int S) {
    (void)V;
    return heads_layout(B, K, d, S).total;
}

cudaError_t launch_heads(medusa_dtype dtype, const void *h, const void *W1, const void *b1,
                         const void *W2, int B, int d, int V, int K, int S, int32_t *ids,
                         float *logp, void *ws, cudaStream_t stream) {
    char *w = static_cast<char *>(ws);
    const int nb = nb_bucket(B);
#define MEDUSA_HEADS_CASE(T, N) \
    if (nb == N) return run_heads<T, N>(h, W1, b1, W2, B, d, V, K, S, ids, logp, w, stream);
    if (dtype == MEDUSA_BF16) {
        MEDUSA_HEADS_CASE(bf16, 1)
        MEDUSA_HEADS_CASE(bf16, 2)
        MEDUSA_HEADS_CASE(bf16, 4)
        MEDUSA_HEADS_CASE(bf16, 8)
    } else {
        MEDUSA_HEADS_CASE(float, 1)
        MEDUSA_HEADS_CASE(float, 2)
        MEDUSA_HEADS_CASE(float, 4)
        MEDUSA_HEADS_CASE(float, 8)
    }
#undef MEDUSA_HEADS_CASE
    return cudaErrorInvalidValue;
}

}  // namespace medusa
