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
//   phase 1  heads_w1_kernel   one full wave of warps, each streaming a
//                              contiguous share of W1's rows (all heads) with
//                              16-byte loads, fp32 accumulation, residual
//                              SiLU fused; z kept in fp32 scratch.
//   phase 2  heads_w2_kernel   persistent grid; each CTA streams an equal
//                              slice of every head's W2 rows.  Per row a warp
//                              forms the logit(s), then folds it into a running
//                              (max, sum-exp) pair and a sorted top-s list held
//                              one entry per lane.  The logits never reach HBM:
//                              each CTA writes only its (max, sum, top-s)
//                              partial per (head, sequence).
//   phase 3  heads_reduce_kernel merges the partials of each (head, sequence)
//                              into log Z and the final top-s log-probs.
// With the base model's LM head W_lm given (medusa_heads_lm), it joins the
// pass as head 0 with z = h: its rows stream in the same phase-2 grid as the
// Medusa heads' W2 rows, and phase 3 emits its greedy token (the tree root)
// and that token's log-probability.
// z and h sit in shared memory in a split-plane layout (elements 0-3 and 4-7
// of each 8-element vector in separate planes) so that a warp's 16-byte
// shared loads are bank-conflict free.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "heads_tc.h"
#include "launch.h"
#include "philox.cuh"
#include "topk.cuh"

namespace medusa {

namespace {

constexpr int kW1Threads = 256;
constexpr int kW2Threads = 512;
constexpr int kW2Warps = kW2Threads / kWarp;
constexpr int kReduceThreads = 512;

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
// rows from vector `base` on, added to acc.
template <typename T, int NB, int U>
__device__ __forceinline__ void row_dot_tail(const uint4 *__restrict__ w,
                                             const float4 *__restrict__ act, int nvec, int base,
                                             float (&acc)[NB]) {
    for (; base < nvec; base += kWarp * U) {
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
}

// Dot products of one weight row with NB activation rows; result replicated
// in every lane.
template <typename T, int NB, int U>
__device__ __forceinline__ void row_dot(const uint4 *__restrict__ w, const float4 *__restrict__ act,
                                        int nvec, int lane, float (&acc)[NB]) {
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.f;
    row_dot_tail<T, NB, U>(w, act, nvec, lane, acc);
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = warp_sum(acc[b]);
}

// Stage NB activation rows of d elements (src row b at src + b * stride,
// rows >= B zero) into shared memory in the split-plane layout, one 16-byte
// load per vector of VN elements.
template <typename S, int VN, int NB>
__device__ __forceinline__ void stage_planes(const S *__restrict__ src, size_t stride, int B,
                                             int d, float4 *__restrict__ dst) {
    constexpr int NPL = VN / 4;
    constexpr int SN = 16 / sizeof(S);  // source elements per 16-byte load
    const int nvec = d / VN;
    const int nsv = d / SN;
    for (int i = threadIdx.x; i < NB * nsv; i += blockDim.x) {
        const int b = i / nsv, sv = i - b * nsv;
        float f[SN];
        if (b < B) {
            const uint4 w = *reinterpret_cast<const uint4 *>(src + b * stride + (size_t)sv * SN);
            Vec16<S>::widen(w, f);
        } else {
#pragma unroll
            for (int e = 0; e < SN; ++e) f[e] = 0.f;
        }
        // elements sv*SN .. sv*SN+SN-1: SN/4 groups of four, each one float4
#pragma unroll
        for (int g = 0; g < SN / 4; ++g) {
            const int c = sv * SN + 4 * g;
            const int p = (c % VN) / 4, idx = c / VN;
            dst[(b * NPL + p) * nvec + idx] =
                make_float4(f[4 * g], f[4 * g + 1], f[4 * g + 2], f[4 * g + 3]);
        }
    }
}

// ------------------------------------------------------------- phase 1 ---

template <typename T, int NB, int U>
__global__ void __launch_bounds__(kW1Threads, NB == 1 ? 6 : (NB <= 2 ? 4 : 1))
heads_w1_kernel(const T *__restrict__ h, const T *__restrict__ W1, const T *__restrict__ b1,
                float *__restrict__ z, float *__restrict__ z_lm, int B, int d, int K,
                int total_warps) {
    {
        // The weights are never written by any kernel, so each warp pulls its
        // first two rows into L2 before the wait for the previous kernel
        const int gw0 = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
        const int rows0 = K * d;
        const int rb = (int)(((long long)gw0 * rows0) / total_warps);
        const int re = min((int)(((long long)(gw0 + 1) * rows0) / total_warps), rb + 2);
        if ((threadIdx.x & 31) == 0 && re > rb)
            prefetch_l2_bulk(W1 + (size_t)rb * d, (unsigned)((re - rb) * d * sizeof(T)));
    }
    pdl_enter();
    extern __shared__ float4 smem4[];
    float *hs = reinterpret_cast<float *>(smem4);
    constexpr int VN = Vec16<T>::N;
    const int nvec = d / VN;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int rows = K * d;
    // the grid fills every resident warp slot once, and warp gw owns rows
    // [gw*rows/total, (gw+1)*rows/total): shares differ by at most one row, so
    // every SM streams the same number of bytes
    const int gw = blockIdx.x * nwarps + warp;
    const int r_begin = (int)(((long long)gw * rows) / total_warps);
    const int r_end = (int)(((long long)(gw + 1) * rows) / total_warps);
    stage_planes<T, VN, NB>(h, (size_t)d, B, d, smem4);
    if (z_lm)  // the LM head's z is h itself (no residual block)
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < B * d; i += gridDim.x * blockDim.x)
            z_lm[i] = Vec16<T>::load1(h + i);
    __syncthreads();
    // the biases of the warp's rows, 32 at a time (lane i holds the bias of
    // the chunk's row i), fetched before the chunk's first row: no row waits
    // on a bias load of its own
    float bias_l = 0.f;
    for (int row = r_begin; row < r_end; ++row) {
        const int ri = (row - r_begin) & (kWarp - 1);
        if (ri == 0) bias_l = (b1 && row + lane < r_end) ? Vec16<T>::load1(b1 + row + lane) : 0.f;
        float acc[NB];
        const uint4 *wrow = reinterpret_cast<const uint4 *>(W1 + (size_t)row * d);
        row_dot<T, NB, U>(wrow, smem4, nvec, lane, acc);
        const float bias = __shfl_sync(0xffffffffu, bias_l, ri);
        if (lane < B) {
            float a = 0.f;
#pragma unroll
            for (int b = 0; b < NB; ++b)
                if (b == lane) a = acc[b];
            const int k = row / d, j = row - k * d;
            const float u = a + bias;
            const float silu = u / (1.f + expf(-u));
            z[((size_t)k * B + lane) * d + j] = hs[plane_index<VN>(lane, j, nvec)] + silu;
        }
    }
}

// ------------------------------------------------------------- phase 2 ---

// Row v of head k's vocabulary projection: with the LM head present it is
// head 0 and the Medusa heads follow.
template <typename T>
__device__ __forceinline__ const T *w2_row(const T *W2, const T *Wlm, int k, int v, int V, int d) {
    if (Wlm) {
        if (k == 0) return Wlm + (size_t)v * d;
        --k;
    }
    return W2 + ((size_t)k * V + v) * d;
}

template <typename T, int NB, int U, bool SAMPLE>
__global__ void __launch_bounds__(kW2Threads, NB <= 1 ? 2 : 1)
heads_w2_kernel(const float *__restrict__ z, const T *__restrict__ W2, const T *__restrict__ Wlm,
                int B, int d, int V, int K, int S, int hpg, float2 *__restrict__ part_ms,
                float *__restrict__ part_val, int *__restrict__ part_id, SampleArgs smp) {
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
    // The weights are never written by any kernel, so this warp's first two
    // rows can be pulled into L2 before the wait for phase 1's z (the CTA
    // starts while phase 1's last CTAs still stream).
    if (lane == 0 && warp < nrows)
        prefetch_l2_bulk(w2_row(W2, Wlm, 0, r0 + warp, V, d), (unsigned)(d * sizeof(T)));
    if (lane == 0 && warp + kW2Warps < nrows)
        prefetch_l2_bulk(w2_row(W2, Wlm, 0, r0 + warp + kW2Warps, V, d),
                         (unsigned)(d * sizeof(T)));
    pdl_enter();

    for (int k0 = 0; k0 < K; k0 += hpg) {
        const int hk = min(hpg, K - k0);
        // stage z for heads k0 .. k0+hk-1 (zero rows for b >= B)
        for (int kk = 0; kk < hk; ++kk)
            stage_planes<float, VN, NB>(z + (size_t)(k0 + kk) * B * d, (size_t)d, B, d,
                                        zs4 + (size_t)kk * NB * d / 4);
        __syncthreads();

        WarpTop st[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) st[b].reset();
        int cur = 0;
        const int items = hk * nrows;
        // sampling: lane l holds the Gumbel draws of this warp's l-th next item,
        // refilled every 32 items (one Philox block per lane per 32 rows)
        float gz[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) gz[b] = 0.f;
        int jb = 0;
        for (int it = warp; it < items; it += kW2Warps, ++jb) {
            const int kk = it / nrows;
            const int v = r0 + (it - kk * nrows);
            if (SAMPLE && (jb & 31) == 0) {
                const int itl = it + lane * kW2Warps;
                if (itl < items) {
                    const int kl = itl / nrows;
                    const int vl = r0 + (itl - kl * nrows);
#pragma unroll
                    for (int b = 0; b < NB; ++b)
                        if (b < B) gz[b] = gumbel_at(smp.seed, smp.step, kRngDraft, b, k0 + kl, vl);
                }
            }
            while (cur < kk) {
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    flush_slot(slots[(warp * hpg + cur) * NB + b], st[b], S, lane);
                    st[b].reset();
                }
                ++cur;
            }
            float acc[NB];
            const uint4 *wrow = reinterpret_cast<const uint4 *>(w2_row(W2, Wlm, k0 + kk, v, V, d));
            const float4 *zk = zs4 + (size_t)kk * NB * d / 4;
            row_dot<T, NB, U>(wrow, zk, nvec, lane, acc);
            if (!SAMPLE) {
#pragma unroll
                for (int b = 0; b < NB; ++b)
                    if (b < B) st[b].push(acc[b], v, S, lane);
            } else {
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const float g = __shfl_sync(0xffffffffu, gz[b], jb & 31);
                    if (b < B) {
                        const float y = acc[b] * smp.inv_T;
                        st[b].push_key(y, y + g, v, S, lane);
                        if (smp.logits_out && lane == 0)
                            smp.logits_out[((size_t)b * K + (k0 + kk)) * V + v] = acc[b];
                    }
                }
            }
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

        // merge the warps' states per (head, sequence), one warp per pair
        const int pairs = hk * B;
        for (int pair = warp; pair < pairs; pair += kW2Warps) {
            const int kk = pair / B, b = pair - kk * B;
            const size_t o = ((size_t)(k0 + kk) * B + b) * G + g;
            float m, sum;
            warp_merge_ms(slots + kk * NB + b, hpg * NB, kW2Warps, lane, m, sum);
            float tv;
            int ti;
            warp_merge_top(slots + kk * NB + b, hpg * NB, kW2Warps, S, lane, tv, ti);
            if (lane == 0) part_ms[o] = make_float2(m, sum);
            if (lane < S) {
                part_val[o * S + lane] = tv;
                part_id[o * S + lane] = ti;
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------- phase 3 ---

// One CTA per (head, sequence).  The G partial top-s lists sit contiguously
// (G*S candidates); each warp selects the top-s of its share with
// warp_select_top, the partial (max, sum) pairs loading in the same round as
// the candidates; then one warp merges the warps' lists by warp selection
// (warp_merge_top) while another merges their (max, sum) pairs.
__global__ void __launch_bounds__(kReduceThreads)
heads_reduce_kernel(const float2 *__restrict__ part_ms, const float *__restrict__ part_val,
                    const int *__restrict__ part_id, int G, int B, int K, int S, int lm,
                    int32_t *__restrict__ topk_ids, float *__restrict__ topk_logp,
                    int32_t *__restrict__ root, float *__restrict__ root_logp) {
    constexpr int U = 4;
    constexpr int NW = kReduceThreads / kWarp;
    pdl_enter();
    __shared__ TopSlot slots[NW];
    __shared__ float s_logz;
    __shared__ float r_val[MEDUSA_MAX_TOP_S];
    __shared__ int r_id[MEDUSA_MAX_TOP_S];
    const int kb = blockIdx.x;  // k * B + b over all heads (the LM head first if lm)
    const int k = kb / B, b = kb - k * B;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int C = G * S;
    const float *pv = part_val + (size_t)kb * C;
    const int *pi = part_id + (size_t)kb * C;
    // this warp's contiguous share of the candidates
    const int c_lo = (int)(((long long)warp * C) / NW);
    const int c_hi = (int)(((long long)(warp + 1) * C) / NW);
    // the (max, sum) pairs load in the same round as the candidates
    // (G <= kMaxW2Ctas = 2 * kReduceThreads)
    const float2 ms0 = threadIdx.x < G ? part_ms[(size_t)kb * G + threadIdx.x]
                                       : make_float2(-INFINITY, 0.f);
    const float2 ms1 = threadIdx.x + kReduceThreads < G
                           ? part_ms[(size_t)kb * G + threadIdx.x + kReduceThreads]
                           : make_float2(-INFINITY, 0.f);
    float val = -INFINITY;
    int id = INT_MAX;
    for (int c0 = c_lo; c0 < c_hi; c0 += kWarp * U) {
        float cv[U + 1];
        int ci[U + 1];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int idx = c0 + u * kWarp + lane;
            cv[u] = idx < c_hi ? pv[idx] : -INFINITY;
            ci[u] = idx < c_hi ? pi[idx] : INT_MAX;
        }
        cv[U] = lane < S ? val : -INFINITY;  // the running list joins the pool
        ci[U] = lane < S ? id : INT_MAX;
        warp_select_top<U>(cv, ci, S, lane, val, id);
    }
    WarpTop st;
    st.reset();
    st.merge_ms(ms0.x, ms0.y);
    st.merge_ms(ms1.x, ms1.y);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, st.m, o);
        const float os = __shfl_xor_sync(0xffffffffu, st.s, o);
        st.merge_ms(om, os);
    }
    st.val = val;
    st.id = id;
    flush_slot(slots[warp], st, S, lane);
    __syncthreads();
    if (warp == 0) {
        float m, sum;
        warp_merge_ms(slots, 1, NW, lane, m, sum);
        if (lane == 0) s_logz = m + logf(sum);
    }
    if (warp == 1) {
        float tv;
        int ti;
        warp_merge_top(slots, 1, NW, S, lane, tv, ti);
        if (lane < S) {
            r_val[lane] = tv;
            r_id[lane] = ti;
        }
    }
    __syncthreads();
    if (lm && k == 0) {  // the LM head: its greedy token is the tree root
        if (threadIdx.x == 0) {
            root[b] = r_id[0];
            root_logp[b] = r_val[0] - s_logz;
        }
    } else if (threadIdx.x < S) {
        const size_t o = ((size_t)b * (K - lm) + (k - lm)) * S + threadIdx.x;
        topk_ids[o] = r_id[threadIdx.x];
        if (topk_logp) topk_logp[o] = r_val[threadIdx.x] - s_logz;
    }
}

// ---------------------------------------------------------------- host ---

constexpr int kMaxW2Ctas = 1024;
static_assert(kMaxW2Ctas <= 2 * kReduceThreads,
              "phase 3 loads at most two (max, sum) pairs a thread");
// Shared memory per phase-2 CTA.  One sequence (NB = 1) runs two CTAs per SM,
// and two CTAs must stay within the 196 KB shared-memory carveout: the
// largest carveout (228 KB) leaves L1 so small that the weight stream runs
// ~15% slower (measured on GB300), more than a second head group costs.
constexpr size_t kSmemBudget = 200 * 1024;
constexpr size_t kSmemBudgetPair = 97 * 1024;

int nb_bucket(int B) { return B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : 8; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct HeadsLayout {
    size_t z_off, ms_off, val_off, id_off, total;
};

// Kt = heads in the pass (the Medusa heads, plus the LM head when present).
HeadsLayout heads_layout(int B, int Kt, int d, int S) {
    HeadsLayout L;
    size_t o = MEDUSA_WS_HEADER;
    L.z_off = o;
    // fp32 z [Kt][B][d] (CUDA cores) or bf16 hi/lo rows [Kt][16][d] (tensor cores)
    size_t zb = (size_t)Kt * B * d * sizeof(float);
    if (B >= kHeadsTcMinBatch) zb = std::max(zb, heads_tc_zt_bytes(Kt, d));
    o = align256(o + zb);
    L.ms_off = o;
    o = align256(o + (size_t)Kt * B * kMaxW2Ctas * sizeof(float2));
    L.val_off = o;
    o = align256(o + (size_t)Kt * B * kMaxW2Ctas * S * sizeof(float));
    L.id_off = o;
    o = align256(o + (size_t)Kt * B * kMaxW2Ctas * S * sizeof(int));
    L.total = o;
    return L;
}

template <typename T, int NB>
cudaError_t run_heads(const void *h, const void *Wlm, const void *W1, const void *b1,
                      const void *W2, int B, int d, int V, int K, int S, int32_t *ids,
                      float *logp, int32_t *root, float *root_logp, const SampleArgs &smp,
                      char *ws, cudaStream_t stream) {
    // one sequence: six CTAs a SM with four loads in flight per lane (48
    // warps) beat four CTAs with eight (the bs1 step 248.5 against 248.9 us);
    // each lane still walks its vectors in the same order, so the sums are
    // unchanged
    constexpr int U1 = NB == 1 ? 4 : (NB <= 4 ? 8 : 4);
    constexpr int U2 = NB <= 4 ? 8 : 4;
    const int lm = Wlm ? 1 : 0;
    const int Kt = K + lm;
    const HeadsLayout L = heads_layout(B, Kt, d, S);
    float *z = reinterpret_cast<float *>(ws + L.z_off);  // [Kt][B][d], the LM head first
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
    const int warps1 = kW1Threads / kWarp;
    const int grid1 = sms * std::max(occ1, 1);  // one full wave
    const int total_warps = grid1 * warps1;
    e = launch_pdl(k1, dim3(grid1), dim3(kW1Threads), smem1, stream, static_cast<const T *>(h),
                   static_cast<const T *>(W1), static_cast<const T *>(b1),
                   z + (size_t)lm * B * d, lm ? z : nullptr, B, d, K, total_warps);
    note_launch();
    if (e) return e;

    // phase 2
    const size_t per_head = (size_t)NB * d * sizeof(float);
    const size_t slot_per_head = (size_t)kW2Warps * NB * sizeof(TopSlot);
    const size_t budget = NB == 1 ? kSmemBudgetPair : kSmemBudget;
    int hpg = (int)std::min<size_t>(Kt, std::max<size_t>(1, budget / (per_head + slot_per_head)));
    const size_t smem2 = hpg * (per_head + slot_per_head);
    auto k2 = smp.on ? heads_w2_kernel<T, NB, U2, true> : heads_w2_kernel<T, NB, U2, false>;
    if ((e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2)))
        return e;
    int occ2 = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ2, k2, kW2Threads, smem2))) return e;
    const int G = std::max(1, std::min(kMaxW2Ctas, sms * std::max(occ2, 1)));
    e = launch_pdl(k2, dim3(G), dim3(kW2Threads), smem2, stream, static_cast<const float *>(z),
                   static_cast<const T *>(W2), static_cast<const T *>(Wlm), B, d, V, Kt, S, hpg,
                   pms, pval, pid, smp);
    note_launch();
    if (e) return e;

    // phase 3
    e = launch_pdl(heads_reduce_kernel, dim3(Kt * B), dim3(kReduceThreads), 0, stream,
                   static_cast<const float2 *>(pms), static_cast<const float *>(pval),
                   static_cast<const int *>(pid), G, B, Kt, S, lm, ids, logp, root, root_logp);
    note_launch();
    return e;
}

}  // namespace

size_t heads_workspace_bytes(int B, int K, int d, int V, int S, bool with_lm_head) {
    (void)V;
    return heads_layout(B, K + (with_lm_head ? 1 : 0), d, S).total;
}

cudaError_t launch_heads(medusa_dtype dtype, const void *h, const void *Wlm, const void *W1,
                         const void *b1, const void *W2, int B, int d, int V, int K, int S,
                         int32_t *ids, float *logp, int32_t *root, float *root_logp,
                         const SampleArgs *sample, void *ws, cudaStream_t stream) {
    char *w = static_cast<char *>(ws);
    if (heads_tc_eligible(dtype, B, d, V, K, Wlm != nullptr, sample != nullptr)) {
        // several bf16 sequences: both GEMVs on the tensor cores (heads_tc.cu),
        // then the same merge of the per-CTA partials
        const int lm = Wlm ? 1 : 0, Kt = K + lm;
        const HeadsLayout L = heads_layout(B, Kt, d, S);
        float2 *pms = reinterpret_cast<float2 *>(w + L.ms_off);
        float *pval = reinterpret_cast<float *>(w + L.val_off);
        int *pid = reinterpret_cast<int *>(w + L.id_off);
        cudaError_t e = launch_heads_tc(h, Wlm, W1, b1, W2, B, d, V, K, S, sample, w + L.z_off,
                                        pms, pval, pid, reinterpret_cast<int *>(w), stream);
        if (e) return e;
        e = launch_pdl(heads_reduce_kernel, dim3(Kt * B), dim3(kReduceThreads), 0, stream,
                       static_cast<const float2 *>(pms), static_cast<const float *>(pval),
                       static_cast<const int *>(pid), heads_tc_ctas_per_head(Kt), B, Kt, S, lm,
                       ids, logp, root, root_logp);
        note_launch();
        return e;
    }
    const int nb = nb_bucket(B);
    SampleArgs smp = {};
    if (sample) smp = *sample;
#define MEDUSA_HEADS_CASE(T, N)                                                                  \
    if (nb == N)                                                                                 \
        return run_heads<T, N>(h, Wlm, W1, b1, W2, B, d, V, K, S, ids, logp, root, root_logp,   \
                               smp, w, stream);
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
