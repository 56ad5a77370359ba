// speculative.cu -- exact speculative sampling on a chain of sampled drafts
// (medusa_speculative_posterior).
//
// "Medusa: Faster LLM text generation", Acceptance rules, and "Medusa 深读"
// §3 and §5: draft x_k was sampled from q_k = softmax(head logits / T); it is
// accepted with probability min(1, p(x_k) / q_k(x_k)) under the verifying
// model's p = softmax(logits / T) of the row before it; at the first
// rejection the next token is sampled from the normalised positive residual
// max(0, p - q_k); if all K drafts are accepted it is sampled from the last
// row's p.  Sampling uses the Gumbel-max rule with the Philox streams of
// philox.cuh (accept: purpose 2, row k, index 0; resample: purpose 3, row
// L, index v).
//
//   spec_stats_kernel   grid (slices, 2K+1, B): (max, sum-exp) of x / T per
//                       slice of every p row (r <= K) and q row (r > K).
//   spec_sample_kernel  grid (slices, B): every CTA merges the row
//                       normalisers, evaluates the K acceptance decisions
//                       (a few loads), and samples row L over its slice:
//                       best of log(p - q)+ + G, and of log p + G as the
//                       fallback for an empty residual.
//   spec_select_kernel  one CTA per sequence: merges the slices' winners and
//                       writes the results.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "launch.h"
#include "philox.cuh"

namespace medusa {

namespace {

constexpr int kSpecThreads = 256;
constexpr int kSpecSlices = 8;

struct SpecPick {
    float key;
    int id;
    float key_p;
    int id_p;
};

template <typename T>
__device__ __forceinline__ float load_elt(const T *p, size_t i) {
    return Vec16<T>::load1(p + i);
}

__device__ __forceinline__ void ms_merge(float &m, float &s, float om, float os) {
    if (om == -INFINITY) return;
    if (om > m) {
        s = s * expf(m - om) + os;
        m = om;
    } else {
        s += os * expf(om - m);
    }
}

// block-wide (max, sum) merge; result valid in thread 0
__device__ __forceinline__ void block_ms(float &m, float &s, float2 *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, o);
        const float os = __shfl_xor_sync(0xffffffffu, s, o);
        ms_merge(m, s, om, os);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = make_float2(m, s);
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) ms_merge(m, s, red[w].x, red[w].y);
    }
}

// better (key, id): larger key, smaller id on equal keys
__device__ __forceinline__ bool pick_better(float ka, int ia, float kb, int ib) {
    return ka > kb || (ka == kb && ia < ib);
}

__device__ __forceinline__ void warp_pick(float &k, int &i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, k, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (pick_better(ok, oi, k, i)) {
            k = ok;
            i = oi;
        }
    }
}

// slice [v0, v1) of V, in whole 8-element groups
__device__ __forceinline__ void slice_of(int V, int slice, int nslices, int &v0, int &v1) {
    const int g = (V + 7) / 8;
    v0 = (int)(((long long)slice * g) / nslices) * 8;
    v1 = min(V, (int)(((long long)(slice + 1) * g) / nslices) * 8);
}

template <typename T>
__global__ void __launch_bounds__(kSpecThreads)
spec_stats_kernel(const T *__restrict__ logits, const float *__restrict__ draft, int V, int K,
                  float inv_T, float2 *__restrict__ parts) {
    pdl_enter();
    __shared__ float2 red[kSpecThreads / kWarp];
    const int slice = blockIdx.x, r = blockIdx.y, b = blockIdx.z;
    const int ns = gridDim.x;
    int v0, v1;
    slice_of(V, slice, ns, v0, v1);
    float m = -INFINITY, s = 0.f;
    if (r <= K) {
        const T *row = logits + ((size_t)b * (K + 1) + r) * V;
        for (int v = v0 + threadIdx.x; v < v1; v += kSpecThreads) {
            const float x = load_elt(row, v) * inv_T;
            ms_merge(m, s, x, 1.f);
        }
    } else {
        const float *row = draft + ((size_t)b * K + (r - K - 1)) * V;
        for (int v = v0 + threadIdx.x; v < v1; v += kSpecThreads) ms_merge(m, s, row[v] * inv_T, 1.f);
    }
    block_ms(m, s, red);
    if (threadIdx.x == 0) parts[((size_t)b * (2 * K + 1) + r) * ns + slice] = make_float2(m, s);
}

template <typename T>
__global__ void __launch_bounds__(kSpecThreads)
spec_sample_kernel(const T *__restrict__ logits, const int32_t *__restrict__ tokens,
                   const float *__restrict__ draft, int V, int K, float inv_T, uint64_t seed,
                   uint64_t step, const float2 *__restrict__ parts, int ns_stats,
                   SpecPick *__restrict__ picks, int32_t *__restrict__ acc_out,
                   int32_t *__restrict__ L_out, int *status) {
    // The predecessor that can still be running, spec_stats_kernel, writes
    // only the row normalisers: thread k's draft token, its raw p and q
    // logits and its uniform are read before the launch wait.
    const int tid0 = threadIdx.x, b0 = blockIdx.y;
    int x_k = -1;
    float lp_raw = 0.f, lq_raw = 0.f, u_k = 1.f;
    if (tid0 >= 1 && tid0 <= K) {
        x_k = tokens[(size_t)b0 * (K + 1) + tid0];
        if (x_k >= 0 && x_k < V) {
            lp_raw = load_elt(logits + ((size_t)b0 * (K + 1) + (tid0 - 1)) * V, x_k);
            lq_raw = draft[((size_t)b0 * K + (tid0 - 1)) * V + x_k];
            u_k = uniform_at(seed, step, kRngAccept, b0, tid0, 0);
        }
    }
    pdl_enter();
    __shared__ float s_lz[2 * MEDUSA_MAX_HEADS + 1];
    __shared__ int s_rej[MEDUSA_MAX_HEADS + 1];
    __shared__ float s_k[kSpecThreads / kWarp], s_kp[kSpecThreads / kWarp];
    __shared__ int s_i[kSpecThreads / kWarp], s_ip[kSpecThreads / kWarp];
    const int slice = blockIdx.x, b = blockIdx.y;
    const int ns = gridDim.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // row normalisers: log Z = m + log s, p rows 0..K then q rows
    if (tid < 2 * K + 1) {
        float m = -INFINITY, s = 0.f;
        const float2 *pr = parts + ((size_t)b * (2 * K + 1) + tid) * ns_stats;
        for (int j = 0; j < ns_stats; ++j) ms_merge(m, s, pr[j].x, pr[j].y);
        s_lz[tid] = m + logf(s);
    }
    __syncthreads();
    // acceptance decisions: thread k (1..K) judges draft k; rejected -> 1
    if (tid >= 1 && tid <= K) {
        const int k = tid;
        int rej = 1;
        if (x_k < 0 || x_k >= V) {
            set_status(status, MEDUSA_DEV_BAD_TOKEN);
        } else {
            const float lp = lp_raw * inv_T - s_lz[k - 1];
            const float lq = lq_raw * inv_T - s_lz[K + k];
            rej = !(lp - lq - logf(u_k) > 0.f);
        }
        s_rej[k] = rej;
    }
    __syncthreads();
    int L = K;
    for (int k = 1; k <= K; ++k)
        if (s_rej[k]) {
            L = k - 1;
            break;
        }
    if (slice == 0 && tid == 0) {
        L_out[b] = L;
        for (int k = 1; k <= K; ++k)
            acc_out[(size_t)b * K + (k - 1)] = k <= L ? 1 : (k == L + 1 ? 0 : -1);
    }
    // ---- sample row L over this slice
    int v0, v1;
    slice_of(V, slice, ns, v0, v1);
    const T *prow = logits + ((size_t)b * (K + 1) + L) * V;
    const float *qrow = L < K ? draft + ((size_t)b * K + L) * V : nullptr;
    const float lzp = s_lz[L];
    const float lzq = L < K ? s_lz[K + 1 + L] : 0.f;
    float bk = -INFINITY, bkp = -INFINITY;
    int bi = INT_MAX, bip = INT_MAX;
    // each thread takes whole groups of four indices (one Philox block)
    for (int v4 = v0 + 4 * tid; v4 < v1; v4 += 4 * kSpecThreads) {
        const Philox4x64 rnd = philox4x64((uint64_t)(v4 >> 2), (uint64_t)L, (uint64_t)b,
                                          (uint64_t)kRngResample, seed, step);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int v = v4 + e;
            if (v >= v1) break;
            const float g = -logf(-logf(word_uniform(rnd.w[e])));
            const float lp = load_elt(prow, v) * inv_T - lzp;
            const float kp = lp + g;
            if (pick_better(kp, v, bkp, bip)) {
                bkp = kp;
                bip = v;
            }
            if (qrow) {
                const float r = expf(lp) - expf(qrow[v] * inv_T - lzq);
                if (r > 0.f) {
                    const float kr = logf(r) + g;
                    if (pick_better(kr, v, bk, bi)) {
                        bk = kr;
                        bi = v;
                    }
                }
            }
        }
    }
    warp_pick(bk, bi);
    warp_pick(bkp, bip);
    if (lane == 0) {
        s_k[warp] = bk;
        s_i[warp] = bi;
        s_kp[warp] = bkp;
        s_ip[warp] = bip;
    }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kSpecThreads / kWarp; ++w) {
            if (pick_better(s_k[w], s_i[w], bk, bi)) {
                bk = s_k[w];
                bi = s_i[w];
            }
            if (pick_better(s_kp[w], s_ip[w], bkp, bip)) {
                bkp = s_kp[w];
                bip = s_ip[w];
            }
        }
        SpecPick pk;
        pk.key = bk;
        pk.id = bi;
        pk.key_p = bkp;
        pk.id_p = bip;
        picks[(size_t)b * ns + slice] = pk;
    }
}

__global__ void __launch_bounds__(32)
spec_select_kernel(const int32_t *__restrict__ tokens, const SpecPick *__restrict__ picks,
                   const int32_t *__restrict__ L_in, int K, int ns, int32_t *__restrict__ accept_len,
                   int32_t *__restrict__ path_tokens, int32_t *__restrict__ next_token) {
    const int b = blockIdx.x, lane = threadIdx.x;
    // the chain's tokens come from before spec_sample_kernel (the one
    // predecessor that can still be running), so they load before the wait;
    // lanes 0..K hold them (K <= 8 < 32)
    const int tok_q = lane <= K ? tokens[(size_t)b * (K + 1) + lane] : -1;
    pdl_enter();
    float bk = -INFINITY, bkp = -INFINITY;
    int bi = INT_MAX, bip = INT_MAX;
    for (int j = lane; j < ns; j += 32) {
        const SpecPick pk = picks[(size_t)b * ns + j];
        if (pick_better(pk.key, pk.id, bk, bi)) {
            bk = pk.key;
            bi = pk.id;
        }
        if (pick_better(pk.key_p, pk.id_p, bkp, bip)) {
            bkp = pk.key_p;
            bip = pk.id_p;
        }
    }
    warp_pick(bk, bi);
    warp_pick(bkp, bip);
    const int L = L_in[b];
    if (lane == 0) {
        accept_len[b] = L;
        // the residual when it has mass (a rejection), else a sample of p
        const int nt = (L < K && bi != INT_MAX) ? bi : bip;
        next_token[b] = nt == INT_MAX ? 0 : nt;
    }
    if (lane <= K) path_tokens[(size_t)b * (K + 1) + lane] = lane <= L ? tok_q : -1;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct SpecLayout {
    size_t stats_off, picks_off, L_off, acc_off, total;
};

SpecLayout spec_layout(int B, int K) {
    SpecLayout l;
    size_t o = MEDUSA_WS_HEADER;
    l.stats_off = o;
    o = align256(o + (size_t)B * (2 * K + 1) * kSpecSlices * sizeof(float2));
    l.picks_off = o;
    o = align256(o + (size_t)B * kSpecSlices * sizeof(SpecPick));
    l.L_off = o;
    o = align256(o + (size_t)B * sizeof(int32_t));
    l.acc_off = o;
    o = align256(o + (size_t)B * std::max(K, 1) * sizeof(int32_t));
    l.total = o;
    return l;
}

template <typename T>
cudaError_t run_speculative(const void *logits, const int32_t *tokens, const float *draft, int B,
                            int V, int K, float temperature, uint64_t seed, uint64_t step,
                            int32_t *accept_len, int32_t *path_tokens, int32_t *next_token,
                            int32_t *accept, void *ws, cudaStream_t stream) {
    const SpecLayout l = spec_layout(B, K);
    char *w = static_cast<char *>(ws);
    int *status = reinterpret_cast<int *>(w);
    float2 *stats = reinterpret_cast<float2 *>(w + l.stats_off);
    SpecPick *picks = reinterpret_cast<SpecPick *>(w + l.picks_off);
    int32_t *Lb = reinterpret_cast<int32_t *>(w + l.L_off);
    int32_t *acc = accept ? accept : reinterpret_cast<int32_t *>(w + l.acc_off);
    const float inv_T = 1.f / temperature;
    const T *lg = static_cast<const T *>(logits);
    cudaError_t e = launch_pdl(spec_stats_kernel<T>, dim3(kSpecSlices, 2 * K + 1, B),
                               dim3(kSpecThreads), 0, stream, lg, draft, V, K, inv_T, stats);
    note_launch();
    if (e) return e;
    e = launch_pdl(spec_sample_kernel<T>, dim3(kSpecSlices, B), dim3(kSpecThreads), 0, stream, lg,
                   tokens, draft, V, K, inv_T, seed, step, static_cast<const float2 *>(stats),
                   kSpecSlices, picks, acc, Lb, status);
    note_launch();
    if (e) return e;
    e = launch_pdl(spec_select_kernel, dim3(B), dim3(32), 0, stream, tokens,
                   static_cast<const SpecPick *>(picks), static_cast<const int32_t *>(Lb), K,
                   kSpecSlices, accept_len, path_tokens, next_token);
    note_launch();
    return e;
}

}  // namespace

size_t speculative_workspace_bytes(int B, int K) { return spec_layout(B, K).total; }

cudaError_t launch_speculative(medusa_dtype dtype, const void *logits, const int32_t *tokens,
                               const float *draft_logits, int B, int V, int K, float temperature,
                               uint64_t seed, uint64_t step, int32_t *accept_len,
                               int32_t *path_tokens, int32_t *next_token, int32_t *accept,
                               void *ws, cudaStream_t stream) {
    if (dtype == MEDUSA_BF16)
        return run_speculative<bf16>(logits, tokens, draft_logits, B, V, K, temperature, seed,
                                     step, accept_len, path_tokens, next_token, accept, ws,
                                     stream);
    return run_speculative<float>(logits, tokens, draft_logits, B, V, K, temperature, seed, step,
                                  accept_len, path_tokens, next_token, accept, ws, stream);
}

}  // namespace medusa
