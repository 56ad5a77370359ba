// attention.cu -- tree-masked attention over the KV cache.
//
// "Medusa: Faster LLM text generation" (Tree attention) and "Medusa 深读"
// §6.1: every tree node attends to the whole prefix and to its own branch
// ancestors (itself included), never to another branch.  Sequence b's cache
// holds the prefix in slots 0..P_b-1 and the R tree nodes (canonical order)
// in slots P_b..P_b+R-1; node i may see tree slot t iff bit t of its
// ancestor-mask row is set.
//
// bf16 path (tcgen05 tensor cores, split-KV):
//   tree_attn_tc_kernel  grid (H * row tiles, key ranges, B): one CTA per
//       (128-row tile of the tree, head, key range, sequence) computes
//       unnormalised partial (O, m, l) rows over its keys (below).
//   tree_attn_combine_kernel  merges the key ranges of each (b, row, head)
//       with a log-sum-exp rescale and writes the bf16 output.
// f32 path (small problems): tree_attn_f32_kernel, one CTA per
// (row, head, sequence) on CUDA cores, exact softmax.
#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace medusa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// A sequence's cache pointers are read on the device, so their checks run
// there: NULL or not 16-byte aligned -> MEDUSA_DEV_BAD_CACHE, and the
// sequence's output is zero.
__device__ __forceinline__ bool cache_pointers_bad(const void *kc, const void *vc) {
    return !kc || !vc ||
           ((reinterpret_cast<uintptr_t>(kc) | reinterpret_cast<uintptr_t>(vc)) & 15u) != 0;
}

struct AttnArgs {
    const bf16 *q;
    const bf16 *const *kc;
    const bf16 *const *vc;
    const int32_t *prefix_len;
    const uint64_t *anc_mask;
    int B, R, H, P_max;
    int chunk, nps;
    int row_tiles;  // 128-row tiles of the R tree rows
    float scale_log2;
    uint32_t wait_polls;  // poll limit of the key loop's mbarrier waits
    float *part_o;
    float2 *part_ml;
    int *status;
};

// ------------------------------------------------------- tensor-core path ---
//
// tree_attn_tc_kernel: one CTA per (key range, head, 128-row tile of the
// tree, sequence); trees of more than 128 rows take two tiles, except a tree
// of 129 rows over long key ranges, whose last row the tile's own threads
// compute on the CUDA cores (the TAIL variant, below).  The keys of
// a sequence are its cache slots 0 .. P+R-1, prefix and tree alike (they are
// contiguous); a key range is `cps` consecutive sub-chunks of 64 keys.  K and
// V of the sub-chunks stream through a three-stage cp.async ring in shared
// memory (two sub-chunks in flight while one computes); every thread copies
// four 16-byte chunks of K and of V per stage at a fixed column (constant
// steps, no per-chunk index arithmetic), and the next stage is issued while
// the S MMA runs.  Q, S, P and O live in tensor memory:
//     columns [0, 64)        S = Q K_j^T (fp32), then P over it (bf16 pairs)
//     columns [64, 64+DH/2)  Q (bf16 pairs, one query row per lane)
//     columns [128, 128+DH)  O += P V_j (fp32)
// 256 threads: threads t and t+128 own query row 128*tile + t (rows >= R are
// zero), each taking half of a sub-chunk's keys and half of the output
// columns; one thread issues the MMAs (A from tensor memory, B from shared
// memory).  Every thread reads its S half-row, masks it (slots past the
// range; tree slots that are not ancestors-or-self of the row) and writes
// P = 2^(s*scale*log2e - m) back over the S columns it read: the row max is
// taken on the raw scores (three-input maxima) and scaled once, the scale
// enters the exponent through a packed two-score FMA, and the exponential is
// the hardware's ex2.approx (P is rounded to bf16 next).  The row reference
// m is raised only when a sub-chunk's max exceeds it by more than 2^8; the
// threads then rescale their O row in tensor memory.  Otherwise P may reach
// 2^8, harmless in bf16 and fp32.  The row sum adds the fp32 weights (packed
// adds) while the MMA uses their bf16 rounding, as flash attention does.  The CTA
// writes one unnormalised partial (O, m, l) per row; tree_attn_combine_kernel
// merges the ranges.  Every mbarrier wait is bounded; on a timeout the CTA
// records MEDUSA_DEV_TIMEOUT, stops, waits once more (bounded) for its MMAs
// and frees its tensor memory before returning.  Freeing is safe when the
// drain sees the last commit arrive; an issued MMA takes far less than the
// drain's 2^16 polls.  If the drain gives up as well, the CTA still frees
// (holding the columns would stall every later allocation on the SM) and
// records MEDUSA_DEV_DRAIN_TIMEOUT over any earlier code, so the caller
// knows the outputs and the tensor memory may be corrupt.
constexpr int kTcSub = 64;               // keys per pipeline stage
constexpr int kTailMax = 1;              // tree rows past a full 128-row tile on CUDA cores
constexpr int kTailMinSubs = 8;          // sub-chunks per CTA that make the tail path pay
constexpr int kTcStages = 3;
constexpr float kRescaleLog2 = 8.f;      // lazy-rescale threshold (log2 units)
constexpr uint32_t kWaitPolls = 1u << 16;  // the drain's limit (the key loop's: a.wait_polls)

template <int DH>
struct TcSmem {
    static constexpr int NB = DH / 64;                 // 64-element column blocks of dh
    static constexpr int K_BYTES = NB * kTcSub * 128;   // [NB][64 keys][128 B]
    static constexpr int V_BYTES = NB * kTcSub * 128;   // [NB][64 keys][128 B]
    static constexpr int STAGE_BYTES = K_BYTES + V_BYTES;
    // two CTAs per SM stay within the same shared-memory carveout as the heads
    // kernels (2 x 96 KB): a larger carveout would shrink L1 under them
    static constexpr int BAR_OFF = kTcStages * STAGE_BYTES;  // mbarriers, TMEM holder, flag
    // 2 x (TOTAL + 1 KB reserved per CTA) must stay within a 196 KB carveout
    static constexpr int TOTAL = BAR_OFF + 64;
    // the tail variant adds the tail row's q in fp32, its weights, the warp
    // maxima and its mask words, within the same carveout (a larger one
    // costs the tile ~10 % at 128 live rows)
    static constexpr int TQ_OFF = TOTAL;
    static constexpr int TP_OFF = TQ_OFF + kTailMax * DH * 4;
    static constexpr int TMX_OFF = TP_OFF + kTailMax * kTcSub * 4;
    static constexpr int TAM_OFF = TMX_OFF + kTailMax * 4 * 4;
    static constexpr int TOTAL_TAIL = TAM_OFF + kTailMax * 3 * 8;
    static_assert(TQ_OFF % 16 == 0 && TMX_OFF % 16 == 0 && TAM_OFF % 8 == 0,
                  "tail areas aligned");
    static_assert(2 * (TOTAL_TAIL + 1024) <= 196 * 1024, "two tail-variant CTAs per SM");
};

// Issue the cp.async copies of sub-chunk keys [k0, k0+kTcSub) (rows past kend
// are zero-filled) into one stage; every thread commits one group.  Thread t
// owns 16-byte column t % CPR of key rows t / CPR + RPP * u: rows RPP apart
// (a multiple of 8) share the 128-byte swizzle phase, so each further chunk
// is a constant step in both shared and global memory.
template <int DH>
__device__ __forceinline__ void tc_load_stage(unsigned char *k_s, unsigned char *v_s,
                                              const bf16 *kc, const bf16 *vc, int k0, int kend,
                                              int H, int h, int tid) {
    constexpr int CPR = (DH / 64) * 8;    // 16-byte chunks per key row
    constexpr int RPP = 256 / CPR;        // key rows covered by one pass of the CTA
    constexpr int PASSES = kTcSub / RPP;
    static_assert(RPP % 8 == 0 && kTcSub % RPP == 0, "passes keep the swizzle phase");
    const int c16 = tid % CPR, r0 = tid / CPR;
    const uint32_t so0 = (c16 >> 3) * kTcSub * 128 + tc::sw128(r0, c16 & 7);
    const size_t row_elems = (size_t)H * DH;
    const size_t off0 = ((size_t)k0 * H + h) * DH + c16 * 8;  // key k0: always in range
#pragma unroll
    for (int u = 0; u < PASSES; ++u) {
        const int r = r0 + u * RPP;
        const bool ok = k0 + r < kend;
        const size_t off = ok ? off0 + (size_t)r * row_elems : off0;
        const uint32_t so = so0 + u * RPP * 128;
        cp_async16(tc::smem_addr(k_s + so), kc + off, ok ? 16 : 0);
        cp_async16(tc::smem_addr(v_s + so), vc + off, ok ? 16 : 0);
    }
    cp_async_commit();
}

// WIDE: trees of more than 128 rows (row tiles, four mask words per row).
// TAIL (dh 128): trees of 129 .. 128 + kTailMax rows in one 128-row tile; the
// rows past the tile are computed on the CUDA cores by the tile's own threads
// in the windows where they wait for the tensor cores: warps 4-7 score the
// sub-chunk's 64 keys against the tail rows while the S MMA runs (key
// (warp-4)*16 + lane/2, dh half lane%2); the tail rows' max rides on the
// tile's row-max barrier and their reference moves by the same lazy rule;
// the weights go to shared memory, and after the P barrier, while thread 0
// issues the P V MMA, warp w adds keys 8w..8w+7 into its own partial of the
// tail rows' O (four columns per lane).  The eight partials are summed once,
// after the key loop.  The row-max exchange of the tile moves out of the K
// tile, which warps 4-7 read while other warps are already past the S wait,
// into tensor memory: each thread writes its half-row max into a column of
// its own lane that its S read has freed (16 or 48; P takes 0-15 and 32-47).
template <int DH, bool WIDE, bool TAIL>
__global__ void __launch_bounds__(256, 2) tree_attn_tc_kernel(AttnArgs a) {
    static_assert(!TAIL || (WIDE && DH == 128), "the tail variant: dh 128, mask words past 128");
    static_assert(kTailMax == 1, "the tail bookkeeping below holds one row");
    pdl_enter();
    using L = TcSmem<DH>;
    constexpr int HALF = kTcSub / 2;  // keys per thread per sub-chunk
    // operand tiles need 1024-byte alignment (swizzle atoms)
    extern __shared__ __align__(1024) unsigned char tc_raw[];
    uint64_t &bar_s = *reinterpret_cast<uint64_t *>(tc_raw + L::BAR_OFF);
    uint64_t &bar_o = *reinterpret_cast<uint64_t *>(tc_raw + L::BAR_OFF + 8);
    uint32_t &tmem_holder = *reinterpret_cast<uint32_t *>(tc_raw + L::BAR_OFF + 16);
    int &failed = *reinterpret_cast<int *>(tc_raw + L::BAR_OFF + 20);

    // heads (and the row tiles of a head) vary fastest in the grid, so CTAs
    // resident together read whole token rows ([H, dh] per slot) of the same
    // key range; row tile rt of head h holds tree rows [128*rt, 128*rt + 128)
    const int h = WIDE ? blockIdx.x / a.row_tiles : blockIdx.x;
    const int rt = WIDE ? blockIdx.x - h * a.row_tiles : 0;
    const int split = blockIdx.y, b = blockIdx.z;
    const int R = a.R, H = a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = TAIL ? R - 128 : 0;  // tail rows
    // warp w reads TMEM lanes 32*(w%4)..: lane = tid % 128 holds tree row
    // row0 + lane; half = column half
    const int lrow = tid & 127, half = tid >> 7;
    const int row0 = rt * 128, row = row0 + lrow;
    int P = a.prefix_len[b];
    if (P < 0 || P > a.P_max) {
        set_status(a.status, MEDUSA_DEV_BAD_PREFIX);
        P = 0;
    }
    const int NS = a.nps;  // key ranges per (sequence, head)
    const size_t pbase = ((size_t)(b * H + h) * NS + split) * R;
    const int kbeg = split * a.chunk;  // a.chunk = cps * kTcSub keys per range
    const int kend = min(kbeg + a.chunk, P + R);
    const bf16 *kc = a.kc[b];
    const bf16 *vc = a.vc[b];
    const bool bad_cache = cache_pointers_bad(kc, vc);
    if (bad_cache) set_status(a.status, MEDUSA_DEV_BAD_CACHE);
    if (kend <= kbeg || bad_cache) {
        if (row < R && half == 0) a.part_ml[pbase + row] = make_float2(-INFINITY, 0.f);
        if (TAIL && tid < T) a.part_ml[pbase + 128 + tid] = make_float2(-INFINITY, 0.f);
        return;
    }
    const int nsub = (kend - kbeg + kTcSub - 1) / kTcSub;
    auto stage_k = [&](int j) { return tc_raw + (j % kTcStages) * L::STAGE_BYTES; };
    auto stage_v = [&](int j) { return tc_raw + (j % kTcStages) * L::STAGE_BYTES + L::K_BYTES; };

    // ---- Q row into registers first (its latency overlaps the K/V issue):
    // 64 elements per thread (dh 128: each half of the row; dh 64: the whole
    // row, by the first 128 threads)
    const bool q_owner = DH == 128 || half == 0;  // warp-uniform
    const int e0 = DH == 128 ? half * 64 : 0;
    uint32_t qr[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) qr[i] = 0u;
    if (q_owner && row < R) {
        const uint4 *src =
            reinterpret_cast<const uint4 *>(a.q + (((size_t)b * R + row) * H + h) * DH + e0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 v = src[i];
            qr[4 * i] = v.x;
            qr[4 * i + 1] = v.y;
            qr[4 * i + 2] = v.z;
            qr[4 * i + 3] = v.w;
        }
    }

    // ---- the first two sub-chunks start loading
    tc_load_stage<DH>(stage_k(0), stage_v(0), kc, vc, kbeg, kend, H, h, tid);
    if (nsub > 1) tc_load_stage<DH>(stage_k(1), stage_v(1), kc, vc, kbeg + kTcSub, kend, H, h, tid);
    // this row's ancestor-mask words (R <= 256: up to four)
    uint64_t am0 = 0, am1 = 0, am2 = 0, am3 = 0;
    const int W = (R + 63) / 64;
    if (kend > P && row < R) {
        const uint64_t *mr = a.anc_mask + ((size_t)b * R + row) * W;
        am0 = mr[0];
        if (W > 1) am1 = mr[1];
        if (WIDE && W > 2) am2 = mr[2];
        if (WIDE && W > 3) am3 = mr[3];
    }
    // ---- tail rows: q in fp32 and mask words in shared memory, and the
    // per-thread state (references identical in every thread)
    float *tq = reinterpret_cast<float *>(tc_raw + L::TQ_OFF);     // [kTailMax][DH]
    float *tp = reinterpret_cast<float *>(tc_raw + L::TP_OFF);     // [kTailMax][64] weights
    float *tmx = reinterpret_cast<float *>(tc_raw + L::TMX_OFF);   // [kTailMax][4] warp maxima
    uint64_t *tam = reinterpret_cast<uint64_t *>(tc_raw + L::TAM_OFF);  // [kTailMax][3]
    float tm[kTailMax], tl[kTailMax], tx[kTailMax], to[kTailMax][4];
#pragma unroll
    for (int t = 0; t < kTailMax; ++t) {
        tm[t] = -INFINITY;
        tl[t] = 0.f;
        tx[t] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c) to[t][c] = 0.f;
    }
    if constexpr (TAIL) {
        for (int e = tid; e < T * DH; e += 256) {
            const int t = e / DH, c = e - t * DH;
            tq[e] = __bfloat162float(a.q[(((size_t)b * R + 128 + t) * H + h) * DH + c]);
        }
        if (tid < T * 3) {
            const int t = tid / 3, w = tid - t * 3;
            tam[tid] = w < W ? a.anc_mask[((size_t)b * R + 128 + t) * W + w] : 0ull;
        }
    }
    if (tid == 0) {
        tc::mbar_init(&bar_s, 1);
        tc::mbar_init(&bar_o, 1);
        failed = 0;
    }
    if (warp == 0) tc::tmem_alloc(&tmem_holder, 256);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_holder;
    const uint32_t t_s = tmem, t_q = tmem + 64, t_o = tmem + 128;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

    // ---- Q row into tensor memory
    if (q_owner) {
        tc::tmem_st32u(t_q + lane_base + e0 / 2, qr);
        tc::tmem_wait_st();
    }
    // warps whose 32 rows are all padding (>= R) skip the softmax: their S
    // rows are zero (zero Q rows), which read as zero P, and their O rows are
    // never written out
    const bool rows_live = row0 + (warp & 3) * 32 < R;  // warp-uniform

    float m_run = -INFINITY;  // row reference (log2 units), same in both threads of a row
    float l_run = 0.f;        // this thread's share of the row sum
    int done = 0;             // sub-chunks whose P V MMA was issued
    for (int j = 0; j < nsub; ++j) {
        unsigned char *k_s = stage_k(j);
        unsigned char *v_s = stage_v(j);
        const int k0 = kbeg + j * kTcSub;
        // P V of sub-chunk j-1 done: its stage may be refilled (with j+2) and O
        // may be rescaled
        if (j > 0 && !tc::mbar_wait_bounded(&bar_o, (j - 1) & 1, a.wait_polls)) failed = 1;
        // groups in flight: j's and j+1's where it exists (j+2's is issued
        // below, while the S MMA of sub-chunk j runs)
        if (j + 1 < nsub)
            cp_async_wait<1>();
        else
            cp_async_wait<0>();
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (failed) break;  // uniform: read after the barrier

        // ---- S = Q K_j^T (A = Q in tensor memory, B = K_j in shared memory)
        if (tid == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16(128, kTcSub, 0);
            // the K-slices' descriptors differ only in the start-address
            // field (bytes >> 4), so the base is built once per sub-chunk
            const uint64_t bd0 = tc::sdesc_sw128(tc::smem_addr(k_s), 16, 1024);
#pragma unroll
            for (int ks = 0; ks < DH / 16; ++ks) {
                const uint32_t koff = (ks >> 2) * kTcSub * 128 + (ks & 3) * 32;
                tc::mma_bf16_ts(t_s, t_q + ks * 8, bd0 + (koff >> 4), idesc, ks > 0);
            }
            tc::mma_commit(&bar_s);
        }
        // ---- refill the stage of sub-chunk j-1 with j+2 while the MMA runs
        if (j + 2 < nsub)
            tc_load_stage<DH>(stage_k(j + 2), stage_v(j + 2), kc, vc, k0 + 2 * kTcSub, kend,
                              H, h, tid);
        __syncwarp();
        if constexpr (TAIL) {
            if (warp >= 4) {
                // ---- tail scores: key kk against each tail row, dh half hd
                // (column block hd of the K tile), halves summed by a shuffle
                const int kk = (warp - 4) * 16 + (lane >> 1), hd = lane & 1;
                const unsigned char *kb = k_s + hd * kTcSub * 128;
#pragma unroll
                for (int t = 0; t < kTailMax; ++t) {
                    if (t >= T) break;
                    const float *q = tq + t * DH + hd * 64;
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float4 qa = *reinterpret_cast<const float4 *>(q + c * 8);
                        const float4 qb = *reinterpret_cast<const float4 *>(q + c * 8 + 4);
                        const uint4 kv = *reinterpret_cast<const uint4 *>(kb + tc::sw128(kk, c));
                        acc[0] = fmaf(qa.x, bf_lo(kv.x), acc[0]);
                        acc[1] = fmaf(qa.y, bf_hi(kv.x), acc[1]);
                        acc[2] = fmaf(qa.z, bf_lo(kv.y), acc[2]);
                        acc[3] = fmaf(qa.w, bf_hi(kv.y), acc[3]);
                        acc[0] = fmaf(qb.x, bf_lo(kv.z), acc[0]);
                        acc[1] = fmaf(qb.y, bf_hi(kv.z), acc[1]);
                        acc[2] = fmaf(qb.z, bf_lo(kv.w), acc[2]);
                        acc[3] = fmaf(qb.w, bf_hi(kv.w), acc[3]);
                    }
                    float sc = (acc[0] + acc[1]) + (acc[2] + acc[3]);
                    sc += __shfl_xor_sync(0xffffffffu, sc, 1);
                    const int key = k0 + kk;
                    bool vis = key < kend;
                    if (vis && key >= P) {
                        const int tt = key - P;
                        const uint64_t w = tt < 64 ? tam[t * 3] : tt < 128 ? tam[t * 3 + 1]
                                                                           : tam[t * 3 + 2];
                        vis = (w >> (tt & 63)) & 1u;
                    }
                    tx[t] = vis ? sc : -INFINITY;
                    float mx = tx[t];
#pragma unroll
                    for (int o = 2; o < kWarp; o <<= 1)
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    if (lane == 0) tmx[t * 4 + warp - 4] = mx;
                }
            }
        }
        if (!tc::mbar_wait_bounded(&bar_s, j & 1, a.wait_polls)) failed = 1;
        tc::fence_after_sync();

        // ---- this thread's 32 keys of the sub-chunk
        float x[HALF];
        if (rows_live) {
            tc::tmem_ld32(t_s + lane_base + half * HALF, x);
        } else {
#pragma unroll
            for (int e = 0; e < HALF; ++e) x[e] = -INFINITY;
        }
        const int kc0 = k0 + half * HALF;
        const bool masked = (k0 + kTcSub > P || k0 + kTcSub > kend) && rows_live;
        if (masked) {
#pragma unroll
            for (int e = 0; e < HALF; ++e) {
                const int key = kc0 + e;
                bool vis = key < kend;
                if (vis && key >= P) {
                    const int t = key - P;
                    const uint64_t w = WIDE && t >= 128 ? (t < 192 ? am2 : am3)
                                                        : (t < 64 ? am0 : am1);
                    vis = (w >> (t & 63)) & 1u;
                }
                x[e] = vis ? x[e] : -INFINITY;
            }
        }
        // the half-row's max with three-input maxima (two accumulators)
        float mxa = max3f(x[0], x[1], x[2]), mxb = max3f(x[3], x[4], x[5]);
#pragma unroll
        for (int e = 6; e + 3 < HALF; e += 4) {
            mxa = max3f(mxa, x[e], x[e + 1]);
            mxb = max3f(mxb, x[e + 2], x[e + 3]);
        }
        static_assert(HALF % 4 == 0, "the max loop leaves the last two scores");
        mxa = max3f(mxa, x[HALF - 2], x[HALF - 1]);
        // row max of the sub-chunk: halves exchange through the dead K_j tile
        // (it is refilled only after the barrier that ends this iteration) or,
        // in the tail variant, through tensor memory
        // (scores are scaled into log2 units here and inside the exponent:
        // the scale is positive, so the max of the scaled scores is the
        // scaled max)
        const float hmx = fmaxf(mxa, mxb) * a.scale_log2;
        float cm;
        if constexpr (TAIL) {
            tc::tmem_st1(t_s + lane_base + half * HALF + 16, hmx);
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncthreads();
            tc::fence_after_sync();
            cm = fmaxf(hmx, tc::tmem_ld1(t_s + lane_base + (1 - half) * HALF + 16));
        } else {
            float *xch = reinterpret_cast<float *>(k_s);
            xch[half * 128 + lrow] = hmx;
            __syncthreads();
            cm = fmaxf(xch[lrow], xch[128 + lrow]);
        }
        const bool raise = cm > m_run + kRescaleLog2;
        const float m_new = raise ? cm : m_run;
        const float alpha = raise ? exp2f(m_run - m_new) : 1.f;  // 0 when m_run = -inf
        l_run *= alpha;
        m_run = m_new;
        const float mu = (m_run == -INFINITY) ? 0.f : m_run;
        if constexpr (TAIL) {
            // ---- tail rows: reference (every thread alike), then the
            // weights of warps 4-7's keys into shared memory
#pragma unroll
            for (int t = 0; t < kTailMax; ++t) {
                if (t >= T) break;
                const float4 w4 = *reinterpret_cast<const float4 *>(tmx + t * 4);
                const float tcm = fmaxf(fmaxf(w4.x, w4.y), fmaxf(w4.z, w4.w)) * a.scale_log2;
                if (tcm > tm[t] + kRescaleLog2) {
                    const float al = exp2f(tm[t] - tcm);  // 0 when the reference was -inf
                    tl[t] *= al;
#pragma unroll
                    for (int c = 0; c < 4; ++c) to[t][c] *= al;
                    tm[t] = tcm;
                }
                if (warp >= 4 && (lane & 1) == 0) {
                    const float tmu = tm[t] == -INFINITY ? 0.f : tm[t];
                    const float p = ex2_approx(fmaf(tx[t], a.scale_log2, -tmu));
                    tp[t * kTcSub + (warp - 4) * 16 + (lane >> 1)] = p;
                    tl[t] += p;
                }
            }
        }
        if (rows_live) {
            // two scores per packed FMA and per packed add
            const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
            const float2 nm2 = make_float2(-mu, -mu);
            float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            uint32_t pk[HALF / 2];
#pragma unroll
            for (int e = 0; e < HALF; e += 2) {
                const float2 t = __ffma2_rn(make_float2(x[e], x[e + 1]), sc2, nm2);
                const float p0 = ex2_approx(t.x), p1 = ex2_approx(t.y);
                pk[e / 2] = pack_bf16(p0, p1);
                // the row sum adds the fp32 weights; the MMA uses their bf16
                // rounding (relative difference <= 2^-9 per weight)
                ls[(e / 2) & 1] = __fadd2_rn(ls[(e / 2) & 1], make_float2(p0, p1));
            }
            l_run += (ls[0].x + ls[0].y) + (ls[1].x + ls[1].y);
            // P over the S columns this thread read: keys half*32.. -> columns
            // half*32 .. half*32+15
            tc::tmem_st16(t_s + lane_base + half * HALF, pk);
        }
        if (rows_live && __any_sync(0xffffffffu, raise && done > 0)) {
            // rescale this warp's O rows (lanes whose row did not move scale by
            // 1); P V of sub-chunk j-1 is complete, P V of j not yet issued
#pragma unroll 1
            for (int c = 0; c < DH / 2; c += 32) {
                float ov[32];
                tc::tmem_ld32(t_o + lane_base + half * (DH / 2) + c, ov);
#pragma unroll
                for (int e = 0; e < 32; ++e) ov[e] *= alpha;
                tc::tmem_st32(t_o + lane_base + half * (DH / 2) + c, ov);
            }
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();

        // ---- O += P_j V_j (A = P in tensor memory, B = V_j in shared memory)
        if (tid == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16(128, DH, 1);
            const uint64_t bd0 = tc::sdesc_sw128(tc::smem_addr(v_s), kTcSub * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kTcSub / 16; ++ks) {
                const uint32_t pa = t_s + (ks >> 1) * HALF + (ks & 1) * 8;
                tc::mma_bf16_ts(t_o, pa, bd0 + ((ks * 16 * 128) >> 4), idesc,
                                (done > 0 || ks > 0) ? 1u : 0u);
            }
            tc::mma_commit(&bar_o);
        }
        __syncwarp();
        if constexpr (TAIL) {
            // ---- tail P V: keys 8w..8w+7 into this warp's partial, four
            // columns per lane (V_j stays until the next iteration's barrier)
            const int col0 = lane * 4;
            const unsigned char *vb = v_s + (col0 / 64) * kTcSub * 128 + (col0 % 8) * 2;
            const int vch = (col0 % 64) / 8;
#pragma unroll
            for (int t = 0; t < kTailMax; ++t) {
                if (t >= T) break;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int kk = warp * 8 + i;
                    const float p = tp[t * kTcSub + kk];
                    const uint2 wv = *reinterpret_cast<const uint2 *>(vb + tc::sw128(kk, vch));
                    to[t][0] = fmaf(p, bf_lo(wv.x), to[t][0]);
                    to[t][1] = fmaf(p, bf_hi(wv.x), to[t][1]);
                    to[t][2] = fmaf(p, bf_lo(wv.y), to[t][2]);
                    to[t][3] = fmaf(p, bf_hi(wv.y), to[t][3]);
                }
            }
        }
        ++done;
    }
    // ---- wait for the last P V, then write the partial rows
    bool drain_failed = false;
    if (done > 0 && !tc::mbar_wait_bounded(&bar_o, (done - 1) & 1, kWaitPolls)) {
        failed = 1;
        // drain before freeing TMEM
        drain_failed = !tc::mbar_wait_bounded(&bar_o, (done - 1) & 1, kWaitPolls);
    }
    cp_async_wait<0>();
    tc::fence_after_sync();
    __syncthreads();
    const bool ok = !failed && done == nsub;  // uniform over the CTA
    if (failed && tid == 0) set_status(a.status, MEDUSA_DEV_TIMEOUT);
    if (drain_failed && a.status) atomicExch(a.status, MEDUSA_DEV_DRAIN_TIMEOUT);
    if (ok) {
        // this thread's half of the row's DH output columns
        float *dst = a.part_o + (pbase + row) * DH;
        for (int c = half * (DH / 2); c < (half + 1) * (DH / 2); c += 32) {
            float ov[32];
            tc::tmem_ld32(t_o + lane_base + c, ov);
            if (row < R) {
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4 *>(dst + c + e) =
                        make_float4(ov[e], ov[e + 1], ov[e + 2], ov[e + 3]);
            }
        }
    }
    // row sums: halves exchange through stage 0 (no copy is in flight now);
    // the tail rows' per-warp partials go there as well, past the first 4 KB
    float *xs = reinterpret_cast<float *>(tc_raw);
    float *tob = reinterpret_cast<float *>(tc_raw + 4096);  // [8 warps][kTailMax][DH]
    float *tlb = tob + 8 * kTailMax * DH;                    // [4 warps][kTailMax]
    xs[half * 128 + lrow] = l_run;
    if constexpr (TAIL) {
#pragma unroll
        for (int t = 0; t < kTailMax; ++t) {
            if (t >= T) break;
            *reinterpret_cast<float4 *>(tob + (warp * kTailMax + t) * DH + lane * 4) =
                make_float4(to[t][0], to[t][1], to[t][2], to[t][3]);
            const float ls = warp_sum(tl[t]);
            if (warp >= 4 && lane == 0) tlb[(warp - 4) * kTailMax + t] = ls;
        }
    }
    __syncthreads();
    if (half == 0 && row < R) {
        const float l = xs[lrow] + xs[128 + lrow];
        a.part_ml[pbase + row] = ok ? make_float2(m_run, l) : make_float2(-INFINITY, 0.f);
    }
    if constexpr (TAIL) {
        for (int e = tid; e < T * DH; e += 256) {
            const int t = e / DH, c = e - t * DH;
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) o += tob[(w * kTailMax + t) * DH + c];
            if (ok) a.part_o[(pbase + 128 + t) * DH + c] = o;
        }
        if (tid < T) {
            float l = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) l += tlb[w * kTailMax + tid];
            a.part_ml[pbase + 128 + tid] = ok ? make_float2(tm[0], l) : make_float2(-INFINITY, 0.f);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// One warp per (sequence, row, head).  Lane s reads split s's (m, l), and
// the O rows of the first PRE splits are loaded in the same round (they do
// not depend on the weights), so NS <= PRE costs one round of independent
// loads (PRE = 4, 8 or 16, the smallest that covers NS); later splits' rows
// are read with independent loads as well.  An empty split (l = 0) has weight 0 and its row, never
// written, is never used.
template <int DH, int PRE>
__global__ void __launch_bounds__(256)
tree_attn_combine_kernel(const float *__restrict__ part_o, const float2 *__restrict__ part_ml,
                         int B, int R, int H, int NS, bf16 *__restrict__ out) {
    pdl_enter();
    constexpr int PER = DH / 32;  // contiguous output columns per lane: one 8- or 16-byte load
    static_assert(PER == 2 || PER == 4, "dh 64 or 128");
    const int lane = threadIdx.x & 31;
    const int c0 = lane * PER;
    // this lane's PER columns of one partial row
    auto load_cols = [&](const float *row_base, float (&v)[PER]) {
        if constexpr (PER == 4) {
            const float4 t = *reinterpret_cast<const float4 *>(row_base + c0);
            v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
        } else {
            const float2 t = *reinterpret_cast<const float2 *>(row_base + c0);
            v[0] = t.x; v[1] = t.y;
        }
    };
    const long long item = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (item >= (long long)B * R * H) return;
    const int h = (int)(item % H);
    const int row = (int)((item / H) % R);
    const int b = (int)(item / ((long long)H * R));
    const size_t base = (size_t)(b * H + h) * NS;
    const float2 ml0 =
        lane < NS ? part_ml[(base + lane) * R + row] : make_float2(-INFINITY, 0.f);
    float pre[PRE][PER];
#pragma unroll
    for (int j = 0; j < PRE; ++j)
        if (j < NS) load_cols(part_o + ((base + j) * R + row) * DH, pre[j]);
    float M = ml0.y > 0.f ? ml0.x : -INFINITY;
    for (int s = lane + 32; s < NS; s += 32) {
        const float2 ml = part_ml[(base + s) * R + row];
        if (ml.y > 0.f) M = fmaxf(M, ml.x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    float acc[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) acc[j] = 0.f;
    for (int s0 = 0; s0 < NS; s0 += 32) {
        const float2 ml = s0 == 0                 ? ml0
                          : s0 + lane < NS ? part_ml[(base + s0 + lane) * R + row]
                                           : make_float2(-INFINITY, 0.f);
        float w_l = 0.f;
        if (ml.y > 0.f) {
            w_l = exp2f(ml.x - M);
            L = fmaf(w_l, ml.y, L);
        }
        const int cnt = min(32, NS - s0);
        int j0 = 0;
        if (s0 == 0) {
#pragma unroll
            for (int j = 0; j < PRE; ++j) {
                const float w = __shfl_sync(0xffffffffu, w_l, j);
                if (j < cnt && w != 0.f) {
#pragma unroll
                    for (int p = 0; p < PER; ++p) acc[p] = fmaf(w, pre[j][p], acc[p]);
                }
            }
            j0 = PRE;
        }
#pragma unroll 4
        for (int j = j0; j < cnt; ++j) {
            const float w = __shfl_sync(0xffffffffu, w_l, j);
            if (w != 0.f) {
                float v[PER];
                load_cols(part_o + ((base + s0 + j) * R + row) * DH, v);
#pragma unroll
                for (int p = 0; p < PER; ++p) acc[p] = fmaf(w, v[p], acc[p]);
            }
        }
    }
    L = warp_sum(L);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    bf16 *dst = out + (((size_t)b * R + row) * H + h) * DH + c0;
    if constexpr (PER == 4)
        *reinterpret_cast<uint2 *>(dst) =
            make_uint2(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv));
    else
        *reinterpret_cast<uint32_t *>(dst) = pack_bf16(acc[0] * inv, acc[1] * inv);
}

// ------------------------------------------------------------ f32 path ---

__global__ void __launch_bounds__(128)
tree_attn_f32_kernel(const float *__restrict__ q, const float *const *kcs, const float *const *vcs,
                     const int32_t *__restrict__ prefix_len, const uint64_t *__restrict__ anc_mask,
                     int R, int H, int dh, int P_max, float scale, float *__restrict__ out,
                     int *status) {
    pdl_enter();
    extern __shared__ float fsm[];
    __shared__ float red[128 / kWarp];
    const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    int P = prefix_len[b];
    if (P < 0 || P > P_max) {
        set_status(status, MEDUSA_DEV_BAD_PREFIX);
        P = 0;
    }
    const int n = P + R;
    float *qs = fsm;
    float *sc = fsm + dh;
    const float *kc = kcs[b];
    const float *vc = vcs[b];
    if (cache_pointers_bad(kc, vc)) {  // uniform over the CTA
        set_status(status, MEDUSA_DEV_BAD_CACHE);
        for (int c = threadIdx.x; c < dh; c += blockDim.x)
            out[(((size_t)b * R + i) * H + h) * dh + c] = 0.f;
        return;
    }
    const int W = (R + 63) / 64;
    const uint64_t *mrow = anc_mask + ((size_t)b * R + i) * W;
    for (int c = threadIdx.x; c < dh; c += blockDim.x)
        qs[c] = q[(((size_t)b * R + i) * H + h) * dh + c];
    __syncthreads();
    float lmax = -INFINITY;
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
        bool vis = j < P;
        if (!vis) {
            const int t = j - P;
            vis = (mrow[t >> 6] >> (t & 63)) & 1u;
        }
        float s = -INFINITY;
        if (vis) {
            const float *kr = kc + ((size_t)j * H + h) * dh;
            float acc = 0.f;
            for (int c = 0; c < dh; ++c) acc = fmaf(qs[c], kr[c], acc);
            s = acc * scale;
        }
        sc[j] = s;
        lmax = fmaxf(lmax, s);
    }
    for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = lmax;
    __syncthreads();
    float m = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
    __syncthreads();
    float lsum = 0.f;
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
        const float p = (sc[j] == -INFINITY) ? 0.f : expf(sc[j] - m);
        sc[j] = p;
        lsum += p;
    }
    lsum = warp_sum(lsum);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = lsum;
    __syncthreads();
    float L = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) L += red[w];
    for (int c = threadIdx.x; c < dh; c += blockDim.x) {
        float acc = 0.f;
        for (int j = 0; j < n; ++j)
            if (sc[j] != 0.f) acc = fmaf(sc[j], vc[((size_t)j * H + h) * dh + c], acc);
        out[(((size_t)b * R + i) * H + h) * dh + c] = acc / L;
    }
}

// ---------------------------------------------------------------- host ---

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Key ranges of the tensor-core path: at least two 64-key sub-chunks per CTA
// (so that loads overlap compute), and one (B = 1) or two (B > 1) waves of
// two CTAs per SM over the whole grid at P_max.
struct TcPlan {
    int ns, chunk, row_tiles;
    bool tail;  // 129 .. 128 + kTailMax rows: one tile, the rest on CUDA cores
};

TcPlan tc_plan(int B, int H, int R, int P_max, int dh) {
    const int nsub = (P_max + R + kTcSub - 1) / kTcSub;
    const int waves = B == 1 ? 1 : 2;
    auto plan = [&](int row_tiles, bool tail) {
        TcPlan p;
        p.tail = tail;
        p.row_tiles = row_tiles;
        const int per_head =
            std::max(1, 2 * waves * device_sm_count() / std::max(1, B * H * row_tiles));
        const int cps = std::max(2, (nsub + per_head - 1) / per_head);
        p.ns = (nsub + cps - 1) / cps;
        p.chunk = cps * kTcSub;
        return p;
    };
    // A tree one row past the tile (dh 128: the tail code reads dh as two
    // 64-column blocks) takes one tile and the tail row when every CTA then
    // runs at least kTailMinSubs sub-chunks: with fewer, the halved grid and
    // the tail's own set-up and merge cost more than the second tile saves
    // (129 rows, one sequence: prefix 512 23.0 against 18.2 us, 2048 30.3
    // against 28.4 us, 8192 49.6 against 60.2 us).
    if (dh == 128 && R > 128 && R - 128 <= kTailMax) {
        const TcPlan t = plan(1, true);
        if (t.chunk / kTcSub >= kTailMinSubs) return t;
    }
    return plan((R + 127) / 128, false);
}

}  // namespace

size_t attention_workspace_bytes(medusa_dtype dtype, int B, int R, int H, int dh, int P_max) {
    if (dtype == MEDUSA_F32) return MEDUSA_WS_HEADER;
    const TcPlan tp = tc_plan(B, H, R, P_max, dh);
    const size_t rows = (size_t)B * H * tp.ns * R;
    return MEDUSA_WS_HEADER + align256(rows * dh * sizeof(float)) + align256(rows * sizeof(float2));
}

cudaError_t launch_tree_attention(medusa_dtype dtype, const void *q, const void *const *k_cache,
                                  const void *const *v_cache, const int32_t *prefix_len,
                                  int P_max, const uint64_t *anc_mask, int B, int R, int H,
                                  int dh, float scale, void *out, void *ws, cudaStream_t stream) {
    int *status = static_cast<int *>(ws);
    cudaError_t e;
    if (dtype == MEDUSA_F32) {
        const size_t smem = (size_t)(dh + P_max + R) * sizeof(float);
        if ((e = cudaFuncSetAttribute(tree_attn_f32_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
            return e;
        e = launch_pdl(tree_attn_f32_kernel, dim3(R, H, B), dim3(128), smem, stream,
                       static_cast<const float *>(q),
                       reinterpret_cast<const float *const *>(k_cache),
                       reinterpret_cast<const float *const *>(v_cache), prefix_len, anc_mask, R, H,
                       dh, P_max, scale, static_cast<float *>(out), status);
        note_launch();
        return e;
    }
    const TcPlan tp = tc_plan(B, H, R, P_max, dh);
    const int NS = tp.ns;
    const size_t rows = (size_t)B * H * NS * R;
    char *w = static_cast<char *>(ws) + MEDUSA_WS_HEADER;
    float *part_o = reinterpret_cast<float *>(w);
    float2 *part_ml = reinterpret_cast<float2 *>(w + align256(rows * dh * sizeof(float)));
    AttnArgs a;
    a.q = static_cast<const bf16 *>(q);
    a.kc = reinterpret_cast<const bf16 *const *>(k_cache);
    a.vc = reinterpret_cast<const bf16 *const *>(v_cache);
    a.prefix_len = prefix_len;
    a.anc_mask = anc_mask;
    a.B = B;
    a.R = R;
    a.H = H;
    a.P_max = P_max;
    a.chunk = tp.chunk;
    a.nps = NS;
    a.row_tiles = tp.row_tiles;
    a.scale_log2 = scale * kLog2e;
    a.wait_polls = wait_budget();
    a.part_o = part_o;
    a.part_ml = part_ml;
    a.status = status;
    const bool wide = tp.row_tiles > 1;
    auto kern = wide ? tree_attn_tc_kernel<64, true, false> : tree_attn_tc_kernel<64, false, false>;
    if (dh == 128)
        kern = tp.tail ? tree_attn_tc_kernel<128, true, true>
               : wide  ? tree_attn_tc_kernel<128, true, false>
                       : tree_attn_tc_kernel<128, false, false>;
    int smem = dh == 128 ? TcSmem<128>::TOTAL : TcSmem<64>::TOTAL;
    if (tp.tail) smem = TcSmem<128>::TOTAL_TAIL;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)))
        return e;
    e = launch_pdl(kern, dim3(H * tp.row_tiles, NS, B), dim3(256), (size_t)smem, stream, a);
    note_launch();
    if (e) return e;
    const long long items = (long long)B * R * H;
    const int cblocks = (int)((items + 7) / 8);
    auto comb = NS <= 4 ? tree_attn_combine_kernel<64, 4>
                : NS <= 8 ? tree_attn_combine_kernel<64, 8> : tree_attn_combine_kernel<64, 16>;
    if (dh == 128)
        comb = NS <= 4 ? tree_attn_combine_kernel<128, 4>
               : NS <= 8 ? tree_attn_combine_kernel<128, 8> : tree_attn_combine_kernel<128, 16>;
    e = launch_pdl(comb, dim3(cblocks), dim3(256), 0, stream, static_cast<const float *>(part_o),
                   static_cast<const float2 *>(part_ml), B, R, H, NS, static_cast<bf16 *>(out));
    note_launch();
    return e;
}

}  // namespace medusa
