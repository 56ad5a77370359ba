// heads_tc.cu -- the Medusa heads on the tensor cores, for batches of several
// sequences (bf16).
//
// Same computation as heads.cu ("Medusa 深读" §3.1, the equation for
// p_t^(k); "Medusa Part I" Part 3, ResidualBlock and the bias-free vocabulary
// projection; top-s per head, "Medusa 深读" §6.1):
//     u = W1[k] h[b] + b1[k];  z = h[b] + SiLU(u);  logits = W2[k] z
//
// Why tensor cores here.  With B sequences each weight element meets B
// activations.  On CUDA cores every 16-byte weight vector costs 2B shared
// loads of fp32 activations, which caps a batch of 8 at about a quarter of
// HBM bandwidth.  As an MMA the weights are the A operand (up to 128 rows x
// 64 columns per stage, straight from HBM by TMA) and the activations the B
// operand (N = 16 rows), so the weight stream runs at the HBM rate and the
// tensor cores idle most of the time.
//
// B operand.  Phase 1 multiplies by h (bf16 input; rows B..15 of the box are
// outside the tensor and read as zero).  Phase 2 multiplies by z, which
// phase 1 writes as two bf16 rows per sequence: zt[k][b] = bf16(z) and
// zt[k][8+b] = bf16(z - bf16(z)); logit = D[b] + D[8+b] carries z to about
// 2^-16 relative (a logit error near 1e-5 at d = 4096), where a single bf16 z
// would move logits by ~1e-3.
//
// Work split.  A CTA per SM (192 threads): warp 0 issues the TMA copies,
// warp 1 the MMAs, warps 2-5 read the accumulators.  A ring of 3 stages
// runs ahead of the MMAs across tile boundaries; a stage holds 4 K-blocks
// (4 x 64 columns) of a tile's weight rows and the matching 16-row B tile
// (at most 64 + 8 KB), each brought by one 3-D copy (the number of copies,
// not their bytes, bounded the stream when a stage took one copy per box).
// Rows are handed out in 8-row units: phase 1 spreads the K*d rows of W1
// evenly over every CTA (h is shared by all heads); phase 2 gives each head
// the same number of CTAs and spreads the head's V rows over them, so a
// CTA's z never changes.  A CTA's rows form tiles of at most 128 rows (near-
// equal multiples of 8, one tensor map per tile height).  Each of a stage's
// four K-slices (K = 16 per MMA) accumulates into its own 128-lane x
// 16-column accumulator, since an N = 16 MMA is too short to hide the wait
// on the previous one into the same accumulator; the epilogue adds the
// four.  Two tiles' accumulators sit in tensor memory, so the epilogue of
// one overlaps the MMAs of the next.  Phase 1's epilogue applies bias, SiLU
// and the residual and writes zt; phase 2's keeps, per sequence, each
// thread's running (max, sum-exp) and
// a per-warp top-s list (candidates pass a threshold test by ballot; the few
// that pass are inserted one by one), then merges the warps and writes one
// partial per (head, sequence, CTA) for heads_reduce_kernel.
//
// Every mbarrier wait is bounded (medusa_set_wait_budget); on a timeout the
// CTA records MEDUSA_DEV_TIMEOUT, stops, drains its copies and MMAs with a
// fixed limit and frees its tensor memory (MEDUSA_DEV_DRAIN_TIMEOUT if the
// drain also gives up).
#include <cuda.h>  // CUtensorMap and its enums (the encoder comes from the driver at run time)

#include <algorithm>
#include <climits>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "heads_tc.h"
#include "launch.h"
#include "philox.cuh"
#include "tcgen05.cuh"
#include "topk.cuh"

namespace medusa {

namespace {

constexpr int kTcThreads = 192;                 // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kRing = 3;                        // ring stages
constexpr int kTileRows = 128;                  // M of one MMA tile
constexpr int kKb = 64;                         // K elements per K-block (one 128-byte row)
constexpr int kKbs = 4;                         // K-blocks per stage
constexpr int kWBytes = kKbs * kTileRows * 128; // weight part of a stage (64 KB)
constexpr int kBRows = 16;                      // N: rows of the B operand
constexpr int kBBytes = kKbs * kBRows * 128;    // B part of a stage (8 KB)
constexpr int kSlotBytes = kWBytes + kBBytes;   // 72 KB, a multiple of 1024
constexpr int kMaxMaps = 6;                     // distinct tile heights per phase
constexpr int kAccCols = 16;                    // fp32 columns of one accumulator (N)
constexpr int kNAcc = kKb / 16;                 // accumulators per tile: one per K-slice
constexpr int kTileCols = kNAcc * kAccCols;     // 64 columns per tile
constexpr int kTmemCols = 2 * kTileCols;        // two tiles in flight
constexpr int kEpiWarps = 4;
constexpr int kMaxB = 8;
constexpr uint32_t kDrainPolls = 1u << 16;      // the drain's own limit

// Weights and B operand are read through 3-D views [K-block][row][64]: one
// copy brings kKbs K-blocks of a tile's rows and lands as kKbs consecutive
// [rows][128 B] swizzled blocks, the layout the MMA reads.
struct TcMaps {
    CUtensorMap w[kMaxMaps];    // weight rows: box (64, height of map i, kKbs)
    CUtensorMap wlm[kMaxMaps];  // phase 2 with the LM head: W_lm's rows, same boxes
    CUtensorMap b;              // B operand: box (64, 16, kKbs)
};

struct TcArgs {
    int phase;          // 1: W1 h -> zt; 2: W2 z -> partial softmax + top-s
    int B, d, V, K, S;
    int cph;            // phase 2: CTAs per head
    int8_t map_of[17];  // tile height / 8 -> index into TcMaps::w
    int lm;             // 1: the LM head is head 0 of phase 2 (z = h), the Medusa heads follow
    // sampling (phase 2): one draft per head, the top-1 of logit/T + Gumbel
    // noise (Philox stream purpose 1, row = head, key (seed, step)), raw
    // logits to logits_out [B][K][V]
    int sample;
    float inv_T;
    uint64_t seed, step;
    float *logits_out;
    const bf16 *h;      // [B][d]
    const bf16 *b1;     // [K][d] or null
    bf16 *zt;           // [K][16][d] (phase 1 writes it, phase 2 reads it by TMA)
    float2 *part_ms;    // phase 2 partials, index (k * B + b) * cph + j
    float *part_val;
    int *part_id;
    int *status;
    uint32_t wait_polls;
};

// Shared memory: 1 KB of alignment slack, the ring, then the barriers and
// the epilogue's merge slots.
struct TcSmem {
    static constexpr int RING = kRing * kSlotBytes;
    static constexpr int BARS = RING;                              // uint64 barriers
    static constexpr int NBARS = 2 * kRing + 4 + 1;                // full, empty, acc f/e, drain
    static constexpr int MISC = BARS + NBARS * 8;                  // tmem holder, flags
    static constexpr int SLOTS = (MISC + 16 + 15) / 16 * 16;       // TopSlot [4 warps][8]
    static constexpr int TOTAL = SLOTS + kEpiWarps * kMaxB * (int)sizeof(TopSlot);
    static constexpr int ALLOC = TOTAL + 1024;
};
// an 8-row-B stage's last K-block lets the MMA read 8 rows (1 KB) past the
// slot; past the last slot those bytes must still lie inside the CTA's block
static_assert(TcSmem::TOTAL - TcSmem::RING >= 1024, "guard after the ring");

// This CTA's rows: [row0, row0 + 8 * units) of its weight matrix, the token
// id of its first row (phase 2) and (phase 2) its head in the pass.
struct Span {
    int row0, units, head, tok0;
};

__device__ __forceinline__ Span cta_span(const TcArgs &a) {
    Span s;
    if (a.phase == 1) {
        const long long U = (long long)a.K * a.d / 8, G = gridDim.x, g = blockIdx.x;
        const int u0 = (int)(g * U / G), u1 = (int)((g + 1) * U / G);
        s.row0 = u0 * 8;
        s.units = u1 - u0;
        s.head = 0;
        s.tok0 = 0;
    } else {
        const int k = blockIdx.x / a.cph, j = blockIdx.x - k * a.cph;
        const long long U = a.V / 8;
        const int u0 = (int)(j * U / a.cph), u1 = (int)((j + 1) * U / a.cph);
        // with the LM head, head 0 reads W_lm and head k >= 1 reads W2's
        // head k - 1
        s.row0 = (a.lm && k == 0 ? 0 : (k - a.lm) * a.V) + u0 * 8;
        s.units = u1 - u0;
        s.head = k;
        s.tok0 = u0 * 8;
    }
    return s;
}

// Tile t of T = ceil(units / 16): rows [first, first + rows) relative to
// the span, near-equal multiples of 8 of at most 128.
__device__ __forceinline__ void tile_of(const Span &sp, int T, int t, int &first, int &rows) {
    const int a = (int)((long long)t * sp.units / T), b = (int)((long long)(t + 1) * sp.units / T);
    first = a * 8;
    rows = (b - a) * 8;
}

__device__ __forceinline__ void grid_wait() {
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
__device__ __forceinline__ void grid_trigger() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

__device__ __forceinline__ void named_sync_epi() {
    asm volatile("bar.sync 1, %0;\n" ::"r"(kEpiWarps * kWarp) : "memory");
}

// the MMA warp and the epilogue warps (tensor-memory hand-over)
__device__ __forceinline__ void named_sync_mma_epi() {
    asm volatile("bar.sync 2, %0;\n" ::"r"((kEpiWarps + 1) * kWarp) : "memory");
}

__global__ void __launch_bounds__(kTcThreads, 1)
heads_tc_kernel(const __grid_constant__ TcMaps maps, const TcArgs a) {
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte alignment (in the shared window) for the 128-byte-swizzled tiles
    unsigned char *smem = smem_raw + ((1024u - (tc::smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + TcSmem::BARS);
    uint64_t *full = bars;                   // [kRing] TMA landed
    uint64_t *empty = bars + kRing;          // [kRing] MMAs done reading
    uint64_t *acc_full = bars + 2 * kRing;   // [2] accumulator complete
    uint64_t *acc_empty = acc_full + 2;      // [2] accumulator read out
    uint64_t *drain = acc_full + 4;          // the MMA thread's final commit
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + TcSmem::MISC);
    volatile int *err = reinterpret_cast<volatile int *>(smem + TcSmem::MISC + 4);
    int *consumed = reinterpret_cast<int *>(smem + TcSmem::MISC + 8);
    TopSlot *slots = reinterpret_cast<TopSlot *>(smem + TcSmem::SLOTS);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Span sp = cta_span(a);
    const int T = (sp.units + 15) / 16;
    const int nkb = a.d / (kKb * kKbs);  // stages per tile
    const int total = T * nkb;           // stages of this CTA

    if (tid == 0) {
        for (int i = 0; i < kRing; ++i) {
            tc::mbar_init(&full[i], 1);
            tc::mbar_init(&empty[i], 1);
        }
        tc::mbar_init(&acc_full[0], 1);
        tc::mbar_init(&acc_full[1], 1);
        tc::mbar_init(&acc_empty[0], kEpiWarps);
        tc::mbar_init(&acc_empty[1], kEpiWarps);
        tc::mbar_init(drain, 1);
        tc::fence_mbarrier_init();
        *err = 0;
        *consumed = 0;
    }
    __syncthreads();
    // Tensor memory is allocated only after the wait for the previous grid
    // (by the MMA warp, which then meets the epilogue warps), so this CTA
    // never holds columns while an earlier grid may still need some.
    uint32_t tmem = 0;
    auto take_tmem = [&]() {
        if (warp == 1) tc::tmem_alloc(tmem_holder, kTmemCols);
        tc::fence_before_sync();
        named_sync_mma_epi();
        tc::fence_after_sync();
        tmem = *tmem_holder;
    };

    // stage i -> ring slot i % kRing: the rows of tile i / nkb at K-blocks
    // kKbs * (i % nkb) .. + kKbs - 1, in one copy (the number of copies, not
    // their bytes, bounds the TMA stream: ~160 ns per copy per SM measured)
    auto issue_w = [&](int i) {
        const int s = i % kRing, t = i / nkb, kg = i - t * nkb;
        int first, rows;
        tile_of(sp, T, t, first, rows);
        tc::mbar_arrive_expect_tx(&full[s], (uint32_t)(kKbs * (rows * 128 + kBRows * 128)));
        const CUtensorMap *wm = a.lm && a.phase == 2 && sp.head == 0 ? maps.wlm : maps.w;
        tc::tma_load_3d(smem + s * kSlotBytes, &wm[a.map_of[rows / 8]], 0, sp.row0 + first,
                        kg * kKbs, &full[s]);
    };
    auto issue_b = [&](int i) {
        const int s = i % kRing, kg = i % nkb;
        tc::tma_load_3d(smem + s * kSlotBytes + kWBytes, &maps.b, 0,
                        a.phase == 1 ? 0 : sp.head * kBRows, kg * kKbs, &full[s]);
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ---
        int issued = 0;
        if (lane == 0) {
            for (int mi = 0; mi < kMaxMaps; ++mi) {
                tc::prefetch_tmap(&maps.w[mi]);
                if (a.lm) tc::prefetch_tmap(&maps.wlm[mi]);
            }
            tc::prefetch_tmap(&maps.b);
            // The weights are never written by any kernel: the first stages'
            // weight boxes go out before the wait for the previous grid; their
            // B tiles (h from the caller, z from phase 1) after it.
            const int pre = min(kRing, total);
            for (int i = 0; i < pre; ++i) issue_w(i);
            grid_wait();
            grid_trigger();
            for (int i = 0; i < pre; ++i) issue_b(i);
            issued = pre;
            for (int i = pre; i < total; ++i) {
                const int s = i % kRing;
                if (*err) break;
                if (!tc::mbar_wait_bounded(&empty[s], ((i / kRing) - 1) & 1, a.wait_polls)) {
                    *err = 1;
                    break;
                }
                issue_w(i);
                issue_b(i);
                issued = i + 1;
            }
        } else {
            grid_wait();
            grid_trigger();
        }
        __syncwarp();
        __syncthreads();  // (A) every role has left its loop
        if (lane == 0) {
            // copies still in flight (only after a failure): wait for them
            // before the shared memory is released
            bool ok = true;
            for (int i = *consumed; i < issued; ++i)
                ok &= tc::mbar_wait_bounded(&full[i % kRing], (i / kRing) & 1, kDrainPolls);
            if (!ok) *err = 2;
        }
        __syncthreads();  // (B)
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer ---
        grid_wait();
        grid_trigger();
        take_tmem();
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16(kTileRows, kBRows, 0);
            int i = 0;
            for (int t = 0; t < T && !*err; ++t) {
                const int acc = t & 1;
                if (t >= 2 &&
                    !tc::mbar_wait_bounded(&acc_empty[acc], ((t >> 1) - 1) & 1, a.wait_polls)) {
                    *err = 1;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t d_tm = tmem + acc * kTileCols;
                int first, rows;
                tile_of(sp, T, t, first, rows);
                for (int kg = 0; kg < nkb; ++kg, ++i) {
                    const int s = i % kRing;
                    if (!tc::mbar_wait_bounded(&full[s], (i / kRing) & 1, a.wait_polls)) {
                        *err = 1;
                        break;
                    }
                    *consumed = i + 1;
                    tc::fence_after_sync();
                    const uint32_t wa = tc::smem_addr(smem + s * kSlotBytes);
                    const uint32_t ba = wa + kWBytes;
                    // K-block e of the stage: the tile's rows at wa + e * rows
                    // * 128 (rows past the tile read neighbouring bytes of the
                    // stage; their accumulator lanes are never used).  K-slice
                    // ks accumulates into its own 16 columns: an N = 16 MMA is
                    // short, and MMAs into one accumulator wait on each other.
#pragma unroll
                    for (int e = 0; e < kKbs; ++e)
#pragma unroll
                        for (int ks = 0; ks < kNAcc; ++ks)
                            tc::mma_bf16_ss(
                                d_tm + ks * kAccCols,
                                tc::sdesc_sw128(wa + e * rows * 128 + ks * 32, 16, 1024),
                                tc::sdesc_sw128(ba + e * kBRows * 128 + ks * 32, 16, 1024), idesc,
                                (kg | e) != 0 ? 1u : 0u);
                    tc::mma_commit(&empty[s]);  // the slot may be refilled
                }
                if (*err) break;
                tc::mma_commit(&acc_full[acc]);
            }
        }
        __syncwarp();
        __syncthreads();  // (A)
        if (lane == 0) {
            // every MMA this thread issued has finished before tensor memory
            // is freed
            tc::mma_commit(drain);
            if (!tc::mbar_wait_bounded(drain, 0, kDrainPolls)) *err = 2;
        }
        __syncthreads();  // (B)
    } else {
        // ------------------------------------------------------ epilogue ---
        grid_wait();
        grid_trigger();
        take_tmem();
        const int q = warp & 3;  // tensor-memory lane quarter of this warp
        const int B = a.B;
        if (a.phase == 1 && a.lm) {
            // the LM head multiplies h itself: its B-operand rows are h (value
            // rows) and zero (remainder rows); every CTA copies a share
            const int n = kBRows * a.d, e0 = (int)((long long)blockIdx.x * n / gridDim.x),
                      e1 = (int)((long long)(blockIdx.x + 1) * n / gridDim.x);
            for (int e = e0 + threadIdx.x - 64; e < e1; e += kEpiWarps * kWarp) {
                const int r = e / a.d, j = e - r * a.d;
                a.zt[e] = r < B ? a.h[(size_t)r * a.d + j] : __float2bfloat16_rn(0.f);
            }
        }
        // phase 2 running state: per sequence, this thread's (max, sum-exp)
        // and the warp's top-s list (entry i in lane i)
        float m_run[kMaxB], s_run[kMaxB], l_val[kMaxB];
        int l_id[kMaxB];
#pragma unroll
        for (int b = 0; b < kMaxB; ++b) {
            m_run[b] = -INFINITY;
            s_run[b] = 0.f;
            l_val[b] = -INFINITY;
            l_id[b] = INT_MAX;
        }
        bool ok = true;
        for (int t = 0; t < T; ++t) {
            const int acc = t & 1;
            // warp-uniform decision: the lanes go on to full-warp shuffles
            const bool got = *err == 0 &&
                             tc::mbar_wait_bounded(&acc_full[acc], (t >> 1) & 1, a.wait_polls);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            float D[kAccCols];
            {
                // the tile's four K-slice accumulators, summed in a fixed order
                float x0[32], x1[32];
                const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + acc * kTileCols;
                tc::tmem_ld32(ta, x0);
                tc::tmem_ld32(ta + 32, x1);
#pragma unroll
                for (int c = 0; c < kAccCols; ++c)
                    D[c] = (x0[c] + x0[kAccCols + c]) + (x1[c] + x1[kAccCols + c]);
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&acc_empty[acc]);
            int first, rows;
            tile_of(sp, T, t, first, rows);
            const int row = q * 32 + lane;
            const bool valid = row < rows;
            const int r = sp.row0 + first + row;  // global weight row
            if (a.phase == 1) {
                if (valid) {
                    const int k = r / a.d, j = r - k * a.d;
                    const float bias = a.b1 ? Vec16<bf16>::load1(a.b1 + r) : 0.f;
                    bf16 *zk = a.zt + (size_t)(k + a.lm) * kBRows * a.d + j;
#pragma unroll
                    for (int b = 0; b < kMaxB; ++b) {
                        bf16 hi = __float2bfloat16_rn(0.f), lo = hi;
                        if (b < B) {
                            const float u = D[b] + bias;
                            const float z = Vec16<bf16>::load1(a.h + (size_t)b * a.d + j) +
                                            u / (1.f + expf(-u));
                            hi = __float2bfloat16_rn(z);
                            lo = __float2bfloat16_rn(z - __bfloat162float(hi));
                        }
                        zk[(size_t)b * a.d] = hi;
                        zk[(size_t)(kMaxB + b) * a.d] = lo;
                    }
                }
            } else {
                const int v = sp.tok0 + first + row;  // token id
#pragma unroll
                for (int b = 0; b < kMaxB; ++b) {
                    if (b >= B) break;
                    const float logit = D[b] + D[kMaxB + b];
                    // sampling ranks y + Gumbel noise and normalises y = logit / T
                    float x = logit, y = logit;
                    if (a.sample) {
                        y = logit * a.inv_T;
                        x = valid ? y + gumbel_at(a.seed, a.step, kRngDraft, b, sp.head, v)
                                  : -INFINITY;
                        if (valid && a.logits_out)
                            a.logits_out[((size_t)b * a.K + sp.head) * a.V + v] = logit;
                    }
                    if (valid) {
                        if (y > m_run[b]) {
                            s_run[b] = s_run[b] * expf(m_run[b] - y) + 1.f;
                            m_run[b] = y;
                        } else {
                            s_run[b] += expf(y - m_run[b]);
                        }
                    }
                    // top-s: lanes whose candidate beats the list's last entry
                    const float tv = __shfl_sync(0xffffffffu, l_val[b], a.S - 1);
                    const int ti = __shfl_sync(0xffffffffu, l_id[b], a.S - 1);
                    unsigned pass = __ballot_sync(0xffffffffu, valid && better(x, v, tv, ti));
                    while (pass) {
                        const int src = __ffs(pass) - 1;
                        pass &= pass - 1;
                        const float cv = __shfl_sync(0xffffffffu, x, src);
                        const int cid = __shfl_sync(0xffffffffu, v, src);
                        WarpTop lt;
                        lt.val = l_val[b];
                        lt.id = l_id[b];
                        lt.insert(cv, cid, a.S, lane);
                        l_val[b] = lt.val;
                        l_id[b] = lt.id;
                    }
                }
            }
        }
        if (!ok && !*err) *err = 1;
        if (a.phase == 2) {
            // the warps' states per sequence, then one partial per (head,
            // sequence, CTA)
            const int e = warp - 2;
#pragma unroll
            for (int b = 0; b < kMaxB; ++b) {
                if (b >= B) break;
                WarpTop st;
                st.m = m_run[b];
                st.s = s_run[b];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float om = __shfl_xor_sync(0xffffffffu, st.m, o);
                    const float os = __shfl_xor_sync(0xffffffffu, st.s, o);
                    st.merge_ms(om, os);
                }
                st.val = l_val[b];
                st.id = l_id[b];
                flush_slot(slots[e * kMaxB + b], st, a.S, lane);
            }
            named_sync_epi();
            if (__all_sync(0xffffffffu, *err == 0)) {
                const int j = blockIdx.x - sp.head * a.cph;
                for (int b = e; b < B; b += kEpiWarps) {
                    float m, sum;
                    warp_merge_ms(slots + b, kMaxB, kEpiWarps, lane, m, sum);
                    float tv;
                    int ti;
                    warp_merge_top(slots + b, kMaxB, kEpiWarps, a.S, lane, tv, ti);
                    const size_t o = ((size_t)sp.head * B + b) * a.cph + j;
                    if (lane == 0) a.part_ms[o] = make_float2(m, sum);
                    if (lane < a.S) {
                        a.part_val[o * a.S + lane] = tv;
                        a.part_id[o * a.S + lane] = ti;
                    }
                }
            }
        }
        __syncthreads();  // (A)
        __syncthreads();  // (B)
    }
    // (B) passed: copies landed, MMAs finished
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
    if (tid == 0 && *err && a.status) {
        if (*err == 2)
            atomicExch(a.status, MEDUSA_DEV_DRAIN_TIMEOUT);
        else
            set_status(a.status, MEDUSA_DEV_TIMEOUT);
    }
}

// ------------------------------------------------------------- host ---

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiled>(nullptr);
        return reinterpret_cast<EncodeTiled>(p);
    }();
    return fn;
}

// Tensor maps are plain host-side descriptors; encoding them costs host time
// only, so the last few are kept by (address, shape, box).
struct MapKey {
    const void *base;
    uint64_t rows, cols;
    uint32_t box_rows;
    bool operator==(const MapKey &o) const {
        return base == o.base && rows == o.rows && cols == o.cols && box_rows == o.box_rows;
    }
};

// 3-D view [cols / 64][rows][64] of a row-major bf16 [rows][cols] matrix
// (strides: a row, then 128 bytes for the next K-block), box (64, box_rows,
// kKbs), 128-byte swizzle, zero fill outside.
bool encode_rows(CUtensorMap *out, const void *base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows) {
    static std::mutex mu;
    static std::vector<std::pair<MapKey, CUtensorMap>> cache;
    const MapKey key{base, rows, cols, box_rows};
    std::lock_guard<std::mutex> lock(mu);
    for (auto &e : cache)
        if (e.first == key) {
            *out = e.second;
            return true;
        }
    EncodeTiled fn = encoder();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kKb, rows, cols / kKb};
    const cuuint64_t strides[2] = {cols * 2, (cuuint64_t)kKb * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kKb, box_rows, (cuuint32_t)kKbs};
    const cuuint32_t es[3] = {1, 1, 1};
    if (fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
           es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    if (cache.size() >= 64) cache.erase(cache.begin());
    cache.emplace_back(key, *out);
    return true;
}

cudaError_t launch_phase(const TcMaps &maps, const TcArgs &a, int grid, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(heads_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TcSmem::ALLOC);
    if (e) return e;
    e = launch_pdl(heads_tc_kernel, dim3(grid), dim3(kTcThreads), (size_t)TcSmem::ALLOC, stream,
                   maps, a);
    note_launch();
    return e;
}

}  // namespace

bool heads_tc_eligible(medusa_dtype dtype, int B, int d, int V, int K, bool with_lm_head,
                       bool sample) {
    if (dtype != MEDUSA_BF16 || (with_lm_head && sample)) return false;
    if (B < kHeadsTcMinBatch || B > kMaxB) return false;
    if (d % (kKb * kKbs) || d > 16384 || V % 8 || V < 8) return false;
    const int sms = device_sm_count();
    const int Kt = K + (with_lm_head ? 1 : 0);
    // every CTA needs at least one 8-row unit in both phases
    return (long long)K * d / 8 >= sms && V / 8 >= std::max(1, sms / Kt);
}

int heads_tc_ctas_per_head(int K) { return std::max(1, device_sm_count() / K); }

size_t heads_tc_zt_bytes(int K, int d) { return (size_t)K * kBRows * d * sizeof(uint16_t); }

// The tile heights (in 8-row units) the device's partition produces: for G
// spans of a range of U units, split like cta_span / tile_of.  Heights go
// into `units` (distinct, at most kMaxMaps; false if more).
bool tile_heights(long long U, int G, std::vector<int> &units) {
    for (int g = 0; g < G; ++g) {
        const int n = (int)((g + 1) * U / G - g * U / G);
        const int T = (n + 15) / 16;
        for (int t = 0; t < T; ++t) {
            const int u = (int)((long long)(t + 1) * n / T - (long long)t * n / T);
            if (std::find(units.begin(), units.end(), u) == units.end()) units.push_back(u);
        }
    }
    return units.size() <= (size_t)kMaxMaps;
}

bool plan_maps(TcMaps &m, TcArgs &a, const void *W, uint64_t rows, int d, long long U, int G) {
    std::vector<int> units;
    if (!tile_heights(U, G, units)) return false;
    for (int i = 0; i < 17; ++i) a.map_of[i] = 0;
    for (size_t i = 0; i < units.size(); ++i) {
        if (units[i] < 1 || units[i] > 16) return false;
        a.map_of[units[i]] = (int8_t)i;
        if (!encode_rows(&m.w[i], W, rows, (uint64_t)d, (uint32_t)(units[i] * 8))) return false;
    }
    for (size_t i = units.size(); i < (size_t)kMaxMaps; ++i) m.w[i] = m.w[0];
    return true;
}

cudaError_t launch_heads_tc(const void *h, const void *Wlm, const void *W1, const void *b1,
                            const void *W2, int B, int d, int V, int K, int S,
                            const SampleArgs *sample, void *zt, float2 *part_ms, float *part_val,
                            int *part_id, int *status, cudaStream_t stream) {
    const int sms = device_sm_count();
    const int lm = Wlm ? 1 : 0;
    const int Kt = K + lm;  // heads of phase 2
    const int cph = heads_tc_ctas_per_head(Kt);
    // phase 1: 8 K-blocks a stage (tiles of up to 64 rows) where d allows
    TcMaps m1, m2;
    TcArgs a1 = {}, a2 = {};
    if (!plan_maps(m1, a1, W1, (uint64_t)K * d, d, (long long)K * d / 8, sms) ||
        !plan_maps(m2, a2, W2, (uint64_t)K * V, d, V / 8, cph)) {
        set_last_error("tensor maps for the heads' weights could not be made "
                       "(cuTensorMapEncodeTiled failed or too many tile heights)");
        return cudaErrorInvalidValue;
    }
    // phase 1 has no LM-head rows; phase 2's W_lm maps share W2's tile heights
    for (int i = 0; i < kMaxMaps; ++i) m1.wlm[i] = m1.w[i];
    if (lm) {  // the same partition of V rows per head: the same tile heights, in order
        TcArgs alm = {};
        TcMaps tmp;
        if (!plan_maps(tmp, alm, Wlm, (uint64_t)V, d, V / 8, cph)) {
            set_last_error("tensor maps for the LM head could not be made");
            return cudaErrorInvalidValue;
        }
        for (int i = 0; i < kMaxMaps; ++i) m2.wlm[i] = tmp.w[i];
    } else {
        for (int i = 0; i < kMaxMaps; ++i) m2.wlm[i] = m2.w[i];
    }
    if (!encode_rows(&m1.b, h, (uint64_t)B, (uint64_t)d, kBRows) ||
        !encode_rows(&m2.b, zt, (uint64_t)Kt * kBRows, (uint64_t)d, kBRows)) {
        set_last_error("cuTensorMapEncodeTiled failed for the heads' activations");
        return cudaErrorInvalidValue;
    }
    TcArgs a = {};
    a.B = B;
    a.d = d;
    a.V = V;
    a.K = K;
    a.S = S;
    a.h = static_cast<const bf16 *>(h);
    a.b1 = static_cast<const bf16 *>(b1);
    a.zt = static_cast<bf16 *>(zt);
    a.part_ms = part_ms;
    a.part_val = part_val;
    a.part_id = part_id;
    a.status = status;
    a.wait_polls = wait_budget();
    a.lm = lm;
    if (sample && sample->on) {
        a.sample = 1;
        a.inv_T = sample->inv_T;
        a.seed = sample->seed;
        a.step = sample->step;
        a.logits_out = sample->logits_out;
    }
    a.phase = 1;
    a.cph = 1;
    std::copy(a1.map_of, a1.map_of + 17, a.map_of);
    cudaError_t e = launch_phase(m1, a, sms, stream);
    if (e) return e;
    a.phase = 2;
    a.cph = cph;
    a.K = Kt;
    std::copy(a2.map_of, a2.map_of + 17, a.map_of);
    return launch_phase(m2, a, cph * Kt, stream);
}

}  // namespace medusa
