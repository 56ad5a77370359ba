// common.cuh -- device helpers shared by the Medusa step kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "medusa.h"

namespace medusa {

constexpr int kWarp = 32;

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------------- loads ---

// 16-byte streaming load: read-only path, no L1 allocation (weights and
// logits are touched once per step).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// Bulk prefetch of `bytes` (multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}

// 2^x by the hardware's approximate exponential (ex2.approx.ftz: relative
// error ~2^-22, subnormal results flushed to 0, -inf gives +0).  Used where
// the result is rounded to bf16 next (attention weights) or only compared in
// the log domain (posterior sums).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Three-input maximum, one instruction on this architecture; like fmaxf, a
// NaN operand is ignored unless all three are NaN.
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// bf16 pair packed in a 32-bit word -> two floats (exact widening).
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float bf16_to_f(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Element type traits: how many elements one 16-byte vector holds and how to
// widen them to fp32.
template <typename T> struct Vec16;

template <> struct Vec16<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void widen(const uint4 &v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static float load1(const float *p) { return __ldg(p); }
};

template <> struct Vec16<bf16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void widen(const uint4 &v, float (&f)[8]) {
        f[0] = bf_lo(v.x); f[1] = bf_hi(v.x);
        f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
        f[4] = bf_lo(v.z); f[5] = bf_hi(v.z);
        f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
    }
    __device__ __forceinline__ static float load1(const bf16 *p) {
        return bf16_to_f(__ldg(reinterpret_cast<const unsigned short *>(p)));
    }
};

// ----------------------------------------------------------- reductions ---

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// (value, id) ordering used for every top-k and argmax: larger value first,
// equal values -> smaller id first.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

// ---------------------------------------------- programmatic dependent launch
//
// Every kernel of the step is launched with programmatic stream serialization
// (see launch_pdl).  At its start a kernel waits for the grid before it in the
// stream to complete and flush (griddepcontrol.wait) and then lets the next
// grid begin launching (griddepcontrol.launch_dependents), so the next
// kernel's launch overlaps this one's execution instead of following its
// completion.  The next grid cannot start before every CTA of this grid has
// started and passed the trigger, and it waits for this grid's completion
// before touching memory; both instructions are no-ops for a kernel launched
// without the attribute.
//
// The order -- wait, then trigger -- is relied on by the kernels that read
// inputs before their own wait: posterior_select_kernel (tree arrays, the
// typical-acceptance logits and, with the fused commit, the cache pointers
// and prefix lengths), spec_sample_kernel and spec_select_kernel
// (draft tokens, their p and q logits and uniforms; the chain's tokens), and
// the L2 prefetches of heads_w1/heads_w2 (weights, never written) and of
// posterior_rows_kernel (its slice of the logits: a prefetch consumes no
// data, so it would be safe even if an earlier grid were writing them).  Because
// every kernel of the library waits before it triggers, a kernel that starts
// early can only overlap its immediate predecessor; all older grids have
// completed and their writes are visible.  Triggering before the wait in any
// kernel would turn those early reads into races with the grid before it.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// ------------------------------------------------------- device status ---

__device__ __forceinline__ void set_status(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

}  // namespace medusa
