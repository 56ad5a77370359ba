// heads_tc.h -- the tensor-core heads path (heads_tc.cu), used by heads.cu
// for batches of several bf16 sequences.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "launch.h"
#include "medusa.h"

namespace medusa {

// Smallest batch the tensor-core path takes.  At one sequence the CUDA-core
// GEMV streams the weights at the HBM rate (216 us for the 7B heads on
// GB300) and the tensor-core path's two-phase set-up costs more (~230 us);
// from two sequences on the CUDA-core GEMV's shared-memory loads of the
// activations slow it (280 us at two, 860 us at eight) while the
// tensor-core path stays at ~230-240 us.
constexpr int kHeadsTcMinBatch = 2;

// Whether launch_heads_tc handles this call (bf16, B in kHeadsTcMinBatch..8,
// d a multiple of 256, V a multiple of 8, enough 8-row units for every CTA;
// top-s mode with or without the LM head, or sampling mode).
bool heads_tc_eligible(medusa_dtype dtype, int B, int d, int V, int K, bool with_lm_head,
                       bool sample);

// CTAs per head in phase 2 (the G of its partials).
int heads_tc_ctas_per_head(int K);

// Bytes of the z operand the two phases share: [K][16][d] bf16.
size_t heads_tc_zt_bytes(int K, int d);

// Phase 1 (z into zt) and phase 2 (partials, index (k * B + b) * G + g with
// G = heads_tc_ctas_per_head(Kt), Kt = K + 1 with the LM head as head 0);
// heads_reduce_kernel merges the partials.  sample (or null): draft mode.
// zt holds heads_tc_zt_bytes(Kt, d).
cudaError_t launch_heads_tc(const void *h, const void *Wlm, const void *W1, const void *b1,
                            const void *W2, int B, int d, int V, int K, int S,
                            const SampleArgs *sample, void *zt, float2 *part_ms, float *part_val,
                            int *part_id, int *status, cudaStream_t stream);

}  // namespace medusa
