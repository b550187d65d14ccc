// Internal interface of the short-sequence (mask-unit) attention kernel.
#pragma once

#include <cuda_runtime.h>

#include "iha.h"

namespace iha {

// Sequences the packed kernel handles: no mask, Nq == Nk <= 64, d <= 128.
bool mu_attention_supported(int Nq, int Nk, int d, int mask);

// Softmax attention of every (b_outer, b_inner, head) sequence of T tokens,
// two sequences per 128-row tile; arguments as mha_fwd (bf16, validated).
// q_stride > 1 (dividing T): the queries are max-pooled to T / q_stride rows
// first (the block index the slow axis), and o / lse hold T / q_stride rows.
iha_status mu_attention_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                            int Bo, int Bi, int Hh, int T, int d, const iha_strides& sq,
                            const iha_strides& sk, const iha_strides& sv, const iha_strides& so,
                            float scale, cudaStream_t stream, int q_stride = 1);

// Gather -> mask-unit attention (Q = K = V = the unit's tokens) -> scatter
// into the canvas in one pass (arguments validated by the entry point).
iha_status mu_attention_fused(const void* x, const int32_t* keep, void* canvas, int B, int grid_h,
                              int grid_w, int mu_h, int mu_w, int n_keep, int C, float scale,
                              cudaStream_t stream);

}  // namespace iha
