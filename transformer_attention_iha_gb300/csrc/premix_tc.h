// Internal interface between the premix entry points and the tensor-core
// premix kernels.
#pragma once

#include <cuda_runtime.h>

#include "iha.h"

namespace iha {

// RoPE inverse frequencies inv_freq_i = base^(-2i/d) (i < d/2, up to 64),
// computed in double on the host and carried as an fp32 pair hi + lo.
struct RopeTable {
  float hi[64];
  float lo[64];
};
void make_rope_table(RopeTable* rt, int d, float base);

// Shapes the tensor-core premix handles: bf16, d in {64, 128}, H <= 32,
// H*P <= 128.
bool premix_tc_supported(int H, int P, int d);

// Backward shapes: bf16, d = 128, H <= 32, H*P <= 128, and the kernel variant
// (dX and / or dW, with or without RoPE) fits in shared memory.
bool premix_bwd_tc_supported(int H, int P, int d, bool do_dx, bool do_dw, bool rope);

// dX (if dx != nullptr) and dW (if dw != nullptr, accumulated with atomics
// into a zeroed dw) in one pass over dY.
iha_status premix_bwd_tc(const void* dy, const void* x, const float* w, void* dx, float* dw,
                         int B, int N, int H, int P, int d, int rope, float rope_base,
                         cudaStream_t stream);

// The same over ntens (1..3) tensors in one launch: tensor t reads dy[t],
// x[t], w[t] and writes dx[t] / dw[t] (all dx null or all non-null, the same
// for dw), rotated when bit t of rope_mask is set; every dw[t] zeroed first.
iha_status premix_bwd_tc_multi(int ntens, const void* const* dy, const void* const* x,
                               const float* const* w, void* const* dx, float* const* dw, int B,
                               int N, int H, int P, int d, int rope_mask, float rope_base,
                               cudaStream_t stream);

iha_status premix_fwd_tc(const void* x, const float* w, void* y, int B, int N, int H, int P,
                         int d, int rope, float rope_base, cudaStream_t stream);

// The same forward over ntens (1..3) tensors in one launch; tensor t reads
// x[t], w[t], writes y[t], and is rotated when bit t of rope_mask is set.
// interleave: Y rows ordered p * H + h ([B, N, P, H, d]) instead of h * P + p.
iha_status premix_fwd_tc_multi(int ntens, const void* const* x, const float* const* w,
                               void* const* y, int B, int N, int H, int P, int d, int rope_mask,
                               float rope_base, cudaStream_t stream, int interleave = 0);

}  // namespace iha
