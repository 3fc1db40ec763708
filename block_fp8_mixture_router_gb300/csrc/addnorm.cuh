// The residual add + RMS norm kernel in front of the layer (k_addnorm.cu).
#pragma once

#include "moe_internal.cuh"

namespace moe {

constexpr int kAddNormMaxHidden = 8192;  // widest row the add-norm kernel takes

// residual add + RMS norm + FP8 groups of the normed rows, one CTA per row;
// pdl: launched with programmatic dependent launch (it waits for the
// previous kernel before reading its inputs)
cudaError_t launch_add_rmsnorm_quant(const bf16* residual, const bf16* x, const bf16* gamma,
                                     float eps, int rows, int H, bf16* h_out, bf16* xn_out,
                                     uint8_t* codes, float* scales, cudaStream_t s,
                                     bool pdl = false);

}  // namespace moe
