// LayerNorm application pass for rows normalised across several GEMM N tiles
// (ln_apply.cu).
#pragma once

#include <cuda_runtime.h>

namespace tl {

struct LnApplyArgs {
  const float* r;       // [M, N] pre-normalisation rows (x + a), fp32
  const float2* stats;  // [M][n_parts] (mean, M2) of each row's n_parts column blocks
  const float *gamma, *beta;  // [N]
  int M, N;             // N a multiple of 8; all row pointers 16-byte aligned
  int n_parts;          // column blocks per row (N / n_parts columns each)
  float* o32;           // optional fp32 [M, N]
  void *o_hi, *o_lo;    // optional (hi, lo) planes [M, N] of the I/O type
  void* o_final;        // optional [M, N] in the I/O type (round to nearest)
};

cudaError_t ln_apply(const LnApplyArgs& a, bool bf16, int num_sms, cudaStream_t s);

}  // namespace tl
