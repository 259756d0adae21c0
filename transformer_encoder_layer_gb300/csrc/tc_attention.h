// Host interface of the tcgen05 flash-attention kernel (tc_attention.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "neartie.cuh"

namespace tl {

struct TcAttnArgs {
  // (hi, lo) 16-bit planes: q, k [B, H, L, dh]; v^T [B, H, dh, Lp]
  const void *q_hi, *q_lo, *k_hi, *k_lo, *vt_hi, *vt_lo;
  void *ctx_hi, *ctx_lo;   // [B, L, d] (hi, lo)
  const int32_t* valid_len;
  const int* kmax;         // [B*H] max_j |k_j| as float bits (near-tie test)
  NearTieList ties;
  int B, H, L, Lp, dh, d;
  int* status;
};

bool tc_attention_supported(int dh);
cudaError_t tc_attention(const TcAttnArgs& a, bool bf16, int num_sms, cudaStream_t s);

}  // namespace tl
