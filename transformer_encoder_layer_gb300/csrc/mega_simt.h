// Sequence-resident megakernel on CUDA cores for fp32 I/O and small models.
#pragma once

#include <cuda_runtime.h>

#include "internal.h"

namespace tl {

constexpr int kMegaSimtMaxLayers = 8;

struct MegaSimtArgs {
  tl_layer_dev layers[kMegaSimtMaxLayers];
  int n_layers;
  const float* x;      // [B, L, d]
  float* out;          // [B, L, d]
  const int32_t* vl;   // [B]
  int* status;
  int B, L, d, H, dh, dff;
  int w_stage;         // 1: every layer's weights staged in shared memory (set by the launcher)
};

bool mega_simt_supported(int d, int H, int dff, int L, int n_layers, tl_dtype t);
cudaError_t mega_simt_forward(const MegaSimtArgs& a, cudaStream_t s);

}  // namespace tl
