// Host interface of the sequence-resident megakernel (mega.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tl_encoder.h"

namespace tl {

// One layer, as the megakernel reads it (device memory, built at create).
struct MegaLayer {
  const CUtensorMap* map_qkv;  // W_qkv [384, 128], box 64 x 128, 128-byte swizzle
  const CUtensorMap* map_o;    // W_o [128, 128]
  const CUtensorMap* map_1;    // W_1 [d_ff, 128], box 64 x 128
  const CUtensorMap* map_2;    // W_2 [128, d_ff]
  const void* w_qkv;           // raw W_qkv (near-tie correction)
  const float *b_qkv, *b_o, *ln1_g, *ln1_b, *b_1, *b_2, *ln2_g, *ln2_b;
};

struct MegaArgs {
  const MegaLayer* layers;  // device array [n_layers]
  int n_layers, B, dff;
  const int32_t* valid_len;
  void* out;
  int* status;
  // Assisted mode (a helper CTA per tile, clusters of two) for batches whose
  // tiles fill at most half the SMs: -1 automatic, 0 never (mega_assisted).
  int assist = -1;
};

bool mega_supported(int d, int H, int dff, int L, tl_dtype dt);
// Whether a forward of B sequences runs assisted (setting: -1 auto, 0 off, 1 on).
bool mega_assisted(int B, int L, int dff, int num_sms, int setting);
cudaError_t mega_forward(const void* x, const MegaArgs& a, int L, bool bf16, int num_sms, cudaStream_t s);

}  // namespace tl
