// Persistent task-graph path (one launch per forward, fp32 I/O).
#pragma once

#include <cuda_runtime.h>

#include "internal.h"

namespace tl {

constexpr int kDagMaxLayers = 8;
constexpr int kDagRows = 64;   // rows of one row block
constexpr int kDagKChunk = 256;  // K of one GEMM task (split-K beyond it)
constexpr long long kDagAutoMaxTokens = 8192;  // TL_PATH_AUTO picks the path up to B*L tokens

struct DagArgs {
  tl_layer_dev layers[kDagMaxLayers];
  int n_layers;
  const float* x;          // [T, d] input
  float* out;              // [T, d] output
  const int32_t* vl;       // [B]
  // fp32 workspace
  float *xs0, *xs1;        // layer inputs, by layer parity
  float *q, *k, *v;        // [B, H, L, dh] each
  float* ctx;              // [T, d]
  float* y;                // [T, d] LayerNorm-1 output
  float* hb;               // [T, dff] GELU output
  float* part;             // [kc_max, T, d] split-K partial sums
  int* cnt;                // [n_layers, 7, RB] completion counters, then head, abort
  int* head;
  int* abort;
  int* status;
  int B, L, T, RB, d, H, dh, dff;
  int inject_stall;        // test hook: the first task waits on a counter nothing bumps
};

bool dag_supported(int d, int H, int dff, int n_layers, tl_dtype t);
int dag_counter_ints(int n_layers, int RB);
size_t dag_dyn_smem(int d, int dh);
cudaError_t dag_forward(const DagArgs& a, int num_sms, cudaStream_t s);

}  // namespace tl
