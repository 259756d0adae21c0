// Near-tie detection and the fp64 fix-up of attention rows.
//
// At large input scales (the pages sweep input_scale up to 1e3: "Hyper-
// optimized megakernel-hybrid transformer inference", section "Headline
// results"; the same page's "Challenges" notes kernels that passed at 1.0
// and failed at larger scales) first-layer scores reach ~1e6 and an fp32
// score carries an absolute error of a logit or more.  A row whose two best
// keys are within a few logits is then ill-conditioned: its softmax weights,
// and so its output, move by more than the accuracy gate allows.  Such rows
// are rare (the gap of the top two of n Gaussian scores of spread sigma is
// below g with probability ~ g sqrt(2 ln n) / sigma).
//
// Detection: every attention kernel tracks per (row, head) the largest two
// fp32 scores m1 >= m2 and the error scale
//     E = 2^-19 |q_i| max_j |k_j| / sqrt(dh)
// (about 4x the largest error measured for fp32 scores on these shapes).  A
// row is queued when E > 2e-3 (below that the fp32 error moves no output by
// more than ~1e-3) and m1 - m2 < 12 + 2E: keys further below the best than
// 12 logits carry weight < e^-12 whatever their error.
//
// Fix-up (one warp per queued row): recompute q_i in fp64 from the layer
// input and the weights (exact inputs, fp64 arithmetic), rescreen every
// visible key with the stored fp32 q/k, recompute the scores of candidate
// keys (fp32 score within 12 + 2E of the best) in fp64 as
// x_j . (W_k^T q_i) + b_k . q_i, then redo that row's softmax and weighted
// sum of V in fp64 and overwrite the row's context.
#pragma once

#include "common.cuh"

namespace tl {

struct NearTieList {
  int* count;    // device counter, zeroed before each attention launch
  int* list;     // entries (b*H + h)*L + i
  int capacity;  // B*H*L
};

constexpr float kTieGap = 12.0f;        // natural-log logits
constexpr float kTieErrMin = 2e-3f;     // logits
constexpr float kTieErrScale = 1.9073486328125e-06f;  // 2^-19

__device__ __forceinline__ float neartie_err(float qnorm, float kmax, int dh) {
  return kTieErrScale * qnorm * kmax * rsqrtf((float)dh);
}

__device__ __forceinline__ bool neartie_flag(float gap_nat, float qnorm, float kmax, int dh) {
  const float e = neartie_err(qnorm, kmax, dh);
  return e > kTieErrMin && gap_nat < kTieGap + 2.f * e;
}

__device__ __forceinline__ void neartie_push(NearTieList t, int entry) {
  if (!t.count) return;
  int at = atomicAdd(t.count, 1);
  if (at < t.capacity) t.list[at] = entry;
}

// How the fix-up reads tensors.  kind: 0 fp32, 1 fp16, 2 bf16, 3 fp16 hi/lo
// pair (value = hi + lo), 4 bf16 hi/lo pair: global memory, read through L2
// only; 5 fp32 through a generic pointer (a CTA's own shared memory).
struct Plane {
  const void* hi;
  const void* lo;
  int kind;
};

// Views the fix-up needs, for one layer.
struct FixupArgs {
  NearTieList ties;
  Plane x;               // layer input [T, d]
  const void* w_qkv;     // [3d, d] in the I/O dtype
  int w_kind;            // 0 fp32, 1 fp16, 2 bf16
  const float* b_qkv;    // [3d]
  Plane q, k, v;         // stored projections
  int v_transposed;      // 0: v [B,H,L,dh]; 1: v^T [B,H,dh,Lp]
  int Lp;                // padded L of v^T rows
  void* ctx_hi;          // output [T, d]: fp32 (ctx_kind 0) or hi/lo planes
  void* ctx_lo;
  int ctx_kind;
  const int32_t* valid_len;
  int B, H, L, dh, d;
};

cudaError_t neartie_fixup(const FixupArgs& a, cudaStream_t s);

}  // namespace tl
