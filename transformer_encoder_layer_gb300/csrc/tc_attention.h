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
  // Split-K over keys (set by tc_attention from the plan): key tiles per
  // chunk (0 = no split), the work-item count, the partial-state buffer and
  // the per-(plane, query tile) arrival counters (zeroed by tc_attention).
  int kc = 0, n_items = 0;
  int group = 1;  // planes per L2-resident group of unsplit items (set by tc_attention)
  float* part = nullptr;
  int* cnt = nullptr;
};

// How the attention kernel partitions the key range ("KernelForge",
// section "What's next": split-K attention that merges partial softmax
// states).  Query tiles whose causal key range spans more than kc 64-key
// tiles are cut into chunks of kc tiles; each chunk is its own work item,
// writes its partial state (unnormalised output, running max, second-best
// score, row sum) to part_bytes of workspace, and the last chunk of a tile
// to arrive merges them.  kc = 0: no split (part_bytes = cnt_bytes = 0).
struct TcAttnSplit {
  int kc = 0;
  int n_items = 0;
  size_t part_bytes = 0, cnt_bytes = 0;
};
// force_kc < 0: choose by a model of the persistent CTAs' static item
// assignment (split only where it shortens the busiest CTA's work by 10% or
// more); 0: never split; > 0: chunks of force_kc key tiles.
TcAttnSplit tc_attention_split_plan(int B, int H, int L, int dh, int num_sms, int force_kc);

bool tc_attention_supported(int dh);
// ws_part / ws_cnt: workspace of at least the plan's part_bytes / cnt_bytes
// (256-byte aligned), used when the plan splits.
cudaError_t tc_attention(const TcAttnArgs& a, bool bf16, int num_sms, int force_kc, void* ws_part,
                         void* ws_cnt, cudaStream_t s);

}  // namespace tl
