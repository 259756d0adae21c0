// Internal (C++) interface between the C ABI and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/tl_encoder.h"
#include "neartie.cuh"

// Device pointers of one layer's packed parameters.  Weights stay in the I/O
// dtype ([out, in] row-major, exactly the caller's values); biases and
// LayerNorm parameters are also kept as fp32 copies for the epilogues.
struct tl_layer_dev {
  const void* w_qkv;  // [3d, d]  dtype
  const void* w_o;    // [d, d]
  const void* w_1;    // [d_ff, d]
  const void* w_2;    // [d, d_ff]
  const float* b_qkv; // [3d]     fp32
  const float* b_o;   // [d]
  const float* ln1_g; const float* ln1_b;
  const float* b_1;   // [d_ff]
  const float* b_2;   // [d]
  const float* ln2_g; const float* ln2_b;
};

// Prefetch every parameter array of layer P (dtype element size es) into L2,
// as thread idx of `stride` cooperating threads.
__device__ __forceinline__ void prefetch_layer_l2(const tl_layer_dev& P, int d, int dff, int es, int idx,
                                                  int stride) {
  tl::prefetch_l2(P.w_qkv, (size_t)3 * d * d * es, idx, stride);
  tl::prefetch_l2(P.w_o, (size_t)d * d * es, idx, stride);
  tl::prefetch_l2(P.w_1, (size_t)dff * d * es, idx, stride);
  tl::prefetch_l2(P.w_2, (size_t)d * dff * es, idx, stride);
  tl::prefetch_l2(P.b_qkv, (size_t)3 * d * 4, idx, stride);
  tl::prefetch_l2(P.b_o, (size_t)d * 4, idx, stride);
  tl::prefetch_l2(P.ln1_g, (size_t)d * 4, idx, stride);
  tl::prefetch_l2(P.ln1_b, (size_t)d * 4, idx, stride);
  tl::prefetch_l2(P.b_1, (size_t)dff * 4, idx, stride);
  tl::prefetch_l2(P.b_2, (size_t)d * 4, idx, stride);
  tl::prefetch_l2(P.ln2_g, (size_t)d * 4, idx, stride);
  tl::prefetch_l2(P.ln2_b, (size_t)d * 4, idx, stride);
}

// Kernel classes for per-kernel timing (names in timing.cu).
enum tl_kernel_class {
  KC_SIMT_GEMM_QKV = 0, KC_SIMT_ATTENTION, KC_SIMT_GEMM_OUT, KC_SIMT_LAYERNORM,
  KC_SIMT_GEMM_FFN1, KC_SIMT_GEMM_FFN2, KC_TC_GEMM_QKV, KC_TC_ATTENTION,
  KC_TC_GEMM_OUT_LN, KC_TC_GEMM_FFN1, KC_TC_GEMM_FFN2_LN, KC_MEGA, KC_AUX, KC_DAG, KC_MEGA_SIMT,
  KC_LN_APPLY, KC_COUNT
};

struct tl_timing;  // event pool, defined in timing.cu

struct tl_encoder {
  int n_layers = 0, d = 0, H = 0, dh = 0, dff = 0;
  tl_dtype dtype = TL_F32;
  tl_path path = TL_PATH_AUTO;
  bool simt_attention = false;  // layered path: CUDA-core attention instead of tcgen05
  bool dag_inject_stall = false;  // task-graph path: make the first wait time out (tests)
  // Split-K attention on the layered path: -1 automatic, 0 never, k > 0
  // chunks of k 64-key tiles (tl_encoder_set_attention_split).
  int attn_split = -1;
  // Layered-path GEMMs on CTA pairs (tcgen05 cta_group::2): -1 automatic
  // (the default: the FFN2 GEMM of large shapes), 0 off, 1 every GEMM the
  // shape allows (tl_encoder_set_gemm_pairs).
  int gemm_pairs = -1;
  // Megakernel assisted mode (a helper CTA per tile when the tiles fill at
  // most half the SMs): -1 automatic (off: no measured gain), 0 off, 1 on
  // where possible (tl_encoder_set_mega_assist).
  int mega_assist = -1;
  int device = 0;
  int num_sms = 0;
  void* wbuf = nullptr;      // one allocation holding every packed parameter
  size_t wbuf_bytes = 0;
  int* status = nullptr;     // device status word
  tl_layer_dev* layers = nullptr;  // host array of n_layers
  tl_timing* timing = nullptr;     // non-null while per-kernel timing is on
  const void* mega_layers = nullptr;  // device array of MegaLayer (megakernel path)
  // Device address of the library's static scratch array in this handle's
  // context (tl_encoder_forward_static), looked up at create.
  void* static_scratch = nullptr;
  // Host-buffer forward: batch slices per call (0 = automatic) and the two
  // non-blocking streams plus fork/join events its copy/compute pipeline uses
  // (created on first use).
  int host_chunks = 0;
  cudaStream_t host_stream[2] = {nullptr, nullptr};
  cudaEvent_t host_event[3] = {nullptr, nullptr, nullptr};
  // Graph mode of the layered path (tl_encoder_set_graphs): the launch
  // sequence of the last (shape, buffers) seen, captured once and replayed.
  bool graphs = false;
  cudaStream_t capture_stream = nullptr;
  cudaGraphExec_t graph_exec = nullptr;
  struct GraphKey {
    int path, B, L, attn_split;
    const void *x, *vl, *out, *ws;
    bool operator==(const GraphKey& o) const {
      return path == o.path && B == o.B && L == o.L && attn_split == o.attn_split && x == o.x &&
             vl == o.vl && out == o.out && ws == o.ws;
    }
  } graph_key{};
  long long graph_captures = 0, graph_replays = 0;
};

namespace tl {
// Records an event pair around one launch when timing is enabled.
struct KernelTimer {
  KernelTimer(tl_encoder* h, int kernel_class, cudaStream_t s);
  ~KernelTimer();
  tl_encoder* h; int k; cudaStream_t s; int slot;
};
void timing_destroy(tl_encoder* h);
// Device address of the static scratch array in the current context, or null.
void* static_scratch_address();
}  // namespace tl

namespace tl {

// ---- generic fp32 CUDA-core (SIMT) kernels -------------------------------
enum SimtEpi { EPI_QKV_HEADMAJOR = 0, EPI_BIAS_GELU = 1, EPI_BIAS_RESID = 2 };

// C[M, N] = A[M, K] . W[N, K]^T with a fused epilogue.
//  a_dtype: TL_F32 for fp32 activations, else the I/O dtype of x.
//  EPI_QKV_HEADMAJOR: out is fp32 q|k|v, each [B, H, L, dh] (N = 3d).
//  EPI_BIAS_GELU:     out fp32 [M, N] = gelu(acc + bias).
//  EPI_BIAS_RESID:    out fp32 [M, N] = acc + bias + resid (resid in r_dtype).
struct SimtGemmArgs {
  const void* A; tl_dtype a_dtype;
  const void* W; tl_dtype w_dtype;
  const float* bias;
  const void* resid; tl_dtype r_dtype;
  float* out;
  int M, N, K;
  int B, L, H, dh;  // for the head-major epilogue
  int epi;
};
cudaError_t simt_gemm(const SimtGemmArgs& a, cudaStream_t s);

// Causal + key-padding attention on CUDA cores, fp32 arithmetic.
// mode 0: fp32 q, k, v [B, H, L, dh] and fp32 ctx [B, L, H*dh];
// mode 1/2: fp16/bf16 (hi, lo) planes, v given transposed [B, H, dh, Lp],
// ctx written as (hi, lo) planes.  dh <= 128.  Near-tie rows are queued.
struct AttnIO {
  const void *q_hi, *q_lo, *k_hi, *k_lo, *v_hi, *v_lo;
  int v_transposed, Lp;
  void *ctx_hi, *ctx_lo;
};
cudaError_t simt_attention(const AttnIO& io, int mode, const int32_t* vl, int B, int H, int L,
                           int dh, int* status, NearTieList ties, cudaStream_t s);

// Row LayerNorm over d (<= 1024): y = (r - mean)/sqrt(var + 1e-5) g + b,
// two-pass in fp32.  Writes y32 (fp32, may be null) and/or yout (I/O dtype,
// may be null).
cudaError_t simt_layernorm(const float* r, const float* g, const float* b, float* y32,
                           void* yout, tl_dtype out_dtype, int M, int d, cudaStream_t s);

}  // namespace tl
