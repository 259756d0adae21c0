// Per-kernel device timing: CUDA event pairs around each launch, summed per
// kernel class on request.  Off by default; costs nothing when off.
#include <cuda_runtime.h>

#include <new>
#include <vector>

#include "internal.h"

struct tl_timing {
  std::vector<cudaEvent_t> ev;  // 2 per slot
  std::vector<int> cls;         // kernel class per used slot
  int used = 0;
};

namespace {
static_assert(KC_COUNT <= TL_KERNEL_CLASSES, "kernel classes exceed the ABI table");
const char* kNames[KC_COUNT] = {
    "simt_gemm_qkv", "simt_attention", "simt_gemm_out", "simt_layernorm",
    "simt_gemm_ffn1", "simt_gemm_ffn2", "tc_gemm_qkv", "tc_attention",
    "tc_gemm_out_ln", "tc_gemm_ffn1", "tc_gemm_ffn2_ln", "megakernel", "aux", "dag", "megakernel_simt",
    "ln_apply"};
}

namespace tl {

KernelTimer::KernelTimer(tl_encoder* h_, int k_, cudaStream_t s_) : h(h_), k(k_), s(s_), slot(-1) {
  tl_timing* t = h->timing;
  if (!t || t->used * 2 >= (int)t->ev.size()) return;
  slot = t->used++;
  t->cls[slot] = k;
  cudaEventRecord(t->ev[2 * slot], s);
}

KernelTimer::~KernelTimer() {
  if (slot >= 0) cudaEventRecord(h->timing->ev[2 * slot + 1], s);
}

void timing_destroy(tl_encoder* h) {
  if (!h->timing) return;
  for (cudaEvent_t e : h->timing->ev) cudaEventDestroy(e);
  delete h->timing;
  h->timing = nullptr;
}

}  // namespace tl

extern "C" {

tl_status tl_encoder_enable_timing(tl_encoder* h, int enable, int capacity) {
  if (!h) return TL_ERR_INVALID_ARG;
  tl::timing_destroy(h);
  if (!enable) return TL_OK;
  if (capacity < 1) return TL_ERR_INVALID_ARG;
  tl_timing* t = new (std::nothrow) tl_timing();
  if (!t) return TL_ERR_OUT_OF_MEMORY;
  t->ev.resize(2 * (size_t)capacity);
  t->cls.resize(capacity);
  for (auto& e : t->ev) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
      h->timing = t;
      tl::timing_destroy(h);
      return TL_ERR_CUDA;
    }
  }
  h->timing = t;
  return TL_OK;
}

tl_status tl_encoder_read_timing(tl_encoder* h, int k, float* total_ms, int* launches) {
  if (!h || !total_ms || !launches || k < 0 || k >= TL_KERNEL_CLASSES) return TL_ERR_INVALID_ARG;
  *total_ms = 0.f;
  *launches = 0;
  if (!h->timing) return TL_OK;
  if (cudaDeviceSynchronize() != cudaSuccess) return TL_ERR_CUDA;
  tl_timing* t = h->timing;
  for (int i = 0; i < t->used; ++i) {
    if (t->cls[i] != k) continue;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, t->ev[2 * i], t->ev[2 * i + 1]) != cudaSuccess) return TL_ERR_CUDA;
    *total_ms += ms;
    ++*launches;
  }
  return TL_OK;
}

tl_status tl_encoder_reset_timing(tl_encoder* h) {
  if (!h) return TL_ERR_INVALID_ARG;
  if (h->timing) h->timing->used = 0;
  return TL_OK;
}

const char* tl_kernel_class_name(int k) { return (k >= 0 && k < KC_COUNT) ? kNames[k] : ""; }

}  // extern "C"
