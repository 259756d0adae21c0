// Shared device/host helpers of the encoder library: dtype conversion,
// the device status word, and small warp reductions.
#pragma once

#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/tl_encoder.h"

namespace tl {

// ---------------------------------------------------------------- dtypes
template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

inline size_t dtype_size(tl_dtype t) { return t == TL_F32 ? 4 : 2; }

// ------------------------------------------------------- device status
// One int per handle.  Kernels record the first error with atomicCAS from 0;
// the host reads and clears it in tl_encoder_get_status().
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// valid_len clamped to [1, L]; an out-of-range value is recorded.
__device__ __forceinline__ int load_valid_len(const int32_t* vl, int b, int L, int* status) {
  int v = vl[b];
  if (v < 1 || v > L) {
    set_status(status, TL_ERR_BAD_VALID_LEN);
    v = v < 1 ? 1 : L;
  }
  return v;
}

// ------------------------------------------- launch configuration cache
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) is a driver call of some
// microseconds; launchers call this instead, which sets the attribute once
// per (kernel, device) and again only when a larger size is asked for.
inline cudaError_t set_max_dyn_smem(const void* func, size_t bytes) {
  struct Entry { const void* f; int dev; size_t bytes; };
  static Entry table[128];
  static int n = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < n; ++i)
    if (table[i].f == func && table[i].dev == dev && table[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < n; ++i)
    if (table[i].f == func && table[i].dev == dev) { table[i].bytes = bytes; return cudaSuccess; }
  if (n < 128) table[n++] = Entry{func, dev, bytes};
  return cudaSuccess;
}

// ------------------------------------------------------ L2 prefetch
// Thread idx of `stride` cooperating threads prefetches its share of the
// 128-byte lines of [p, p + bytes) into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, size_t bytes, int idx, int stride) {
  const char* c = reinterpret_cast<const char*>(p);
  for (size_t off = (size_t)idx * 128; off < bytes; off += (size_t)stride * 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(c + off));
}

// ------------------------------------------------------ warp reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Exact GELU on fp32: 0.5 u (1 + erf(u / sqrt 2)), with CUDA's erff.
__device__ __forceinline__ float gelu_erf(float u) {
  return 0.5f * u * (1.0f + erff(u * 0.70710678118654752f));
}

// ------------------------------------------------ paired fp32 arithmetic
// Two fp32 values in one 64-bit register for sm_100+'s paired fp32
// instructions (fma/mul/add .f32x2): each lane is rounded exactly as the
// scalar instruction rounds it, so a paired evaluation gives the scalar
// results bit for bit in half the instructions.
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t splat2(float a) { return pk2(a, a); }

// GELU with a branch-free erf: Abramowitz & Stegun, Handbook of
// Mathematical Functions (1964), formula 7.1.28 (after Hastings):
//   erf(x) = 1 - (1 + a1 x + a2 x^2 + ... + a6 x^6)^-16,  x >= 0,  |error| <= 3e-7.
// With r = (...)^-16 at x = |u| / sqrt 2, 0.5 u (1 + erf(u / sqrt 2)) is
// u - 0.5 u r for u >= 0 and 0.5 u r for u < 0 (no cancellation), i.e.
// max(u, 0) - 0.5 |u| r for either sign: one fused multiply-add, no select.
// In fp32 the power amplifies the polynomial's rounding 16-fold, so the GELU
// error is at most 0.5 |u| (3e-7 + 2.5e-6 r) + 2e-7 |gelu(u)| (r <= 1).  Every
// lane runs the same instructions (one reciprocal, no exponential), which
// keeps long unrolled epilogue loops free of divergent branches.  Two values
// at a time, on the paired fp32 instructions: every operation is the scalar
// one, rounded the same way.  Its agreement with the erff form is checked on
// the GPU over a dense grid (tl_eval_gelu).
__device__ __forceinline__ void gelu_as7128_x2(float& u0, float& u1) {
  const uint64_t au = pk2(fabsf(u0), fabsf(u1));
  const uint64_t x = mul2(au, splat2(0.70710678118654752f));
  uint64_t t = fma2(x, splat2(0.0000430638f), splat2(0.0002765672f));
  t = fma2(x, t, splat2(0.0001520143f));
  t = fma2(x, t, splat2(0.0092705272f));
  t = fma2(x, t, splat2(0.0422820123f));
  t = fma2(x, t, splat2(0.0705230784f));
  t = fma2(x, t, splat2(1.0f));
  t = mul2(t, t);  // ^2
  t = mul2(t, t);  // ^4
  t = mul2(t, t);  // ^8
  t = mul2(t, t);  // ^16
  float t0, t1, r0, r1;
  upk2(t, t0, t1);
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(t0));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(t1));
  const uint64_t m = mul2(au, splat2(-0.5f));  // -0.5 |u|, exact
  upk2(fma2(m, pk2(r0, r1), pk2(fmaxf(u0, 0.f), fmaxf(u1, 0.f))), u0, u1);
}

}  // namespace tl
