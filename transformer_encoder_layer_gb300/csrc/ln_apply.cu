// Second half of the add + LayerNorm epilogue for rows wider than one GEMM N
// tile ("KernelForge", section "What we built": fused add + LayerNorm after
// the projection GEMMs).  The GEMM's epilogue has already formed the
// pre-normalisation rows r = x + a (bias and residual added) and, per row and
// GEMM N tile, the (mean, M2) of the tile's columns; this kernel merges them
// (equal counts c per block: mean = the blocks' mean, M2 = sum M2_b + c sum
// (mean_b - mean)^2), takes rstd = 1/sqrt(M2 / N + eps) and applies
//   y = (r - mean) * rstd * gamma + beta
// and writes y as fp32 and/or (hi, lo) 16-bit planes, or as the stack's
// output in the I/O dtype.  It is a plain streaming pass: each thread takes 8
// consecutive columns (two 16-byte loads, 16-byte stores), so every warp
// instruction covers whole 128-byte lines and many loads are in flight per
// SM, which the GEMM's four epilogue warps (one row per thread) could not
// provide while its tensor cores run the next tile.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ln_apply.h"
#include "tc_common.cuh"

namespace tl {
namespace {

template <typename T>
__global__ void __launch_bounds__(256) ln_apply_kernel(const LnApplyArgs a) {
  const int groups = a.N / 8;  // 8-column groups per row
  const long long total = (long long)a.M * groups;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int row = (int)(i / groups), c0 = (int)(i % groups) * 8;
    const size_t at = (size_t)row * a.N + c0;
    const float4* rp = reinterpret_cast<const float4*>(a.r + at);
    const float4 r0 = __ldcs(rp), r1 = __ldcs(rp + 1);
    float2 st;  // (mean, rstd) of the row from its blocks' statistics
    {
      const float2* ps = a.stats + (size_t)row * a.n_parts;
      float msum = 0.f;
      for (int k = 0; k < a.n_parts; ++k) msum += ps[k].x;
      const float mean = msum / (float)a.n_parts;
      float m2 = 0.f;
      const float cnt = (float)(a.N / a.n_parts);
      for (int k = 0; k < a.n_parts; ++k) {
        const float2 p = ps[k];
        const float dm = p.x - mean;
        m2 += p.y + cnt * dm * dm;
      }
      st = make_float2(mean, rsqrtf(m2 / (float)a.N + 1e-5f));
    }
    const float4 g0 = __ldg(reinterpret_cast<const float4*>(a.gamma + c0));
    const float4 g1 = __ldg(reinterpret_cast<const float4*>(a.gamma + c0) + 1);
    const float4 b0 = __ldg(reinterpret_cast<const float4*>(a.beta + c0));
    const float4 b1 = __ldg(reinterpret_cast<const float4*>(a.beta + c0) + 1);
    const float rv[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    float y[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = (rv[j] - st.x) * st.y * gv[j] + bv[j];
    if (a.o32) {
      float4* o = reinterpret_cast<float4*>(a.o32 + at);
      o[0] = make_float4(y[0], y[1], y[2], y[3]);
      o[1] = make_float4(y[4], y[5], y[6], y[7]);
    }
    if (a.o_hi) {
      uint4 hv, lv;
      T* hp = reinterpret_cast<T*>(&hv);
      T* lp = reinterpret_cast<T*>(&lv);
#pragma unroll
      for (int j = 0; j < 8; ++j) tc::Split<T>::go(y[j], hp[j], lp[j]);
      *reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.o_hi) + at) = hv;
      *reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.o_lo) + at) = lv;
    }
    if (a.o_final) {
      uint4 fv;
      T* fp = reinterpret_cast<T*>(&fv);
#pragma unroll
      for (int j = 0; j < 8; ++j) fp[j] = from_f32<T>(y[j]);
      *reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.o_final) + at) = fv;
    }
  }
}

}  // namespace

cudaError_t ln_apply(const LnApplyArgs& a, bool bf16, int num_sms, cudaStream_t s) {
  if (a.M < 1 || a.N < 8 || a.N % 8 || a.n_parts < 1 || a.N % a.n_parts || !a.r || !a.stats ||
      !a.gamma || !a.beta ||
      (!a.o32 && !a.o_hi && !a.o_final) || (a.o_hi && !a.o_lo))
    return cudaErrorInvalidValue;
  const long long work = (long long)a.M * (a.N / 8);
  long long blocks = (work + 255) / 256;
  const long long cap = (long long)num_sms * 8;  // 8 resident blocks of 256 per SM
  if (blocks > cap) blocks = cap;
  if (bf16)
    ln_apply_kernel<__nv_bfloat16><<<(int)blocks, 256, 0, s>>>(a);
  else
    ln_apply_kernel<__half><<<(int)blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace tl
