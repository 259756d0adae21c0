// The fp64 near-tie correction of one attention row, shared by the fix-up
// kernel (neartie.cu) and the task-graph kernel (dag.cu).  The method is
// described in neartie.cuh.  Loads of activations bypass L1, since inside
// one kernel they may have been written by other CTAs.
#pragma once

#include "common.cuh"
#include "neartie.cuh"

namespace tl {
namespace ntie {

__device__ __forceinline__ double ld64(const Plane& p, size_t i) {
  auto h16 = [](const void* base, size_t j) {
    return __ldcg(reinterpret_cast<const unsigned short*>(base) + j);
  };
  switch (p.kind) {
    case 0: return (double)__ldcg(reinterpret_cast<const float*>(p.hi) + i);
    case 1: return (double)__half2float(__ushort_as_half(h16(p.hi, i)));
    case 2: return (double)__bfloat162float(__ushort_as_bfloat16(h16(p.hi, i)));
    case 5: return (double)reinterpret_cast<const float*>(p.hi)[i];  // fp32, generic (shared) memory
    case 3:
      return (double)__half2float(__ushort_as_half(h16(p.hi, i))) +
             (double)__half2float(__ushort_as_half(h16(p.lo, i)));
    default:
      return (double)__bfloat162float(__ushort_as_bfloat16(h16(p.hi, i))) +
             (double)__bfloat162float(__ushort_as_bfloat16(h16(p.lo, i)));
  }
}

__device__ __forceinline__ double ldw(const void* w, int kind, size_t i) {
  if (kind == 0) return (double)reinterpret_cast<const float*>(w)[i];
  if (kind == 1) return (double)__half2float(reinterpret_cast<const __half*>(w)[i]);
  return (double)__bfloat162float(reinterpret_cast<const __nv_bfloat16*>(w)[i]);
}

__device__ __forceinline__ double warp_max_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Correct one queued (row, head): the whole warp runs this; q64 [dh] and
// u [d] are this warp's fp64 scratch in shared memory.
__device__ inline void neartie_fix_entry(const FixupArgs& a, int entry, double* q64, double* u, int lane) {
  const int d = a.d, dh = a.dh, H = a.H, L = a.L;
  const double rsq = 1.0 / sqrt((double)dh);
  const int i = entry % L, bh = entry / L, h = bh % H, b = bh / H;
  int vl = a.valid_len[b];
  vl = vl < 1 ? 1 : (vl > L ? L : vl);
  const int nk = min(i + 1, vl);
  const size_t xrow = ((size_t)b * L + i) * d;
  // q_i in fp64 from the exact layer input and weights.
  for (int c = lane; c < dh; c += 32) {
    double acc = a.b_qkv[h * dh + c];
    const size_t wr = (size_t)(h * dh + c) * d;
    for (int t = 0; t < d; ++t) acc = fma(ldw(a.w_qkv, a.w_kind, wr + t), ld64(a.x, xrow + t), acc);
    q64[c] = acc;
  }
  __syncwarp();
  // u = W_k,h^T q_i and u0 = b_k,h . q_i, so that q_i . k_j = x_j . u + u0.
  for (int t = lane; t < d; t += 32) {
    double acc = 0.0;
    for (int c = 0; c < dh; ++c)
      acc = fma(q64[c], ldw(a.w_qkv, a.w_kind, (size_t)(d + h * dh + c) * d + t), acc);
    u[t] = acc;
  }
  double u0 = 0.0, qn2 = 0.0;
  for (int c = 0; c < dh; ++c) {
    u0 = fma(q64[c], (double)a.b_qkv[d + h * dh + c], u0);
    qn2 = fma(q64[c], q64[c], qn2);
  }
  __syncwarp();
  const size_t plane = (size_t)bh * L * dh;
  auto screen = [&](int j) -> float {  // fp32 score from the stored keys
    float t = 0.f;
    for (int c = 0; c < dh; ++c) t = fmaf((float)q64[c], (float)ld64(a.k, plane + (size_t)j * dh + c), t);
    return t * (float)rsq;
  };
  auto exact = [&](int j) -> double {
    const size_t xr = ((size_t)b * L + j) * d;
    double t = u0;
    for (int c = 0; c < d; ++c) t = fma(ld64(a.x, xr + c), u[c], t);
    return t * rsq;
  };
  // Pass A: best screening score and the largest key norm.
  float m1 = -INFINITY, kmax = 0.f;
  for (int j = lane; j < nk; j += 32) {
    m1 = fmaxf(m1, screen(j));
    float kn = 0.f;
    for (int c = 0; c < dh; ++c) {
      float kv = (float)ld64(a.k, plane + (size_t)j * dh + c);
      kn = fmaf(kv, kv, kn);
    }
    kmax = fmaxf(kmax, sqrtf(kn));
  }
  m1 = warp_max(m1);
  kmax = warp_max(kmax);
  const float err = neartie_err((float)sqrt(qn2), kmax, dh);
  const float thr = m1 - kTieGap - 2.f * err;
  // Pass B: the exact best score over the candidates.
  double M = -INFINITY;
  for (int j = lane; j < nk; j += 32) {
    float s = screen(j);
    M = fmax(M, s >= thr ? exact(j) : (double)s);
  }
  M = warp_max_d(M);
  // Pass C: fp64 softmax weights and the weighted sum of V.
  double l = 0.0, o[4] = {0.0, 0.0, 0.0, 0.0};  // dims lane, lane+32, ...
  for (int j0 = 0; j0 < nk; j0 += 32) {
    const int j = j0 + lane;
    double w = 0.0;
    if (j < nk) {
      float s = screen(j);
      w = exp((s >= thr ? exact(j) : (double)s) - M);
    }
    l += w;
    unsigned mask = __ballot_sync(0xffffffffu, w != 0.0);
    while (mask) {
      const int src = __ffs(mask) - 1;
      mask &= mask - 1;
      const double wj = __shfl_sync(0xffffffffu, w, src);
      const int jj = j0 + src;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int c = lane + 32 * r;
        if (c < dh) {
          size_t vi = a.v_transposed ? ((size_t)bh * dh + c) * a.Lp + jj : plane + (size_t)jj * dh + c;
          o[r] = fma(wj, ld64(a.v, vi), o[r]);
        }
      }
    }
  }
  l = warp_sum_d(l);
  const size_t orow = ((size_t)b * L + i) * d + (size_t)h * dh;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int c = lane + 32 * r;
    if (c >= dh) continue;
    const float val = (float)(o[r] / l);
    if (a.ctx_kind == 0) {
      reinterpret_cast<float*>(a.ctx_hi)[orow + c] = val;
    } else if (a.ctx_kind == 3) {
      __half hi = __float2half_rn(val);
      reinterpret_cast<__half*>(a.ctx_hi)[orow + c] = hi;
      reinterpret_cast<__half*>(a.ctx_lo)[orow + c] = __float2half_rn(val - __half2float(hi));
    } else {
      __nv_bfloat16 hi = __float2bfloat16_rn(val);
      reinterpret_cast<__nv_bfloat16*>(a.ctx_hi)[orow + c] = hi;
      reinterpret_cast<__nv_bfloat16*>(a.ctx_lo)[orow + c] = __float2bfloat16_rn(val - __bfloat162float(hi));
    }
  }
  __syncwarp();
}

}  // namespace ntie
}  // namespace tl
