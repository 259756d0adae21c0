// Sequence-resident megakernel for fp32 I/O and small models, on CUDA cores
// ("Hyper-optimized megakernel-hybrid transformer inference", section
// "Problem decomposition": a short sequence fits in shared memory, so one
// CTA owns it for every layer and no activation goes back to HBM between
// steps).  fp32 weights are not exact in a 16-bit tensor-core operand, and
// these shapes (d_model <= 64) are far too small to feed the tensor pipe, so
// the arithmetic is fp32 FMA.
//
// One CTA per sequence, 256 threads.  Shared memory holds, for the CTA's
// sequence, the layer input X [L, d], Q, K, V head-major [H, L, dh], K
// transposed per head [H, dh, L] (conflict-free scores), the context / LN1
// output C [L, d], the pre-LayerNorm rows R [L, d] and the FFN hidden
// HB [L, d_ff].  Weights are read through L1 (16-byte loads).  Per layer:
//   X -> Q, K, V (+ b_qkv)          GEMM, one output column x 8 rows a thread
//   attention rows                   4 threads per (head, query row), online
//                                    softmax in registers; the top two scores
//                                    feed the near-tie test, and flagged rows
//                                    are recomputed in fp64 in place
//   R = C W_o^T + b_o + X, C = LN1(R)
//   HB = gelu(C W_1^T + b_1)
//   R = HB W_2^T + b_2 + C, X = LN2(R) (or the output rows)
#include <cuda_runtime.h>

#include "common.cuh"
#include "mega_simt.h"
#include "neartie.cuh"
#include "neartie_entry.cuh"

namespace tl {
namespace {

constexpr int kThreads = 256, kWarps = kThreads / 32;
constexpr int kRB = 8;  // output rows per GEMM task

struct Smem {
  float *X, *Q, *K, *V, *Kt, *C, *R, *HB;
  int* kmax;
  int* nflag;
  int* flags;  // queued (head, row) entries for the fp64 fix-up
  double* fix;
  size_t bytes;
};

__host__ __device__ inline Smem carve(unsigned char* base, int L, int d, int dh, int dff) {
  Smem s;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    unsigned char* p = base + off;
    off = (off + bytes + 15) / 16 * 16;
    return p;
  };
  const size_t ld = (size_t)L * d * sizeof(float);
  s.X = (float*)take(ld); s.Q = (float*)take(ld); s.K = (float*)take(ld); s.V = (float*)take(ld);
  s.Kt = (float*)take(ld); s.C = (float*)take(ld); s.R = (float*)take(ld);
  s.HB = (float*)take((size_t)L * dff * sizeof(float));
  s.kmax = (int*)take(64 * sizeof(int));
  s.nflag = (int*)take(16);
  s.flags = (int*)take((size_t)(d / dh) * L * sizeof(int));
  s.fix = (double*)take((size_t)kWarps * (dh + d) * sizeof(double));
  s.bytes = off;
  return s;
}

// out(t, n) = sum_k A[t][k] W[n][k] for t < L, n < N, handed to epi; A is a
// dense [L, K] shared-memory array, W [N, K] in global memory, K % 4 == 0.
// A task is one column n for kRB rows; its weight row is loaded 8 x 16 bytes
// at a time, all in flight together, so a K-long row costs K / 32 memory
// latencies instead of K / 4.
template <typename Epi>
__device__ __forceinline__ void gemm(const float* A, int K, const float* W, int N, int L, Epi epi) {
  const int groups = (L + kRB - 1) / kRB;
  for (int task = threadIdx.x; task < N * groups; task += kThreads) {
    const int n = task % N, t0 = (task / N) * kRB;
    float acc[kRB];
#pragma unroll
    for (int r = 0; r < kRB; ++r) acc[r] = 0.f;
    const float4* w4 = reinterpret_cast<const float4*>(W + (size_t)n * K);
    const int K4 = K / 4;
    for (int kb = 0; kb < K4; kb += 8) {
      float4 w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) w[u] = kb + u < K4 ? __ldg(w4 + kb + u) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r = 0; r < kRB; ++r) {
        const float* arow = A + (size_t)min(t0 + r, L - 1) * K + 4 * kb;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (kb + u < K4) {
            const float4 x = *reinterpret_cast<const float4*>(arow + 4 * u);
            acc[r] = fmaf(x.x, w[u].x, acc[r]);
            acc[r] = fmaf(x.y, w[u].y, acc[r]);
            acc[r] = fmaf(x.z, w[u].z, acc[r]);
            acc[r] = fmaf(x.w, w[u].w, acc[r]);
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kRB; ++r)
      if (t0 + r < L) epi(t0 + r, n, acc[r]);
  }
}

// Rows of R -> (r - mean) / sqrt(var + 1e-5) * g + b into out (row stride d),
// two-pass in fp32, a warp per row; d <= 64.
__device__ __forceinline__ void layernorm_rows(const float* R, const float* g, const float* be,
                                               float* out, int L, int d) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int t = warp; t < L; t += kWarps) {
    const float* x = R + (size_t)t * d;
    const float v0 = lane < d ? x[lane] : 0.f;
    const float v1 = lane + 32 < d ? x[lane + 32] : 0.f;
    const float mean = warp_sum(v0 + v1) / d;
    const float d0 = lane < d ? v0 - mean : 0.f, d1 = lane + 32 < d ? v1 - mean : 0.f;
    const float rstd = rsqrtf(warp_sum(fmaf(d0, d0, d1 * d1)) / d + 1e-5f);
    if (lane < d) out[(size_t)t * d + lane] = d0 * rstd * g[lane] + be[lane];
    if (lane + 32 < d) out[(size_t)t * d + lane + 32] = d1 * rstd * g[lane + 32] + be[lane + 32];
  }
}

template <int DH>
__global__ void __launch_bounds__(kThreads) mega_simt_kernel(const __grid_constant__ MegaSimtArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int L = a.L, d = a.d, H = a.H, dh = DH, dff = a.dff;
  const Smem sm = carve(smem_raw, L, d, dh, dff);
  const int seq = blockIdx.x, tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  int vl = a.vl[seq];
  if (vl < 1 || vl > L) {
    if (tid == 0) set_status(a.status, TL_ERR_BAD_VALID_LEN);
    vl = vl < 1 ? 1 : L;
  }
  // Every layer's parameters into L2 first: the steps below then wait on L2,
  // not on HBM, for their first touches.
  for (int l = 0; l < a.n_layers; ++l) prefetch_layer_l2(a.layers[l], d, dff, 4, tid, kThreads);
  const float* xin = a.x + (size_t)seq * L * d;
  for (int i = tid; i < L * d; i += kThreads) sm.X[i] = xin[i];
  const float scale_log2 = rsqrtf((float)dh) * 1.4426950408889634f;

  for (int l = 0; l < a.n_layers; ++l) {
    const tl_layer_dev& P = a.layers[l];
    if (tid < H) sm.kmax[tid] = 0;
    __syncthreads();
    // ---- QKV projection, head-major (K also transposed)
    gemm(sm.X, d, (const float*)P.w_qkv, 3 * d, L, [&](int t, int n, float acc) {
      const float v = acc + P.b_qkv[n];
      const int which = n / d, w = n % d, h = w / dh, c = w % dh;
      const size_t hm = ((size_t)h * L + t) * dh + c;
      if (which == 0) {
        sm.Q[hm] = v;
      } else if (which == 1) {
        sm.K[hm] = v;
        sm.Kt[((size_t)h * dh + c) * L + t] = v;
      } else {
        sm.V[hm] = v;
      }
    });
    __syncthreads();
    // the largest |k| of each head (near-tie error scale)
    for (int i = tid; i < H * L; i += kThreads) {
      const float* k = sm.K + (size_t)i * dh;
      float n2 = 0.f;
      for (int c = 0; c < dh; ++c) n2 = fmaf(k[c], k[c], n2);
      atomicMax(sm.kmax + i / L, __float_as_int(sqrtf(n2)));
    }
    __syncthreads();
    // ---- attention: 4 threads per (head, query row), each taking every 4th
    // visible key with an online softmax in registers; the four partial
    // states merge by shuffles.  Rows whose two best scores are close
    // relative to the fp32 score error are queued and recomputed in fp64.
    if (tid == 0) *sm.nflag = 0;
    __syncthreads();
    for (int base = 0; base < H * L; base += kThreads / 4) {
      const int row = base + tid / 4, sub = tid & 3;
      const bool active = row < H * L;
      const int h = active ? row / L : 0, i = active ? row % L : 0;
      const int nk = active ? min(i + 1, vl) : 0;
      float q[DH], o[DH];
      float qn2 = 0.f;
      const float* qrow = sm.Q + ((size_t)h * L + i) * DH;
#pragma unroll
      for (int c = 0; c < DH; ++c) {
        q[c] = active ? qrow[c] : 0.f;
        qn2 = fmaf(q[c], q[c], qn2);
        q[c] *= scale_log2;
        o[c] = 0.f;
      }
      const float* kt = sm.Kt + (size_t)h * DH * L;
      const float* vh = sm.V + (size_t)h * L * DH;
      float m = -INFINITY, lsum = 0.f, m1 = -INFINITY, m2 = -INFINITY;
      for (int jj = sub; jj < nk; jj += 4) {
        float sc = 0.f;
#pragma unroll
        for (int c = 0; c < DH; ++c) sc = fmaf(q[c], kt[c * L + jj], sc);
        m2 = fmaxf(m2, fminf(m1, sc));
        m1 = fmaxf(m1, sc);
        if (sc > m) {
          const float corr = exp2f(m - sc);  // 0 while m = -inf
          lsum *= corr;
#pragma unroll
          for (int c = 0; c < DH; ++c) o[c] *= corr;
          m = sc;
        }
        const float pj = exp2f(sc - m);
        lsum += pj;
        const float* vj = vh + (size_t)jj * DH;
#pragma unroll
        for (int c = 0; c < DH; ++c) o[c] = fmaf(pj, vj[c], o[c]);
      }
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, off);
        const float lo = __shfl_xor_sync(0xffffffffu, lsum, off);
        const float a1 = __shfl_xor_sync(0xffffffffu, m1, off);
        const float a2 = __shfl_xor_sync(0xffffffffu, m2, off);
        const float mn = fmaxf(m, mo);
        const float fa = mn == -INFINITY ? 0.f : exp2f(m - mn);
        const float fb = mn == -INFINITY ? 0.f : exp2f(mo - mn);
#pragma unroll
        for (int c = 0; c < DH; ++c) o[c] = o[c] * fa + __shfl_xor_sync(0xffffffffu, o[c], off) * fb;
        lsum = lsum * fa + lo * fb;
        m = mn;
        m2 = fmaxf(fmaxf(m2, a2), fminf(m1, a1));
        m1 = fmaxf(m1, a1);
      }
      if (active && sub == 0) {
        const float inv = 1.f / lsum;
        float* dst = sm.C + (size_t)i * d + h * DH;
#pragma unroll
        for (int c = 0; c < DH; ++c) dst[c] = o[c] * inv;
        if (neartie_flag((m1 - m2) * 0.69314718055994531f, sqrtf(qn2), __int_as_float(sm.kmax[h]), DH))
          sm.flags[atomicAdd(sm.nflag, 1)] = h * L + i;
      }
    }
    __syncthreads();
    if (*sm.nflag > 0) {
      FixupArgs fa{};
      fa.x = Plane{sm.X, nullptr, 5};
      fa.w_qkv = P.w_qkv;
      fa.w_kind = 0;
      fa.b_qkv = P.b_qkv;
      fa.q = Plane{sm.Q, nullptr, 5};
      fa.k = Plane{sm.K, nullptr, 5};
      fa.v = Plane{sm.V, nullptr, 5};
      fa.v_transposed = 0;
      fa.Lp = L;
      fa.ctx_hi = sm.C;
      fa.ctx_kind = 0;
      fa.valid_len = a.vl + seq;  // clamped again by the fix-up
      fa.B = 1; fa.H = H; fa.L = L; fa.dh = DH; fa.d = d;
      double* q64 = sm.fix + (size_t)warp * (DH + d);
      for (int e = warp; e < *sm.nflag; e += kWarps) ntie::neartie_fix_entry(fa, sm.flags[e], q64, q64 + DH, lane);
    }
    __syncthreads();
    // ---- out-projection + b_o + residual, LayerNorm 1 into C
    gemm(sm.C, d, (const float*)P.w_o, d, L, [&](int t, int n, float acc) {
      sm.R[(size_t)t * d + n] = acc + P.b_o[n] + sm.X[(size_t)t * d + n];
    });
    __syncthreads();
    layernorm_rows(sm.R, P.ln1_g, P.ln1_b, sm.C, L, d);
    __syncthreads();
    // ---- FFN
    gemm(sm.C, d, (const float*)P.w_1, dff, L, [&](int t, int n, float acc) {
      sm.HB[(size_t)t * dff + n] = gelu_erf(acc + P.b_1[n]);
    });
    __syncthreads();
    gemm(sm.HB, dff, (const float*)P.w_2, d, L, [&](int t, int n, float acc) {
      sm.R[(size_t)t * d + n] = acc + P.b_2[n] + sm.C[(size_t)t * d + n];
    });
    __syncthreads();
    const bool last = l + 1 == a.n_layers;
    layernorm_rows(sm.R, P.ln2_g, P.ln2_b, last ? a.out + (size_t)seq * L * d : sm.X, L, d);
    __syncthreads();
  }
}

size_t smem_bytes(int L, int d, int dh, int dff) { return carve(nullptr, L, d, dh, dff).bytes; }

}  // namespace

bool mega_simt_supported(int d, int H, int dff, int L, int n_layers, tl_dtype t) {
  if (t != TL_F32 || H < 1 || d % H || H > 64 || n_layers < 1 || n_layers > kMegaSimtMaxLayers) return false;
  const int dh = d / H;
  return d <= 64 && d % 4 == 0 && (dh == 8 || dh == 16 || dh == 32) && L <= 64 && dff <= 256 &&
         dff % 4 == 0 && smem_bytes(L, d, dh, dff) <= 200 * 1024;
}

template <int DH>
static cudaError_t launch(const MegaSimtArgs& a, cudaStream_t s) {
  const size_t smem = smem_bytes(a.L, a.d, DH, a.dff);
  cudaError_t e = set_max_dyn_smem((const void*)mega_simt_kernel<DH>, smem);
  if (e != cudaSuccess) return e;
  mega_simt_kernel<DH><<<a.B, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t mega_simt_forward(const MegaSimtArgs& a, cudaStream_t s) {
  if (a.dh == 8) return launch<8>(a, s);
  if (a.dh == 16) return launch<16>(a, s);
  return launch<32>(a, s);
}

}  // namespace tl
