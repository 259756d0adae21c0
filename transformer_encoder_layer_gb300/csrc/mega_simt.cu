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
// HB [L, d_ff].  When they fit, every layer's weights are copied into shared
// memory at kernel start (cp.async, one group per layer, rows padded by 16
// bytes so that neighbouring output columns hit different banks), and layer
// l waits only for its own group; otherwise they are read through L1.  Per
// layer:
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

struct Smem {
  float *X, *Q, *K, *V, *Kt, *C, *R, *HB;
  int* kmax;
  int* nflag;
  int* flags;  // queued (head, row) entries for the fp64 fix-up
  double* fix;
  float* W;    // staged weights, n_layers x layer_w_floats (or null)
  size_t bytes;
};

// Floats of one layer's staged weights: W_qkv [3d][d+4], W_o [d][d+4],
// W_1 [dff][d+4], W_2 [d][dff+4].
__host__ __device__ inline size_t layer_w_floats(int d, int dff) {
  return (size_t)4 * d * (d + 4) + (size_t)dff * (d + 4) + (size_t)d * (dff + 4);
}

__host__ __device__ inline Smem carve(unsigned char* base, int L, int d, int dh, int dff,
                                      int w_layers) {
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
  s.W = w_layers ? (float*)take((size_t)w_layers * layer_w_floats(d, dff) * sizeof(float)) : nullptr;
  s.bytes = off;
  return s;
}

// 16-byte asynchronous copy global -> shared, and its group bookkeeping.
__device__ __forceinline__ void cp16(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }
// Wait until at most n of this thread's groups are pending (n <= 7).
__device__ __forceinline__ void cp_wait_n(int n) {
  switch (n) {
    case 0: cp_wait<0>(); break;
    case 1: cp_wait<1>(); break;
    case 2: cp_wait<2>(); break;
    case 3: cp_wait<3>(); break;
    case 4: cp_wait<4>(); break;
    case 5: cp_wait<5>(); break;
    case 6: cp_wait<6>(); break;
    default: cp_wait<7>(); break;
  }
}

// W [N, K] (global, K % 4 == 0) -> dst [N][K + 4] in shared memory.
__device__ __forceinline__ void stage_w(float* dst, const float* W, int N, int K) {
  const int K4 = K / 4;
  for (int i = threadIdx.x; i < N * K4; i += kThreads) {
    const int n = i / K4, k4 = i - n * K4;
    cp16(dst + (size_t)n * (K + 4) + 4 * k4, W + (size_t)n * K + 4 * k4);
  }
}

// out(t, n) = sum_k A[t][k] W[n][k] for t < L, n < N; A is a dense [L, K]
// shared-memory array, W [N, K] with row pitch ldw, in shared memory (SW) or
// global memory, K % 4 == 0.  A task is one column n for RB rows; its weight
// row is read 8 x 16 bytes at a time, all in flight together.  The epilogue
// gets the task's rows at once: epi(t0, rows, n, acc[RB]).
template <int RB, bool SW, typename Epi>
__device__ __forceinline__ void gemm(const float* A, int K, const float* W, int ldw, int N, int L,
                                     Epi epi) {
  const int groups = (L + RB - 1) / RB;
  for (int task = threadIdx.x; task < N * groups; task += kThreads) {
    const int n = task % N, t0 = (task / N) * RB;
    float acc[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) acc[r] = 0.f;
    const float4* w4 = reinterpret_cast<const float4*>(W + (size_t)n * ldw);
    const int K4 = K / 4;
    for (int kb = 0; kb < K4; kb += 8) {
      float4 w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        w[u] = kb + u < K4 ? (SW ? w4[kb + u] : __ldg(w4 + kb + u)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r = 0; r < RB; ++r) {
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
    epi(t0, min(RB, L - t0), n, acc);
  }
}

// The GEMM with 8-row tasks, or 4-row tasks when 8-row ones would leave
// threads idle.
template <bool SW, typename Epi>
__device__ __forceinline__ void gemm_rows(const float* A, int K, const float* W, int ldw, int N, int L,
                                          Epi epi) {
  if (N * ((L + 7) / 8) >= kThreads) gemm<8, SW>(A, K, W, ldw, N, L, epi);
  else gemm<4, SW>(A, K, W, ldw, N, L, epi);
}

// Rows of R -> (r - mean) / sqrt(var + 1e-5) * g + b into out (row stride d),
// two-pass in fp32; 8 lanes per row (columns lane, lane + 8, ...), 4 rows per
// warp at once; d <= 64.
__device__ __forceinline__ void layernorm_rows(const float* R, const float* g, const float* be,
                                               float* out, int L, int d) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, sub = lane & 7;
  for (int t0 = 4 * warp; t0 < L; t0 += 4 * kWarps) {
    const int t = t0 + (lane >> 3);
    const bool ok = t < L;
    float v[8], sum = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int col = sub + 8 * c;
      v[c] = ok && col < d ? R[(size_t)t * d + col] : 0.f;
      sum += v[c];
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float mean = sum / d;
    float q = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float dv = sub + 8 * c < d ? v[c] - mean : 0.f;
      v[c] = dv;
      q = fmaf(dv, dv, q);
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
    const float rstd = rsqrtf(q / d + 1e-5f);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int col = sub + 8 * c;
      if (ok && col < d) out[(size_t)t * d + col] = v[c] * rstd * g[col] + be[col];
    }
  }
}

template <int DH>
__global__ void __launch_bounds__(kThreads) mega_simt_kernel(const __grid_constant__ MegaSimtArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int L = a.L, d = a.d, H = a.H, dh = DH, dff = a.dff;
  const Smem sm = carve(smem_raw, L, d, dh, dff, a.w_stage ? a.n_layers : 0);
  const int seq = blockIdx.x, tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  int vl = a.vl[seq];
  if (vl < 1 || vl > L) {
    if (tid == 0) set_status(a.status, TL_ERR_BAD_VALID_LEN);
    vl = vl < 1 ? 1 : L;
  }
  const size_t lw = layer_w_floats(d, dff);
  if (a.w_stage) {
    // every layer's weights into shared memory, one cp.async group per layer
    for (int l = 0; l < a.n_layers; ++l) {
      const tl_layer_dev& P = a.layers[l];
      float* w = sm.W + l * lw;
      stage_w(w, (const float*)P.w_qkv, 3 * d, d);
      stage_w(w + 3 * d * (d + 4), (const float*)P.w_o, d, d);
      stage_w(w + 4 * d * (d + 4), (const float*)P.w_1, dff, d);
      stage_w(w + 4 * d * (d + 4) + (size_t)dff * (d + 4), (const float*)P.w_2, d, dff);
      cp_commit();
    }
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
    if (a.w_stage) cp_wait_n(a.n_layers - 1 - l);  // this layer's weights have landed
    __syncthreads();
    // This layer's weights and their row pitches, staged or in global memory.
    const float* wl = sm.W + l * lw;
    const bool sw = a.w_stage != 0;
    const float* Wq = sw ? wl : (const float*)P.w_qkv;
    const float* Wo = sw ? wl + 3 * d * (d + 4) : (const float*)P.w_o;
    const float* W1 = sw ? wl + 4 * d * (d + 4) : (const float*)P.w_1;
    const float* W2 = sw ? wl + 4 * d * (d + 4) + (size_t)dff * (d + 4) : (const float*)P.w_2;
    const int ldd = sw ? d + 4 : d, ldf = sw ? dff + 4 : dff;
    // ---- QKV projection, head-major (K also transposed)
    auto qkv_epi = [&](int t0, int nr, int n, const auto& acc) {
      constexpr int rb = sizeof(acc) / sizeof(float);
      const float b = P.b_qkv[n];
      const int which = n / d, w = n % d, h = w / dh, c = w % dh;
      float* dst = which == 0 ? sm.Q : (which == 1 ? sm.K : sm.V);
#pragma unroll
      for (int r = 0; r < rb; ++r) {
        if (r < nr) {
          const int t = t0 + r;
          const float v = acc[r] + b;
          dst[((size_t)h * L + t) * dh + c] = v;
          if (which == 1) sm.Kt[((size_t)h * dh + c) * L + t] = v;
        }
      }
    };
    if (sw) gemm_rows<true>(sm.X, d, Wq, ldd, 3 * d, L, qkv_epi);
    else gemm_rows<false>(sm.X, d, Wq, ldd, 3 * d, L, qkv_epi);
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
    auto out_epi = [&](int t0, int nr, int n, const auto& acc) {
      constexpr int rb = sizeof(acc) / sizeof(float);
      const float b = P.b_o[n];
#pragma unroll
      for (int r = 0; r < rb; ++r)
        if (r < nr) sm.R[(size_t)(t0 + r) * d + n] = acc[r] + b + sm.X[(size_t)(t0 + r) * d + n];
    };
    if (sw) gemm_rows<true>(sm.C, d, Wo, ldd, d, L, out_epi);
    else gemm_rows<false>(sm.C, d, Wo, ldd, d, L, out_epi);
    __syncthreads();
    layernorm_rows(sm.R, P.ln1_g, P.ln1_b, sm.C, L, d);
    __syncthreads();
    // ---- FFN
    auto ffn1_epi = [&](int t0, int nr, int n, const auto& acc) {
      constexpr int rb = sizeof(acc) / sizeof(float);
      const float b = P.b_1[n];
#pragma unroll
      for (int r = 0; r < rb; ++r)
        if (r < nr) sm.HB[(size_t)(t0 + r) * dff + n] = gelu_erf(acc[r] + b);
    };
    if (sw) gemm_rows<true>(sm.C, d, W1, ldd, dff, L, ffn1_epi);
    else gemm_rows<false>(sm.C, d, W1, ldd, dff, L, ffn1_epi);
    __syncthreads();
    auto ffn2_epi = [&](int t0, int nr, int n, const auto& acc) {
      constexpr int rb = sizeof(acc) / sizeof(float);
      const float b = P.b_2[n];
#pragma unroll
      for (int r = 0; r < rb; ++r)
        if (r < nr) sm.R[(size_t)(t0 + r) * d + n] = acc[r] + b + sm.C[(size_t)(t0 + r) * d + n];
    };
    if (sw) gemm_rows<true>(sm.HB, dff, W2, ldf, d, L, ffn2_epi);
    else gemm_rows<false>(sm.HB, dff, W2, ldf, d, L, ffn2_epi);
    __syncthreads();
    const bool last = l + 1 == a.n_layers;
    layernorm_rows(sm.R, P.ln2_g, P.ln2_b, last ? a.out + (size_t)seq * L * d : sm.X, L, d);
    __syncthreads();
  }
}

size_t smem_bytes(int L, int d, int dh, int dff, int w_layers) {
  return carve(nullptr, L, d, dh, dff, w_layers).bytes;
}

constexpr size_t kSmemBudget = 200 * 1024;

}  // namespace

bool mega_simt_supported(int d, int H, int dff, int L, int n_layers, tl_dtype t) {
  if (t != TL_F32 || H < 1 || d % H || H > 64 || n_layers < 1 || n_layers > kMegaSimtMaxLayers) return false;
  const int dh = d / H;
  return d <= 64 && d % 4 == 0 && (dh == 8 || dh == 16 || dh == 32) && L <= 64 && dff <= 256 &&
         dff % 4 == 0 && smem_bytes(L, d, dh, dff, 0) <= kSmemBudget;
}

template <int DH>
static cudaError_t launch(MegaSimtArgs a, cudaStream_t s) {
  // Stage the weights when every layer's fit beside the activations.
  a.w_stage = smem_bytes(a.L, a.d, DH, a.dff, a.n_layers) <= kSmemBudget ? 1 : 0;
  const size_t smem = smem_bytes(a.L, a.d, DH, a.dff, a.w_stage ? a.n_layers : 0);
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
