// Generic fp32 CUDA-core path: every step of the layer for any supported
// shape (head_dim <= 128, d_model <= 1024).  It is the accurate fallback for
// shapes the tensor-core paths do not cover (fp32 I/O, odd head sizes) and a
// second GPU implementation the tensor-core kernels are cross-checked with.
#include "common.cuh"
#include "internal.h"
#include "neartie.cuh"

namespace tl {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;

template <typename T>
__device__ __forceinline__ float ld(const void* p, size_t i) {
  return to_f32<T>(reinterpret_cast<const T*>(p)[i]);
}

// C tile 64x64, 256 threads, each a 4x4 block; A and W both K-major.
template <typename TA, typename TW, typename TR, int EPI>
__global__ void __launch_bounds__(256) simt_gemm_kernel(SimtGemmArgs a) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Ws[TK][TN + 4];
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  float acc[4][4] = {};
  const int lr = tid / 4, lk = (tid % 4) * 4;  // loader: row, first k
  for (int k0 = 0; k0 < a.K; k0 += TK) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int m = m0 + lr, k = k0 + lk + j;
      As[lk + j][lr] = (m < a.M && k < a.K) ? ld<TA>(a.A, (size_t)m * a.K + k) : 0.f;
      int n = n0 + lr;
      Ws[lk + j][lr] = (n < a.N && k < a.K) ? ld<TW>(a.W, (size_t)n * a.K + k) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float av[4], wv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) wv[j] = Ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }
  const int d = a.H * a.dh;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int m = m0 + ty * 4 + i;
    if (m >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int n = n0 + tx * 4 + j;
      if (n >= a.N) continue;
      float v = acc[i][j] + a.bias[n];
      if (EPI == EPI_QKV_HEADMAJOR) {
        int which = n / d, w = n % d, h = w / a.dh, c = w % a.dh;
        int b = m / a.L, t = m % a.L;
        size_t plane = (size_t)a.B * a.H * a.L * a.dh;
        a.out[which * plane + (((size_t)b * a.H + h) * a.L + t) * a.dh + c] = v;
      } else if (EPI == EPI_BIAS_GELU) {
        a.out[(size_t)m * a.N + n] = gelu_erf(v);
      } else {
        a.out[(size_t)m * a.N + n] = v + ld<TR>(a.resid, (size_t)m * a.N + n);
      }
    }
  }
}

template <typename TA, typename TW, typename TR, int EPI>
cudaError_t launch_gemm(const SimtGemmArgs& a, cudaStream_t s) {
  dim3 grid((a.N + TN - 1) / TN, (a.M + TM - 1) / TM);
  simt_gemm_kernel<TA, TW, TR, EPI><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

// Only the operand combinations the layer uses are instantiated: the QKV
// projection reads x (I/O dtype) or the fp32 residual stream; the
// out-projection adds x or the fp32 stream; FFN1/FFN2 read fp32.
template <typename TW>
cudaError_t gemm_w(const SimtGemmArgs& a, cudaStream_t s) {
  const bool a32 = a.a_dtype == TL_F32, r32 = a.r_dtype == TL_F32;
  switch (a.epi) {
    case EPI_QKV_HEADMAJOR:
      return a32 ? launch_gemm<float, TW, float, EPI_QKV_HEADMAJOR>(a, s)
                 : launch_gemm<TW, TW, float, EPI_QKV_HEADMAJOR>(a, s);
    case EPI_BIAS_GELU:
      if (!a32) return cudaErrorInvalidValue;
      return launch_gemm<float, TW, float, EPI_BIAS_GELU>(a, s);
    default:
      if (!a32) return cudaErrorInvalidValue;
      return r32 ? launch_gemm<float, TW, float, EPI_BIAS_RESID>(a, s)
                 : launch_gemm<float, TW, TW, EPI_BIAS_RESID>(a, s);
  }
}

// ------------------------------------------------------------- attention
// One thread per query row, 128 rows per block; K/V of one (b, h) streamed
// through shared memory in key tiles.  Online softmax in fp32 with one
// rescale per key tile.  Keys visible to row i: j < min(i + 1, valid_len).
// Each row also tracks its two largest scores and the error scale of its
// fp32 scores, and queues itself for the fp64 near-tie fix-up when a tie
// within that error could move the softmax (see neartie.cuh).
constexpr int AQ = 128;

// Where the attention reads Q/K/V and writes the context:
//  MODE 0  fp32 q, k, v [B, H, L, dh]; fp32 ctx [T, d]
//  MODE 1/2  fp16/bf16 (hi, lo) planes, q, k [B, H, L, dh], v^T [B, H, dh, Lp];
//            ctx as (hi, lo) planes [T, d]
template <int MODE> struct AttnAcc;
template <> struct AttnAcc<0> {
  __device__ static float ld(const void* hi, const void*, size_t i) {
    return reinterpret_cast<const float*>(hi)[i];
  }
  __device__ static void st(void* hi, void*, size_t i, float v) { reinterpret_cast<float*>(hi)[i] = v; }
};
template <typename T> struct AttnAccPair {
  __device__ static float ld(const void* hi, const void* lo, size_t i) {
    return to_f32<T>(reinterpret_cast<const T*>(hi)[i]) + to_f32<T>(reinterpret_cast<const T*>(lo)[i]);
  }
  __device__ static void st(void* hi, void* lo, size_t i, float v) {
    T h = from_f32<T>(v);
    reinterpret_cast<T*>(hi)[i] = h;
    reinterpret_cast<T*>(lo)[i] = from_f32<T>(v - to_f32<T>(h));
  }
};
template <> struct AttnAcc<1> : AttnAccPair<__half> {};
template <> struct AttnAcc<2> : AttnAccPair<__nv_bfloat16> {};

// Key-tile size shrinks as head_dim grows to bound registers.
template <int DH, int MODE, int AK = (DH <= 32 ? 32 : DH == 64 ? 16 : 8)>
__global__ void __launch_bounds__(AQ) simt_attention_kernel(AttnIO io, const int32_t* __restrict__ vlp,
                                                            int B, int H, int L, int dh, int* status,
                                                            NearTieList ties) {
  using Acc = AttnAcc<MODE>;
  __shared__ float Ks[AK][DH];
  __shared__ float Vs[AK][DH];
  __shared__ float Kn[AK];
  const int b = blockIdx.z, h = blockIdx.y;
  const int i0 = blockIdx.x * AQ, i = i0 + threadIdx.x;
  const int vl = load_valid_len(vlp, b, L, threadIdx.x == 0 && blockIdx.x == 0 && h == 0 ? status : nullptr);
  const size_t bh = (size_t)b * H + h;
  const size_t base = bh * L * dh;
  const float scale_log2 = rsqrtf((float)dh) * 1.4426950408889634f;
  float qr[DH], acc[DH];
  float qn2 = 0.f;
#pragma unroll
  for (int c = 0; c < DH; ++c) {
    float qv = (i < L && c < dh) ? Acc::ld(io.q_hi, io.q_lo, base + (size_t)i * dh + c) : 0.f;
    qn2 = fmaf(qv, qv, qn2);
    qr[c] = qv * scale_log2;
    acc[c] = 0.f;
  }
  const int n_keys = i < L ? min(i + 1, vl) : 0;
  const int block_keys = min(min(i0 + AQ, L), vl);  // keys any row of the block sees
  float m = -INFINITY, m2 = -INFINITY, l = 0.f, kmax = 0.f;
  for (int j0 = 0; j0 < block_keys; j0 += AK) {
    for (int e = threadIdx.x; e < AK * DH; e += AQ) {
      int jj = e / DH, c = e % DH, j = j0 + jj;
      bool ok = j < block_keys && c < dh;
      Ks[jj][c] = ok ? Acc::ld(io.k_hi, io.k_lo, base + (size_t)j * dh + c) : 0.f;
      size_t vi = io.v_transposed ? (bh * dh + c) * io.Lp + j : base + (size_t)j * dh + c;
      Vs[jj][c] = ok ? Acc::ld(io.v_hi, io.v_lo, vi) : 0.f;
    }
    __syncthreads();
    if (threadIdx.x < AK) {
      float t = 0.f;
#pragma unroll
      for (int c = 0; c < DH; ++c) t = fmaf(Ks[threadIdx.x][c], Ks[threadIdx.x][c], t);
      Kn[threadIdx.x] = sqrtf(t);
    }
    __syncthreads();
    float s[AK];
    float tmax = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < AK; ++jj) {
      kmax = fmaxf(kmax, Kn[jj]);
      float t = 0.f;
#pragma unroll
      for (int c = 0; c < DH; ++c) t = fmaf(qr[c], Ks[jj][c], t);
      s[jj] = (j0 + jj < n_keys) ? t : -INFINITY;
      // second-largest so far: max(m2, min(running max, s))
      m2 = fmaxf(m2, fminf(fmaxf(m, tmax), s[jj]));
      tmax = fmaxf(tmax, s[jj]);
    }
    if (tmax > -INFINITY) {
      float mn = fmaxf(m, tmax);
      float corr = exp2f(m - mn);  // m = -inf on the first tile -> 0
      l *= corr;
#pragma unroll
      for (int c = 0; c < DH; ++c) acc[c] *= corr;
#pragma unroll
      for (int jj = 0; jj < AK; ++jj) {
        float p = exp2f(s[jj] - mn);  // exactly 0 for hidden keys
        l += p;
#pragma unroll
        for (int c = 0; c < DH; ++c) acc[c] = fmaf(p, Vs[jj][c], acc[c]);
      }
      m = mn;
    }
    __syncthreads();
  }
  if (i < L) {
    float inv = 1.f / l;
    const size_t o = ((size_t)b * L + i) * H * dh + (size_t)h * dh;
#pragma unroll
    for (int c = 0; c < DH; ++c)
      if (c < dh) Acc::st(io.ctx_hi, io.ctx_lo, o + c, acc[c] * inv);
    // scores are in log2 units here; the test takes natural-log gaps
    if (neartie_flag((m - m2) * 0.69314718055994531f, sqrtf(qn2), kmax, dh))
      neartie_push(ties, (int)(bh * L) + i);
  }
}

// ------------------------------------------------------------- LayerNorm
template <int PER_LANE>
__global__ void simt_layernorm_kernel(const float* __restrict__ r, const float* __restrict__ g,
                                      const float* __restrict__ bta, float* __restrict__ y32,
                                      void* __restrict__ yout, int out_dtype, int M, int d) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
  if (warp >= M) return;
  const float* row = r + (size_t)warp * d;
  float x[PER_LANE];
  float sum = 0.f;
#pragma unroll
  for (int t = 0; t < PER_LANE; ++t) {
    int c = lane + 32 * t;
    x[t] = c < d ? row[c] : 0.f;
    sum += x[t];
  }
  const float mean = warp_sum(sum) / d;
  float sq = 0.f;
#pragma unroll
  for (int t = 0; t < PER_LANE; ++t) {
    int c = lane + 32 * t;
    float dv = c < d ? x[t] - mean : 0.f;
    sq = fmaf(dv, dv, sq);
  }
  const float rstd = rsqrtf(warp_sum(sq) / d + 1e-5f);
#pragma unroll
  for (int t = 0; t < PER_LANE; ++t) {
    int c = lane + 32 * t;
    if (c >= d) continue;
    float yv = (x[t] - mean) * rstd * g[c] + bta[c];
    size_t o = (size_t)warp * d + c;
    if (y32) y32[o] = yv;
    if (yout) {
      if (out_dtype == TL_F32) reinterpret_cast<float*>(yout)[o] = yv;
      else if (out_dtype == TL_F16) reinterpret_cast<__half*>(yout)[o] = __float2half_rn(yv);
      else reinterpret_cast<__nv_bfloat16*>(yout)[o] = __float2bfloat16_rn(yv);
    }
  }
}

}  // namespace

cudaError_t simt_gemm(const SimtGemmArgs& a, cudaStream_t s) {
  switch (a.w_dtype) {
    case TL_F32: return gemm_w<float>(a, s);
    case TL_F16: return gemm_w<__half>(a, s);
    default: return gemm_w<__nv_bfloat16>(a, s);
  }
}

template <int MODE>
static cudaError_t attn_mode(const AttnIO& io, const int32_t* vl, int B, int H, int L, int dh,
                             int* status, NearTieList ties, cudaStream_t s) {
  dim3 grid((L + AQ - 1) / AQ, H, B);
  if (dh <= 16) simt_attention_kernel<16, MODE><<<grid, AQ, 0, s>>>(io, vl, B, H, L, dh, status, ties);
  else if (dh <= 32) simt_attention_kernel<32, MODE><<<grid, AQ, 0, s>>>(io, vl, B, H, L, dh, status, ties);
  else if (dh <= 64) simt_attention_kernel<64, MODE><<<grid, AQ, 0, s>>>(io, vl, B, H, L, dh, status, ties);
  else simt_attention_kernel<128, MODE><<<grid, AQ, 0, s>>>(io, vl, B, H, L, dh, status, ties);
  return cudaGetLastError();
}

cudaError_t simt_attention(const AttnIO& io, int mode, const int32_t* vl, int B, int H, int L,
                           int dh, int* status, NearTieList ties, cudaStream_t s) {
  if (mode == 0) return attn_mode<0>(io, vl, B, H, L, dh, status, ties, s);
  if (mode == 1) return attn_mode<1>(io, vl, B, H, L, dh, status, ties, s);
  return attn_mode<2>(io, vl, B, H, L, dh, status, ties, s);
}

cudaError_t simt_layernorm(const float* r, const float* g, const float* b, float* y32,
                           void* yout, tl_dtype out_dtype, int M, int d, cudaStream_t s) {
  const int threads = 256, rows_per_block = threads / 32;
  dim3 grid((M + rows_per_block - 1) / rows_per_block);
  if (d <= 128) simt_layernorm_kernel<4><<<grid, threads, 0, s>>>(r, g, b, y32, yout, out_dtype, M, d);
  else if (d <= 256) simt_layernorm_kernel<8><<<grid, threads, 0, s>>>(r, g, b, y32, yout, out_dtype, M, d);
  else if (d <= 512) simt_layernorm_kernel<16><<<grid, threads, 0, s>>>(r, g, b, y32, yout, out_dtype, M, d);
  else simt_layernorm_kernel<32><<<grid, threads, 0, s>>>(r, g, b, y32, yout, out_dtype, M, d);
  return cudaGetLastError();
}

}  // namespace tl
