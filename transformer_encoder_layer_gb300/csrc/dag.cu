// Persistent task-graph megakernel for small batches ("Hyper-optimized
// megakernel-hybrid transformer inference", section "Problem decomposition":
// when the batch is tiny, one CTA per sequence leaves most SMs idle, so a
// per-shape task graph is fixed ahead of time and persistent CTAs pop tasks
// from a queue until none are left).
//
// The graph is a pure function of the shape, so nothing is uploaded: task t
// decodes to (layer, kind, row block, tile).  Per layer, in queue order (a
// topological order of the graph):
//   QKV (rb, n)      64 x 64 tile of x W_qkv^T + b_qkv, scattered head-major
//   ATT (rb, h)      attention of the block's 64 query rows for head h;
//                    row blocks are queued last-first, the longest first
//   OUT (rb, n, kc)  64 x 64 tile of ctx W_o^T over one 256-wide K chunk;
//                    chunk 0 also adds b_o and the residual
//   LN1 (rb)         y = LayerNorm1(sum of the OUT chunks), rows of rb
//   F1  (rb, n)      64 x 64 tile of gelu(y W_1^T + b_1)
//   F2  (rb, n, kc)  64 x 64 tile of h W_2^T over one K chunk; chunk 0 also
//                    adds b_2 and y
//   LN2 (rb)         x' = LayerNorm2(sum of the F2 chunks): the next layer's
//                    input, or the output
// A task waits (bounded) on the completion counters of what it reads, then
// bumps its own.  It only ever waits on tasks earlier in the queue, each of
// which a running CTA has already taken, so the graph cannot deadlock, with
// any number of resident CTAs.  A QKV task of layer l also waits for every
// layer l-1 attention task that reads keys of its rows, so the single Q/K/V,
// ctx and activation buffers are never overwritten under a reader.
//
// The path serves fp32 I/O, whose weights no 16-bit tensor-core operand
// holds exactly: its arithmetic is fp32 on the CUDA cores, tiles staged in
// shared memory with cp.async.  The attention keeps the near-tie test and
// corrects flagged rows in fp64 inside the same task.
#include <cuda_runtime.h>

#include "common.cuh"
#include "dag.h"
#include "neartie.cuh"
#include "neartie_entry.cuh"

namespace tl {
namespace {

constexpr int kThreads = 256;
constexpr int R = kDagRows;
constexpr long long kWait = 4000000000LL;  // ~2 s of SM cycles per dependency wait
enum { K_QKV = 0, K_ATT, K_OUT, K_LN1, K_F1, K_F2, K_LN2, K_KINDS };

// Tasks of one layer, per kind.
struct Plan {
  int nt3, ntd, ntf;  // 64-wide column tiles of 3d, d and d_ff
  int kco, kcf;       // K chunks of the out-projection (K = d) and FFN2 (K = d_ff)
  int n[K_KINDS];
  int per_layer;
};

__host__ __device__ inline Plan make_plan(int RB, int H, int d, int dff) {
  Plan p;
  p.nt3 = (3 * d + 63) / 64;
  p.ntd = (d + 63) / 64;
  p.ntf = (dff + 63) / 64;
  p.kco = (d + kDagKChunk - 1) / kDagKChunk;
  p.kcf = (dff + kDagKChunk - 1) / kDagKChunk;
  p.n[K_QKV] = RB * p.nt3;
  p.n[K_ATT] = RB * H;
  p.n[K_OUT] = RB * p.ntd * p.kco;
  p.n[K_LN1] = RB;
  p.n[K_F1] = RB * p.ntf;
  p.n[K_F2] = RB * p.ntd * p.kcf;
  p.n[K_LN2] = RB;
  p.per_layer = 0;
  for (int k = 0; k < K_KINDS; ++k) p.per_layer += p.n[k];
  return p;
}

// ------------------------------------------------------------ primitives
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// 16-byte global -> shared copy through L2 only (data written earlier in
// this kernel by other CTAs is never read through a stale L1 line); a false
// predicate zero-fills the destination.
__device__ __forceinline__ void cp16(void* smem, const void* gmem, bool pred) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem),
               "r"(pred ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ GEMM
struct GemmSmem {
  float a[2][R][36];  // [stage][row][k], 32-wide K slabs, rows padded to 144 B
  float w[2][64][36];
};

// acc = A[m0.., k0..k1) . W[n0.., k0..k1)^T for a 64 x 64 tile.  Thread
// (ty, tx) = (tid / 16, tid % 16) owns rows ty + 16 i and columns tx + 16 j.
// K (lda, ldw and k1) must be a multiple of 4.
__device__ __forceinline__ void gemm_tile(const float* A, int lda, const float* W, int ldw, int M,
                                          int N, int k0, int k1, int m0, int n0,
                                          float (&acc)[4][4], GemmSmem& sm) {
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  const int nslab = (k1 - k0 + 31) / 32;
  auto issue = [&](int s) {
    const int st = s & 1, kb = k0 + s * 32;
#pragma unroll
    for (int c = tid; c < R * 8; c += kThreads) {
      const int row = c / 8, kc = (c % 8) * 4, k = kb + kc;
      const bool kin = k < k1;
      const bool pa = kin && m0 + row < M, pw = kin && n0 + row < N;
      cp16(&sm.a[st][row][kc], pa ? A + (size_t)(m0 + row) * lda + k : A, pa);
      cp16(&sm.w[st][row][kc], pw ? W + (size_t)(n0 + row) * ldw + k : W, pw);
    }
    cp_commit();
  };
  issue(0);
  for (int s = 0; s < nslab; ++s) {
    if (s + 1 < nslab) {
      issue(s + 1);
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    const int st = s & 1;
#pragma unroll
    for (int kk = 0; kk < 32; kk += 4) {
      float4 av[4], wv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = *reinterpret_cast<const float4*>(&sm.a[st][ty + 16 * i][kk]);
#pragma unroll
      for (int j = 0; j < 4; ++j) wv[j] = *reinterpret_cast<const float4*>(&sm.w[st][tx + 16 * j][kk]);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(av[i].x, wv[j].x, acc[i][j]);
          acc[i][j] = fmaf(av[i].y, wv[j].y, acc[i][j]);
          acc[i][j] = fmaf(av[i].z, wv[j].z, acc[i][j]);
          acc[i][j] = fmaf(av[i].w, wv[j].w, acc[i][j]);
        }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------- LayerNorm
// Rows of block rb: r = sum over the kc partial planes (in order), then
// (r - mean) / sqrt(var + 1e-5) * g + b, two-pass in fp32, one warp per row.
__device__ void ln_rows(const float* part, int kc, size_t plane, const float* g, const float* be,
                        float* out, int rb, int T, int d) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int rr = warp; rr < R; rr += kThreads / 32) {
    const int row = rb * R + rr;
    if (row >= T) break;
    const float* p = part + (size_t)row * d;
    float v[32];
    float sum = 0.f;
#pragma unroll
    for (int it = 0; it < 32; ++it) {
      const int c = lane + 32 * it;
      float s = 0.f;
      if (c < d) {
        s = __ldcg(p + c);
        for (int q = 1; q < kc; ++q) s += __ldcg(p + q * plane + c);
      }
      v[it] = s;
      sum += s;
    }
    const float mean = warp_sum(sum) / d;
    float sq = 0.f;
#pragma unroll
    for (int it = 0; it < 32; ++it) {
      const int c = lane + 32 * it;
      if (c < d) sq = fmaf(v[it] - mean, v[it] - mean, sq);
    }
    const float rstd = rsqrtf(warp_sum(sq) / d + 1e-5f);
#pragma unroll
    for (int it = 0; it < 32; ++it) {
      const int c = lane + 32 * it;
      if (c < d) out[(size_t)row * d + c] = (v[it] - mean) * rstd * g[c] + be[c];
    }
  }
}

// ------------------------------------------------------------- attention
template <int DH>
struct AttSmem {
  float k[2][64][DH + 4];
  float v[2][64][DH + 4];
  float kn2[2][64];
};

// One (row block, head): 4 threads per query row, each taking every 4th key
// of a 64-key tile; online softmax in the log2 domain; the four partial
// states merged at the end.  Rows whose two best scores are close relative
// to the fp32 score error are corrected in fp64 before the task completes.
template <int DH>
__device__ void attention_task(const DagArgs& a, int l, int rb, int h, const float* x_in,
                               unsigned char* smem_raw, int* flag_s, int* nflag_s) {
  AttSmem<DH>& sm = *reinterpret_cast<AttSmem<DH>*>(smem_raw);
  const int tid = threadIdx.x, row = tid >> 2, sub = tid & 3;
  const int H = a.H, L = a.L, T = a.T;
  const int rg = rb * R + row;
  const bool active = rg < T;
  const int b = active ? rg / L : 0, i = active ? rg % L : 0;
  int vl = a.vl[b];
  if (vl < 1 || vl > L) {
    if (active && l == 0 && h == 0 && i == 0 && sub == 0) set_status(a.status, TL_ERR_BAD_VALID_LEN);
    vl = vl < 1 ? 1 : L;
  }
  const int key_lo = b * L, key_end = active ? b * L + min(i + 1, vl) : 0;  // visible [lo, end)
  const int g_lo = ((rb * R) / L) * L, g_hi = min(rb * R + R, T);          // block's keys
  const int ntile = (g_hi - g_lo + 63) / 64;

  auto issue = [&](int t) {
    const int st = t & 1;
    constexpr int CPK = DH / 4;  // 16-byte chunks per key row
    for (int c = tid; c < 64 * CPK; c += kThreads) {
      const int jj = c / CPK, cc = (c % CPK) * 4, g = g_lo + t * 64 + jj;
      const bool ok = g < g_hi;
      const size_t off = ok ? ((((size_t)(g / L) * H + h) * L + g % L) * DH + cc) : 0;
      cp16(&sm.k[st][jj][cc], a.k + off, ok);
      cp16(&sm.v[st][jj][cc], a.v + off, ok);
    }
    cp_commit();
  };
  issue(0);

  const float scale_log2 = rsqrtf((float)DH) * 1.4426950408889634f;
  float q[DH], o[DH];
  float qn2 = 0.f;
  const float* qrow = a.q + (((size_t)b * H + h) * L + i) * DH;
#pragma unroll
  for (int c = 0; c < DH; c += 4) {
    float4 t4 = active ? __ldcg(reinterpret_cast<const float4*>(qrow + c)) : make_float4(0.f, 0.f, 0.f, 0.f);
    q[c] = t4.x; q[c + 1] = t4.y; q[c + 2] = t4.z; q[c + 3] = t4.w;
  }
#pragma unroll
  for (int c = 0; c < DH; ++c) {
    qn2 = fmaf(q[c], q[c], qn2);
    q[c] *= scale_log2;
    o[c] = 0.f;
  }
  float m = -INFINITY, lsum = 0.f, m1 = -INFINITY, m2 = -INFINITY, kn2max = 0.f;

  for (int t = 0; t < ntile; ++t) {
    if (t + 1 < ntile) {
      issue(t + 1);
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    const int st = t & 1;
    {  // squared key norms of the tile, 4 threads per key
      const int key = tid >> 2, part = tid & 3;
      float s = 0.f;
#pragma unroll
      for (int c = part * 4; c < DH; c += 16) {
        const float4 kv = *reinterpret_cast<const float4*>(&sm.k[st][key][c]);
        s = fmaf(kv.x, kv.x, fmaf(kv.y, kv.y, fmaf(kv.z, kv.z, fmaf(kv.w, kv.w, s))));
      }
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (part == 0) sm.kn2[st][key] = s;
    }
    __syncthreads();
    const int gbase = g_lo + t * 64;
    if (gbase < key_end && gbase + 64 > key_lo) {
      float s[16];
      float mt = -INFINITY;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int jj = sub + 4 * u, g = gbase + jj;
        if (g >= key_lo && g < key_end) {
          float dot = 0.f;
#pragma unroll
          for (int c = 0; c < DH; c += 4) {
            const float4 kv = *reinterpret_cast<const float4*>(&sm.k[st][jj][c]);
            dot = fmaf(q[c], kv.x, dot);
            dot = fmaf(q[c + 1], kv.y, dot);
            dot = fmaf(q[c + 2], kv.z, dot);
            dot = fmaf(q[c + 3], kv.w, dot);
          }
          s[u] = dot;
          m2 = fmaxf(m2, fminf(m1, dot));
          m1 = fmaxf(m1, dot);
          kn2max = fmaxf(kn2max, sm.kn2[st][jj]);
        } else {
          s[u] = -INFINITY;
        }
        mt = fmaxf(mt, s[u]);
      }
      if (mt > m) {
        const float corr = exp2f(m - mt);  // 0 while m = -inf
        lsum *= corr;
#pragma unroll
        for (int c = 0; c < DH; ++c) o[c] *= corr;
        m = mt;
      }
      if (m != -INFINITY) {
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float p = exp2f(s[u] - m);  // 0 for masked keys
          lsum += p;
          const int jj = sub + 4 * u;
#pragma unroll
          for (int c = 0; c < DH; c += 4) {
            const float4 vv = *reinterpret_cast<const float4*>(&sm.v[st][jj][c]);
            o[c] = fmaf(p, vv.x, o[c]);
            o[c + 1] = fmaf(p, vv.y, o[c + 1]);
            o[c + 2] = fmaf(p, vv.z, o[c + 2]);
            o[c + 3] = fmaf(p, vv.w, o[c + 3]);
          }
        }
      }
    }
    __syncthreads();
  }
  // merge the four partial states of the row (adjacent lanes)
#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, off);
    const float lo = __shfl_xor_sync(0xffffffffu, lsum, off);
    const float a1 = __shfl_xor_sync(0xffffffffu, m1, off);
    const float a2 = __shfl_xor_sync(0xffffffffu, m2, off);
    kn2max = fmaxf(kn2max, __shfl_xor_sync(0xffffffffu, kn2max, off));
    const float mn = fmaxf(m, mo);
    const float fa = mn == -INFINITY ? 0.f : exp2f(m - mn);
    const float fb = mn == -INFINITY ? 0.f : exp2f(mo - mn);
#pragma unroll
    for (int c = 0; c < DH; ++c) {
      const float oo = __shfl_xor_sync(0xffffffffu, o[c], off);
      o[c] = o[c] * fa + oo * fb;
    }
    lsum = lsum * fa + lo * fb;
    m = mn;
    m2 = fmaxf(fmaxf(m2, a2), fminf(m1, a1));
    m1 = fmaxf(m1, a1);
  }
  if (tid == 0) *nflag_s = 0;
  __syncthreads();
  if (active && sub == 0) {
    const float inv = 1.f / lsum;
    float* dst = a.ctx + (size_t)rg * a.d + (size_t)h * DH;
#pragma unroll
    for (int c = 0; c < DH; c += 4)
      *reinterpret_cast<float4*>(dst + c) = make_float4(o[c] * inv, o[c + 1] * inv, o[c + 2] * inv, o[c + 3] * inv);
    if (neartie_flag((m1 - m2) * 0.69314718055994531f, sqrtf(qn2), sqrtf(kn2max), DH))
      flag_s[atomicAdd(nflag_s, 1)] = ((b * H + h) * L) + i;
  }
  __syncthreads();
  const int nflag = *nflag_s;
  if (nflag > 0) {
    FixupArgs fa{};
    fa.x = Plane{x_in, nullptr, 0};
    fa.w_qkv = a.layers[l].w_qkv;
    fa.w_kind = 0;
    fa.b_qkv = a.layers[l].b_qkv;
    fa.q = Plane{a.q, nullptr, 0};
    fa.k = Plane{a.k, nullptr, 0};
    fa.v = Plane{a.v, nullptr, 0};
    fa.v_transposed = 0;
    fa.Lp = L;
    fa.ctx_hi = a.ctx;
    fa.ctx_kind = 0;
    fa.valid_len = a.vl;
    fa.B = a.B; fa.H = H; fa.L = L; fa.dh = DH; fa.d = a.d;
    const int warp = tid / 32, lane = tid % 32;
    double* q64 = reinterpret_cast<double*>(smem_raw) + (size_t)warp * (DH + a.d);
    for (int e = warp; e < nflag; e += kThreads / 32)
      ntie::neartie_fix_entry(fa, flag_s[e], q64, q64 + DH, lane);
  }
}

// ---------------------------------------------------------------- kernel
template <int DH>
__global__ void __launch_bounds__(kThreads, 1) dag_kernel(const __grid_constant__ DagArgs a) {
  extern __shared__ __align__(16) unsigned char dag_smem[];
  __shared__ int task_s, go_s, nflag_s;
  __shared__ int flag_s[R];
  const int tid = threadIdx.x;
  const Plan pl = make_plan(a.RB, a.H, a.d, a.dff);
  const int total = a.n_layers * pl.per_layer;
  const int d = a.d, H = a.H, L = a.L, T = a.T, RB = a.RB;
  const size_t plane = (size_t)T * d;
  auto counter = [&](int l, int kind, int rb) { return a.cnt + ((size_t)l * K_KINDS + kind) * RB + rb; };
  // Thread 0 only: wait until *c >= target, or give up (abort or deadline).
  auto wait_ge = [&](const int* c, int target) -> bool {
    if (ld_acquire(c) >= target) return true;
    const long long t0 = clock64();
    while (ld_acquire(c) < target) {
      if (*(volatile int*)a.abort) return false;
      __nanosleep(64);
      if (clock64() - t0 > kWait) {
        atomicExch(a.abort, 1);
        set_status(a.status, TL_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
    return true;
  };
  // Every thread's writes are ordered before the release of the counter.
  auto signal = [&](int* c) {
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      atomicAdd(c, 1);
    }
  };
  // The row blocks holding rows of the sequences that meet block rb.
  auto rb_first = [&](int rb) { return ((rb * R) / L) * L / R; };
  auto rb_last = [&](int rb) {
    const int last_row = min(rb * R + R, T) - 1;
    return min(((last_row / L + 1) * L - 1) / R, RB - 1);
  };

  while (true) {
    __syncthreads();
    if (tid == 0) task_s = atomicAdd(a.head, 1);
    __syncthreads();
    const int t = task_s;
    if (t >= total) break;
    const int l = t / pl.per_layer;
    int rem = t % pl.per_layer, kind = 0;
    while (rem >= pl.n[kind]) rem -= pl.n[kind++];
    const tl_layer_dev& P = a.layers[l];
    const float* x_in = l == 0 ? a.x : ((l & 1) ? a.xs1 : a.xs0);  // this layer's input
    float* x_next = (l & 1) ? a.xs0 : a.xs1;
    // task coordinates
    int rb = 0, nt = 0, kc = 0, h = 0;
    switch (kind) {
      case K_QKV: rb = rem / pl.nt3; nt = rem % pl.nt3; break;
      case K_ATT: rb = RB - 1 - rem / H; h = rem % H; break;
      case K_OUT: rb = rem / (pl.ntd * pl.kco); nt = (rem / pl.kco) % pl.ntd; kc = rem % pl.kco; break;
      case K_F1: rb = rem / pl.ntf; nt = rem % pl.ntf; break;
      case K_F2: rb = rem / (pl.ntd * pl.kcf); nt = (rem / pl.kcf) % pl.ntd; kc = rem % pl.kcf; break;
      default: rb = rem; break;
    }
    // ------------------------------------------------------ dependencies
    if (tid == 0) {
      bool ok = !*(volatile int*)a.abort;
      if (ok && a.inject_stall && t == 0) ok = wait_ge(counter(0, K_LN2, 0), 1 << 30);
      switch (kind) {
        case K_QKV:
          if (l > 0) {
            ok = ok && wait_ge(counter(l - 1, K_LN2, rb), 1);
            for (int r2 = rb; ok && r2 <= rb_last(rb); ++r2) ok = wait_ge(counter(l - 1, K_ATT, r2), H);
          }
          break;
        case K_ATT:
          for (int r2 = rb_first(rb); ok && r2 <= rb; ++r2) ok = wait_ge(counter(l, K_QKV, r2), pl.nt3);
          break;
        case K_OUT: ok = ok && wait_ge(counter(l, K_ATT, rb), H); break;
        case K_LN1: ok = ok && wait_ge(counter(l, K_OUT, rb), pl.ntd * pl.kco); break;
        case K_F1: ok = ok && wait_ge(counter(l, K_LN1, rb), 1); break;
        case K_F2: ok = ok && wait_ge(counter(l, K_F1, rb), pl.ntf); break;
        default: ok = ok && wait_ge(counter(l, K_F2, rb), pl.ntd * pl.kcf); break;
      }
      if (ok) __threadfence();
      go_s = ok;
    }
    __syncthreads();
    if (!go_s) continue;  // aborted: drain the queue without work
    // --------------------------------------------------------------- work
    if (kind == K_ATT) {
      attention_task<DH>(a, l, rb, h, x_in, dag_smem, flag_s, &nflag_s);
    } else if (kind == K_LN1) {
      ln_rows(a.part, pl.kco, plane, P.ln1_g, P.ln1_b, a.y, rb, T, d);
    } else if (kind == K_LN2) {
      ln_rows(a.part, pl.kcf, plane, P.ln2_g, P.ln2_b, l + 1 < a.n_layers ? x_next : a.out, rb, T, d);
    } else {
      GemmSmem& gs = *reinterpret_cast<GemmSmem*>(dag_smem);
      float acc[4][4];
      const int m0 = rb * R, n0 = nt * 64;
      int N = d;
      if (kind == K_QKV) {
        N = 3 * d;
        gemm_tile(x_in, d, (const float*)P.w_qkv, d, T, N, 0, d, m0, n0, acc, gs);
      } else if (kind == K_OUT) {
        gemm_tile(a.ctx, d, (const float*)P.w_o, d, T, N, kc * kDagKChunk,
                  min(d, (kc + 1) * kDagKChunk), m0, n0, acc, gs);
      } else if (kind == K_F1) {
        N = a.dff;
        gemm_tile(a.y, d, (const float*)P.w_1, d, T, N, 0, d, m0, n0, acc, gs);
      } else {
        gemm_tile(a.hb, a.dff, (const float*)P.w_2, a.dff, T, N, kc * kDagKChunk,
                  min(a.dff, (kc + 1) * kDagKChunk), m0, n0, acc, gs);
      }
      const int tx = tid % 16, ty = tid / 16;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int mm = m0 + ty + 16 * i;
        if (mm >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int n = n0 + tx + 16 * j;
          if (n >= N) continue;
          const float v = acc[i][j];
          if (kind == K_QKV) {
            const int which = n / d, w = n % d, hh = w / DH, c = w % DH;
            float* dst = which == 0 ? a.q : which == 1 ? a.k : a.v;
            dst[(((size_t)(mm / L) * H + hh) * L + mm % L) * DH + c] = v + P.b_qkv[n];
          } else if (kind == K_OUT) {
            const size_t at = (size_t)mm * d + n;
            a.part[kc * plane + at] = kc == 0 ? v + P.b_o[n] + __ldcg(x_in + at) : v;
          } else if (kind == K_F1) {
            a.hb[(size_t)mm * a.dff + n] = gelu_erf(v + P.b_1[n]);
          } else {
            const size_t at = (size_t)mm * d + n;
            a.part[kc * plane + at] = kc == 0 ? v + P.b_2[n] + __ldcg(a.y + at) : v;
          }
        }
      }
    }
    signal(counter(l, kind, rb));
  }
}

template <int DH>
cudaError_t launch(const DagArgs& a, int grid, cudaStream_t s) {
  const size_t smem = dag_dyn_smem(a.d, DH);
  auto k = dag_kernel<DH>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool dag_supported(int d, int H, int dff, int n_layers, tl_dtype t) {
  if (t != TL_F32 || H < 1 || d % H || n_layers < 1 || n_layers > kDagMaxLayers) return false;
  const int dh = d / H;
  // 16-byte cp.async rows need d and d_ff multiples of 4; LayerNorm keeps a
  // row in 32 registers per lane.
  return (dh == 16 || dh == 32 || dh == 64) && d <= 1024 && dff % 4 == 0 && dff >= 4;
}

int dag_counter_ints(int n_layers, int RB) { return n_layers * K_KINDS * RB + 2; }

size_t dag_dyn_smem(int d, int dh) {
  size_t att = dh == 16 ? sizeof(AttSmem<16>) : dh == 32 ? sizeof(AttSmem<32>) : sizeof(AttSmem<64>);
  size_t fix = (size_t)(kThreads / 32) * (dh + d) * sizeof(double);
  size_t m = sizeof(GemmSmem);
  if (att > m) m = att;
  if (fix > m) m = fix;
  return m;
}

cudaError_t dag_forward(const DagArgs& a, int num_sms, cudaStream_t s) {
  const Plan pl = make_plan(a.RB, a.H, a.d, a.dff);
  const int total = a.n_layers * pl.per_layer;
  const int grid = total < num_sms ? total : num_sms;  // one resident CTA per SM
  const int dh = a.d / a.H;
  if (dh == 16) return launch<16>(a, grid, s);
  if (dh == 32) return launch<32>(a, grid, s);
  return launch<64>(a, grid, s);
}

}  // namespace tl
