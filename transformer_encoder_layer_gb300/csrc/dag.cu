// Persistent task-graph megakernel for small batches ("Hyper-optimized
// megakernel-hybrid transformer inference", section "Problem decomposition":
// when the batch is tiny, one CTA per sequence leaves most SMs idle, so a
// per-shape task graph is fixed ahead of time and persistent CTAs pop tasks
// from a queue until none are left).
//
// The graph is a pure function of the shape, so nothing is uploaded: task t
// decodes to (layer, kind, row block, tile).  Per layer, in queue order (a
// topological order of the graph):
//   QKV (rb, n)         64 x 64 tile of x W_qkv^T + b_qkv, scattered head-major
//   ATT (rb, half, h)   attention of 32 query rows for head h; row blocks are
//                       queued last-first, the longest first
//   OUT (rb, n, kc)     64 x 64 tile of ctx W_o^T over one 256-wide K chunk;
//                       chunk 0 also adds b_o and the residual
//   F1  (rb, n)         64 x 64 tile of gelu(y W_1^T + b_1)
//   F2  (rb, n, kc)     64 x 64 tile of h W_2^T over one K chunk; chunk 0 also
//                       adds b_2 and y
// The two LayerNorms are not queued: the OUT (F2) task that completes a row
// block last sums its K-chunk partials in a fixed order and normalises the
// block's rows (y, or the next layer's input / the output).
//
// A task waits (bounded) on the completion counters of what it reads, then
// bumps its own.  It only ever waits on tasks earlier in the queue, so the
// lowest unfinished task is always running with its inputs ready: no
// deadlock, with any number of resident CTAs, also while each CTA holds the
// index of its next task (popped early to hide the atomic's latency).  A QKV
// task of layer l also waits for every layer l-1 attention task that reads
// keys of its rows, so the single Q/K/V, ctx and activation buffers are
// never overwritten under a reader.
//
// The path serves fp32 I/O, whose weights no 16-bit tensor-core operand
// holds exactly: its arithmetic is fp32 on the CUDA cores, tiles staged in
// shared memory with cp.async.  Each CTA runs a handful of tasks of
// different kinds per forward, so the code is kept compact (instruction
// fetch of cold, heavily unrolled code dominated the first version).  The
// attention keeps the near-tie test and corrects flagged rows in fp64 inside
// the same task.
#include <cuda_runtime.h>

#include "common.cuh"
#include "dag.h"
#include "neartie.cuh"
#include "neartie_entry.cuh"

namespace tl {
namespace {

constexpr int kThreads = 256;
constexpr int R = kDagRows;
constexpr int kAttRows = 32;  // query rows of one attention task
constexpr long long kWait = 4000000000LL;  // ~2 s of SM cycles per dependency wait
enum { K_QKV = 0, K_ATT, K_OUT, K_LN1, K_F1, K_F2, K_LN2, K_KINDS };
// Queue order within a layer: QKV, ATT, OUT, F1, F2 (the LayerNorms are not queued).
__host__ __device__ constexpr int queued_kind(int q) { return q < 3 ? q : q + 1; }

// Tasks of one layer, per kind.
struct Plan {
  int nt3, ntd, ntf;  // 64-wide column tiles of 3d, d and d_ff
  int kco, kcf;       // K chunks of the out-projection (K = d) and FFN2 (K = d_ff)
  int n[K_KINDS];     // queued tasks per kind (0 for the LayerNorms)
  int target[K_KINDS];  // completions per row block
  int per_layer;
};

__host__ __device__ inline Plan make_plan(int RB, int H, int d, int dff) {
  Plan p;
  p.nt3 = (3 * d + 63) / 64;
  p.ntd = (d + 63) / 64;
  p.ntf = (dff + 63) / 64;
  p.kco = (d + kDagKChunk - 1) / kDagKChunk;
  p.kcf = (dff + kDagKChunk - 1) / kDagKChunk;
  p.target[K_QKV] = p.nt3;
  p.target[K_ATT] = (R / kAttRows) * H;
  p.target[K_OUT] = p.ntd * p.kco;
  p.target[K_LN1] = 1;
  p.target[K_F1] = p.ntf;
  p.target[K_F2] = p.ntd * p.kcf;
  p.target[K_LN2] = 1;
  p.per_layer = 0;
  for (int k = 0; k < K_KINDS; ++k) {
    p.n[k] = (k == K_LN1 || k == K_LN2) ? 0 : RB * p.target[k];
    p.per_layer += p.n[k];
  }
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

// Wait until at most n of this thread's cp.async groups are pending.
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

// ------------------------------------------------------------------ GEMM
// 128 columns of K of both operands are staged at once, one cp.async group
// per 32-wide slab, so the copies of every slab are in flight together and
// compute on slab s overlaps the arrival of the later ones.
constexpr int kStageK = 128;           // K staged in shared memory at once
constexpr int kGemmLd = kStageK + 4;   // row stride in floats (16-byte multiple, 4-bank skew)
struct GemmSmem {
  float a[R][kGemmLd];
  float w[64][kGemmLd];
};

// acc = A[m0.., k0..k1) . W[n0.., k0..k1)^T for a 64 x 64 tile, staged 128
// columns of K at a time.  Thread (ty, tx) = (tid / 16, tid % 16) owns rows ty + 16 i and
// columns tx + 16 j.  K (lda, ldw and k1) must be a multiple of 4.
__device__ __forceinline__ void gemm_tile(const float* A, int lda, const float* W, int ldw, int M,
                                          int N, int k0, int k1, int m0, int n0,
                                          float (&acc)[4][4], GemmSmem& sm) {
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int kb = k0; kb < k1; kb += kStageK) {
    const int ke = min(k1, kb + kStageK);
    const int nslab = (ke - kb + 31) / 32;  // <= 4
    for (int s = 0; s < nslab; ++s) {
#pragma unroll
      for (int c = tid; c < R * 8; c += kThreads) {
        const int row = c / 8, kl = s * 32 + (c % 8) * 4, k = kb + kl;
        const bool kin = k < ke;
        const bool pa = kin && m0 + row < M, pw = kin && n0 + row < N;
        cp16(&sm.a[row][kl], pa ? A + (size_t)(m0 + row) * lda + k : A, pa);
        cp16(&sm.w[row][kl], pw ? W + (size_t)(n0 + row) * ldw + k : W, pw);
      }
      cp_commit();
    }
    for (int s = 0; s < nslab; ++s) {
      cp_wait_n(nslab - 1 - s);
      __syncthreads();
#pragma unroll 2
      for (int kk = s * 32; kk < s * 32 + 32; kk += 4) {
        float4 av[4], wv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = *reinterpret_cast<const float4*>(&sm.a[ty + 16 * i][kk]);
#pragma unroll
        for (int j = 0; j < 4; ++j) wv[j] = *reinterpret_cast<const float4*>(&sm.w[tx + 16 * j][kk]);
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
    }
    __syncthreads();  // the staging buffers are free again
  }
}

// ------------------------------------------------------------- LayerNorm
// Rows of block rb: r = part[0] + part[1] + ... (K-chunk partials, in that
// order), then (r - mean) / sqrt(var + 1e-5) * g + b, two-pass in fp32.  The
// sums are formed with 16 independent 16-byte loads in flight per thread and
// parked in shared memory (at most 64 KB a pass); one warp then normalises
// each row from there.
__device__ __noinline__ void ln_block(const float* part, int kc, size_t plane, const float* g,
                                      const float* be, float* out, int rb, int T, int d,
                                      float* sbuf) {
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int rows = min(R, T - rb * R);
  const int rp = min(R, 16384 / d);
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r0 = 0; r0 < rows; r0 += rp) {
    const int nr = min(rp, rows - r0);
    const int nch = nr * d / 4;  // <= 4096 chunks: 16 per thread
    const float4* src = reinterpret_cast<const float4*>(part + (size_t)(rb * R + r0) * d);
    float4 acc[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int c = tid + u * kThreads;
      acc[u] = c < nch ? __ldcg(src + c) : z;
    }
    for (int q = 1; q < kc; ++q) {
      const float4* sq = src + q * (plane / 4);
      float4 t[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int c = tid + u * kThreads;
        t[u] = c < nch ? __ldcg(sq + c) : z;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        acc[u].x += t[u].x; acc[u].y += t[u].y; acc[u].z += t[u].z; acc[u].w += t[u].w;
      }
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int c = tid + u * kThreads;
      if (c < nch) reinterpret_cast<float4*>(sbuf)[c] = acc[u];
    }
    __syncthreads();
    for (int rr = warp; rr < nr; rr += kThreads / 32) {
      const float* x = sbuf + (size_t)rr * d;
      float sum = 0.f;
      for (int c = lane; c < d; c += 32) sum += x[c];
      const float mean = warp_sum(sum) / d;
      float sq = 0.f;
      for (int c = lane; c < d; c += 32) sq = fmaf(x[c] - mean, x[c] - mean, sq);
      const float rstd = rsqrtf(warp_sum(sq) / d + 1e-5f);
      float* o = out + (size_t)(rb * R + r0 + rr) * d;
      for (int c = lane; c < d; c += 32) o[c] = (x[c] - mean) * rstd * g[c] + be[c];
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------- attention
constexpr int kAttStages = 4;  // K/V tiles in flight
template <int DH>
struct AttSmem {
  float k[kAttStages][64][DH + 4];
  float v[kAttStages][64][DH + 4];
  float kn2[kAttStages][64];
};

// fp64 correction of the flagged rows, one warp per row (rare: kept out of line).
__device__ __noinline__ void fix_rows(const DagArgs& a, int l, const float* x_in, const int* list,
                                      int n, double* dsm) {
  FixupArgs fa{};
  fa.x = Plane{x_in, nullptr, 0};
  fa.w_qkv = a.layers[l].w_qkv;
  fa.w_kind = 0;
  fa.b_qkv = a.layers[l].b_qkv;
  fa.q = Plane{a.q, nullptr, 0};
  fa.k = Plane{a.k, nullptr, 0};
  fa.v = Plane{a.v, nullptr, 0};
  fa.v_transposed = 0;
  fa.Lp = a.L;
  fa.ctx_hi = a.ctx;
  fa.ctx_kind = 0;
  fa.valid_len = a.vl;
  fa.B = a.B; fa.H = a.H; fa.L = a.L; fa.dh = a.dh; fa.d = a.d;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  double* q64 = dsm + (size_t)warp * (a.dh + a.d);
  for (int e = warp; e < n; e += kThreads / 32) ntie::neartie_fix_entry(fa, list[e], q64, q64 + a.dh, lane);
}

// 32 query rows x one head: 8 threads per row, each taking every 8th key of
// a 64-key tile, online softmax key by key in the log2 domain; the eight
// partial states are merged at the end.  Rows whose two best scores are
// close relative to the fp32 score error are corrected in fp64.
template <int DH>
__device__ void attention_task(const DagArgs& a, int l, int rb, int half, int h, const float* x_in,
                               unsigned char* smem_raw, int* flag_s, int* nflag_s) {
  AttSmem<DH>& sm = *reinterpret_cast<AttSmem<DH>*>(smem_raw);
  const int tid = threadIdx.x, row = tid >> 3, sub = tid & 7;
  const int H = a.H, L = a.L, T = a.T;
  const int r_first = rb * R + half * kAttRows;
  const int rg = r_first + row;
  const bool active = rg < T;
  const int b = active ? rg / L : 0, i = active ? rg % L : 0;
  int vl = a.vl[b];
  if (vl < 1 || vl > L) {
    if (active && l == 0 && h == 0 && i == 0 && sub == 0) set_status(a.status, TL_ERR_BAD_VALID_LEN);
    vl = vl < 1 ? 1 : L;
  }
  const int key_lo = b * L, key_end = active ? b * L + min(i + 1, vl) : 0;  // visible [lo, end)
  const int g_lo = (r_first / L) * L, g_hi = min(r_first + kAttRows, T);  // the task's keys
  const int ntile = (g_hi - g_lo + 63) / 64;

  auto issue = [&](int t) {
    const int st = t % kAttStages;
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
  for (int t = 0; t < kAttStages && t < ntile; ++t) issue(t);

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
    // issued so far: tiles 0 .. min(ntile - 1, t - 1 + stages); tile t must have landed
    cp_wait_n(min(ntile - 1 - t, kAttStages - 1));
    __syncthreads();
    const int st = t % kAttStages;
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
    const int u_lo = max(0, (key_lo - gbase - sub + 7) / 8);
    const int u_hi = min(8, (key_end - gbase - sub + 7) / 8);
#pragma unroll 1
    for (int u = u_lo; u < u_hi; ++u) {
      const int jj = sub + 8 * u;
      float dot = 0.f;
#pragma unroll
      for (int c = 0; c < DH; c += 4) {
        const float4 kv = *reinterpret_cast<const float4*>(&sm.k[st][jj][c]);
        dot = fmaf(q[c], kv.x, dot);
        dot = fmaf(q[c + 1], kv.y, dot);
        dot = fmaf(q[c + 2], kv.z, dot);
        dot = fmaf(q[c + 3], kv.w, dot);
      }
      m2 = fmaxf(m2, fminf(m1, dot));
      m1 = fmaxf(m1, dot);
      kn2max = fmaxf(kn2max, sm.kn2[st][jj]);
      if (dot > m) {  // a new running maximum: rescale (a few times per row)
        const float corr = exp2f(m - dot);  // 0 while m = -inf
        lsum *= corr;
#pragma unroll
        for (int c = 0; c < DH; ++c) o[c] *= corr;
        m = dot;
      }
      const float p = exp2f(dot - m);
      lsum += p;
#pragma unroll
      for (int c = 0; c < DH; c += 4) {
        const float4 vv = *reinterpret_cast<const float4*>(&sm.v[st][jj][c]);
        o[c] = fmaf(p, vv.x, o[c]);
        o[c + 1] = fmaf(p, vv.y, o[c + 1]);
        o[c + 2] = fmaf(p, vv.z, o[c + 2]);
        o[c + 3] = fmaf(p, vv.w, o[c + 3]);
      }
    }
    __syncthreads();
    if (t + kAttStages < ntile) issue(t + kAttStages);
  }
  // merge the eight partial states of the row (adjacent lanes)
#pragma unroll
  for (int off = 1; off <= 4; off <<= 1) {
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
  if (nflag > 0) fix_rows(a, l, x_in, flag_s, nflag, reinterpret_cast<double*>(smem_raw));
}

// ---------------------------------------------------------------- kernel
// One CTA per SM: two co-resident CTAs (head_dim <= 32 at 128 registers)
// measured slower on the batch-1 d_model = 256 workload, each task taking
// longer while sharing the SM and the attention spilling.
template <int DH>
constexpr int dag_ctas_per_sm() { return 1; }

template <int DH>
__global__ void __launch_bounds__(kThreads, dag_ctas_per_sm<DH>()) dag_kernel(const __grid_constant__ DagArgs a) {
  extern __shared__ __align__(16) unsigned char dag_smem[];
  __shared__ int task_s, go_s, last_s, nflag_s;
  __shared__ int flag_s[kAttRows];
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
      __nanosleep(32);
      if (clock64() - t0 > kWait) {
        atomicExch(a.abort, 1);
        set_status(a.status, TL_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
    return true;
  };
  // Release the block's writes through counter c; true in the whole block
  // when this was the completion that reached `target`.
  auto complete = [&](int* c, int target) -> bool {
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const int old = atomicAdd(c, 1);
      if (old == target - 1) __threadfence();  // acquire the other tasks' writes
      last_s = old == target - 1;
    }
    __syncthreads();
    return last_s;
  };
  // The row blocks holding rows of the sequences that meet block rb.
  auto rb_first = [&](int rb) { return ((rb * R) / L) * L / R; };
  auto rb_last = [&](int rb) {
    const int last_row = min(rb * R + R, T) - 1;
    return min(((last_row / L + 1) * L - 1) / R, RB - 1);
  };

  // Every layer's parameters into L2, spread over all threads of the grid.
  for (int l = 0; l < a.n_layers; ++l)
    prefetch_layer_l2(a.layers[l], d, a.dff, 4, blockIdx.x * kThreads + tid, gridDim.x * kThreads);
  int next = 0;
  if (tid == 0) next = atomicAdd(a.head, 1);
  while (true) {
    __syncthreads();
    if (tid == 0) {
      task_s = next;
      next = atomicAdd(a.head, 1);  // consumed on the next iteration
    }
    __syncthreads();
    const int t = task_s;
    if (t >= total) break;
    const int l = t / pl.per_layer;
    int rem = t % pl.per_layer, kind = 0;
    for (int q = 0; q < 5; ++q) {
      kind = queued_kind(q);
      if (rem < pl.n[kind]) break;
      rem -= pl.n[kind];
    }
    const tl_layer_dev& P = a.layers[l];
    const float* x_in = l == 0 ? a.x : ((l & 1) ? a.xs1 : a.xs0);  // this layer's input
    float* x_next = (l & 1) ? a.xs0 : a.xs1;
    // task coordinates
    int rb = 0, nt = 0, kc = 0, h = 0, half = 0;
    switch (kind) {
      case K_QKV: rb = rem / pl.nt3; nt = rem % pl.nt3; break;
      case K_ATT: {
        const int per = pl.target[K_ATT], hh = rem % per;
        rb = RB - 1 - rem / per;
        half = R / kAttRows - 1 - hh / H;
        h = hh % H;
        break;
      }
      case K_OUT: rb = rem / (pl.ntd * pl.kco); nt = (rem / pl.kco) % pl.ntd; kc = rem % pl.kco; break;
      case K_F1: rb = rem / pl.ntf; nt = rem % pl.ntf; break;
      default: rb = rem / (pl.ntd * pl.kcf); nt = (rem / pl.kcf) % pl.ntd; kc = rem % pl.kcf; break;
    }
    // ------------------------------------------------------ dependencies
    if (tid == 0) {
      bool ok = !*(volatile int*)a.abort;
      if (ok && a.inject_stall && t == 0) ok = wait_ge(counter(0, K_LN2, 0), 1 << 30);
      switch (kind) {
        case K_QKV:
          if (l > 0) {
            ok = ok && wait_ge(counter(l - 1, K_LN2, rb), 1);
            for (int r2 = rb; ok && r2 <= rb_last(rb); ++r2)
              ok = wait_ge(counter(l - 1, K_ATT, r2), pl.target[K_ATT]);
          }
          break;
        case K_ATT:
          for (int r2 = rb_first(rb); ok && r2 <= rb; ++r2) ok = wait_ge(counter(l, K_QKV, r2), pl.nt3);
          break;
        case K_OUT: ok = ok && wait_ge(counter(l, K_ATT, rb), pl.target[K_ATT]); break;
        case K_F1: ok = ok && wait_ge(counter(l, K_LN1, rb), 1); break;
        default: ok = ok && wait_ge(counter(l, K_F1, rb), pl.ntf); break;
      }
      if (ok) __threadfence();
      go_s = ok;
    }
    __syncthreads();
    if (!go_s) continue;  // aborted: drain the queue without work
    // --------------------------------------------------------------- work
    if (kind == K_ATT) {
      attention_task<DH>(a, l, rb, half, h, x_in, dag_smem, flag_s, &nflag_s);
      complete(counter(l, K_ATT, rb), pl.target[K_ATT]);
      continue;
    }
    GemmSmem& gs = *reinterpret_cast<GemmSmem*>(dag_smem);
    float acc[4][4];
    const int m0 = rb * R, n0 = nt * 64;
    const int tx = tid % 16, ty = tid / 16;
    if (kind == K_QKV) {
      gemm_tile(x_in, d, (const float*)P.w_qkv, d, T, 3 * d, 0, d, m0, n0, acc, gs);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int mm = m0 + ty + 16 * i;
        if (mm >= T) continue;
        const size_t rowbase = (size_t)(mm / L) * H * L + mm % L;  // ((b H) L + t)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int n = n0 + tx + 16 * j;
          if (n >= 3 * d) continue;
          const int which = n / d, w = n % d, hh = w / DH, c = w % DH;
          float* dst = which == 0 ? a.q : which == 1 ? a.k : a.v;
          dst[(rowbase + (size_t)hh * L) * DH + c] = acc[i][j] + P.b_qkv[n];
        }
      }
      complete(counter(l, K_QKV, rb), pl.nt3);
    } else if (kind == K_F1) {
      gemm_tile(a.y, d, (const float*)P.w_1, d, T, a.dff, 0, d, m0, n0, acc, gs);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int mm = m0 + ty + 16 * i;
        if (mm >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int n = n0 + tx + 16 * j;
          if (n < a.dff) a.hb[(size_t)mm * a.dff + n] = gelu_erf(acc[i][j] + P.b_1[n]);
        }
      }
      complete(counter(l, K_F1, rb), pl.ntf);
    } else {
      // OUT or F2: a K-chunk partial; chunk 0 carries the bias and residual.
      const bool out = kind == K_OUT;
      const int K = out ? d : a.dff;
      gemm_tile(out ? a.ctx : a.hb, K, (const float*)(out ? P.w_o : P.w_2), K, T, d, kc * kDagKChunk,
                min(K, (kc + 1) * kDagKChunk), m0, n0, acc, gs);
      const float* bias = out ? P.b_o : P.b_2;
      const float* res = out ? x_in : a.y;
      float* dst = a.part + kc * plane;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int mm = m0 + ty + 16 * i;
        if (mm >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int n = n0 + tx + 16 * j;
          if (n >= d) continue;
          const size_t at = (size_t)mm * d + n;
          dst[at] = kc == 0 ? acc[i][j] + bias[n] + __ldcg(res + at) : acc[i][j];
        }
      }
      if (complete(counter(l, kind, rb), pl.target[kind])) {
        // the row block's last chunk: LayerNorm its rows now
        if (out) {
          ln_block(a.part, pl.kco, plane, P.ln1_g, P.ln1_b, a.y, rb, T, d, (float*)dag_smem);
          complete(counter(l, K_LN1, rb), 1);
        } else {
          ln_block(a.part, pl.kcf, plane, P.ln2_g, P.ln2_b, l + 1 < a.n_layers ? x_next : a.out, rb,
                   T, d, (float*)dag_smem);
          complete(counter(l, K_LN2, rb), 1);
        }
      }
    }
  }
}

template <int DH>
cudaError_t launch(const DagArgs& a, int total, int num_sms, cudaStream_t s) {
  const int per_sm = dag_ctas_per_sm<DH>();
  const int grid = total < per_sm * num_sms ? total : per_sm * num_sms;  // all resident
  const size_t smem = dag_dyn_smem(a.d, DH);
  auto k = dag_kernel<DH>;
  cudaError_t e = set_max_dyn_smem((const void*)k, smem);
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool dag_supported(int d, int H, int dff, int n_layers, tl_dtype t) {
  if (t != TL_F32 || H < 1 || d % H || n_layers < 1 || n_layers > kDagMaxLayers) return false;
  const int dh = d / H;
  // 16-byte cp.async rows need d and d_ff multiples of 4; a LayerNorm pass
  // parks at least 16 rows of d in 64 KB of shared memory.
  return (dh == 16 || dh == 32 || dh == 64) && d <= 1024 && dff % 4 == 0 && dff >= 4;
}

int dag_counter_ints(int n_layers, int RB) { return n_layers * K_KINDS * RB + 2; }

size_t dag_dyn_smem(int d, int dh) {
  size_t att = dh == 16 ? sizeof(AttSmem<16>) : dh == 32 ? sizeof(AttSmem<32>) : sizeof(AttSmem<64>);
  size_t fix = (size_t)(kThreads / 32) * (dh + d) * sizeof(double);
  size_t ln = (size_t)(R < 16384 / d ? R : 16384 / d) * d * sizeof(float);
  size_t m = sizeof(GemmSmem);
  if (att > m) m = att;
  if (fix > m) m = fix;
  if (ln > m) m = ln;
  return m;
}

cudaError_t dag_forward(const DagArgs& a, int num_sms, cudaStream_t s) {
  const Plan pl = make_plan(a.RB, a.H, a.d, a.dff);
  const int total = a.n_layers * pl.per_layer;
  const int dh = a.d / a.H;
  if (dh == 16) return launch<16>(a, total, num_sms, s);
  if (dh == 32) return launch<32>(a, total, num_sms, s);
  return launch<64>(a, total, num_sms, s);
}

}  // namespace tl
