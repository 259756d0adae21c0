// tcgen05 GEMM with fused epilogues: C[M, N] = A[M, K] . W[N, K]^T.
//
// A is an activation carried as one or two 16-bit planes (hi, lo: the value
// is hi + lo, about fp32 accuracy); W is a weight in the same 16-bit type,
// exact.  Both are K-major.  Per 128 x BN output tile the MMA issues, per
// 64-wide K block, 4 x n_parts tcgen05.mma (K = 16 each) into an fp32 TMEM
// accumulator; the product hi.W + lo.W is accumulated in the same TMEM
// columns.
//
// Warp roles (192 threads, one CTA per SM, persistent over tiles):
//   warp 0     TMA producer: A planes and the W tile of each K block into a
//              `stages`-deep shared-memory ring (128-byte swizzle)
//   warp 1     TMEM allocation; one elected thread issues the MMAs
//   warps 2-5  epilogue: thread = output row (TMEM lane), 32 columns at a
//              time with tcgen05.ld; two TMEM accumulators let the epilogue
//              of one tile overlap the main loop of the next
//
// CTA-pair variant (PAIR, launched as clusters of two): the pair owns a
// 256-row block.  Each CTA loads its own 128 rows of A and its half (BN/2
// rows) of the W tile -- every byte is loaded once, by one CTA -- with both CTAs' loads
// completing on the leader's (rank 0) ring barrier; the leader alone issues
// tcgen05.mma.cta_group::2 with M = 256, which reads A and B from both
// CTAs' shared memory and writes each CTA's rows into its own tensor memory,
// and commits both CTAs' ring and accumulator barriers.  One MMA instruction
// thus covers 256 rows: half the instructions per row of the single-CTA
// kernel, and half the W bytes staged per CTA.  The epilogue is unchanged;
// the peer's epilogue warps release the accumulator on the leader's barrier.
// Both CTAs hand each other a bounded "done" signal before freeing tensor
// memory and exiting, so neither leaves while the other may still signal it.
// Epilogues (the pages' fused steps: "KernelForge", section "What we
// built" -- fused QKV projection, fused add + LayerNorm; the megakernel
// page, section "Hybrid" -- QKV GEMM with the head-major transpose fused):
//   QKV   + bias, scattered head-major: Q and K as [B, H, L, dh] and V as
//         V^T [B, H, dh, Lp], each as (hi, lo) planes
//   GELU  + bias, exact-erf GELU, (hi, lo) planes [M, N]
//   LN    + bias + residual, LayerNorm over the full row (per-32-column
//         (mean, M2) merged with Chan's formula), written as fp32 and/or
//         (hi, lo) planes, or as the final output in the I/O dtype.  When a
//         row fits one N tile the CTA normalises it from TMEM.  A row wider
//         than one N tile goes to a scratch row, each tile with the (mean,
//         M2) of its columns (each tile a work unit of its own), and
//         ln_apply.cu merges the statistics and normalises those rows in a
//         streaming pass while this kernel's tensor cores are free for the
//         next launch.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_gemm.h"

namespace tl {
namespace {

using namespace tc;

// Threads per CTA: a TMA warp, an MMA warp and the epilogue warps, four per
// half of a tile's columns (one per TMEM lane quarter).  Two halves: with
// one, a tile's epilogue (about 21K cycles for 128 x 256 QKV or GELU outputs
// on GB300, 33K with LayerNorm statistics) outlasted its MMAs (about 19K at
// K = 1024).  The CTA-pair LayerNorm GEMM (the FFN2 over a long K, whose
// MMAs outlast its epilogue) keeps one: the second half's warps slowed the
// MMA warp they share a sub-partition with (0.599 -> 0.633 ms per d1024
// forward).  A LayerNorm epilogue that normalises whole rows itself runs on
// the first half (its statistics run along the row); with per-tile
// statistics each half writes its own.
template <int EPI, bool PAIR>
constexpr int epi_halves() { return EPI == TC_EPI_LN && PAIR ? 1 : 2; }
template <int EPI, bool PAIR>
constexpr int gemm_threads() { return 64 + 128 * epi_halves<EPI, PAIR>(); }
constexpr int kBM = 128, kBK = 64;
constexpr int kATileBytes = kBM * kBK * 2;  // 16 KB

struct Smem {
  // carved from dynamic shared memory: [stages x stage bytes] then barriers
  uint64_t* full;
  uint64_t* empty;
  uint64_t* acc_full;   // [2]
  uint64_t* acc_empty;  // [2]
  uint64_t* mma_done;   // [1]
  uint64_t* done;       // [1] pair: the peer has finished signalling this CTA
  uint32_t* tmem_base;
  int* abort;
};

template <typename T>
__device__ __forceinline__ void store_pair(T* hi, T* lo, size_t i, float v) {
  T h, l;
  Split<T>::go(v, h, l);
  hi[i] = h;
  lo[i] = l;
}

// 32 consecutive values of one row as (hi, lo) 16-bit planes, 16-byte stores.
template <typename T>
__device__ __forceinline__ void store_row32_pair(T* hi, T* lo, size_t at, const float (&v)[32]) {
  uint4 hv[4], lv[4];
  T* hp = reinterpret_cast<T*>(hv);
  T* lp = reinterpret_cast<T*>(lv);
#pragma unroll
  for (int j = 0; j < 32; ++j) Split<T>::go(v[j], hp[j], lp[j]);
  uint4* hd = reinterpret_cast<uint4*>(hi + at);
  uint4* ld = reinterpret_cast<uint4*>(lo + at);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    hd[j] = hv[j];
    ld[j] = lv[j];
  }
}

template <typename T>
__device__ __forceinline__ void store_row32(T* dst, size_t at, const float (&v)[32]) {
  uint4 hv[4];
  T* hp = reinterpret_cast<T*>(hv);
#pragma unroll
  for (int j = 0; j < 32; ++j) hp[j] = from_f32<T>(v[j]);
  uint4* hd = reinterpret_cast<uint4*>(dst + at);
#pragma unroll
  for (int j = 0; j < 4; ++j) hd[j] = hv[j];
}

// W consecutive values of one row as (hi, lo) 16-bit planes, 16-byte stores
// (W a multiple of 8, `at` a multiple of 8 elements).
template <typename T, int W>
__device__ __forceinline__ void store_row_pair(T* hi, T* lo, size_t at, const float* v) {
#pragma unroll
  for (int q = 0; q < W / 8; ++q) {
    uint4 hv, lv;
    T* hp = reinterpret_cast<T*>(&hv);
    T* lp = reinterpret_cast<T*>(&lv);
#pragma unroll
    for (int j = 0; j < 8; ++j) Split<T>::go(v[8 * q + j], hp[j], lp[j]);
    reinterpret_cast<uint4*>(hi + at)[q] = hv;
    reinterpret_cast<uint4*>(lo + at)[q] = lv;
  }
}

// QKV epilogue for one row's 32-column chunk starting at column n0 of
// [q | k | v]: head pieces of W = min(dh, 32) columns (dh divides 32 or is a
// multiple of it).  Q and K go to
// [B, H, L, dh] planes, V to the transposed [B, H, dh, Lp] planes (a lane
// per row, so each V^T store covers consecutive positions).  kn2 carries
// |k|^2 of the head being written across chunks (dh > 32); the head's |k|
// goes to the plane maximum used by the near-tie test.
template <typename T, int W>
__device__ __forceinline__ void qkv_scatter(const float (&v)[32], const TcGemmArgs& a, int row, int n0,
                                            float& kn2) {
  const int d = a.H * a.dh;
  const int b = row / a.L, i = row % a.L;
#pragma unroll
  for (int j0 = 0; j0 < 32; j0 += W) {
    const int n = n0 + j0;
    const int which = n / d, h = (n % d) / a.dh, c0 = n % a.dh;
    const size_t bh = (size_t)b * a.H + h;
    if (which < 2) {
      T* hi = reinterpret_cast<T*>(which == 0 ? a.q_hi : a.k_hi);
      T* lo = reinterpret_cast<T*>(which == 0 ? a.q_lo : a.k_lo);
      const size_t at = (bh * a.L + i) * a.dh + c0;
      if constexpr (W % 8 == 0) {
        store_row_pair<T, W>(hi, lo, at, v + j0);
      } else {
#pragma unroll
        for (int j = 0; j < W; ++j) store_pair(hi, lo, at + j, v[j0 + j]);
      }
      if (which == 1 && a.kmax) {
#pragma unroll
        for (int j = 0; j < W; ++j) kn2 = fmaf(v[j0 + j], v[j0 + j], kn2);
        if (c0 + W == a.dh) {
          // one atomic per (sequence, head) present in the warp: the lanes
          // sharing a plane reduce first (non-negative floats order like
          // their bit patterns)
          const unsigned lane = threadIdx.x & 31u;
          const unsigned mask = __activemask();
          const unsigned grp = __match_any_sync(mask, (unsigned long long)bh);
          const unsigned mx = __reduce_max_sync(grp, (unsigned)__float_as_int(sqrtf(kn2)));
          if ((grp & ((1u << lane) - 1u)) == 0u) atomicMax(a.kmax + bh, (int)mx);
          kn2 = 0.f;
        }
      }
    } else {
      T* vt_hi = reinterpret_cast<T*>(a.vt_hi);
      T* vt_lo = reinterpret_cast<T*>(a.vt_lo);
#pragma unroll
      for (int j = 0; j < W; ++j) {
        const size_t vr = (bh * a.dh + c0 + j) * a.Lp;
        store_pair(vt_hi, vt_lo, vr + i, v[j0 + j]);
        if (i == a.L - 1)  // zero the pitch padding: keys beyond L read as 0
          for (int z = a.L; z < a.Lp; ++z) store_pair(vt_hi, vt_lo, vr + z, 0.f);
      }
    }
  }
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
      "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
      "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]),
      "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]),
      "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

template <typename T, int EPI, bool PAIR>
__global__ void __launch_bounds__(gemm_threads<EPI, PAIR>(), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a0, const __grid_constant__ CUtensorMap map_a1,
                   const __grid_constant__ CUtensorMap map_w, const TcGemmArgs args) {
  extern __shared__ __align__(1024) unsigned char dyn_smem[];
  const TcGemmArgs& a = args;
  // 1024-byte align the operand ring (the 128-byte swizzle atom).
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  const int BN = a.BN;
  const int w_rows = PAIR ? BN / 2 : BN;  // rows of the W tile this CTA stages
  const int stage_bytes = a.n_parts * kATileBytes + w_rows * kBK * 2;
  unsigned char* bar_base = base + (size_t)a.stages * stage_bytes;
  Smem sm;
  sm.full = reinterpret_cast<uint64_t*>(bar_base);
  sm.empty = sm.full + a.stages;
  sm.acc_full = sm.empty + a.stages;
  sm.acc_empty = sm.acc_full + 2;
  sm.mma_done = sm.acc_empty + 2;
  sm.done = sm.mma_done + 1;
  sm.tmem_base = reinterpret_cast<uint32_t*>(sm.done + 1);
  sm.abort = reinterpret_cast<int*>(sm.tmem_base + 1);
  // Pair: rank 0 leads (issues the MMAs); the peer is the other CTA.
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  const bool leader = rank == 0;
  const int rows_per_unit = PAIR ? 2 * kBM : kBM;
  // First unit and stride of this CTA (a pair shares one unit sequence),
  // read from the special registers at each use and kept unsigned: the same
  // values held in int variables across the kernel made the compiler give
  // the one-CTA QKV epilogue 30 more registers, and it ran 40% slower.
#define TL_UNIT0 (PAIR ? (blockIdx.x >> 1) : blockIdx.x)
#define TL_USTEP (PAIR ? (gridDim.x >> 1) : gridDim.x)

  T* const q_hi = reinterpret_cast<T*>(a.q_hi);
  T* const q_lo = reinterpret_cast<T*>(a.q_lo);
  T* const k_hi = reinterpret_cast<T*>(a.k_hi);
  T* const k_lo = reinterpret_cast<T*>(a.k_lo);
  T* const vt_hi = reinterpret_cast<T*>(a.vt_hi);
  T* const vt_lo = reinterpret_cast<T*>(a.vt_lo);
  T* const o_hi = reinterpret_cast<T*>(a.o_hi);
  T* const o_lo = reinterpret_cast<T*>(a.o_lo);
  T* const o_final = reinterpret_cast<T*>(a.o_final);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Work units: an LN GEMM that normalises its rows itself -> one row block
  // (128 rows, or 256 for a pair) with all its N tiles; else one tile (an LN
  // GEMM whose rows span several tiles hands per-tile statistics to the
  // apply pass, so its row blocks' tiles spread over the SMs: 4 x the units,
  // fewer idle SMs in the last wave).  a.m_blocks counts row blocks.
  const bool split_stats = EPI == TC_EPI_LN && a.n_tiles > 1 && a.row_stats;
  const bool ln_rows = EPI == TC_EPI_LN && !split_stats;
  const int n_units = ln_rows ? a.m_blocks : a.m_blocks * a.n_tiles;
  const int tiles_per_unit = ln_rows ? a.n_tiles : 1;
  const int k_blocks = (a.K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.acc_full[s], 1);
      // pair leader: its own 128 epilogue threads plus one arrival per peer
      // epilogue warp
      // every epilogue thread, plus (pair) one remote arrival per peer epilogue warp
      constexpr int kEpiWarps = gemm_threads<EPI, PAIR>() / 32 - 2;
      mbar_init(&sm.acc_empty[s], kEpiWarps * 32 + (PAIR ? kEpiWarps : 0));
    }
    mbar_init(sm.mma_done, 1);
    mbar_init(sm.done, 1);
    *sm.abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_a0);
    if (a.n_parts > 1) tma_prefetch_desc(&map_a1);
    tma_prefetch_desc(&map_w);
  }
  if (warp == 1) {
    if constexpr (PAIR) tmem_alloc_pair(sm.tmem_base, a.tmem_cols);
    else tmem_alloc(sm.tmem_base, a.tmem_cols);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();  // the peer's barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_base;
  volatile int* abort = sm.abort;

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      // a pair's loads of both CTAs complete on the leader's barrier
      const uint32_t tx = (uint32_t)stage_bytes * (PAIR ? 2u : 1u);
      bool ok = true;
      for (int u = TL_UNIT0; u < n_units && ok; u += TL_USTEP) {
        for (int t = 0; t < tiles_per_unit && ok; ++t) {
          const int m_blk = ln_rows ? u : u / a.n_tiles;
          const int n_tile = ln_rows ? t : u % a.n_tiles;
          const int arow = m_blk * rows_per_unit + (int)rank * kBM;
          const int wrow = n_tile * BN + (int)rank * w_rows;
          for (int kb = 0; kb < k_blocks; ++kb) {
            if (!mbar_wait(&sm.empty[stage], phase ^ 1, abort, a.status)) { ok = false; break; }
            unsigned char* st = base + (size_t)stage * stage_bytes;
            if constexpr (PAIR) {
              const uint32_t fb = map_to_rank(smem_u32(&sm.full[stage]), 0);
              if (leader) mbar_arrive_expect_tx(&sm.full[stage], tx);
              tma_load_2d_pair(st, &map_a0, fb, kb * kBK, arow);
              if (a.n_parts > 1) tma_load_2d_pair(st + kATileBytes, &map_a1, fb, kb * kBK, arow);
              tma_load_2d_pair(st + a.n_parts * kATileBytes, &map_w, fb, kb * kBK, wrow);
            } else {
              mbar_arrive_expect_tx(&sm.full[stage], tx);
              tma_load_2d(st, &map_a0, &sm.full[stage], kb * kBK, arow);
              if (a.n_parts > 1) tma_load_2d(st + kATileBytes, &map_a1, &sm.full[stage], kb * kBK, arow);
              tma_load_2d(st + a.n_parts * kATileBytes, &map_w, &sm.full[stage], kb * kBK, wrow);
            }
            ++issued;
            if (++stage == a.stages) { stage = 0; phase ^= 1; }
          }
        }
      }
      // Every load issued must have landed before the CTA exits: wait (with
      // a bound, ignoring the abort flag) on the last `stages` full phases.
      // A pair's peer cannot see its loads' barrier; the leader's MMAs read
      // them before the end-of-kernel handshake, which covers the peer.
      if (!PAIR || leader)
        for (long long r = 1; r <= issued && r <= a.stages; ++r) {
          const long long idx = issued - r;
          mbar_wait_bounded(&sm.full[idx % a.stages], (uint32_t)((idx / a.stages) & 1), a.status);
        }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issue
    if (!PAIR || leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      // commit to this CTA's barrier and, for a pair, to the peer's copy
      // (the whole warp takes part; one elected lane issues, as for the MMAs)
      auto commit_both = [&](uint64_t* bar) {
        if constexpr (PAIR) {
          mma_commit_pair_elect(smem_u32(bar));
          mma_commit_pair_elect(map_to_rank(smem_u32(bar), 1));
        } else {
          mma_commit_elect(bar);
        }
      };
      for (int u = TL_UNIT0; u < n_units && ok; u += TL_USTEP) {
        for (int t = 0; t < tiles_per_unit && ok; ++t) {
          if (!mbar_wait(&sm.acc_empty[acc], acc_phase ^ 1, abort, a.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
          for (int kb = 0; kb < k_blocks; ++kb) {
            if (!mbar_wait(&sm.full[stage], phase, abort, a.status)) { ok = false; break; }
            tc_fence_after();
            {
              // warp-uniform descriptors; one elected lane issues
              unsigned char* st = base + (size_t)stage * stage_bytes;
              // a k16 step moves the descriptors' start address field by 32 / 16
              const uint64_t dw = sdesc_sw128(smem_u32(st + a.n_parts * kATileBytes));
              for (int p = 0; p < a.n_parts; ++p) {
                const uint64_t da = sdesc_sw128(smem_u32(st + p * kATileBytes));
#pragma unroll
                for (int k16 = 0; k16 < kBK / 16; ++k16) {
                  if constexpr (PAIR)
                    mma_f16_pair_elect(d_tmem, da + 2 * k16, dw + 2 * k16, a.idesc, (kb | p | k16) != 0);
                  else
                    mma_f16_elect(d_tmem, da + 2 * k16, dw + 2 * k16, a.idesc, (kb | p | k16) != 0);
                }
              }
              commit_both(&sm.empty[stage]);
            }
            __syncwarp();
            if (++stage == a.stages) { stage = 0; phase ^= 1; }
          }
          commit_both(&sm.acc_full[acc]);
          __syncwarp();
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        }
      }
      // All issued MMAs complete before TMEM is released.
      if constexpr (PAIR) mma_commit_pair_elect(smem_u32(sm.mma_done));
      else mma_commit_elect(sm.mma_done);
      __syncwarp();
      mbar_wait_bounded(sm.mma_done, 0, a.status);
    }
  } else {
    // ----------------------------------------------------------- epilogue
    const int qd = warp & 3;
    const int row_in_tile = qd * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(qd * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    const int n_chunks = BN / 32;
    // This warp's 32-column chunks of a tile: all of them with four epilogue
    // warps; with eight, one half, split between whole heads (QKV with
    // head_dim above 32 carries a head's |k|^2 across its chunks).
    const int half = (warp - 2) / 4;
    const int halves = ln_rows ? 1 : epi_halves<EPI, PAIR>();  // whole LN rows: the first half
    const int grp = (EPI == TC_EPI_QKV && a.dh > 32) ? a.dh / 32 : 1;
    const int n_grp = n_chunks / grp;
    const int c_lo = half < halves ? half * n_grp / halves * grp : 0;
    const int c_hi = half < halves ? (half + 1) * n_grp / halves * grp : 0;
    bool ok = true;
    for (int u = TL_UNIT0; u < n_units && ok; u += TL_USTEP) {
      const int m_blk = ln_rows ? u : u / a.n_tiles;
      const int row = m_blk * rows_per_unit + (int)rank * kBM + row_in_tile;
      const bool row_ok = row < a.M;
      // LayerNorm running statistics over the row (Chan's parallel merge).
      float ln_n = 0.f, ln_mean = 0.f, ln_m2 = 0.f;
      for (int t = 0; t < tiles_per_unit; ++t) {
        const int n_tile = ln_rows ? t : u % a.n_tiles;
        if (!mbar_wait(&sm.acc_full[acc], acc_phase, abort, a.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tbase = tmem + lane_addr + (uint32_t)(acc * BN);
        float kn2 = 0.f;  // running |k|^2 of the head being written (QKV)
        for (int c = c_lo; c < c_hi; ++c) {
          float v[32];
          tmem_ld32(tbase + c * 32, v);
          const int n0 = n_tile * BN + c * 32;
          {  // + bias: eight 16-byte loads (the same addresses in every lane)
            const float4* b4 = reinterpret_cast<const float4*>(a.bias + n0);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 bb = __ldg(b4 + j);
              v[4 * j] += bb.x; v[4 * j + 1] += bb.y; v[4 * j + 2] += bb.z; v[4 * j + 3] += bb.w;
            }
          }
          if (EPI == TC_EPI_QKV) {
            if (row_ok) {
              // a 32-column chunk covers part of one head (dh >= 32) or 32/dh
              // whole heads; the head width is a template constant so the
              // chunk stays in registers
              if (a.dh >= 32) qkv_scatter<T, 32>(v, a, row, n0, kn2);
              else if (a.dh == 16) qkv_scatter<T, 16>(v, a, row, n0, kn2);
              else if (a.dh == 8) qkv_scatter<T, 8>(v, a, row, n0, kn2);
              else if (a.dh == 4) qkv_scatter<T, 4>(v, a, row, n0, kn2);
              else if (a.dh == 2) qkv_scatter<T, 2>(v, a, row, n0, kn2);
              else qkv_scatter<T, 1>(v, a, row, n0, kn2);
            }
          } else if (EPI == TC_EPI_GELU) {
            if (row_ok) {
#pragma unroll
              for (int j = 0; j < 32; j += 2) gelu_as7128_x2(v[j], v[j + 1]);
              store_row32_pair(o_hi, o_lo, (size_t)row * a.N + n0, v);
            }
          } else {  // LN pass 1: r = acc + bias + residual, chunk stats
            if (row_ok) {
              const size_t at = (size_t)row * a.N + n0;
              if (a.resid_kind == 0) {
                const float4* r4 = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.resid) + at);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  float4 r = r4[j];
                  v[4 * j] += r.x; v[4 * j + 1] += r.y; v[4 * j + 2] += r.z; v[4 * j + 3] += r.w;
                }
              } else if (a.resid_kind == 1) {
                const uint4* r4 = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.resid) + at);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  uint4 r = r4[j];
                  const T* rt = reinterpret_cast<const T*>(&r);
#pragma unroll
                  for (int e = 0; e < 8; ++e) v[8 * j + e] += to_f32<T>(rt[e]);
                }
              } else {  // (hi, lo) pair: the residual is hi + lo
                const uint4* h4 = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.resid) + at);
                const uint4* l4 = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.resid_lo) + at);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  uint4 rh = h4[j], rl = l4[j];
                  const T* ht = reinterpret_cast<const T*>(&rh);
                  const T* lt = reinterpret_cast<const T*>(&rl);
#pragma unroll
                  for (int e = 0; e < 8; ++e) v[8 * j + e] += to_f32<T>(ht[e]) + to_f32<T>(lt[e]);
                }
              }
            }
            float cm = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) cm += v[j];
            cm *= (1.f / 32.f);
            float c2 = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) c2 = fmaf(v[j] - cm, v[j] - cm, c2);
            const float nn = ln_n + 32.f, delta = cm - ln_mean;
            ln_mean += delta * (32.f / nn);
            ln_m2 += c2 + delta * delta * (ln_n * 32.f / nn);
            ln_n = nn;
            if (a.n_tiles == 1) {
              tmem_st32(tbase + c * 32, v);  // keep r on chip
            } else if (row_ok) {
              float4* dst = reinterpret_cast<float4*>(a.rscratch + (size_t)row * a.N + n0);
#pragma unroll
              for (int j = 0; j < 8; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            }
          }
        }
        if (EPI == TC_EPI_LN && t == tiles_per_unit - 1 && half < halves) {
          // LN pass 2: normalise and write (or hand the row statistics to
          // the streaming apply pass when the rows went to scratch).
          const float mean = ln_mean;
          const float rstd = rsqrtf(ln_m2 / ln_n + 1e-5f);
          if (split_stats) {
            // (mean, M2) of this warp's half of the tile, for the apply pass
            if (row_ok)
              a.row_stats[((size_t)row * a.n_tiles + n_tile) * halves + half] = make_float2(ln_mean, ln_m2);
          } else for (int tt = 0; tt < a.n_tiles; ++tt) {
            for (int c = 0; c < n_chunks; ++c) {
              float v[32];
              const int n0 = tt * BN + c * 32;
              if (a.n_tiles == 1) {
                tmem_ld32(tbase + c * 32, v);
              } else if (row_ok) {
                const float4* src = reinterpret_cast<const float4*>(a.rscratch + (size_t)row * a.N + n0);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  float4 r = src[j];
                  v[4 * j] = r.x; v[4 * j + 1] = r.y; v[4 * j + 2] = r.z; v[4 * j + 3] = r.w;
                }
              }
              if (!row_ok) continue;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                v[j] = (v[j] - mean) * rstd * __ldg(a.gamma + n0 + j) + __ldg(a.beta + n0 + j);
              const size_t at = (size_t)row * a.N + n0;
              if (a.o32) {
                float4* dst = reinterpret_cast<float4*>(a.o32 + at);
#pragma unroll
                for (int j = 0; j < 8; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
              }
              if (o_hi) store_row32_pair(o_hi, o_lo, at, v);
              if (o_final) store_row32(o_final, at, v);
            }
          }
        }
        tc_fence_before();
        if (PAIR && !leader) {
          // the leader reuses the accumulator: one arrival per warp on its barrier
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(map_to_rank(smem_u32(&sm.acc_empty[acc]), 0));
        } else {
          mbar_arrive(&sm.acc_empty[acc]);
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) {
    // Each CTA has finished every signal it sends the other (the leader's
    // MMA commits completed before its mma_done wait; the peer's releases
    // happened in its epilogue).  Tell the peer, and wait (bounded) for the
    // peer to say the same before freeing the pair's tensor memory.
    if (threadIdx.x == 0) {
      mbar_arrive_cluster(map_to_rank(smem_u32(sm.done), rank ^ 1u));
      mbar_wait_bounded(sm.done, 0, a.status);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, a.tmem_cols);
    else tmem_dealloc(tmem, a.tmem_cols);
  }
#undef TL_UNIT0
#undef TL_USTEP
}

template <typename T, int EPI, bool PAIR>
cudaError_t launch(const CUtensorMap& m0, const CUtensorMap& m1, const CUtensorMap& mw,
                   const TcGemmArgs& a, int grid, size_t smem, cudaStream_t s) {
  auto k = tc_gemm_kernel<T, EPI, PAIR>;
  cudaError_t e = set_max_dyn_smem((const void*)k, smem);
  if (e != cudaSuccess) return e;
  if constexpr (PAIR) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(gemm_threads<EPI, PAIR>());
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, m0, m1, mw, a);
  } else {
    k<<<grid, gemm_threads<EPI, PAIR>(), smem, s>>>(m0, m1, mw, a);
    return cudaGetLastError();
  }
}

}  // namespace

int tc_gemm_stages(int BN, int n_parts, bool pair) {
  const int stage = n_parts * kATileBytes + (pair ? BN / 2 : BN) * kBK * 2;
  int st = (kTcGemmSmemBudget - 2048) / stage;
  return st > 6 ? 6 : st;
}

size_t tc_gemm_smem_bytes(int BN, int n_parts, int stages, bool pair) {
  const int stage = n_parts * kATileBytes + (pair ? BN / 2 : BN) * kBK * 2;
  // pair: slack of one more half W tile after the ring, so that no operand
  // read of the last stage can reach past the allocation
  return 1024 + (size_t)stages * stage + 256 + (pair ? (size_t)(BN / 2) * kBK * 2 : 0);
}

bool tc_gemm_pair_ok(int M, int BN) { return M > kBM && BN >= 64 && BN <= 256 && BN % 32 == 0; }

int tc_gemm_ln_parts(int N, int BN, bool pair) {
  return BN > 0 && N > BN ? (N / BN) * (pair ? epi_halves<TC_EPI_LN, true>() : epi_halves<TC_EPI_LN, false>()) : 1;
}

cudaError_t tc_gemm(const CUtensorMap& map_a0, const CUtensorMap& map_a1, const CUtensorMap& map_w,
                    TcGemmArgs a, bool bf16, int epi, int num_sms, cudaStream_t s) {
  // Reject shapes this kernel does not handle (a host-side check, so a bad
  // call never reaches the GPU).
  if (a.BN % 32 || a.BN < 32 || a.BN > 256 || a.N % a.BN || a.K < 16 || a.K % 8 ||
      a.n_parts < 1 || a.n_parts > 2 || a.M < 1)
    return cudaErrorInvalidValue;
  if (a.pair && !tc_gemm_pair_ok(a.M, a.BN)) return cudaErrorInvalidValue;
  const bool pair = a.pair != 0;
  const int rows = pair ? 2 * kBM : kBM;
  a.n_tiles = a.N / a.BN;
  a.m_blocks = (a.M + rows - 1) / rows;
  a.stages = tc_gemm_stages(a.BN, a.n_parts, pair);
  int cols = 32;
  while (cols < 2 * a.BN) cols <<= 1;
  a.tmem_cols = cols;
  a.idesc = idesc_f16(rows, a.BN, bf16);
  // work units as the kernel counts them (see split_stats there)
  const bool whole_rows = epi == TC_EPI_LN && !(a.n_tiles > 1 && a.row_stats);
  const int units = whole_rows ? a.m_blocks : a.m_blocks * a.n_tiles;
  const int slots = pair ? num_sms / 2 : num_sms;  // CTAs (pairs) resident at once
  const int grid = (units < slots ? units : slots) * (pair ? 2 : 1);
  const size_t smem = tc_gemm_smem_bytes(a.BN, a.n_parts, a.stages, pair);
#define TL_GEMM_LAUNCH(T_, E_)                                                      \
  return pair ? launch<T_, E_, true>(map_a0, map_a1, map_w, a, grid, smem, s)       \
              : launch<T_, E_, false>(map_a0, map_a1, map_w, a, grid, smem, s)
  if (bf16) {
    switch (epi) {
      case TC_EPI_QKV: TL_GEMM_LAUNCH(__nv_bfloat16, TC_EPI_QKV);
      case TC_EPI_GELU: TL_GEMM_LAUNCH(__nv_bfloat16, TC_EPI_GELU);
      default: TL_GEMM_LAUNCH(__nv_bfloat16, TC_EPI_LN);
    }
  }
  switch (epi) {
    case TC_EPI_QKV: TL_GEMM_LAUNCH(__half, TC_EPI_QKV);
    case TC_EPI_GELU: TL_GEMM_LAUNCH(__half, TC_EPI_GELU);
    default: TL_GEMM_LAUNCH(__half, TC_EPI_LN);
  }
#undef TL_GEMM_LAUNCH
}

}  // namespace tl

// ------------------------------------------------------------ tensor maps
namespace tl {

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}
}  // namespace

bool make_tmap_2d(CUtensorMap* map, const void* ptr, bool bf16, uint64_t rows, uint64_t cols,
                  uint64_t pitch_elems, uint32_t box_cols, uint32_t box_rows, int swizzle_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_elems * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUtensorMapSwizzle sw = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                          : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                          : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                  const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace tl
