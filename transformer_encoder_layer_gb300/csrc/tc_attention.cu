// Flash attention on tcgen05 with the causal and key-padding masks applied
// in registers ("KernelForge", section "What we built": both masks inside
// the kernel; section "Challenges": only key tiles that cross a row's limit
// need the per-element predicate).  The L x L scores never leave the chip.
//
// One CTA per SM, persistent over (plane, 128-query tile) work items taken
// heaviest first (the causal triangle makes late query tiles longest).
// Q, K and V arrive as (hi, lo) 16-bit planes; scores and probabilities are
// products of split operands, S = Qh.Kh + Qh.Kl + Ql.Kh (the lo.lo term is
// below fp32 rounding) and O = P.Vh + P.Vl, accumulated in fp32 in TMEM.
// V^T's hi and lo rows sit one after the other in shared memory, so one MMA
// of width 2 x head_dim gives P.Vh and P.Vl side by side in TMEM (the softmax
// adds the two halves): a tcgen05.mma of N <= 128 costs about the same issue
// time whatever its N, and P.V is the larger part of a small head's MMAs.
//
// Warp roles (192 threads):
//   warp 0     TMA: Q (once per work item) and K/V^T tiles of 64 keys into a
//              3-deep ring
//   warp 1     TMEM owner; one thread issues S = Q K^T into one of two TMEM
//              score buffers, then adds P_j V_j to the work item's O
//              accumulator in TMEM once the softmax warps have written P_j
//              (the item's first product overwrites it).  At head_dim
//              16, where the softmax's instruction issue is the bound, each
//              V^T tile carries 16 extra rows after its 2 x head_dim (hi, lo)
//              rows (a row of ones, then zeros, written once at start; TMA
//              never touches them), so the same MMAs also produce the row sum
//              of P_j in output column 2 x head_dim and the softmax adds no
//              probabilities itself; at larger heads the wider MMA costs more
//              than it saves.
//   warps 2-5  softmax: thread = query row.  Reads its 64 scores, masks,
//              updates the running max and writes P_j = 2^(s - mr) (16-bit,
//              hi and, with bf16, lo) into the swizzled shared-memory operand.
//              The reference mr follows the running max lazily: only when the
//              max passes it by more than 2^8 does the thread wait for the
//              last product, scale its row of O (and the row sum) in TMEM by
//              2^(mr_old - mr_new) and move mr.  So no key tile ends with a
//              wait for P.V or a pass over O, the online-softmax correction is
//              applied a few times per row, and the item's O is read once at
//              its end.
//
// Split-K over keys ("KernelForge", section "What's next": partition the key
// range and merge partial softmax states).  When few (plane, query tile)
// items would leave most CTAs idle behind the longest causal rows, the host
// plan cuts every query tile's key range into chunks of kc 64-key tiles and
// makes each chunk its own work item.  A chunk's softmax warps write, per
// row, the unnormalised output, the running max and second-best score (log2
// units), the row sum and |q|^2 to the partial buffer, then count the chunk
// in the tile's arrival counters (one per warp of 32 rows); the warp whose
// chunk arrives last for its rows merges the tile's chunks (out = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c
// with M = max_c m_c) and writes the context.  No CTA ever waits for
// another: the merge is done by whoever finishes last.  A chunk past the
// sequence's valid keys (the plan assumes valid_len = L) loads nothing and
// arrives with an empty state.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>
#include <vector>

#include "common.cuh"
#include "neartie.cuh"
#include "tc_attention.h"
#include "tc_common.cuh"
#include "tc_gemm.h"

namespace tl {
namespace {

using namespace tc;

constexpr int kThreads = 192;
// Query rows and keys per tile; the MMA thread issues P.V of key tile j - 1
// after S of tile j, into two TMEM score buffers (P is written over its
// scores, so a buffer is free again once its P.V is complete).  Running S
// two tiles ahead of P.V, with a third buffer where TMEM has room (head_dim
// up to 32), measured slower on GB300 (85.7 against 81.6 ms per 100k-token
// forward): the MMA thread's issue, not the wait for a free buffer, binds.
constexpr int kBQ = 128, kBKV = 64, kSBufs = 2, kPvLag = kSBufs - 1;

// CTAs per SM: two at every head size (256 TMEM columns each; P lives in
// TMEM, so Q and the K/V ring are all the shared memory a CTA needs), so one
// CTA's softmax overlaps the other's MMAs and loads.
template <int DH>
constexpr int ctas_per_sm() { return 2; }

// max(a, b, c) in one instruction (sm_100 and later).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 16 consecutive TMEM columns of this warp's 32 lanes (no wait).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Store 16 consecutive TMEM columns of this warp's 32 lanes (no wait).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
        "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
        "r"(r[14]), "r"(r[15])
      : "memory");
}

// Multiply the first NCOLS columns of this warp's rows of the O accumulator
// by the lane's factor, in place (warp-collective).
template <int NCOLS>
__device__ __forceinline__ void rescale_o(uint32_t taddr, float corr) {
  static_assert(NCOLS % 16 == 0, "whole 16-column loads");
#pragma unroll
  for (int c0 = 0; c0 < NCOLS; c0 += 16) {
    uint32_t v[16];
    tmem_ld16(taddr + c0, v);
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * corr);
    tmem_st16(taddr + c0, v);
  }
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2^x by the SFU's approximate base-2 exponential with subnormal results
// flushed to zero (a probability below 2^-126 of the row maximum's weight is
// below fp32 resolution of the row sum anyway); 2^-inf = 0.
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory descriptor for a K-major operand whose rows are `row_bytes`
// (32, 64 or 128) long, swizzled at the same width: 8-row atoms of
// 8*row_bytes bytes.
__device__ __forceinline__ uint64_t sdesc_rows(uint32_t saddr, int row_bytes) {
  const uint64_t mode = row_bytes == 128 ? 2 : (row_bytes == 64 ? 4 : 6);
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)((8 * row_bytes) >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= mode << 61;
  return d;
}

// Byte offset of element (r, c) of a K-major tile with `row_bytes`-long
// rows written with the swizzle of the same width: the 16-byte chunk index
// (address bits 4..) is XORed with the 128-byte line index (bits 7..),
// masked to the chunks of one row.
__device__ __forceinline__ int swz_offset(int r, int c_bytes, int row_bytes) {
  const int o = r * row_bytes + c_bytes;
  return o ^ (((o >> 7) & ((row_bytes >> 4) - 1)) << 4);
}

// fp16: the probabilities enter P.V as one 16-bit value (O = Ph.Vh + Ph.Vl,
// no Pl.Vh product, no lo plane of P to compute).  The CPU rounding-emulation
// probe (tests/precision_probe.py) puts the gate's envelope of this plan at
// 0.05-0.13 on the 100k-token workload's layer (0.024 with the lo part) over
// input scales 1e-3 .. 1e3; with bf16 it fails the gate, so bf16 keeps Pl.
template <typename T>
__host__ __device__ constexpr bool p_hi_only() { return std::is_same<T, __half>::value; }

// Row sums of P from the P.V MMAs (a ones row appended to V^T) instead of
// one add per probability: only where the softmax issue rate binds.
template <int DH>
__host__ __device__ constexpr bool row_sum_by_mma() { return DH == 16; }

// How far (log2 units) a row's maximum may pass the reference its
// probabilities are taken against before O and the row sum are rescaled:
// probabilities stay below 2^8, exact in either 16-bit type's range.
constexpr float kLazy = 8.f;

// Split-K partial state per row: output (head_dim), reference, second-best
// score, row sum, |q|^2, best score.
template <int DH>
__host__ __device__ constexpr int kPartCols() { return DH + 5; }

template <typename T, int DH>
struct Layout {
  static constexpr int kQBytes = kBQ * DH * 2;      // one Q plane
  static constexpr int kKBytes = kBKV * DH * 2;     // one K plane tile
  static constexpr int kXRows = row_sum_by_mma<DH>() ? 16 : 0;  // a ones row and 15 zero rows
  static constexpr int kVRows = 2 * DH + kXRows;    // V^T rows: hi, lo, extension
  static constexpr int kVTx = DH * kBKV * 2;        // bytes of one V^T plane tile (TMA)
  static constexpr int kVBytes = kVRows * kBKV * 2; // the V^T block of a stage
  static constexpr int kStageBytes = 2 * kKBytes + kVBytes;
  static constexpr int kStageTx = 2 * kKBytes + 2 * kVTx;  // TMA bytes per stage
  static constexpr int kOUsed = kVRows;              // O columns the MMAs write
  static constexpr int kOCols = (kVRows + 31) / 32 * 32;  // TMEM columns of the O accumulator
  static_assert(kSBufs * kBKV + kOCols <= 256, "two CTAs per SM share the 512 TMEM columns");
  static_assert(kVTx % 1024 == 0 && kStageBytes % 1024 == 0, "128-byte swizzle atoms stay aligned");
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = ((2 * kQBytes + 1023) / 1024) * 1024;
  // K/V ring depth: what the shared memory left per CTA holds, up to 6
  // (the TMA runs further ahead of the MMAs; K/V come from L2).
  static constexpr int kFixedBytes = kKVOff + 256;
  static constexpr int kStages =
      std::min(6, (232448 / ctas_per_sm<DH>() - 1024 - kFixedBytes) / kStageBytes);
  static_assert(kStages >= 2, "K/V ring");
  static constexpr int kBarOff = kKVOff + kStages * kStageBytes;
  static constexpr int kBytes = kBarOff + 256;
  static constexpr int kRowBytes = DH * 2;          // Q/K rows: 32, 64, 128
};

// 64-key tiles query tile qt sees at most (every valid_len = L), and the
// chunks the split plan cuts them into (1 without a split).
__host__ __device__ inline int nkt_bound(int qt, int L) {
  const int kend = qt * kBQ + kBQ < L ? qt * kBQ + kBQ : L;
  return (kend + kBKV - 1) / kBKV;
}
__host__ __device__ inline int chunks_of(int qt, int L, int kc) {
  return kc ? (nkt_bound(qt, L) + kc - 1) / kc : 1;
}

// Work item w -> (plane, query tile, chunk).  Without a split, planes go in
// groups of `group` planes whose K/V fit in L2 together, and within a group
// the items run heaviest query tile first (plane fastest): the CTAs working
// at one time then stream the keys of a few planes, which stay in L2, and the
// causal triangle's long rows still start first.  With a split, order index
// o covers query tile nqt-1-o, whose planes x chunks items are numbered
// chunk-major.  Each role walks its CTA's increasing item indices with its
// own cursor, so the decoding is amortised O(1).
struct ItemCursor {
  int o = 0, base = 0;
  __device__ __forceinline__ void decode(int w, int planes, int nqt, int L, int kc, int group,
                                         int& plane, int& qt, int& c, int& nch) {
    if (kc == 0) {
      const int per_group = group * nqt;
      const int g = w / per_group, i = w - g * per_group;
      const int gp = min(group, planes - g * group);  // planes in this (maybe last) group
      qt = nqt - 1 - i / gp;
      plane = g * group + i % gp;
      c = 0;
      nch = 1;
      return;
    }
    while (true) {
      const int q = nqt - 1 - o;
      const int n = chunks_of(q, L, kc);
      if (w < base + planes * n) {
        const int r = w - base;
        qt = q;
        c = r / planes;
        plane = r % planes;
        nch = n;
        return;
      }
      base += planes * n;
      ++o;
    }
  }
};

template <typename T, int DH>
__global__ void __launch_bounds__(kThreads, ctas_per_sm<DH>())
    tc_attention_kernel(const __grid_constant__ CUtensorMap mqh, const __grid_constant__ CUtensorMap mql,
                        const __grid_constant__ CUtensorMap mkh, const __grid_constant__ CUtensorMap mkl,
                        const __grid_constant__ CUtensorMap mvh, const __grid_constant__ CUtensorMap mvl,
                        const TcAttnArgs a) {
  using Lay = Layout<T, DH>;
  constexpr int kStages = Lay::kStages;
  extern __shared__ __align__(1024) unsigned char dyn_smem[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + Lay::kBarOff);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* kv_full = bars + 2;            // [kStages]
  uint64_t* kv_empty = kv_full + kStages;  // [kStages]
  uint64_t* s_full = kv_empty + kStages;   // [kSBufs]
  uint64_t* p_full = s_full + kSBufs;      // [2]: P written over S
  // [2]: the buffer's P.V complete; the softmax threads wait on it (P_{j+2}
  // may follow, O may be rescaled or read) and so does the MMA thread (the
  // S/P buffer may take S_{j+2}): one commit serves both
  uint64_t* p_empty = p_full + 2;
  static_assert(kSBufs == 2, "S and P buffers pair up one to one");
  uint64_t* o_free = p_empty + 2;          // the item's O has been read
  uint64_t* mma_done = o_free + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int planes = a.B * a.H;
  const int nqt = (a.L + kBQ - 1) / kBQ;
  const int n_items = a.kc ? a.n_items : planes * nqt;
  const int kc = a.kc;
  // S (then P over it): kSBufs x 64 columns, O: kOCols (P.Vh, P.Vl and the row sum)
  constexpr uint32_t kTmemCols = 256;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1 + 128);  // the MMA's last S commit + every softmax thread
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < kSBufs; ++s) mbar_init(&s_full[s], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&p_full[s], 128);
      mbar_init(&p_empty[s], 1);
    }
    mbar_init(o_free, 128);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_holder, kTmemCols);
  // A valid_len outside [1, L] is clamped where it is read (key_tiles); the
  // first CTA records it in the status word, once per offending sequence.
  if (blockIdx.x == 0 && warp >= 2)
    for (int b = threadIdx.x - 64; b < a.B; b += kThreads - 64) load_valid_len(a.valid_len, b, a.L, a.status);
  if (row_sum_by_mma<DH>() && warp >= 2) {
    // The V^T blocks' 16 extra rows, never touched by TMA: the first all
    // ones (its product with P is the row sum), the rest 0.  A row of equal
    // values is the same under the 128-byte swizzle.
    T ones[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) ones[e] = from_f32<T>(1.f);
    const uint4 one4 = *reinterpret_cast<const uint4*>(ones);
    const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
    const int t = threadIdx.x - 64;  // 128 threads, one 16-byte chunk of a 2 KB extension each
    for (int st = 0; st < kStages; ++st) {
      unsigned char* ext = base + Lay::kKVOff + st * Lay::kStageBytes + 2 * Lay::kKBytes + 2 * Lay::kVTx;
      reinterpret_cast<uint4*>(ext)[t] = t < 8 ? one4 : zero4;
    }
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  volatile int* abort = abort_flag;
  const uint32_t tS = tmem, tO = tmem + kSBufs * kBKV;

  auto key_tiles = [&](int plane, int qt, int& vl) {
    vl = a.valid_len[plane / a.H];
    vl = vl < 1 ? 1 : (vl > a.L ? a.L : vl);
    const int kend = min(qt * kBQ + kBQ, vl);  // keys any row of the tile sees
    return (kend + kBKV - 1) / kBKV;
  };
  // Key tiles [j0, j1) of chunk c of a tile with nkt visible key tiles.
  auto key_range = [&](int c, int nkt, int& j0, int& j1) {
    j0 = kc ? c * kc : 0;
    j1 = kc ? min(j0 + kc, nkt) : nkt;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      long long kv_it = 0, n_items_done = 0;  // items with keys (Q loaded)
      bool ok = true;
      ItemCursor cur;
      for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
        int plane, qt, c, nch, vl, j0, j1;
        cur.decode(w, planes, nqt, a.L, kc, a.group, plane, qt, c, nch);
        key_range(c, key_tiles(plane, qt, vl), j0, j1);
        if (j0 >= j1) continue;  // a chunk past the valid keys loads nothing
        if (!mbar_wait(q_empty, (uint32_t)(n_items_done & 1) ^ 1, abort, a.status)) break;
        ++n_items_done;
        mbar_arrive_expect_tx(q_full, 2 * Lay::kQBytes);
        const int qrow = plane * a.L + qt * kBQ;
        tma_load_2d(base + Lay::kQOff, &mqh, q_full, 0, qrow);
        tma_load_2d(base + Lay::kQOff + Lay::kQBytes, &mql, q_full, 0, qrow);
        for (int j = j0; j < j1; ++j, ++kv_it) {
          const int st = (int)(kv_it % kStages);
          const uint32_t ph = (uint32_t)((kv_it / kStages) & 1);
          if (!mbar_wait(&kv_empty[st], ph ^ 1, abort, a.status)) { ok = false; break; }
          unsigned char* sb = base + Lay::kKVOff + st * Lay::kStageBytes;
          mbar_arrive_expect_tx(&kv_full[st], Lay::kStageTx);
          const int krow = plane * a.L + j * kBKV;
          tma_load_2d(sb, &mkh, &kv_full[st], 0, krow);
          tma_load_2d(sb + Lay::kKBytes, &mkl, &kv_full[st], 0, krow);
          tma_load_2d(sb + 2 * Lay::kKBytes, &mvh, &kv_full[st], j * kBKV, plane * DH);
          tma_load_2d(sb + 2 * Lay::kKBytes + Lay::kVTx, &mvl, &kv_full[st], j * kBKV, plane * DH);
        }
      }
      // Drain: wait for the last loads issued into each ring slot and Q.
      for (long long r = 1; r <= kv_it && r <= kStages; ++r) {
        const long long it = kv_it - r;
        mbar_wait_bounded(&kv_full[it % kStages], (uint32_t)((it / kStages) & 1), a.status);
      }
      if (n_items_done > 0) mbar_wait_bounded(q_full, (uint32_t)((n_items_done - 1) & 1), a.status);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    constexpr bool kBf = std::is_same<T, __nv_bfloat16>::value;
    const uint32_t idesc_s = idesc_f16(kBQ, kBKV, kBf);
    const uint32_t idesc_o = idesc_f16(kBQ, Lay::kVRows, kBf);  // P.Vh | P.Vl (| the row sum)
    // bf16's Pl times Vh only, unless the row sum needs the ones row (then
    // Pl.Vl, below fp32 rounding, rides along)
    const uint32_t idesc_ol = idesc_f16(kBQ, row_sum_by_mma<DH>() ? Lay::kVRows : DH, kBf);
    long long kv_it = 0, s_it = 0, o_it = 0, n_done = 0;
    bool ok = true;
    const uint32_t q_addr = smem_u32(base + Lay::kQOff);
    // P_{it_o}.V into the O accumulator; the item's first product overwrites
    // it, once the softmax has read the previous item's O.
    auto issue_pv = [&](long long it_kv, long long it_o, bool first) -> bool {
      const int pb = (int)(it_o & 1);
      if (!mbar_wait(&p_full[pb], (uint32_t)((it_o >> 1) & 1), abort, a.status)) return false;
      if (first && n_done > 1 && !mbar_wait(o_free, (uint32_t)((n_done - 2) & 1), abort, a.status))
        return false;
      tc_fence_after();
      // The whole warp builds the (uniform) descriptors; one elected lane issues.
      const int st = (int)(it_kv % kStages);
      const uint32_t sb = smem_u32(base + Lay::kKVOff + st * Lay::kStageBytes);
      const uint32_t vt = sb + 2 * Lay::kKBytes;  // rows: Vh^T, Vl^T (, extension)
      // P (A operand) in TMEM, over its S buffer: Ph in the first 32
      // columns, Pl (bf16) in the next 32, two 16-bit values per column
      const uint32_t tph = tS + (uint32_t)(pb * kBKV);
      // O += Ph.[Vh | Vl] (+ Pl.Vh with bf16) over 64 keys (4 steps of
      // K = 16, 8 TMEM columns of P each): columns [0, DH) take P.Vh,
      // [DH, 2 DH) P.Vl; with the extension, column 2 DH = the sum of the P
      // values used.  The V descriptor is built once; a k16 step moves its
      // start address field by 32 / 16.
      const uint64_t dvt = sdesc_rows(vt, 128);
#pragma unroll
      for (int k = 0; k < kBKV / 16; ++k)
        mma_f16_ta_elect(tO, tph + 8 * k, dvt + 2 * k, idesc_o, !first || k != 0);
      if constexpr (!p_hi_only<T>()) {
#pragma unroll
        for (int k = 0; k < kBKV / 16; ++k)
          mma_f16_ta_elect(tO, tph + 32 + 8 * k, dvt + 2 * k, idesc_ol, true);
      }
      mma_commit_elect(&p_empty[pb]);
      mma_commit_elect(&kv_empty[st]);
      __syncwarp();
      return true;
    };
    ItemCursor cur;
    for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      int plane, qt, c, nch, vl, j0, j1;
      cur.decode(w, planes, nqt, a.L, kc, a.group, plane, qt, c, nch);
      key_range(c, key_tiles(plane, qt, vl), j0, j1);
      if (j0 >= j1) continue;
      const int nkt = j1 - j0;  // key tiles of this item
      if (!mbar_wait(q_full, (uint32_t)(n_done & 1), abort, a.status)) break;
      ++n_done;
      tc_fence_after();
      for (int j = 0; j < nkt; ++j) {  // j: position within the item's key tiles
        const long long it = kv_it + j;
        const int st = (int)(it % kStages);
        if (!mbar_wait(&kv_full[st], (uint32_t)((it / kStages) & 1), abort, a.status)) { ok = false; break; }
        const int sbuf = (int)(s_it % kSBufs);
        if (!mbar_wait(&p_empty[sbuf], (uint32_t)(((s_it / kSBufs) & 1) ^ 1), abort, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        {
          const uint32_t sb = smem_u32(base + Lay::kKVOff + st * Lay::kStageBytes);
          const uint32_t kh = sb, kl = sb + Lay::kKBytes;
          const uint32_t qh = q_addr, ql = q_addr + Lay::kQBytes;
          const uint32_t d = tS + (uint32_t)(sbuf * kBKV);
          const uint32_t as[3] = {qh, qh, ql};
          const uint32_t bs[3] = {kh, kl, kh};
#pragma unroll
          for (int t = 0; t < 3; ++t) {
            const uint64_t da = sdesc_rows(as[t], Lay::kRowBytes), db = sdesc_rows(bs[t], Lay::kRowBytes);
#pragma unroll
            for (int k = 0; k < DH / 16; ++k)
              mma_f16_elect(d, da + 2 * k, db + 2 * k, idesc_s, (t | k) != 0);
          }
          mma_commit_elect(&s_full[sbuf]);
          if (j == nkt - 1) mma_commit_elect(q_empty);  // Q no longer read
        }
        __syncwarp();
        ++s_it;
        if (j >= kPvLag) {
          if (!issue_pv(kv_it + j - kPvLag, o_it, j == kPvLag)) { ok = false; break; }
          ++o_it;
        }
      }
      if (!ok) break;
      for (int j = nkt >= kPvLag ? nkt - kPvLag : 0; j < nkt && ok; ++j) {
        if (!issue_pv(kv_it + j, o_it, j == 0)) { ok = false; break; }
        ++o_it;
      }
      if (!ok) break;
      kv_it += nkt;
    }
    mma_commit_elect(mma_done);
    __syncwarp();
    mbar_wait_bounded(mma_done, 0, a.status);
  } else {
    // ------------------------------------------------------------ softmax
    const int qd = warp & 3;
    const int r = qd * 32 + lane;  // row of the query tile == TMEM lane
    const uint32_t lane_addr = (uint32_t)(qd * 32) << 16;
    const uint32_t to = tO + lane_addr;  // this warp's rows of the O accumulator
    T* const ctx_hi = reinterpret_cast<T*>(a.ctx_hi);
    T* const ctx_lo = reinterpret_cast<T*>(a.ctx_lo);
    const float scale_log2 = rsqrtf((float)DH) * 1.4426950408889634f;
    long long s_it = 0, n_done = 0;
    bool ok = true;
    ItemCursor cur;
    for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      int plane, qt, cidx, nch, vl, j0, j1;
      cur.decode(w, planes, nqt, a.L, kc, a.group, plane, qt, cidx, nch);
      key_range(cidx, key_tiles(plane, qt, vl), j0, j1);
      const bool has_keys = j0 < j1;
      const int i = qt * kBQ + r;                    // query position in the sequence
      const int limit = min(i + 1, vl);              // keys [0, limit) visible
      const int full_keys = min(qt * kBQ + 1, vl);   // keys every row of the tile sees
      // m, m2: the row's best and second-best score so far (log2 units);
      // mr: the reference the probabilities are taken against.  mr follows
      // m lazily, only when m passes it by more than kLazy, so O (in TMEM)
      // and the row sum are rescaled a few times per row instead of after
      // every key tile; probabilities stay below 2^kLazy.
      float m = -INFINITY, m2 = -INFINITY, mr = -INFINITY, l = 0.f;
      // |q_i| for the near-tie test, from the (hi, lo) Q tile in shared memory.
      float qn2 = 0.f;
      if (!has_keys) {
        // nothing loaded for this chunk: only its (empty) partial state is due
      } else if (mbar_wait(q_full, (uint32_t)(n_done & 1), abort, a.status)) {
        ++n_done;
        const unsigned char* qh = base + Lay::kQOff;
#pragma unroll
        for (int c = 0; c < DH; ++c) {
          const int off = swz_offset(r, c * 2, Lay::kRowBytes);
          float qv = to_f32<T>(*reinterpret_cast<const T*>(qh + off)) +
                     to_f32<T>(*reinterpret_cast<const T*>(qh + Lay::kQBytes + off));
          qn2 = fmaf(qv, qv, qn2);
        }
        mbar_arrive(q_empty);  // this thread no longer reads Q
      } else {
        ok = false;
        break;
      }
      // The second-best score matters only where fp32 scores can be off.
      const float kmax_plane = __int_as_float(a.kmax[plane]);
      bool track = neartie_err(sqrtf(qn2), kmax_plane, DH) > kTieErrMin;
      for (int j = j0; j < j1 && ok; ++j) {
        const long long it = s_it++;  // this CTA's key tile count
        const int sbuf = (int)(it % kSBufs);
        if (!mbar_wait(&s_full[sbuf], (uint32_t)((it / kSBufs) & 1), abort, a.status)) { ok = false; break; }
        tc_fence_after();
        float s[kBKV];
        tmem_ld32(tS + lane_addr + (uint32_t)(sbuf * kBKV), *reinterpret_cast<float(*)[32]>(&s[0]));
        tmem_ld32(tS + lane_addr + (uint32_t)(sbuf * kBKV + 32), *reinterpret_cast<float(*)[32]>(&s[32]));
        const int k0 = j * kBKV;
        const bool needs_mask = k0 + kBKV > full_keys;
        // s stays unscaled (masked keys -inf); the running max m, the
        // second best m2 and the references are in scaled (log2) units.
        // Scaling by a positive constant commutes with the max, rounding
        // included, so the tile max is scaled once.
        float tmax;
        if (track) {
          tmax = -INFINITY;
#pragma unroll
          for (int c = 0; c < kBKV; ++c) {
            float v = s[c];
            if (needs_mask && k0 + c >= limit) v = -INFINITY;
            s[c] = v;
            const float vs = v * scale_log2;
            m2 = fmaxf(m2, fminf(fmaxf(m, tmax), vs));
            tmax = fmaxf(tmax, vs);
          }
        } else {
          // no near tie possible for this row: the second-best score is not
          // needed, and the tile max takes one three-input max per two scores
          if (needs_mask) {
#pragma unroll
            for (int c = 0; c < kBKV; ++c)
              if (k0 + c >= limit) s[c] = -INFINITY;
          }
          float traw = -INFINITY;
#pragma unroll
          for (int c = 0; c < kBKV; c += 2) traw = max3f(traw, s[c], s[c + 1]);
          tmax = traw * scale_log2;
        }
        m = fmaxf(m, tmax);
        // A row with no visible key so far keeps mr = -inf; its
        // probabilities are exactly 0 below.
        float corr = 1.f;
        bool resc = false;
        if (m > mr + kLazy) {
          if (mr != -INFINITY) {
            corr = exp2f(mr - m);
            resc = true;
          }
          mr = m;
        }
        if (__any_sync(0xffffffffu, resc)) {
          // O holds the products up to key tile it-1 against the old
          // references: wait for the last of them, then scale this warp's
          // rows in place (corr = 1 for rows that keep their reference).
          if (!mbar_wait(&p_empty[(it - 1) & 1], (uint32_t)(((it - 1) >> 1) & 1), abort, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          rescale_o<Lay::kOUsed>(to, corr);
          if constexpr (!row_sum_by_mma<DH>()) l *= corr;
        }
        const float mref = mr == -INFINITY ? 0.f : mr;
        const uint64_t sc2 = splat2(scale_log2), nm2 = splat2(-mref);
        // P_it over its own scores in TMEM (this thread's row).  P.V_{it-2},
        // which read the buffer last, is complete (S_it was computed after
        // it); the wait keeps this barrier's phases in step with the rescale
        // and end-of-item waits on it.
        const int pb = (int)(it & 1);
        if (!mbar_wait(&p_empty[pb], (uint32_t)(((it >> 1) & 1) ^ 1), abort, a.status)) { ok = false; break; }
        uint32_t pwh[32];
        uint32_t pwl[p_hi_only<T>() ? 1 : 32];
#pragma unroll
        for (int c8 = 0; c8 < kBKV / 8; ++c8) {
          float p8[8];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {  // 2^(s scale - mref), flushed below 2^-126
            float a0, a1;  // the exponents, two at a time (paired fp32 fma)
            upk2(fma2(pk2(s[c8 * 8 + e], s[c8 * 8 + e + 1]), sc2, nm2), a0, a1);
            p8[e] = ex2_ftz(a0);
            p8[e + 1] = ex2_ftz(a1);
          }
          if constexpr (!row_sum_by_mma<DH>()) {
#pragma unroll
            for (int e = 0; e < 8; ++e) l += p8[e];
          }
          if constexpr (p_hi_only<T>()) {
            *reinterpret_cast<uint4*>(&pwh[4 * c8]) = pack8_hi(p8, T());
          } else {
            split8(p8, *reinterpret_cast<uint4*>(&pwh[4 * c8]), *reinterpret_cast<uint4*>(&pwl[4 * c8]), T());
          }
        }
        const uint32_t tp = tS + lane_addr + (uint32_t)(sbuf * kBKV);
        tmem_st32(tp, pwh);
        if constexpr (!p_hi_only<T>()) tmem_st32(tp + 32, *reinterpret_cast<uint32_t(*)[32]>(pwl));
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();  // orders P's (and a rescale's) TMEM stores before P.V_it
        mbar_arrive(&p_full[pb]);
      }
      if (!ok) break;
      // The item's output (unnormalised, against mr) and row sum, once its
      // last product is complete; then O is free for the next item.
      float acc[DH];
#pragma unroll
      for (int c = 0; c < DH; ++c) acc[c] = 0.f;
      if (has_keys) {
        const long long last = s_it - 1;
        if (!mbar_wait(&p_empty[last & 1], (uint32_t)((last >> 1) & 1), abort, a.status)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < DH; c0 += 16) {
          uint32_t rh[16], rl[16];
          tmem_ld16(to + c0, rh);
          tmem_ld16(to + DH + c0, rl);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int c = 0; c < 16; ++c) acc[c0 + c] = __uint_as_float(rh[c]) + __uint_as_float(rl[c]);
        }
        if constexpr (row_sum_by_mma<DH>()) {  // the row sum, column 2 DH
          uint32_t rs;
          asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(rs) : "r"(to + 2 * DH));
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
          l = __uint_as_float(rs);
        }
        tc_fence_before();
        mbar_arrive(o_free);
      }
      if (nch > 1) {
        // ---- split-K: publish this chunk's partial state, count the chunk
        // in, and merge the tile if it is the last to arrive.
        const int cols = kPartCols<DH>();
        float* mine = a.part + (size_t)w * kBQ * cols + r;  // column-major: [col][row]
#pragma unroll
        for (int e = 0; e < DH; ++e) mine[(size_t)e * kBQ] = acc[e];
        mine[(size_t)DH * kBQ] = mr;  // the reference acc and l are taken against
        mine[(size_t)(DH + 1) * kBQ] = m2;
        mine[(size_t)(DH + 2) * kBQ] = l;
        mine[(size_t)(DH + 3) * kBQ] = has_keys ? qn2 : -1.f;
        mine[(size_t)(DH + 4) * kBQ] = m;
        // Each warp counts its own 32 rows in (no barrier across warps, so
        // no wait that could outlive a failed peer): the last warp of the
        // tile's chunks to arrive for these rows merges them.
        __threadfence();
        __syncwarp();
        int before = 0;
        if (lane == 0) before = atomicAdd(&a.cnt[(plane * nqt + qt) * 4 + qd], 1);
        before = __shfl_sync(0xffffffffu, before, 0);
        if (before != nch - 1) continue;
        __threadfence();
        // The tile's items are numbered first_w + c * planes (chunk-major).
        const int first_w = w - cidx * planes;
        float mmax = mr, top1 = m, top2 = m2;
        for (int c2 = 0; c2 < nch; ++c2) {
          if (c2 == cidx) continue;
          const float* o = a.part + (size_t)(first_w + c2 * planes) * kBQ * cols + r;
          const float mc = __ldcg(o + (size_t)(DH + 4) * kBQ), m2c = __ldcg(o + (size_t)(DH + 1) * kBQ);
          const float qc = __ldcg(o + (size_t)(DH + 3) * kBQ);
          mmax = fmaxf(mmax, __ldcg(o + (size_t)DH * kBQ));
          if (qc >= 0.f) qn2 = qc;  // |q|^2 from any chunk that loaded Q
          // top two of the union of the chunks' (best, second best)
          if (mc > top1) { top2 = fmaxf(top1, m2c); top1 = mc; }
          else top2 = fmaxf(top2, mc);
        }
        // Every row sees key 0, which lies in chunk 0, so mmax (the largest
        // reference) is finite.
        // The chunks are summed in chunk order whichever warp merges, so
        // the result does not depend on which chunk finished last.
        float own[DH];
#pragma unroll
        for (int e = 0; e < DH; ++e) {
          own[e] = acc[e];
          acc[e] = 0.f;
        }
        float lsum = 0.f;
        for (int c2 = 0; c2 < nch; ++c2) {
          if (c2 == cidx) {
            const float wc = exp2f(mr - mmax);
            lsum = fmaf(wc, l, lsum);
#pragma unroll
            for (int e = 0; e < DH; ++e) acc[e] = fmaf(wc, own[e], acc[e]);
            continue;
          }
          const float* o = a.part + (size_t)(first_w + c2 * planes) * kBQ * cols + r;
          const float wc = exp2f(__ldcg(o + (size_t)DH * kBQ) - mmax);
          lsum = fmaf(wc, __ldcg(o + (size_t)(DH + 2) * kBQ), lsum);
#pragma unroll
          for (int e = 0; e < DH; ++e) acc[e] = fmaf(wc, __ldcg(o + (size_t)e * kBQ), acc[e]);
        }
        l = lsum;
        m = top1;
        m2 = top2;
        track = neartie_err(sqrtf(qn2), kmax_plane, DH) > kTieErrMin;
      }
      if (i < a.L) {
        const float inv = 1.f / l;
        const size_t at = ((size_t)(plane / a.H) * a.L + i) * a.d + (size_t)(plane % a.H) * DH;
#pragma unroll
        for (int c8 = 0; c8 < DH / 8; ++c8) {
          uint4 hv, lv;
          T* hp = reinterpret_cast<T*>(&hv);
          T* lp = reinterpret_cast<T*>(&lv);
#pragma unroll
          for (int e = 0; e < 8; ++e) Split<T>::go(acc[c8 * 8 + e] * inv, hp[e], lp[e]);
          *reinterpret_cast<uint4*>(ctx_hi + at + c8 * 8) = hv;
          *reinterpret_cast<uint4*>(ctx_lo + at + c8 * 8) = lv;
        }
        if (track && neartie_flag((m - m2) * 0.69314718055994531f, sqrtf(qn2), kmax_plane, DH))
          neartie_push(a.ties, plane * a.L + i);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename T, int DH>
cudaError_t launch_dh(const TcAttnArgs& a, const CUtensorMap* maps, int grid, cudaStream_t s) {
  using Lay = Layout<T, DH>;
  auto k = tc_attention_kernel<T, DH>;
  const size_t smem = Lay::kBytes + 1024;
  cudaError_t e = set_max_dyn_smem((const void*)k, smem);
  if (e != cudaSuccess) return e;
  static_assert(ctas_per_sm<DH>() * (Lay::kBytes + 1024) <= 232448, "shared memory per SM");
  k<<<grid * ctas_per_sm<DH>(), kThreads, smem, s>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], a);
  return cudaGetLastError();
}

}  // namespace

bool tc_attention_supported(int dh) { return dh == 16 || dh == 32 || dh == 64; }

TcAttnSplit tc_attention_split_plan(int B, int H, int L, int dh, int num_sms, int force_kc) {
  TcAttnSplit p;
  if (!tc_attention_supported(dh) || B < 1 || H < 1 || L < 1 || force_kc == 0) return p;
  const long long planes = (long long)B * H;
  const int nqt = (L + kBQ - 1) / kBQ;
  const long long items0 = planes * nqt;
  const int slots = num_sms * ctas_per_sm<16>();  // every head size runs two CTAs per SM
  // The item index is an int and the decoding walks the query tiles; keep
  // the split to shapes whose (plane, query tile) count is modest.
  if (nqt > 4096 || items0 * ((nkt_bound(nqt - 1, L) + 1) / 2) > (1LL << 28)) return p;
  auto items_of = [&](int kc) {
    long long n = 0;
    for (int qt = 0; qt < nqt; ++qt) n += planes * chunks_of(qt, L, kc);
    return n;
  };
  int kc = 0;
  if (force_kc > 0) {
    kc = force_kc;
  } else {
    if (items0 >= 2LL * slots) return p;  // enough items to keep every CTA busy
    // Model of the persistent grid: CTA g takes items g, g + slots, ... in
    // the kernel's order.  An item costs its 64-key tiles plus about 4 tiles
    // of fixed cost (Q load, pipeline fill and drain); a chunk also pays for
    // its partial state and its share of the merge, about half a tile per
    // chunk of its query tile.  Both constants are fitted to GB300 timings
    // of chunk sizes 4..32 at head_dim 16 and 64 (batch 1 and 2, 2k-32k
    // tokens), which the model then ranks as measured; with two or more
    // items per CTA the unsplit grid was already the fastest.
    auto makespan = [&](int kcc) {
      std::vector<double> load(slots, 0.0);
      long long w = 0;
      for (int o = 0; o < nqt; ++o) {
        const int qt = nqt - 1 - o, nkt = nkt_bound(qt, L), nch = chunks_of(qt, L, kcc);
        for (int c = 0; c < nch; ++c) {
          const int t = kcc ? std::min(kcc, nkt - c * kcc) : nkt;
          const double cost = t + 4.0 + (nch > 1 ? 0.5 * nch : 0.0);
          for (long long pl = 0; pl < planes; ++pl, ++w) load[w % slots] += cost;
        }
      }
      return *std::max_element(load.begin(), load.end());
    };
    double best = makespan(0);
    const double base = best;
    for (int cand : {64, 32, 16, 8}) {
      const double m = makespan(cand);
      if (m < best) { best = m; kc = cand; }
    }
    if (kc && best > 0.9 * base) kc = 0;  // not worth the partial states
  }
  if (!kc) return p;
  const long long n = items_of(kc);
  if (n > (1LL << 30)) return TcAttnSplit{};
  p.kc = kc;
  p.n_items = (int)n;
  p.part_bytes = (size_t)n * kBQ * (dh + 5) * sizeof(float);
  p.cnt_bytes = (size_t)planes * nqt * 4 * sizeof(int);
  return p;
}

cudaError_t tc_attention(const TcAttnArgs& a_in, bool bf16, int num_sms, int force_kc, void* ws_part,
                         void* ws_cnt, cudaStream_t s) {
  TcAttnArgs a = a_in;
  const int dh = a.dh;
  if (!tc_attention_supported(dh) || a.L < 1 || a.Lp % 8 || a.Lp < a.L) return cudaErrorInvalidValue;
  const TcAttnSplit plan = tc_attention_split_plan(a.B, a.H, a.L, dh, num_sms, force_kc);
  a.kc = plan.kc;
  a.n_items = plan.n_items;
  // Planes whose K and V (hi, lo) fit together in half the L2 (64 MB).
  const size_t kv_plane = (size_t)a.L * dh * 2 * 2 * 2;
  const size_t g = ((size_t)64 << 20) / (kv_plane ? kv_plane : 1);
  const int planes = a.B * a.H;
  a.group = (int)std::max<size_t>(1, std::min<size_t>(g, (size_t)planes));
  a.part = (float*)ws_part;
  a.cnt = (int*)ws_cnt;
  if (plan.kc) {
    if (!ws_part || !ws_cnt) return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(ws_cnt, 0, plan.cnt_bytes, s);
    if (e != cudaSuccess) return e;
  }
  const uint64_t rows = (uint64_t)a.B * a.H * a.L;
  CUtensorMap maps[6];
  bool ok = make_tmap_2d(&maps[0], a.q_hi, bf16, rows, dh, dh, dh, kBQ, dh * 2) &&
            make_tmap_2d(&maps[1], a.q_lo, bf16, rows, dh, dh, dh, kBQ, dh * 2) &&
            make_tmap_2d(&maps[2], a.k_hi, bf16, rows, dh, dh, dh, kBKV, dh * 2) &&
            make_tmap_2d(&maps[3], a.k_lo, bf16, rows, dh, dh, dh, kBKV, dh * 2) &&
            make_tmap_2d(&maps[4], a.vt_hi, bf16, (uint64_t)a.B * a.H * dh, a.Lp, a.Lp, kBKV, dh, 128) &&
            make_tmap_2d(&maps[5], a.vt_lo, bf16, (uint64_t)a.B * a.H * dh, a.Lp, a.Lp, kBKV, dh, 128);
  if (!ok) return cudaErrorInvalidValue;
  const long long items = plan.kc ? plan.n_items : (long long)a.B * a.H * ((a.L + kBQ - 1) / kBQ);
  const int grid = items < num_sms ? (int)items : num_sms;  // per resident CTA slot (launch_dh scales)
  if (bf16) {
    if (dh == 16) return launch_dh<__nv_bfloat16, 16>(a, maps, grid, s);
    if (dh == 32) return launch_dh<__nv_bfloat16, 32>(a, maps, grid, s);
    return launch_dh<__nv_bfloat16, 64>(a, maps, grid, s);
  }
  if (dh == 16) return launch_dh<__half, 16>(a, maps, grid, s);
  if (dh == 32) return launch_dh<__half, 32>(a, maps, grid, s);
  return launch_dh<__half, 64>(a, maps, grid, s);
}

}  // namespace tl
