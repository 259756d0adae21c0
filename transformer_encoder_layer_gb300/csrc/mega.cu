// Sequence-resident megakernel: every layer of the stack for a 128-row tile
// of whole sequences in one CTA, activations kept on chip from the input
// load to the output store ("Hyper-optimized megakernel-hybrid transformer
// inference", section "Problem decomposition": short sequences fit in
// shared memory, one CTA owns them across all layers).
//
// Shape: d_model = 128, head_dim = 32 (4 heads), d_ff a multiple of 128 up
// to 512, sequence length L in {32, 64}: a tile holds 128 / L sequences,
// which are rows [128 t, 128 t + 128) of the [B*L, d] input.  16-bit I/O
// (fp16 or bf16); activations are carried as (hi, lo) 16-bit pairs wherever
// they feed a tensor-core product.
//
// One CTA per SM, persistent over tiles.  640 threads in five warpgroups:
//   control  warp 0  TMA: the input tile (once per tile) and weight boxes
//                    from L2 into a 2-deep ring, in the order the MMAs use them
//            warp 1  TMEM (all 512 columns); one thread issues every MMA
//            warps 2, 3 idle (they lend their registers: setmaxnreg, in the
//                    assisted kernel)
//   compute  16 warps in four column groups g = 0..3 of four warps; the four
//            warps of a group cover the 128 rows (TMEM lane quarters), and
//            group g takes columns [32g, 32g + 32) of a 128-wide row, head
//            g for the context, 32 of a 128-wide FFN chunk, and a share of
//            each row's 8-key chunks of the attention scores.  Four warps
//            per SM sub-partition hide the latency of the CUDA-core phases.
//
// Per layer (TMEM columns in brackets):
//   QKV   acc[0, 384) = X . W_qkv^T      X = (hi, lo) of the layer input
//   per head h: Q_h, K_h, V_h -> shared memory as (hi, lo);
//         S = Q_h K_h^T [384, 512); softmax with the causal + key-padding +
//         own-sequence mask -> P; O_h = P V_h into [96h, 96h + 64) (row r's
//         result in [96h + 32 s, +32) for its sequence s).
//         Head h+1's Q, K, V are written as soon as S_h has been read, so
//         S_{h+1} runs during the softmax of head h (P V issued after it).
//         Plain kernel: groups 0, 1 run the softmax (every 2nd 8-key chunk)
//         while groups 2, 3 convert head h+1; assisted kernel: all four
//         groups do both in turn (every 4th chunk).  The row maximum (and
//         the second best score) is merged across the softmax groups
//         through shared memory.
//   ctx = O / l as (hi, lo): plain kernel, TMEM words over each head's O
//         columns (written by the conversion warps as soon as that head's
//         P V is done); assisted kernel, shared memory
//   out   acc[384, 512) (assisted: [128, 256)) = ctx . W_o^T;
//         y = LN1(acc + b_o + x) -> TMEM [128, 256) as (hi, lo) 16-bit
//         pairs, the A operand of FFN1 read straight from tensor memory
//   FFN   per 128-wide chunk c of d_ff: acc1[256 + 128 (c % 2), +128) =
//         y . W_1c^T; h_c = gelu(acc1 + b_1c) replaces acc1 in the same TMEM
//         columns as (hi, lo) words; acc2[0, 128) += h_c . W_2c^T (A from
//         tensor memory again).  GELU of chunk c overlaps the products of
//         chunks c - 1 and c + 1.  Only the weights come from shared memory.
//   x' = LN2(acc2 + b_2 + y) -> X buffer, or the output rows on the last layer
//         (y read back from tensor memory); x' also goes to TMEM [384, 512)
//         as (hi, lo) pairs, the next layer's QKV A operand
// The LayerNorm statistics of a row merge the four groups' (mean, M2) with
// Chan's pairwise formula in a fixed order.
//
// Precision plan.  Every activation operand is a (hi, lo) pair except, with
// fp16 I/O, the probabilities P (O_h = Ph.Vh + Ph.Vl, no Pl.Vh product) and
// the FFN hidden h (FFN2 reads h_hi alone): the CPU rounding-emulation probe
// of this plan (tests/precision_probe.py) puts the gate's envelope on the
// d128 workload at about 0.15 for P alone and 0.65 for both, against 0.024
// with every lo part kept, at every input scale from 1e-3 to 1e3; with bf16
// (8 significant bits) either removal fails the gate, so bf16 keeps them.
// That is 48 of the 264 MMAs of a layer and tile.
//
// Assisted mode (small batches; "Hyper-optimized megakernel-hybrid
// transformer inference", section "Problem decomposition": extra CTAs take
// part of the resident CTAs' work when the tiles alone leave SMs idle).
// Launched as clusters of two CTAs per tile: the resident CTA R (rank 0)
// and its helper H (rank 1) split each layer --
//   QKV      R the weight boxes of heads 0, 1; H those of heads 2, 3
//   heads    R heads 0, 1; H heads 2, 3, whose context H writes into R's
//            ctx buffer (distributed shared memory) once R's own P and V
//            buffers there are free
//   out-proj R alone (all of ctx), LayerNorm 1 -> y, which R also writes
//            into H's X buffer once H's attention no longer reads it
//   FFN      R the first half of the d_ff chunks, H the second half; H's
//            FFN2 partial sum goes (fp32) into R's P/ctx area
//   LN 2     R adds H's partial, normalises, and writes the next layer's
//            input to its own X buffer and tensor memory and into H's X
//            buffer (once H's FFN1 no longer reads y there)
// Each data hand-over is staged in the sender's own shared memory and moved
// by one bulk copy (cp.async.bulk shared::cta -> shared::cluster) that
// completes on the receiver's mbarrier, whose expected bytes the receiver
// registers; "buffer free" signals are single remote arrives (release,
// cluster scope); every wait is a bounded cluster-scope acquire.
//
// Near ties (see neartie.cuh) are corrected in place: a flagged (row, head)
// has its probabilities recomputed in fp64 from the layer input and the
// weights, by the group-0 warp that owns the row, before the P . V product.
#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "common.cuh"
#include "mega.h"
#include "neartie.cuh"
#include "tc_common.cuh"
#include "tc_gemm.h"

namespace tl {
namespace {

using namespace tc;

constexpr int kCtrlWarps = 4;  // one warpgroup: TMA, MMA, two idle warps
constexpr int kCompute = 512;
constexpr int kThreads = kCtrlWarps * 32 + kCompute;
constexpr int kD = 128, kDH = 32, kH = 4;
constexpr int kTY = 128;   // TMEM columns of y (hi [128, 192), lo [192, 256))
constexpr int kTF = 256;   // TMEM FFN buffers b = 0, 1 at 256 + 128 b: FFN1 accumulator, then h (hi, lo)
constexpr int kTX = 384;   // TMEM columns of the next layer's input (hi [384, 448), lo [448, 512))
// plain kernel: the context of head h as (hi, lo) words in TMEM over its O
// columns: dims [16j, 16j + 16) have their hi words at 96h + 16j + [0, 8)
// and their lo words at 96h + 16j + [8, 16); the out-projection reads A
// there and accumulates into [384, 512) (the score columns, free by then)
constexpr int kTOut = 384;
constexpr int kNW = 2;     // regular weight ring slots
constexpr int kNSlot = 5;  // during the FFN: three more, borrowed from the Q/K/V buffers

// Shared memory map (offsets from a 1024-byte aligned base).
constexpr int kTile16 = 128 * 64 * 2;                 // 16 KB: 128 rows x 64 16-bit
constexpr int kXA = 0;                                // [part][khalf] x 16 KB = 64 KB
constexpr int kPB = kXA + 4 * kTile16;                // attention: P [part] 128 x 64 (own keys), then
                                                      // V [buffer][part] 64 x 64; afterwards ctx [part][khalf]
                                                      // (assisted) or the LayerNorm vectors (plain)
constexpr int kPV = kPB + 2 * kTile16;                // the two V buffers, 16 KB each (hi, lo 8 KB)
constexpr int kQB = kPB + 4 * kTile16;                // [part] 128 x 32, 8 KB each
constexpr int kKB = kQB + 2 * 8192;                   // [part] 128 x 32
constexpr int kVB = kKB + 2 * 8192;                   // spare during attention; a weight slot in the FFN
constexpr int kWR = kVB + 4 * 4096;                   // [kNW] x 16 KB
constexpr int kMisc = kWR + kNW * kTile16;
// misc (floats unless noted)
constexpr int kQn2 = kMisc;                           // [2 head parity][2 group][128] partial |q_r|^2
constexpr int kEx = kQn2 + 2 * 2 * 128 * 4;           // [2][4 group][128] exchange: (m1, m2) or (mean, M2)
constexpr int kLs = kEx + 2 * 4 * 128 * 4;            // [4 head][4 group][128] partial softmax sums;
                                                      // assisted kernel, from the out-projection on: b_o,
                                                      // ln1 g, b, b_2, ln2 g, b (plain kernel: in the P area)
constexpr int kKmax = kLs + 4 * 4 * 128 * 4;          // [4 head][2] int: max partial |k|^2 (float bits)
constexpr int kMaxDff = 512;
constexpr int kVec = kKmax + 64;                      // the layer's b_qkv [384] then b_1 [d_ff]
constexpr int kBars = kVec + (384 + kMaxDff) * 4;
constexpr int kNumBars = 42;
constexpr int kSmemBytes = kBars + kNumBars * 8 + 16;

// mbarrier indices
enum {
  B_X_FULL = 0, B_W_FULL, B_W_EMPTY = B_W_FULL + kNSlot, B_A_READY = B_W_EMPTY + kNSlot,
  B_QKV_DONE, B_QKV_DONE2, B_QKVH_READY, B_VH_READY, B_VH_READY1,
  B_S_DONE, B_S_FREE, B_P_READY, B_P_READY1, B_O_DONE, B_O_DONE1, B_CTX_READY, B_OUT_DONE, B_Y_READY, B_F1_DONE,
  B_F1_DONE1, B_H_READY, B_H_FREE, B_H_FREE1, B_F2_DONE, B_XA_FREE,
  B_MMA_DONE, B_SYNC, B_SYNC_SM,
  // assisted mode (a resident CTA R and a helper CTA H per tile, one cluster);
  // data hand-overs are bulk copies completing on the receiver's barrier
  B_PEER_CTX,     // R: H's context of heads 2, 3 has landed in R's ctx buffer
  B_PEER_XFREE,   // R: H no longer reads its X buffer (twice a layer)
  B_PEER_PART,    // R: H's FFN2 partial has landed in R's P/ctx area
  B_PEER_PBFREE,  // H: R is done with its P/V area (H may send the context)
  B_PEER_Y,       // H: y has landed in H's X buffer
  B_PEER_X,       // H: the next layer's input has landed in H's X buffer
  B_COUNT
};
static_assert(B_COUNT <= kNumBars, "barrier slots");
static_assert(kSmemBytes + 1024 <= 232448, "shared memory budget");

// Weight slot st: the two regular ring slots, then (FFN boxes only) the
// Q/K/V buffers, which are free from the end of the layer's out-projection
// until its next QKV product.  FFN boxes of a layer take slots 0, 1, 2, 3,
// 4, 0, ... in turn from slot 0; the other boxes alternate between 0 and 1.
__device__ __forceinline__ int wslot_off(int st) { return st < kNW ? kWR + st * kTile16 : kQB + (st - kNW) * kTile16; }

__device__ __forceinline__ int sw128(int r, int c8) { return r * 128 + ((c8 ^ (r & 7)) << 4); }
__device__ __forceinline__ int sw64(int r, int c_bytes) {
  const int o = r * 64 + c_bytes;
  return o ^ (((o >> 7) & 3) << 4);
}
__device__ __forceinline__ uint64_t desc_sw64(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(512 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)4 << 61;
  return d;
}

// Matrix descriptor of an MN-major operand in the 128-byte swizzle: each
// 128-byte row holds 64 16-bit elements along MN (one swizzle atom wide) for
// one K index, and 8-row K groups are 1024 bytes apart (stride byte offset).
// The leading byte offset (between atoms along MN) is never used by an
// operand 64 elements wide; it is set to the same 1024.
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)(1024 >> 4) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// 32 / 16 columns without waiting; call tmem_wait_ld() before using them.
__device__ __forceinline__ void tmem_ld32_nw(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16_nw(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld8_nw(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 16 32-bit columns of this thread's TMEM lane; call tmem_wait_st()
// before signalling that they are written.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* w) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16};" ::"r"(taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
      "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 2^x by the SFU's approximate base-2 exponential, subnormal results flushed
// to zero (a probability below 2^-126 of the row maximum's weight is below
// the fp32 resolution of the row sum anyway).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max of three (one instruction on sm_100 and later)
__device__ __forceinline__ float max3_f32(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

// Eight 16-bit (hi, lo) values into one 16-byte chunk of each plane.
template <typename T>
__device__ __forceinline__ void put8(unsigned char* hi, unsigned char* lo, int off, const float* v) {
  uint4 hv, lv;
  split8(v, hv, lv, T());
  *reinterpret_cast<uint4*>(hi + off) = hv;
  *reinterpret_cast<uint4*>(lo + off) = lv;
}
// c + a for a 16-bit value a: one mixed-precision add (sm_100 and later),
// a widened exactly, one rounding -- no separate conversion instruction.
template <typename T> __device__ __forceinline__ float addw(float c, unsigned short a);
template <> __device__ __forceinline__ float addw<__half>(float c, unsigned short a) {
  float d;
  asm("add.rn.f32.f16 %0, %1, %2;" : "=f"(d) : "h"(a), "f"(c));
  return d;
}
template <> __device__ __forceinline__ float addw<__nv_bfloat16>(float c, unsigned short a) {
  float d;
  asm("add.rn.f32.bf16 %0, %1, %2;" : "=f"(d) : "h"(a), "f"(c));
  return d;
}
// v[0..8) += the eight 16-bit values of a 16-byte chunk (element 2e in the
// low half of word e); with the lo plane added after the hi plane, a (hi, lo)
// residual costs two adds per element.
template <typename T>
__device__ __forceinline__ void add8w(float* v, uint4 c) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[2 * e] = addw<T>(v[2 * e], (unsigned short)(w[e] & 0xFFFFu));
    v[2 * e + 1] = addw<T>(v[2 * e + 1], (unsigned short)(w[e] >> 16));
  }
}
// v[0..N) += vec[0..N), N a multiple of 4, vec 16-byte aligned (shared or
// global memory).
template <int N>
__device__ __forceinline__ void add_vec(float* v, const float* vec) {
  const float4* b4 = reinterpret_cast<const float4*>(vec);
#pragma unroll
  for (int c = 0; c < N / 4; ++c) {
    const float4 b = b4[c];  // paired adds, rounded as the scalar ones
    upk2(add2(pk2(v[4 * c], v[4 * c + 1]), pk2(b.x, b.y)), v[4 * c], v[4 * c + 1]);
    upk2(add2(pk2(v[4 * c + 2], v[4 * c + 3]), pk2(b.z, b.w)), v[4 * c + 2], v[4 * c + 3]);
  }
}

// fp16 I/O: P and the FFN hidden enter their products without a lo part
// (see the precision plan above); bf16 keeps both parts.
template <typename T>
__host__ __device__ constexpr bool p_hi_only() { return std::is_same<T, __half>::value; }
template <typename T>
__host__ __device__ constexpr bool h_hi_only() { return std::is_same<T, __half>::value; }

// P buffers: with fp16 I/O P has no lo part, so head h's P goes to buffer
// h % 2 (the two 16 KB planes of the P area) and the softmax of head h + 1
// does not wait for P_h V_h; bf16 keeps one (hi, lo) buffer.
template <typename T>
__host__ __device__ constexpr int p_bufs() { return p_hi_only<T>() ? 2 : 1; }
// The (hi, lo) slots of P for row rr and key kk of the row's own sequence,
// in P buffer b.  With two buffers the lo slots (only the fp64 fix-up's
// parked score bits use them) are in the V spare area, free until the
// out-projection.
template <typename T>
__device__ __forceinline__ void p_slot(int rr, int kk, int b, int& hi_off, int& lo_off) {
  const int off = sw128(rr, kk >> 3) + (kk & 7) * 2;
  if constexpr (p_bufs<T>() == 2) {
    hi_off = kPB + b * kTile16 + off;
    lo_off = kVB + off;
  } else {
    hi_off = kPB + off;
    lo_off = kPB + kTile16 + off;
  }
}

// fp64 correction of one flagged (row rr, head h), done by a whole warp.
// The row's fp32 scores (log2 units, scaled, -inf where masked) were parked
// in its own P slots as bit patterns (high half in the hi plane, low half in
// the lo plane); lane owns keys kk = lane + 32 m of sequence sq.  Recomputes
// q_i in fp64 from the layer input and the weights, recomputes the scores of
// the candidate keys (within 12 + 2E of the best) exactly as
// x_j . (W_k^T q_i) + b_k . q_i, writes the row's softmax weights relative
// to the exact best score into the P slots and returns their sum.
template <typename T, int L>
__device__ __noinline__ float fixup_row(unsigned char* sm, const MegaLayer& P, int rr, int sq, int h,
                                        bool first, int lane, float kmx) {
  const int pbuf = h & 1;
  constexpr int NK = L / 32;  // keys per lane
  const unsigned char* xa = sm + kXA;
  auto xval = [&](int row, int col) -> double {
    const int kh = col >> 6, c8 = (col & 63) >> 3, e8 = col & 7;
    const int off = sw128(row, c8) + e8 * 2;
    double v = (double)to_f32<T>(*reinterpret_cast<const T*>(xa + kh * kTile16 + off));
    if (!first) v += (double)to_f32<T>(*reinterpret_cast<const T*>(xa + (2 + kh) * kTile16 + off));
    return v;
  };
  float sc[NK];  // screening scores, natural-log units
#pragma unroll
  for (int m = 0; m < NK; ++m) {
    int ho, lo;
    p_slot<T>(rr, lane + 32 * m, pbuf, ho, lo);
    const uint32_t bits = ((uint32_t)*reinterpret_cast<const uint16_t*>(sm + ho) << 16) |
                          (uint32_t)*reinterpret_cast<const uint16_t*>(sm + lo);
    sc[m] = __uint_as_float(bits) * 0.69314718055994531f;
  }
  const T* W = reinterpret_cast<const T*>(P.w_qkv);
  // q_i in fp64: lane c owns dim c
  double q64 = (double)P.b_qkv[32 * h + lane];
  for (int tt = 0; tt < kD; ++tt)
    q64 = fma((double)to_f32<T>(W[(size_t)(32 * h + lane) * kD + tt]), xval(rr, tt), q64);
  // u = W_k,h^T q_i (lane owns tt = lane + 32 m), u0 = b_k,h . q_i
  double u[4] = {0, 0, 0, 0};
  double u0 = 0.0, qq = 0.0;
  for (int c = 0; c < kDH; ++c) {
    const double qc = __shfl_sync(0xffffffffu, q64, c);
    u0 = fma(qc, (double)P.b_qkv[128 + 32 * h + c], u0);
    qq = fma(qc, qc, qq);
#pragma unroll
    for (int m = 0; m < 4; ++m)
      u[m] = fma(qc, (double)to_f32<T>(W[(size_t)(128 + 32 * h + c) * kD + lane + 32 * m]), u[m]);
  }
  float best = -INFINITY;
#pragma unroll
  for (int m = 0; m < NK; ++m) best = fmaxf(best, sc[m]);
  best = warp_max(best);
  const float err = neartie_err((float)sqrt(qq), kmx, kDH);
  const float thr = best - kTieGap - 2.f * err;
  double s64[NK];
  double Mx = -INFINITY;
#pragma unroll
  for (int m = 0; m < NK; ++m) {
    s64[m] = (double)sc[m];
    unsigned need = __ballot_sync(0xffffffffu, sc[m] != -INFINITY && sc[m] >= thr);
    while (need) {
      const int src = __ffs(need) - 1;
      need &= need - 1;
      const int key = sq * L + src + 32 * m;  // the key's row in the tile
      double part = 0.0;
#pragma unroll
      for (int mm = 0; mm < 4; ++mm) part = fma(xval(key, lane + 32 * mm), u[mm], part);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (lane == src) s64[m] = (part + u0) * (1.0 / sqrt((double)kDH));
    }
    Mx = fmax(Mx, s64[m]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Mx = fmax(Mx, __shfl_xor_sync(0xffffffffu, Mx, o));
  double ws = 0.0;
#pragma unroll
  for (int m = 0; m < NK; ++m) {
    const double e = s64[m] == -INFINITY ? 0.0 : exp(s64[m] - Mx);
    ws += e;
    T hv, lv;
    Split<T>::go((float)e, hv, lv);
    int ho, lo;
    p_slot<T>(rr, lane + 32 * m, pbuf, ho, lo);
    *reinterpret_cast<T*>(sm + ho) = hv;
    *reinterpret_cast<T*>(sm + lo) = lv;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
  return (float)ws;
}

// Registers: 96 per thread at launch (an SM sub-partition holds five warps
// of 16384 / 5 / 32 registers).  The control warpgroup drops to 64; in the
// assisted kernel setmaxnreg gives those to the compute warps (104 each):
// 128 x 64 + 512 x 104 = 61440 = 640 x 96, and per sub-partition
// 32 x (64 + 4 x 104) <= 16384.  The plain kernel's compute code fits 96
// without spills and is faster compiled to that budget.
template <typename T, int L, bool ASSIST>
__global__ void __launch_bounds__(kThreads, 1)
    mega_kernel(const __grid_constant__ CUtensorMap map_x, const MegaArgs a) {
  extern __shared__ __align__(1024) unsigned char dyn_smem[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kBars);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + kBars + kNumBars * 8);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
  constexpr bool kBf = std::is_same<T, __nv_bfloat16>::value;
  constexpr int S = 128 / L;  // sequences per tile
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_tiles = (a.B + S - 1) / S;
  const int n_chunks = a.dff / 128;  // 128-wide FFN chunks
  const int T_rows = a.B * L;
  // Assisted mode: rank 0 = resident R, rank 1 = helper H (see above).
  const uint32_t rank = ASSIST ? cluster_rank() : 0u;
  const bool helper = ASSIST && rank == 1;
  const uint32_t peer = rank ^ 1u;
  const int nb0 = helper ? 1 : 0, nb1 = ASSIST ? nb0 + 2 : 3;    // QKV weight boxes [nb0, nb1)
  const int h0 = helper ? 2 : 0, h1 = ASSIST ? h0 + 2 : kH;      // heads [h0, h1)
  const int half = (n_chunks + 1) / 2;
  const int c0 = helper ? half : 0, c1 = ASSIST && !helper ? half : n_chunks;  // FFN chunks [c0, c1)
  // tile loop: a cluster shares one tile sequence (unsigned special registers)
#define TL_T0 (ASSIST ? (blockIdx.x >> 1) : blockIdx.x)
#define TL_TSTEP (ASSIST ? (gridDim.x >> 1) : gridDim.x)

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      uint32_t cnt = 1;
      switch (i) {
        case B_A_READY: case B_QKVH_READY: case B_VH_READY: case B_VH_READY1: case B_S_FREE:
        case B_P_READY: case B_P_READY1:
        case B_CTX_READY:
        case B_Y_READY: case B_H_READY: case B_XA_FREE:
        case B_SYNC:
          cnt = kCompute;
          break;
        case B_SYNC_SM:
          cnt = kCompute / 2;
          break;
        case B_S_DONE:
          cnt = 2;  // the S commit + a release arrive of the MMA thread
          break;
        default: break;  // the peer barriers: one arrive (or expect-tx arrive) per phase
      }
      mbar_init(bar + i, cnt);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  if constexpr (ASSIST) cluster_sync_all();  // the peer's barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  volatile int* abort = abort_flag;
  int* status = a.status;
  if (warp < kCtrlWarps) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 64;" ::: "memory");
  if (warp == 0) {
    // ================================================================ TMA
    if (lane == 0) {
      long long tiles_done = 0;
      int reg_it = 0, ffn_it = 0;
      uint32_t par = 0, used = 0, out_par = 0;  // per-slot phase parity, slots ever loaded
      bool ok = true;
      auto wload = [&](const CUtensorMap* m, int x, int y, uint32_t bytes, bool ffn, int slot = -1) -> bool {
        const int idx = slot >= 0 ? 0 : ffn ? ffn_it++ : reg_it++;
        const int st = slot >= 0 ? slot : ffn ? idx % kNSlot : idx % kNW;
        if (slot < 0 && ffn && idx == kNW) {
          // the layer's first borrowed slot: its attention must be over
          if (!mbar_wait(bar + B_OUT_DONE, out_par, abort, status)) return false;
          out_par ^= 1;
        }
        if (!mbar_wait(bar + B_W_EMPTY + st, ((par >> st) & 1) ^ 1, abort, status)) return false;
        mbar_arrive_expect_tx(bar + B_W_FULL + st, bytes);
        tma_load_2d(sm + wslot_off(st), m, bar + B_W_FULL + st, x, y);
        par ^= 1u << st;
        used |= 1u << st;
        return true;
      };
      for (int t = TL_T0; t < n_tiles && ok; t += TL_TSTEP, ++tiles_done) {
        if (!mbar_wait(bar + B_XA_FREE, (uint32_t)(tiles_done & 1) ^ 1, abort, status)) break;
        mbar_arrive_expect_tx(bar + B_X_FULL, 2 * kTile16);
        tma_load_2d(sm + kXA, &map_x, bar + B_X_FULL, 0, t * 128);
        tma_load_2d(sm + kXA + kTile16, &map_x, bar + B_X_FULL, 64, t * 128);
        for (int l = 0; l < a.n_layers && ok; ++l) {
          const MegaLayer& P = a.layers[l];
          if constexpr (!ASSIST) {
            // QKV: N blocks 0, 1 of K half 0 into slots 0, 1 and of K half 1
            // into slots 2, 3 (adjacent pairs: two N = 256 operands), N block
            // 2 into slots 4 and 0; the out-projection into slots 1, 0.  The
            // borrowed slots 2-4 are free from the previous FFN's products to
            // the end of this QKV product (the conversions write there after).
            ok = wload(P.map_qkv, 0, 0, kTile16, false, 0) && wload(P.map_qkv, 0, 128, kTile16, false, 1) &&
                 wload(P.map_qkv, 64, 0, kTile16, false, 2) && wload(P.map_qkv, 64, 128, kTile16, false, 3) &&
                 wload(P.map_qkv, 0, 256, kTile16, false, 4) && wload(P.map_qkv, 64, 256, kTile16, false, 0);
            for (int kh = 0; kh < 2 && ok; ++kh) ok = wload(P.map_o, 64 * kh, 0, kTile16, false, kh == 0 ? 1 : 0);
          } else {
            for (int nb = nb0; nb < nb1 && ok; ++nb)
              for (int kh = 0; kh < 2 && ok; ++kh) ok = wload(P.map_qkv, 64 * kh, 128 * nb, kTile16, false);
            if (!helper)
              for (int kh = 0; kh < 2 && ok; ++kh) ok = wload(P.map_o, 64 * kh, 0, kTile16, false);
          }
          ffn_it = 0;  // at least three FFN boxes per layer: slot 2 is used, OUT_DONE waited once
          for (int c = c0; c <= c1 && ok; ++c) {
            if (c < c1)  // W_1 rows [128c, 128c + 128): two 128 x 64 boxes
              for (int kh = 0; kh < 2 && ok; ++kh) ok = wload(P.map_1, 64 * kh, 128 * c, kTile16, true);
            if (c > c0)  // W_2 columns [128(c-1), 128c): two 128 x 64 boxes
              for (int kh = 0; kh < 2 && ok; ++kh) ok = wload(P.map_2, 128 * (c - 1) + 64 * kh, 0, kTile16, true);
          }
        }
      }
      // Drain the loads in flight: each slot's last load.
      for (int st = 0; st < kNSlot; ++st)
        if ((used >> st) & 1) mbar_wait_bounded(bar + B_W_FULL + st, ((par >> st) & 1) ^ 1, status);
      if (tiles_done > 0) mbar_wait_bounded(bar + B_X_FULL, (uint32_t)((tiles_done - 1) & 1), status);
    }
  } else if (warp == 1) {
    // ================================================================ MMA
    int reg_it = 0, ffn_it = 0;  // the same slot sequence as the TMA thread
    uint32_t par = 0;            // per-slot phase parity
    const uint32_t id256 = idesc_f16(128, 256, kBf);
    const uint32_t id128 = idesc_f16(128, 128, kBf);
    const uint32_t id64 = idesc_f16(128, 64, kBf);
    const uint32_t id64_bmn = id64 | (1u << 16);  // B MN-major (bit 16)
    const uint32_t id32 = idesc_f16(128, 32, kBf);
    bool ok = true;
    const uint32_t xa = smem_u32(sm + kXA), pb = smem_u32(sm + kPB);
    const uint32_t qb = smem_u32(sm + kQB), kb = smem_u32(sm + kKB), pv = smem_u32(sm + kPV);
    // One weight box against A (one or two planes x 4 k16 steps) into d.
    // A is a 128 x 64 tile at a_base; its lo plane is part_stride further on
    // (part_stride 0: the hi plane only).
    auto wbox = [&](uint32_t d, uint32_t a_base, uint32_t part_stride, uint32_t idesc, bool first,
                    bool ffn, int slot = -1) -> bool {
      const int st = slot >= 0 ? slot : ffn ? ffn_it++ % kNSlot : reg_it++ % kNW;
      if (!mbar_wait(bar + B_W_FULL + st, (par >> st) & 1, abort, status)) return false;
      par ^= 1u << st;
      tc_fence_after();
      // the whole warp builds the (uniform) descriptors; one elected lane issues
      {
        // descriptors built once; a k16 step or a part moves the start
        // address field (bytes / 16), which no smem address overflows
        const uint64_t dw = sdesc_sw128(smem_u32(sm + wslot_off(st)));
        const uint64_t da = sdesc_sw128(a_base);
        const int parts = part_stride == 0 ? 1 : 2;
        for (int p = 0; p < parts; ++p) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f16_elect(d, da + ((p * part_stride + k * 32) >> 4), dw + 2 * k, idesc,
                          (first && p == 0 && k == 0) ? 0u : 1u);
        }
        mma_commit_elect(bar + B_W_EMPTY + st);
      }
      __syncwarp();
      return true;
    };
    // The same with A in tensor memory: columns a_col + 8 k (k16 step k) of
    // the hi part, part_cols further on for the lo part.
    auto wbox_ta = [&](uint32_t d, uint32_t a_col, uint32_t part_cols, uint32_t idesc, bool first,
                       bool ffn, int parts = 2, int slot = -1) -> bool {
      const int st = slot >= 0 ? slot : ffn ? ffn_it++ % kNSlot : reg_it++ % kNW;
      if (!mbar_wait(bar + B_W_FULL + st, (par >> st) & 1, abort, status)) return false;
      par ^= 1u << st;
      tc_fence_after();
      {
        const uint64_t dw = sdesc_sw128(smem_u32(sm + wslot_off(st)));
        for (int p = 0; p < parts; ++p) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f16_ta_elect(d, tmem + a_col + p * part_cols + 8 * k, dw + 2 * k, idesc,
                             (first && p == 0 && k == 0) ? 0u : 1u);
        }
        mma_commit_elect(bar + B_W_EMPTY + st);
      }
      __syncwarp();
      return true;
    };
    // FFN2's A operand: the h words of FFN buffer column buf_col, box kh
    // (K values [64 kh, 64 kh + 64)).  The compute group g that held K
    // columns [32 g, 32 g + 32) wrote them over its own accumulator columns,
    // hi in the upper 16, lo (bf16) in the lower 16: k16 step k of box kh is
    // word 8 (k % 2) of group 2 kh + k / 2.
    auto wbox_h = [&](uint32_t d, uint32_t buf_col, int kh, uint32_t idesc, bool first,
                      int parts) -> bool {
      const int st = ffn_it++ % kNSlot;
      if (!mbar_wait(bar + B_W_FULL + st, (par >> st) & 1, abort, status)) return false;
      par ^= 1u << st;
      tc_fence_after();
      {
        const uint64_t dw = sdesc_sw128(smem_u32(sm + wslot_off(st)));
        for (int p = 0; p < parts; ++p) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f16_ta_elect(d, tmem + buf_col + 32 * (2 * kh + k / 2) + 8 * (k % 2) + (p == 0 ? 16 : 0),
                             dw + 2 * k, idesc, (first && p == 0 && k == 0) ? 0u : 1u);
        }
        mma_commit_elect(bar + B_W_EMPTY + st);
      }
      __syncwarp();
      return true;
    };
    // QKV N blocks 0 and 1 of K half kh against A (layer 0: the input's hi
    // plane in the X buffer; later layers: the (hi, lo) input in TMEM) into
    // columns [0, 256): one N = 256 product per k16 step, its B operand the
    // adjacent slots s0, s0 + 1 (rows 0-127, 128-255).
    auto wpair = [&](bool from_x, int kh, int s0) -> bool {
      const int s1 = s0 + 1;
      if (!mbar_wait(bar + B_W_FULL + s0, (par >> s0) & 1, abort, status)) return false;
      par ^= 1u << s0;
      if (!mbar_wait(bar + B_W_FULL + s1, (par >> s1) & 1, abort, status)) return false;
      par ^= 1u << s1;
      tc_fence_after();
      const uint64_t dw = sdesc_sw128(smem_u32(sm + wslot_off(s0)));
      if (from_x) {
        const uint64_t da = sdesc_sw128(xa + kh * kTile16);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_f16_elect(tmem, da + ((k * 32) >> 4), dw + 2 * k, id256, (kh == 0 && k == 0) ? 0u : 1u);
      } else {
        for (int p = 0; p < 2; ++p) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f16_ta_elect(tmem, tmem + kTX + 32 * kh + p * 64 + 8 * k, dw + 2 * k, id256,
                             (kh == 0 && p == 0 && k == 0) ? 0u : 1u);
        }
      }
      mma_commit_elect(bar + B_W_EMPTY + s0);
      mma_commit_elect(bar + B_W_EMPTY + s1);
      __syncwarp();
      return true;
    };
    // Plain kernel: one out-projection box (K half kh: heads 2 kh, 2 kh + 1)
    // against the context words in TMEM (hi part, then lo part) into d.
    auto wbox_o = [&](uint32_t d, int kh, int st) -> bool {
      if (!mbar_wait(bar + B_W_FULL + st, (par >> st) & 1, abort, status)) return false;
      par ^= 1u << st;
      tc_fence_after();
      const uint64_t dw = sdesc_sw128(smem_u32(sm + wslot_off(st)));
      for (int p = 0; p < 2; ++p) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_f16_ta_elect(d, tmem + 96 * (2 * kh + k / 2) + 16 * (k % 2) + 8 * p, dw + 2 * k, id128,
                           (kh == 0 && p == 0 && k == 0) ? 0u : 1u);
      }
      mma_commit_elect(bar + B_W_EMPTY + st);
      __syncwarp();
      return true;
    };
    auto commit = [&](int b) {
      mma_commit_elect(bar + b);
      __syncwarp();
    };
    auto wait = [&](int b, long long& n, bool is_free = false) -> bool {
      const uint32_t par = (uint32_t)(n & 1) ^ (is_free ? 1u : 0u);
      ++n;
      if (!mbar_wait(bar + b, par, abort, status)) return false;
      tc_fence_after();
      return true;
    };
    long long c_x = 0, c_a = 0, c_qkvh = 0, c_vh0 = 0, c_vh1 = 0, c_sfree = 0, c_p0 = 0, c_p1 = 0, c_ctx = 0, c_y = 0,
              c_hfree[2] = {0, 0}, c_hr = 0;
    long long c_pctx = 0;  // assisted R: phases of B_PEER_CTX waited
    for (int t = TL_T0; t < n_tiles && ok; t += TL_TSTEP) {
      for (int l = 0; l < a.n_layers && ok; ++l) {
        // ---- QKV (the first layer's input is exact in its hi plane)
        ok = l == 0 ? wait(B_X_FULL, c_x) : wait(B_A_READY, c_a);
        // layer 0: x from shared memory (exact in its hi plane); later layers:
        // the (hi, lo) input LayerNorm 2 also left in TMEM [384, 512) (the
        // helper has it in its X buffer, written by R)
        if constexpr (!ASSIST) {
          // the loader's slots: N blocks 0, 1 as one N = 256 product per K
          // half (slots 0-1, 2-3), then N block 2 (slots 4, 0)
          // columns [0, 256) (heads 0, 1 and head 2's q, k) are released
          // first, so the first head's conversion overlaps N block 2
          ok = wpair(l == 0, 0, 0) && wpair(l == 0, 1, 2);
          if (!ok) break;
          commit(B_QKV_DONE);
          for (int kh = 0; kh < 2 && ok; ++kh)
            ok = l == 0 ? wbox(tmem + 256, xa + kh * kTile16, 0u, id128, kh == 0, false, kh == 0 ? 4 : 0)
                        : wbox_ta(tmem + 256, kTX + 32 * kh, 64, id128, kh == 0, false, 2, kh == 0 ? 4 : 0);
          if (!ok) break;
          commit(B_QKV_DONE2);
        } else {
          for (int nb = nb0; nb < nb1 && ok; ++nb)
            for (int kh = 0; kh < 2 && ok; ++kh)
              ok = l == 0 ? wbox(tmem + 128 * nb, xa + kh * kTile16, 0u, id128, kh == 0, false)
                   : helper ? wbox(tmem + 128 * nb, xa + kh * kTile16, 2u * kTile16, id128, kh == 0, false)
                            : wbox_ta(tmem + 128 * nb, kTX + 32 * kh, 64, id128, kh == 0, false);
          if (!ok) break;
          commit(B_QKV_DONE);
        }
        // ---- attention: S_0, then per head h: S_{h+1} as soon as head h+1's
        // Q, K, V are in shared memory, then P_h V_h, so the next scores are
        // computed while the compute warps run the softmax of head h.
        auto issue_s = [&](int h) -> bool {
          if (!(wait(B_QKVH_READY, c_qkvh) && wait(B_S_FREE, c_sfree, true))) return false;
          // Release what the compute threads wrote before QKVH_READY (norms,
          // the tile's max |k|) to whoever acquires S_DONE.
          if (lane == 0) mbar_arrive(bar + B_S_DONE);
          __syncwarp();
          {
            const uint32_t as[3] = {qb, qb, qb + 8192};
            const uint32_t bs[3] = {kb, kb + 8192, kb};
#pragma unroll
            for (int c = 0; c < 3; ++c)
#pragma unroll
              for (int k = 0; k < 2; ++k)
                mma_f16_elect(tmem + 384, desc_sw64(as[c]) + 2 * k, desc_sw64(bs[c]) + 2 * k, id128,
                              (c | k) != 0);
          }
          commit(B_S_DONE);
          return true;
        };
        ok = issue_s(h0);
        for (int h = h0; h < h1 && ok; ++h) {
          if (h + 1 < h1 && !(ok = issue_s(h + 1))) break;
          // P_h, and V_h (published after Q_h, K_h: S_h does not wait for
          // it), on one of two barriers by head parity: a barrier serves
          // every other head, so it is never two phases ahead of this wait
          ok = ((h & 1) ? wait(B_P_READY1, c_p1) : wait(B_P_READY, c_p0)) &&
               ((h & 1) ? wait(B_VH_READY1, c_vh1) : wait(B_VH_READY, c_vh0));
          if (!ok) break;
          {
            // O_h = Ph.Vh + Ph.Vl (+ Pl.Vh with bf16) over the row's own 64
            // keys (4 steps): B holds both sequences' V side by side (N = 64),
            // so row r's result is in columns [96h + 32 s, +32) of its sequence s.
            // B is MN-major: a 16-key step is 16 rows of 128 bytes further.
            const uint32_t vbuf = pv + (uint32_t)((h & 1) * kTile16);
            const uint32_t pbh = pb + (uint32_t)((p_bufs<T>() == 2 ? h & 1 : 0) * kTile16);
            const uint32_t as[3] = {pbh, pbh, pb + kTile16};
            const uint32_t bs[3] = {vbuf, vbuf + kTile16 / 2, vbuf};
            constexpr int kProducts = p_hi_only<T>() ? 2 : 3;
#pragma unroll
            for (int c = 0; c < kProducts; ++c)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_f16_elect(tmem + 96 * h, sdesc_sw128(as[c]) + 2 * k, sdesc_mn_sw128(bs[c]) + 128 * k,
                              id64_bmn, (c | k) != 0);
          }
          commit(B_O_DONE + (h & 1));
        }
        if (!ok) break;
        if (helper) {
          // no out-projection here: OUT_DONE marks the end of this CTA's
          // attention products (the loader's borrowed FFN slots wait on it)
          commit(B_OUT_DONE);
        } else {
          // ---- out-projection (assisted: also heads 2, 3 from the helper)
          ok = wait(B_CTX_READY, c_ctx);
          if (ok && ASSIST) {
            // H's context (two 16 KB planes) arrives by bulk copy
            if (lane == 0) mbar_arrive_expect_tx(bar + B_PEER_CTX, 2 * kTile16);
            __syncwarp();
            ok = mbar_wait_cluster(bar + B_PEER_CTX, (uint32_t)(c_pctx & 1), abort, status);
            ++c_pctx;
            tc_fence_after();
          }
          if constexpr (!ASSIST) {
            for (int kh = 0; kh < 2 && ok; ++kh) ok = wbox_o(tmem + kTOut, kh, kh == 0 ? 1 : 0);
          } else {
            for (int kh = 0; kh < 2 && ok; ++kh)
              ok = wbox(tmem + 128, pb + kh * kTile16, 2u * kTile16, id128, kh == 0, false);
          }
          if (!ok) break;
          commit(B_OUT_DONE);
        }
        // ---- FFN in 128-wide chunks; chunk c uses TMEM buffer c % 2 for its
        // FFN1 accumulator and then, rewritten by GELU, as FFN2's A operand
        ok = wait(B_Y_READY, c_y);
        ffn_it = 0;
        for (int c = c0; c <= c1 && ok; ++c) {
          if (c < c1) {
            const int buf = c & 1;
            // the buffer's last reader, FFN2 of chunk c - 2, must be done
            if (c >= c0 + 2) ok = wait(B_H_FREE + buf, c_hfree[buf]);
            // A = y: tensor memory, or (helper) the (hi, lo) copy R wrote
            // into this CTA's X buffer
            for (int kh = 0; kh < 2 && ok; ++kh)
              ok = helper ? wbox(tmem + kTF + 128 * buf, xa + kh * kTile16, 2u * kTile16, id128, kh == 0, true)
                          : wbox_ta(tmem + kTF + 128 * buf, kTY + 32 * kh, 64, id128, kh == 0, true);
            if (!ok) break;
            commit(B_F1_DONE + buf);
          }
          if (c > c0) {
            const int hb = (c - 1) & 1;
            ok = wait(B_H_READY, c_hr);
            for (int kh = 0; kh < 2 && ok; ++kh)
              ok = wbox_h(tmem, kTF + 128 * hb, kh, id128, c == c0 + 1 && kh == 0, h_hi_only<T>() ? 1 : 2);
            if (!ok) break;
            commit(B_H_FREE + hb);
          }
        }
        if (!ok) break;
        commit(B_F2_DONE);
        // keep the per-buffer release counts in step: the last two chunks'
        // releases were not waited for in the loop
        for (int c = (c1 - c0 >= 2 ? c1 - 2 : c0); c < c1 && ok; ++c)
          ok = wait(B_H_FREE + (c & 1), c_hfree[c & 1]);
        if (!ok) break;
      }
    }
    commit(B_MMA_DONE);
    mbar_wait_bounded(bar + B_MMA_DONE, 0, status);
  }
  } else {
    // the assisted kernel's compute code needs the 104; the plain kernel's
    // fits 96 without spills and runs faster compiled to that budget
    if constexpr (ASSIST) asm volatile("setmaxnreg.inc.sync.aligned.u32 104;" ::: "memory");
    // ======================================================== compute warps
    const int cw = warp - kCtrlWarps;      // 0..15
    const int g = cw >> 2;                 // column group
    const int qd = warp & 3;               // TMEM lane quarter (fixed by the warp index)
    const int r = qd * 32 + lane;          // row in the tile
    const int sq = r / L;                  // sequence within the tile
    const int i = r % L;                   // position in the sequence
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    float* qn2_s = reinterpret_cast<float*>(sm + kQn2);
    float* ex = reinterpret_cast<float*>(sm + kEx);
    float* l_s = reinterpret_cast<float*>(sm + kLs);
    // the layer's LayerNorm vectors: the P area (plain kernel), the softmax
    // sums' area (assisted kernel, whose P area holds the context)
#define TL_LNV (ASSIST ? l_s : reinterpret_cast<float*>(sm + kPB))
    int* kmax_s = reinterpret_cast<int*>(sm + kKmax);
    const float* vec_s = reinterpret_cast<const float*>(sm + kVec);  // b_qkv, then b_1 at 384
    unsigned char* xa = sm + kXA;
    unsigned char* pbuf = sm + kPB;
    const float scale_log2 = rsqrtf((float)kDH) * 1.4426950408889634f;
    constexpr int NM = L / 32;  // own 8-key chunks of a row per group
    int c_qkv = 0, c_s = 0, c_o0 = 0, c_o1 = 0, c_out = 0, c_f1[2] = {0, 0}, c_f2 = 0,
        c_sync = 0, c_sync_sm = 0;  // completed phases per barrier (parity = count & 1)
    // assisted mode: phases of the barriers the other CTA arrives on
    int c_pbfree = 0, c_py = 0, c_px = 0, c_xfree = 0, c_part = 0;
    bool ok = true;
    // Wait for a hand-over from the other CTA of the cluster.
    auto wait_peer = [&](int b, int& n) -> bool {
      const uint32_t par = (uint32_t)(n & 1);
      ++n;
      if (!mbar_wait_cluster(bar + b, par, abort, status)) return false;
      tc_fence_after();
      return true;
    };
    // One thread of the compute warps handles the bulk copies and signals.
    const bool elected = threadIdx.x == kCtrlWarps * 32;
    auto peer_addr = [&](const void* p) { return map_to_rank(smem_u32(p), peer); };
    // A "buffer free" signal to the other CTA (release at cluster scope).
    auto signal_peer = [&](int b) { mbar_arrive_cluster(peer_addr(bar + b)); };
    // Send `bytes` of this CTA's shared memory at src to the same offset in
    // the other CTA, completing on its barrier b (after every compute thread
    // staged its part: callers fence and bar_compute first).
    auto send_peer = [&](const void* src, uint32_t bytes, int b) {
      bulk_copy_to_cta(peer_addr(src), src, bytes, peer_addr(bar + b));
    };
    auto wait = [&](int b, int& n) -> bool {
      const uint32_t par = (uint32_t)(n & 1);
      ++n;
      if (!mbar_wait(bar + b, par, abort, status)) return false;
      tc_fence_after();
      return true;
    };
    // O_h = P_h V_h done, on one of two barriers by head parity.  Every
    // compute thread waits each head's phase once per layer, in head order
    // (o_next: the first head not yet waited), and nothing completes a
    // head's phase before every thread has waited the previous phase of
    // that barrier (two heads earlier), so no wait sees two phases ahead.
    int o_next = 0;
    auto wait_o_upto = [&](int hl) -> bool {
      for (; o_next <= hl; ++o_next)
        if (!((o_next & 1) ? wait(B_O_DONE1, c_o1) : wait(B_O_DONE, c_o0))) return false;
      return true;
    };
    auto arrive = [&](int b) {
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(bar + b);
    };
    // Barrier of the 512 compute threads on an mbarrier, so that the wait is
    // bounded like every other wait (a bar.sync could not give up).
    auto bar_compute = [&]() {
      mbar_arrive(bar + B_SYNC);
      const uint32_t par = (uint32_t)(c_sync & 1);
      ++c_sync;
      mbar_wait(bar + B_SYNC, par, abort, status);
    };
    // The same for the 256 softmax threads (groups 0, 1) of the split heads.
    auto bar_softmax = [&]() {
      mbar_arrive(bar + B_SYNC_SM);
      const uint32_t par = (uint32_t)(c_sync_sm & 1);
      ++c_sync_sm;
      mbar_wait(bar + B_SYNC_SM, par, abort, status);
    };
    // 16 columns (part 0 or 1) of Q_h (hi, lo) with a partial |q|^2, or of
    // K_h with the tile's largest partial |k|^2.
    auto convert_qk = [&](int h, bool isq, int part) {
      float v[16];
      const int c0 = 16 * part;
      const int col = 96 * h + (isq ? 0 : 32) + c0;  // head h's q | k | v columns
      tmem_ld16_nw(trow + col, v);
      tmem_wait_ld();
      add_vec<16>(v, vec_s + col);
      float n2 = 0.f;
#pragma unroll
      for (int c = 0; c < 16; ++c) n2 = fmaf(v[c], v[c], n2);
      unsigned char* dst = sm + (isq ? kQB : kKB);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) put8<T>(dst, dst + 8192, sw64(r, (2 * part + cc) * 16), v + 8 * cc);
      if (isq) {
        qn2_s[((h & 1) * 2 + part) * 128 + r] = n2;
      } else {
        const float kn = warp_max(n2);
        if (lane == 0) atomicMax(kmax_s + 2 * h + part, __float_as_int(kn));
      }
    };
    // V_h (hi, lo) into buffer h % 2, the B operand of P V read MN-major:
    // row = key position k, its 64 columns [V_s0[k] | V_s1[k]] (the two
    // sequences side by side).  This thread: key r (sequence r / 64,
    // position r % 64), dims [8 vp, 8 vp + 8) -- one 16-byte chunk per plane.
    auto convert_v = [&](int h, int vp) {
      float v[8];
      tmem_ld8_nw(trow + 96 * h + 64 + 8 * vp, v);
      tmem_wait_ld();
      add_vec<8>(v, vec_s + 96 * h + 64 + 8 * vp);
      unsigned char* vh = sm + kPV + (h & 1) * kTile16;
      put8<T>(vh, vh + kTile16 / 2, sw128(r & 63, 4 * (r >> 6) + vp), v);
    };
    // Plain kernel: the context of head hh for this thread's row, dims
    // [16j, 16j + 16): O / l as (hi, lo) words over TMEM columns 96 hh + 16j
    // + [0, 16), which hold this row's own O values for sequence 0 and
    // unused ones for sequence 1 -- no other thread reads or writes them.
    // The stores are waited for before CTX_READY.
    auto ctx_tmem = [&](int hh, int j) {
      float o[16];
      tmem_ld16_nw(trow + 96 * hh + 32 * sq + 16 * j, o);
      const float lsum = l_s[(hh * 4) * 128 + r] + l_s[(hh * 4 + 1) * 128 + r] +
                         l_s[(hh * 4 + 2) * 128 + r] + l_s[(hh * 4 + 3) * 128 + r];
      tmem_wait_ld();
      const float inv = 1.f / lsum;
#pragma unroll
      for (int c = 0; c < 16; ++c) o[c] *= inv;
      uint32_t w[16];
      split8(o, *reinterpret_cast<uint4*>(w), *reinterpret_cast<uint4*>(w + 8), T());
      split8(o + 8, *reinterpret_cast<uint4*>(w + 4), *reinterpret_cast<uint4*>(w + 12), T());
      tmem_st16(trow + 96 * hh + 16 * j, w);
    };
    // LayerNorm of acc (TMEM columns tcol + [32g, +32)) + bias + residual
    // (the X buffer): per-group (mean, M2) over 32 columns, merged through
    // the exchange with Chan's formula, (01)(23) then the two pairs.
    // bias, gam, bet: the layer's vectors staged in shared memory
    auto layernorm = [&](uint32_t tcol, const float* bias, const float* gam, const float* bet,
                         bool resid_lo, bool resid_tmem, float* v, const float* part = nullptr) {
      tmem_ld32_nw(trow + tcol + 32 * g, v);
      if (resid_tmem) {
        // the residual y: (hi, lo) words [16g, 16g + 16) of TMEM columns kTY, kTY + 64
        uint32_t hw[16], lw[16];
        tmem_ld16_nw(trow + kTY + 16 * g, reinterpret_cast<float*>(hw));
        tmem_ld16_nw(trow + kTY + 64 + 16 * g, reinterpret_cast<float*>(lw));
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          v[2 * e] = addw<T>(addw<T>(v[2 * e], (unsigned short)(hw[e] & 0xFFFFu)), (unsigned short)(lw[e] & 0xFFFFu));
          v[2 * e + 1] = addw<T>(addw<T>(v[2 * e + 1], (unsigned short)(hw[e] >> 16)), (unsigned short)(lw[e] >> 16));
        }
      } else {
        tmem_wait_ld();
        const int kh = g >> 1;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int off = sw128(r, (g & 1) * 4 + cc);
          const uint4 hv = *reinterpret_cast<const uint4*>(xa + kh * kTile16 + off);
          const uint4 lv = resid_lo ? *reinterpret_cast<const uint4*>(xa + (2 + kh) * kTile16 + off) : make_uint4(0, 0, 0, 0);
          add8w<T>(v + 8 * cc, hv);
          add8w<T>(v + 8 * cc, lv);
        }
      }
      if (part) {  // the helper's FFN2 partial sum: fp32 [128 rows][128 columns]
        const float4* p4 = reinterpret_cast<const float4*>(part + r * 128 + 32 * g);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 q = p4[c4];
          v[4 * c4] += q.x; v[4 * c4 + 1] += q.y; v[4 * c4 + 2] += q.z; v[4 * c4 + 3] += q.w;
        }
      }
      add_vec<32>(v, bias + 32 * g);
      // sums over four interleaved accumulators (shorter dependency chains),
      // two of them at a time on the paired instructions
      uint64_t sa = 0, sb = 0;
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        sa = add2(sa, pk2(v[c], v[c + 1]));
        sb = add2(sb, pk2(v[c + 2], v[c + 3]));
      }
      float s0, s1, s2, s3;
      upk2(sa, s0, s1);
      upk2(sb, s2, s3);
      const float mean = ((s0 + s1) + (s2 + s3)) * (1.f / 32.f);
      const uint64_t mean2 = splat2(mean);
      uint64_t qa = 0, qb = 0;
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const uint64_t da = sub2(pk2(v[c], v[c + 1]), mean2), db = sub2(pk2(v[c + 2], v[c + 3]), mean2);
        qa = fma2(da, da, qa);
        qb = fma2(db, db, qb);
      }
      upk2(qa, s0, s1);
      upk2(qb, s2, s3);
      const float m2v = (s0 + s1) + (s2 + s3);
      ex[g * 128 + r] = mean;
      ex[(4 + g) * 128 + r] = m2v;
      bar_compute();
      float mg[4], qg[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        mg[k] = ex[k * 128 + r];
        qg[k] = ex[(4 + k) * 128 + r];
      }
      const float d01 = mg[1] - mg[0], d23 = mg[3] - mg[2];
      const float m01 = mg[0] + 0.5f * d01, m23 = mg[2] + 0.5f * d23;
      const float q01 = qg[0] + qg[1] + d01 * d01 * 16.f, q23 = qg[2] + qg[3] + d23 * d23 * 16.f;
      const float dd = m23 - m01;
      const float mu = m01 + 0.5f * dd;
      const float var = (q01 + q23 + dd * dd * 32.f) * (1.f / 128.f);
      const float rstd = rsqrtf(var + 1e-5f);
      const float4* g4 = reinterpret_cast<const float4*>(gam + 32 * g);
      const float4* e4 = reinterpret_cast<const float4*>(bet + 32 * g);
      const uint64_t mu2 = splat2(mu), rs2 = splat2(rstd);
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {  // (v - mu) rstd gamma + beta, paired
        const float4 gg = g4[c4], e = e4[c4];
        upk2(fma2(mul2(sub2(pk2(v[4 * c4], v[4 * c4 + 1]), mu2), rs2), pk2(gg.x, gg.y), pk2(e.x, e.y)),
             v[4 * c4], v[4 * c4 + 1]);
        upk2(fma2(mul2(sub2(pk2(v[4 * c4 + 2], v[4 * c4 + 3]), mu2), rs2), pk2(gg.z, gg.w), pk2(e.z, e.w)),
             v[4 * c4 + 2], v[4 * c4 + 3]);
      }
    };
    // A layer's b_qkv (head-grouped order) and b_1 in shared memory, with the
    // per-head |k| maxima reset: layer 0's here, every next layer's (the next
    // tile's layer 0 after the last) at the previous layer's FFN2 completion,
    // from values loaded into registers after its last GELU.  Every reader of
    // the old values is done by then, and the barrier of LayerNorm 2 (or of
    // the helper's partial sum) publishes the new ones before the next QKV
    // product completes.
    // this thread's entries: cv, cv + 512 (cv = threadIdx.x - 128, recomputed
    // where used rather than held in a register)
#define TL_CV ((int)threadIdx.x - kCtrlWarps * 32)
    auto vec_val = [&](const MegaLayer& Q, int k) -> float {
      if (k >= 384 + a.dff) return 0.f;
      return k < 384 ? __ldg(Q.b_qkv + ((k % 96) >> 5) * 128 + (k / 96) * 32 + (k & 31))
                     : __ldg(Q.b_1 + (k - 384));
    };
    auto stage_vec = [&](float v0, float v1) {
      float* vs = reinterpret_cast<float*>(sm + kVec);
      if (TL_CV < 384 + a.dff) vs[TL_CV] = v0;
      if (TL_CV + kCompute < 384 + a.dff) vs[TL_CV + kCompute] = v1;
      if (threadIdx.x == kCtrlWarps * 32)
        for (int k = 0; k < 2 * kH; ++k) kmax_s[k] = 0;
    };
    stage_vec(vec_val(a.layers[0], TL_CV), vec_val(a.layers[0], TL_CV + kCompute));
    bar_compute();
    for (int t = TL_T0; t < n_tiles && ok; t += TL_TSTEP) {
      const int seq = t * S + sq;
      const bool row_valid = seq < a.B;
      int vl = row_valid ? a.valid_len[seq] : 1;
      if (vl < 1 || vl > L) {
        if (row_valid) set_status(status, TL_ERR_BAD_VALID_LEN);
        vl = vl < 1 ? 1 : L;
      }
      const int limit = min(i + 1, vl);   // visible keys of this row: [sq*L, sq*L + limit)
      const size_t grow = (size_t)t * 128 + r;
      for (int l = 0; l < a.n_layers && ok; ++l) {
        const MegaLayer& P = a.layers[l];
        const bool first = l == 0;
        o_next = h0;
        if (!wait(B_QKV_DONE, c_qkv)) { ok = false; break; }
        // the first head's Q, K, V: every group (groups 0, 1 Q, groups 2, 3 K)
        convert_qk(h0, g < 2, g & 1);
        convert_v(h0, g);
        arrive(B_QKVH_READY);
        arrive(B_VH_READY + (h0 & 1));
        if constexpr (!ASSIST) {
          // Heads on two warp roles at once: groups 0, 1 run the softmax of
          // head h (32 keys of the row each) while groups 2, 3 convert head
          // h + 1's Q, K, V; one role's barrier arrivals count twice, so the
          // barriers keep their 512-thread counts.
          const bool smx = g < 2;
          const int gs = g & 1;
          constexpr int NS = L / 16;  // own 8-key chunks gs + 2 m
          for (int h = h0; h < h1 && ok; ++h) {
            if (!wait(B_S_DONE, c_s)) { ok = false; break; }
            if (!smx) {
              // S_h has read the Q, K buffers: head h + 1's Q, K first, so
              // that S_{h+1} can start; then its V, once P_{h-1} V_{h-1}
              // (waited from the second head on) has read that V buffer.
              // That wait also means the MMA thread has taken the previous
              // phase of this head parity's V barrier (V_{h-1}).
              if (h + 1 < h1) {
                convert_qk(h + 1, true, gs);
                convert_qk(h + 1, false, gs);
                fence_proxy_async();
                tc_fence_before();
                mbar_arrive_n(bar + B_QKVH_READY, 2);
              }
              if (!wait_o_upto(h - 1)) { ok = false; break; }
              // head 2's V is the first conversion from QKV columns [256, 384),
              // completed once a layer like QKV_DONE (so the same parity)
              if (h + 1 == 2) {
                if (!mbar_wait(bar + B_QKV_DONE2, (uint32_t)((c_qkv - 1) & 1), abort, status)) { ok = false; break; }
                tc_fence_after();
              }
              if (h + 1 < h1) {
                convert_v(h + 1, 2 * gs);
                convert_v(h + 1, 2 * gs + 1);
                fence_proxy_async();
                tc_fence_before();
                mbar_arrive_n(bar + B_VH_READY + ((h + 1) & 1), 2);
              }
              // the context of head h - 1, whose P V was just waited for
              if (h > h0) ctx_tmem(h - 1, gs);
              continue;
            }
            float s[8 * NS];
#pragma unroll
            for (int m = 0; m < NS; ++m) tmem_ld8_nw(trow + 384 + sq * L + 8 * (gs + 2 * m), s + 8 * m);
            // the row's |q| and the tile's max |k| of head h, read before S_FREE:
            // the conversion of head h + 2 (which needs S_{h+1}, so S_FREE)
            // reuses these |q|^2 slots
            const float qn2a = qn2_s[((h & 1) * 2) * 128 + r], qn2b = qn2_s[((h & 1) * 2 + 1) * 128 + r];
            const float kmx = sqrtf(__int_as_float(kmax_s[2 * h]) + __int_as_float(kmax_s[2 * h + 1]));
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive_n(bar + B_S_FREE, 2);
            // every softmax thread is done with head h - 1 (its exchange
            // slots and parked scores are reused); P_h's buffer was last read
            // by P_{h - p_bufs} V
            if (p_bufs<T>() == 2 && h > h0) bar_softmax();
            if (!wait_o_upto(h - p_bufs<T>())) { ok = false; break; }
            const float qn = sqrtf(qn2a + qn2b);
            const bool track = neartie_err(qn, kmx, kDH) > kTieErrMin;
            // the second-best score only where a near tie can matter; a
            // row's track flag is the same in both softmax groups, so the
            // unused second-best slots are never merged into a used result
            const bool wtrack = __any_sync(0xffffffffu, track);
            float m1 = -INFINITY, m2 = -INFINITY;
            if (wtrack) {
#pragma unroll
              for (int m = 0; m < NS; ++m)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const int kk = 8 * (gs + 2 * m) + e;
                  const float v = kk < limit ? s[8 * m + e] * scale_log2 : -INFINITY;
                  s[8 * m + e] = v;
                  m2 = fmaxf(m2, fminf(m1, v));
                  m1 = fmaxf(m1, v);
                }
              ex[(4 + gs) * 128 + r] = m2;
            } else {
              // two independent three-input max chains (the maximum is exact
              // in any order)
              float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
              for (int m = 0; m < NS; ++m)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const int kk = 8 * (gs + 2 * m) + e;
                  s[8 * m + e] = kk < limit ? s[8 * m + e] * scale_log2 : -INFINITY;
                }
#pragma unroll
              for (int m = 0; m < NS; ++m) {
                ma = max3_f32(ma, s[8 * m], s[8 * m + 1]);
                mb = max3_f32(mb, s[8 * m + 2], s[8 * m + 3]);
                ma = max3_f32(ma, s[8 * m + 4], s[8 * m + 5]);
                mb = max3_f32(mb, s[8 * m + 6], s[8 * m + 7]);
              }
              m1 = fmaxf(ma, mb);
            }
            ex[gs * 128 + r] = m1;
            if (track) {
              // park the raw scores in this row's P slots for a possible fp64 fix-up
#pragma unroll
              for (int m = 0; m < NS; ++m) {
                uint4 hv, lv;
                uint32_t* hw = reinterpret_cast<uint32_t*>(&hv);
                uint32_t* lw = reinterpret_cast<uint32_t*>(&lv);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                  const uint32_t b0 = __float_as_uint(s[8 * m + 2 * w]), b1 = __float_as_uint(s[8 * m + 2 * w + 1]);
                  hw[w] = (b0 >> 16) | (b1 & 0xFFFF0000u);
                  lw[w] = (b0 & 0xFFFFu) | (b1 << 16);
                }
                int ho, lo;
                p_slot<T>(r, 8 * (gs + 2 * m), h & 1, ho, lo);
                *reinterpret_cast<uint4*>(sm + ho) = hv;
                *reinterpret_cast<uint4*>(sm + lo) = lv;
              }
            }
            bar_softmax();
            float M1 = -INFINITY, M2 = -INFINITY;
            if (wtrack) {
#pragma unroll
              for (int k = 0; k < 2; ++k) {
                const float a1 = ex[k * 128 + r], a2 = ex[(4 + k) * 128 + r];
                M2 = fmaxf(fmaxf(M2, a2), fminf(M1, a1));
                M1 = fmaxf(M1, a1);
              }
            } else {
              M1 = fmaxf(ex[r], ex[128 + r]);
            }
            const bool flag = track && row_valid &&
                              neartie_flag((M1 - M2) * 0.69314718055994531f, qn, kmx, kDH);
            float lt = 0.f;
            if (!flag) {
              const uint64_t m12 = splat2(M1);
              float la = 0.f, lb = 0.f;  // two partial row sums
#pragma unroll
              for (int m = 0; m < NS; ++m) {
#pragma unroll
                for (int e = 0; e < 8; e += 2) {  // probabilities, in place (paired subtraction)
                  float a0, a1;
                  upk2(sub2(pk2(s[8 * m + e], s[8 * m + e + 1]), m12), a0, a1);
                  s[8 * m + e] = ex2_approx(a0);
                  s[8 * m + e + 1] = ex2_approx(a1);
                  la += s[8 * m + e];
                  lb += s[8 * m + e + 1];
                }
                int ho, lo;
                p_slot<T>(r, 8 * (gs + 2 * m), h & 1, ho, lo);
                if constexpr (p_hi_only<T>())
                  *reinterpret_cast<uint4*>(sm + ho) = pack8_hi(s + 8 * m, T());
                else
                  put8<T>(sm + ho, sm + lo, 0, s + 8 * m);
              }
              lt = la + lb;
            }
            if (g == 0) {
              // fp64 correction of this warp's flagged rows (rare)
              unsigned fl = __ballot_sync(0xffffffffu, flag);
              while (fl) {
                const int src = __ffs(fl) - 1;
                fl &= fl - 1;
                const int rr = qd * 32 + src;
                const float kmx_src = __shfl_sync(0xffffffffu, kmx, src);
                const float lrow = fixup_row<T, L>(sm, P, rr, rr / L, h, first, lane, kmx_src);
                if (lane == src) lt = lrow;
              }
            }
            l_s[(h * 4 + gs) * 128 + r] = lt;
            l_s[(h * 4 + gs + 2) * 128 + r] = 0.f;  // the context sums four slots
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive_n(bar + B_P_READY + (h & 1), 2);
          }
        } else
        for (int h = h0; h < h1 && ok; ++h) {
          // ---- softmax of S = Q_h K_h^T over the row's visible keys; this
          // group holds own chunks g + 4m (keys 8 (g + 4m) .. + 8)
          if (!wait(B_S_DONE, c_s)) { ok = false; break; }
          float s[8 * NM];
#pragma unroll
          for (int m = 0; m < NM; ++m) tmem_ld8_nw(trow + 384 + sq * L + 8 * (g + 4 * m), s + 8 * m);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(bar + B_S_FREE);
          // P_{h-1} V_{h-1} done before this head writes P or its exchange
          // slots (this loop keeps the one-buffer order for either type)
          if (!wait_o_upto(h - 1)) { ok = false; break; }
          if (h + 1 < h1) {
            // head h+1's Q, K (their buffers' reader S_h is done) and V (its
            // buffer's reader P_{h-1} V_{h-1} was just waited for), so that
            // S_{h+1} runs during this softmax
            convert_qk(h + 1, g < 2, g & 1);
            convert_v(h + 1, g);
            arrive(B_QKVH_READY);
            arrive(B_VH_READY + ((h + 1) & 1));
          }
          const float qn = sqrtf(qn2_s[((h & 1) * 2) * 128 + r] + qn2_s[((h & 1) * 2 + 1) * 128 + r]);
          const float kmx = sqrtf(__int_as_float(kmax_s[2 * h]) + __int_as_float(kmax_s[2 * h + 1]));
          // the second-best score matters only where fp32 scores can be off
          const bool track = neartie_err(qn, kmx, kDH) > kTieErrMin;
          float m1 = -INFINITY, m2 = -INFINITY;
#pragma unroll
          for (int m = 0; m < NM; ++m)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int kk = 8 * (g + 4 * m) + e;
              const float v = kk < limit ? s[8 * m + e] * scale_log2 : -INFINITY;
              s[8 * m + e] = v;
              m2 = fmaxf(m2, fminf(m1, v));
              m1 = fmaxf(m1, v);
            }
          ex[g * 128 + r] = m1;
          ex[(4 + g) * 128 + r] = m2;
          if (track) {
            // park the raw scores in this row's P slots for a possible fp64 fix-up
#pragma unroll
            for (int m = 0; m < NM; ++m) {
              uint4 hv, lv;
              uint32_t* hw = reinterpret_cast<uint32_t*>(&hv);
              uint32_t* lw = reinterpret_cast<uint32_t*>(&lv);
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                const uint32_t b0 = __float_as_uint(s[8 * m + 2 * w]), b1 = __float_as_uint(s[8 * m + 2 * w + 1]);
                hw[w] = (b0 >> 16) | (b1 & 0xFFFF0000u);
                lw[w] = (b0 & 0xFFFFu) | (b1 << 16);
              }
              int ho, lo;
              p_slot<T>(r, 8 * (g + 4 * m), h & 1, ho, lo);
              *reinterpret_cast<uint4*>(sm + ho) = hv;
              *reinterpret_cast<uint4*>(sm + lo) = lv;
            }
          }
          bar_compute();
          float M1 = -INFINITY, M2 = -INFINITY;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float a1 = ex[k * 128 + r], a2 = ex[(4 + k) * 128 + r];
            M2 = fmaxf(fmaxf(M2, a2), fminf(M1, a1));
            M1 = fmaxf(M1, a1);
          }
          const bool flag = track && row_valid &&
                            neartie_flag((M1 - M2) * 0.69314718055994531f, qn, kmx, kDH);
          float lt = 0.f;
          if (!flag) {
#pragma unroll
            for (int m = 0; m < NM; ++m) {
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                s[8 * m + e] = exp2f(s[8 * m + e] - M1);  // probabilities, in place
                lt += s[8 * m + e];
              }
              int ho, lo;
              p_slot<T>(r, 8 * (g + 4 * m), h & 1, ho, lo);
              if constexpr (p_hi_only<T>())
                *reinterpret_cast<uint4*>(sm + ho) = pack8_hi(s + 8 * m, T());
              else
                put8<T>(sm + ho, sm + lo, 0, s + 8 * m);
            }
          }
          if (g == 0) {
            // fp64 correction of this warp's flagged rows (rare)
            unsigned fl = __ballot_sync(0xffffffffu, flag);
            while (fl) {
              const int src = __ffs(fl) - 1;
              fl &= fl - 1;
              const int rr = qd * 32 + src;
              const float kmx_src = __shfl_sync(0xffffffffu, kmx, src);
              const float lrow = fixup_row<T, L>(sm, P, rr, rr / L, h, first, lane, kmx_src);
              if (lane == src) lt = lrow;
            }
          }
          l_s[(h * 4 + g) * 128 + r] = lt;
          arrive(B_P_READY + (h & 1));
        }
        if (!ok) break;
        // ---- ctx = O / l -> PB (hi, lo); group g takes head g, whose rows of
        // sequence s are in TMEM columns 96g + 32s
        // The layer's six LayerNorm vectors (b_o, ln1 gamma, beta, b_2, ln2
        // gamma, beta; 768 floats).  Plain kernel: loaded now, while the last
        // P V completes, and stored into the P area (unused from then on in
        // this layer) before CTX_READY, which with OUT_DONE orders them before
        // every LayerNorm read.  Assisted kernel: see below.
        const int ct = threadIdx.x - kCtrlWarps * 32;
        auto ln_vec = [&](int k) -> float {
          const int v6 = k >> 7, e = k & 127;
          const float* src = v6 == 0 ? P.b_o : v6 == 1 ? P.ln1_g : v6 == 2 ? P.ln1_b
                           : v6 == 3 ? P.b_2 : v6 == 4 ? P.ln2_g : P.ln2_b;
          return __ldg(src + e);
        };
        float lv0 = 0.f, lv1 = 0.f;
        if constexpr (!ASSIST) {
          lv0 = ln_vec(ct);
          lv1 = ct < 256 ? ln_vec(ct + 512) : 0.f;
        }
        if (!wait_o_upto(h1 - 1)) { ok = false; break; }
        // assisted R: its P and V buffers are free, H may send its context
        if (ASSIST && !helper && elected) signal_peer(B_PEER_PBFREE);
        if constexpr (!ASSIST) {
          // the last head's context (the conversion warps wrote the others
          // during the heads); every context store lands before CTX_READY
          TL_LNV[ct] = lv0;
          if (ct < 256) TL_LNV[ct + 512] = lv1;
          if (g >= 2) ctx_tmem(h1 - 1, g & 1);
          tmem_wait_st();
        } else if (g >= h0 && g < h1) {  // this group's head is one of this CTA's
          float o[32];
          tmem_ld32_nw(trow + 96 * g + 32 * sq, o);
          tmem_wait_ld();
          const float lsum = l_s[(g * 4) * 128 + r] + l_s[(g * 4 + 1) * 128 + r] +
                             l_s[(g * 4 + 2) * 128 + r] + l_s[(g * 4 + 3) * 128 + r];
          const float inv = 1.f / lsum;
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] *= inv;
          const int kh = g >> 1;
          // (H stages heads 2, 3 at the same place in its own buffer, which
          // its attention no longer uses, and sends both planes below)
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            put8<T>(pbuf + kh * kTile16, pbuf + (2 + kh) * kTile16, sw128(r, (g & 1) * 4 + cc), o + 8 * cc);
        }
        if (helper) {
          fence_proxy_async();  // the staged context is read by the bulk copy
          bar_compute();
          if (elected) {
            // once R is done with its P/V area: the hi and lo planes of
            // columns 64..127 into R's ctx buffer
            if (!wait_peer(B_PEER_PBFREE, c_pbfree)) { ok = false; break; }
            send_peer(pbuf + kTile16, kTile16, B_PEER_CTX);
            send_peer(pbuf + 3 * kTile16, kTile16, B_PEER_CTX);
            // H's X buffer is no longer read (its QKV products and every
            // fix-up of its heads are done): R may send y there
            signal_peer(B_PEER_XFREE);
            mbar_arrive_expect_tx(bar + B_PEER_Y, 4 * kTile16);
          }
          if (!wait_peer(B_PEER_Y, c_py)) { ok = false; break; }
        } else {
          // Assisted kernel: the vectors go to the softmax-sum area, free once
          // every thread has read its sums (CTX_READY precedes OUT_DONE): the
          // global loads are issued now and land during the out-projection.
          if constexpr (ASSIST) {
            lv0 = ln_vec(ct);
            lv1 = ct < 256 ? ln_vec(ct + 512) : 0.f;
          }
          arrive(B_CTX_READY);
          // ---- out-projection + b_o + residual x, LayerNorm 1 -> y in XA
          if (!wait(B_OUT_DONE, c_out)) { ok = false; break; }
          if constexpr (ASSIST) {
            l_s[ct] = lv0;
            if (ct < 256) l_s[ct + 512] = lv1;
            bar_compute();
          }
          float y[32];
          layernorm(ASSIST ? 128 : kTOut, TL_LNV, TL_LNV + 128, TL_LNV + 256, !first, false, y);
          // y -> TMEM [128, 256) as (hi, lo) words: group g holds K columns
          // [32g, 32g + 32).  Every group read its out-projection accumulator
          // (the same columns) before the LayerNorm's exchange barrier.
          uint32_t hw[16], lw[16];
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            split8(y + 8 * cc, *reinterpret_cast<uint4*>(hw + 4 * cc), *reinterpret_cast<uint4*>(lw + 4 * cc), T());
          tmem_st16(trow + kTY + 16 * g, hw);
          tmem_st16(trow + kTY + 64 + 16 * g, lw);
          tmem_wait_st();
          if (ASSIST) {
            // y into H's X buffer, the A operand of its FFN1 chunks: staged
            // in this CTA's X buffer (its residual x was read above, by this
            // same thread) and sent once H no longer reads its own
            const int kh = g >> 1;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
              put8<T>(xa + kh * kTile16, xa + (2 + kh) * kTile16, sw128(r, (g & 1) * 4 + cc), y + 8 * cc);
            fence_proxy_async();
            bar_compute();
            if (!wait_peer(B_PEER_XFREE, c_xfree)) { ok = false; break; }
            if (elected) send_peer(xa, 4 * kTile16, B_PEER_Y);
          }
        }
        arrive(B_Y_READY);
        // ---- FFN chunks (128 wide): h_c = gelu(acc1 + b_1) replaces acc1 in
        // its TMEM buffer as (hi, lo) words, the A operand of FFN2
        for (int c = c0; c < c1 && ok; ++c) {
          const int buf = c & 1;
          const uint32_t tb = kTF + 128 * buf;
          if (!wait(B_F1_DONE + buf, c_f1[buf])) { ok = false; break; }
          float hv[32];
          tmem_ld32_nw(trow + tb + 32 * g, hv);
          tmem_wait_ld();
          const float4* b4 = reinterpret_cast<const float4*>(vec_s + 384 + 128 * c + 32 * g);
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 b = b4[c4];  // + b_1 on the paired adds
            upk2(add2(pk2(hv[4 * c4 + 0], hv[4 * c4 + 1]), pk2(b.x, b.y)), hv[4 * c4 + 0], hv[4 * c4 + 1]);
            upk2(add2(pk2(hv[4 * c4 + 2], hv[4 * c4 + 3]), pk2(b.z, b.w)), hv[4 * c4 + 2], hv[4 * c4 + 3]);
            gelu_as7128_x2(hv[4 * c4 + 0], hv[4 * c4 + 1]);
            gelu_as7128_x2(hv[4 * c4 + 2], hv[4 * c4 + 3]);
          }
          // group g holds the chunk's K columns [32g, 32g + 32) and writes
          // their h words over its own accumulator columns (hi in the upper
          // 16, lo in the lower 16): no group writes another's columns, so no
          // barrier stands between the accumulator loads and these stores
          uint32_t hw[16], lw[16];
          if constexpr (h_hi_only<T>()) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) *reinterpret_cast<uint4*>(hw + 4 * cc) = pack8_hi(hv + 8 * cc, T());
            tmem_st16(trow + tb + 32 * g + 16, hw);
          } else {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
              split8(hv + 8 * cc, *reinterpret_cast<uint4*>(hw + 4 * cc), *reinterpret_cast<uint4*>(lw + 4 * cc), T());
            tmem_st16(trow + tb + 32 * g + 16, hw);
            tmem_st16(trow + tb + 32 * g, lw);
          }
          tmem_wait_st();
          arrive(B_H_READY);
        }
        if (!ok) break;
        // the next layer's vectors, staged once FFN2 is done
        const MegaLayer& Pn = a.layers[l + 1 < a.n_layers ? l + 1 : 0];
        const float nv0 = vec_val(Pn, TL_CV), nv1 = vec_val(Pn, TL_CV + kCompute);
        // assisted H: every FFN1 product of its chunks is done, so y in its X
        // buffer is no longer read; R may write the next layer's input there
        if (helper && elected) signal_peer(B_PEER_XFREE);
        // ---- FFN2 + b_2 + residual y, LayerNorm 2
        if (!wait(B_F2_DONE, c_f2)) { ok = false; break; }
        stage_vec(nv0, nv1);
        if (helper) {
          // the partial FFN2 sum over this CTA's chunks -> R's P/ctx area
          // (fp32 [row][128 columns]); R adds it before LayerNorm 2
          // staged in this CTA's P/ctx area (its context copy to R landed
          // before R sent y), then one 64 KB copy to the same place in R
          float v[32];
          tmem_ld32_nw(trow + 32 * g, v);
          tmem_wait_ld();
          float4* dst = reinterpret_cast<float4*>(pbuf + (size_t)(r * 128 + 32 * g) * 4);
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) dst[c4] = make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]);
          fence_proxy_async();
          bar_compute();
          if (elected) {
            send_peer(pbuf, 4 * kTile16, B_PEER_PART);
            if (l + 1 < a.n_layers) mbar_arrive_expect_tx(bar + B_PEER_X, 4 * kTile16);
          }
          if (l + 1 < a.n_layers) {
            // the next layer's input, sent by R into this CTA's X buffer
            if (!wait_peer(B_PEER_X, c_px)) { ok = false; break; }
            tc_fence_before();
            arrive(B_A_READY);
          }
        } else {
          if (ASSIST) {
            if (elected) mbar_arrive_expect_tx(bar + B_PEER_PART, 4 * kTile16);
            if (!wait_peer(B_PEER_PART, c_part)) { ok = false; break; }
          }
          float xo[32];
          layernorm(0, TL_LNV + 384, TL_LNV + 512, TL_LNV + 640, true, true, xo,
                    ASSIST ? reinterpret_cast<const float*>(pbuf) : nullptr);
          const int kh = g >> 1;
          // assisted: H's FFN1 no longer reads y -- so the copy of y out of
          // this CTA's X buffer is complete and H's X buffer may take the
          // next layer's input (waited every layer to keep the phases in step)
          if (ASSIST && !wait_peer(B_PEER_XFREE, c_xfree)) { ok = false; break; }
          if (l + 1 < a.n_layers) {
            // the next layer's input: X buffer (residual, fix-up) and TMEM
            // [384, 512) as (hi, lo) words, the A operand of its QKV product
            uint32_t hw[16], lw[16];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              put8<T>(xa + kh * kTile16, xa + (2 + kh) * kTile16, sw128(r, (g & 1) * 4 + cc), xo + 8 * cc);
              split8(xo + 8 * cc, *reinterpret_cast<uint4*>(hw + 4 * cc), *reinterpret_cast<uint4*>(lw + 4 * cc), T());
            }
            tmem_st16(trow + kTX + 16 * g, hw);
            tmem_st16(trow + kTX + 64 + 16 * g, lw);
            tmem_wait_st();
            if (ASSIST) {  // the same rows into H's X buffer
              fence_proxy_async();
              bar_compute();
              if (elected) send_peer(xa, 4 * kTile16, B_PEER_X);
            }
            arrive(B_A_READY);
          } else if (row_valid && grow < (size_t)T_rows) {
            T* dst = reinterpret_cast<T*>(a.out) + grow * kD + 32 * g;
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
              uint4 u;
              T* up = reinterpret_cast<T*>(&u);
#pragma unroll
              for (int e = 0; e < 8; ++e) up[e] = from_f32<T>(xo[c8 * 8 + e]);
              *reinterpret_cast<uint4*>(dst + c8 * 8) = u;
            }
          }
        }
      }
      if (!ok) break;
      tc_fence_before();
      mbar_arrive(bar + B_XA_FREE);  // the next tile's input may overwrite XA
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
#undef TL_T0
#undef TL_TSTEP
#undef TL_LNV
}

template <typename T, int L, bool ASSIST>
cudaError_t launch_l(const CUtensorMap& mx, const MegaArgs& a, int grid, cudaStream_t s) {
  auto k = mega_kernel<T, L, ASSIST>;
  const size_t smem = kSmemBytes + 1024;
  cudaError_t e = set_max_dyn_smem((const void*)k, smem);
  if (e != cudaSuccess) return e;
  if constexpr (ASSIST) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, mx, a);
  } else {
    k<<<grid, kThreads, smem, s>>>(mx, a);
    return cudaGetLastError();
  }
}

}  // namespace

bool mega_supported(int d, int H, int dff, int L, tl_dtype dt) {
  return d == kD && H == kH && dff % 128 == 0 && dff >= 128 && dff <= kMaxDff &&
         L == 64 && dt != TL_F32;
}

bool mega_assisted(int B, int L, int dff, int num_sms, int setting) {
  const int tiles = (B + (128 / L) - 1) / (128 / L);
  const bool possible = dff >= 256 && 2 * tiles <= num_sms;  // every CTA gets a helper
  // Automatic (-1) is off: on GB300 the assisted forward measured within
  // 2% of one CTA per tile (0.140-0.142 vs 0.142-0.146 ms for 1-152
  // sequences of the d128 workload), not worth a second SM per tile.
  return possible && setting == 1;
}

cudaError_t mega_forward(const void* x, const MegaArgs& a, int L, bool bf16, int num_sms, cudaStream_t s) {
  CUtensorMap mx;
  if (!make_tmap_2d(&mx, x, bf16, (uint64_t)a.B * L, kD, kD, 64, 128, 128)) return cudaErrorInvalidValue;
  const int S = 128 / L;
  const int tiles = (a.B + S - 1) / S;
  if (mega_assisted(a.B, L, a.dff, num_sms, a.assist)) {
    const int grid = 2 * tiles;  // one cluster (resident + helper) per tile
    return bf16 ? launch_l<__nv_bfloat16, 64, true>(mx, a, grid, s) : launch_l<__half, 64, true>(mx, a, grid, s);
  }
  const int grid = tiles < num_sms ? tiles : num_sms;
  if (bf16) {
    return launch_l<__nv_bfloat16, 64, false>(mx, a, grid, s);
  }
  return launch_l<__half, 64, false>(mx, a, grid, s);
}

}  // namespace tl
