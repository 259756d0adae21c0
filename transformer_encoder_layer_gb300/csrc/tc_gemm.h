// Host interface of the tcgen05 GEMM with fused epilogues (tc_gemm.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tl {

enum TcEpi { TC_EPI_QKV = 0, TC_EPI_GELU = 1, TC_EPI_LN = 2 };

constexpr int kTcGemmSmemBudget = 200 * 1024;

// Arguments of one GEMM launch.  16-bit pointers are of the I/O type
// (fp16 or bf16).  Fields marked (set by tc_gemm) are computed on the host.
struct TcGemmArgs {
  int M, N, K;
  int BN;        // N tile: a multiple of 32 in [32, 256] dividing N
  int n_parts;   // A planes: 1 (exact 16-bit input) or 2 (hi, lo)
  int pair;      // 1: CTA pairs on 256-row blocks (tcgen05 cta_group::2); the
                 // W map's box is then BN/2 rows (tc_gemm_pair_ok must hold)
  int n_tiles, m_blocks, stages, tmem_cols;  // (set by tc_gemm)
  uint32_t idesc;                            // (set by tc_gemm)
  const float* bias;  // [N]
  // TC_EPI_QKV: head-major (hi, lo) planes; V transposed with row pitch Lp.
  void *q_hi, *q_lo, *k_hi, *k_lo, *vt_hi, *vt_lo;
  int B, L, H, dh, Lp;
  int* kmax;     // [B*H] max |k_j| per plane as float bits (atomicMax), or null
  // TC_EPI_GELU: (hi, lo) planes [M, N].  TC_EPI_LN: optional (hi, lo) out.
  void *o_hi, *o_lo;
  // TC_EPI_LN
  // [M, N]: fp32 (resid_kind 0), the 16-bit type (1), or the hi plane of a
  // (hi, lo) pair of the 16-bit type whose lo plane is resid_lo (2)
  const void* resid;
  const void* resid_lo;
  int resid_kind;
  const float *gamma, *beta;
  float* o32;         // optional fp32 [M, N]
  void* o_final;      // optional 16-bit [M, N] (the stack's output)
  float* rscratch;    // fp32 [M, N] pre-LN rows when N > BN
  // When N > BN and row_stats is set, every (row block, N tile) is a work
  // unit of its own: the epilogue writes the pre-LN rows to rscratch and,
  // per row, the (mean, M2) of each of tc_gemm_ln_parts(N, BN, pair) equal column
  // blocks here; ln_apply merges them and normalises (the outputs above are
  // not written by the GEMM).
  float2* row_stats;  // [M][tc_gemm_ln_parts(N, BN, pair)] or null
  int* status;
};

int tc_gemm_stages(int BN, int n_parts, bool pair);
size_t tc_gemm_smem_bytes(int BN, int n_parts, int stages, bool pair);
// Whether the CTA-pair variant can run M rows with N tile BN.
bool tc_gemm_pair_ok(int M, int BN);

// map_a0/map_a1: A planes [M, K] (box 64 x 128), map_w: W [N, K] (box
// 64 x BN, or 64 x BN/2 with pair), all 128-byte swizzled.  map_a1 is
// ignored when n_parts == 1.
// Column blocks per row whose (mean, M2) an LN GEMM with N > BN writes (on
// CTA pairs or not).
int tc_gemm_ln_parts(int N, int BN, bool pair);

cudaError_t tc_gemm(const CUtensorMap& map_a0, const CUtensorMap& map_a1, const CUtensorMap& map_w,
                    TcGemmArgs a, bool bf16, int epi, int num_sms, cudaStream_t s);

// Tensor map of a row-major 2-D array of 16-bit elements [rows, cols] with
// row pitch `pitch_elems`, box (box_cols x box_rows) and the given swizzle
// (32, 64 or 128 bytes).  Returns false if the driver rejects it.
bool make_tmap_2d(CUtensorMap* map, const void* ptr, bool bf16, uint64_t rows, uint64_t cols,
                  uint64_t pitch_elems, uint32_t box_cols, uint32_t box_rows, int swizzle_bytes);

}  // namespace tl
