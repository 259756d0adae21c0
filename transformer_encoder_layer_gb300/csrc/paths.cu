// Shape dispatch (the frozen plan table) and the launch sequence of each path.
#include "common.cuh"
#include "internal.h"
#include "paths.h"

namespace tl {
namespace {

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Workspace of the SIMT path: fp32 activations of one layer.
struct SimtWs {
  float *resid, *qkv, *ctx, *r, *y, *hid;
  int* ties;  // [0] count, then the list
  size_t bytes;
};

SimtWs simt_layout(const tl_encoder* h, int B, int L, void* base) {
  const size_t T = (size_t)B * L;
  size_t off = 0;
  auto take = [&](size_t n) { size_t at = off; off = align256(off + n * 4); return at; };
  size_t o_resid = take(T * h->d), o_qkv = take(3 * T * h->d), o_ctx = take(T * h->d),
         o_r = take(T * h->d), o_y = take(T * h->d), o_h = take(T * h->dff),
         o_t = take(1 + T * h->H);
  char* b = (char*)base;
  SimtWs w;
  w.resid = (float*)(b + o_resid); w.qkv = (float*)(b + o_qkv); w.ctx = (float*)(b + o_ctx);
  w.r = (float*)(b + o_r); w.y = (float*)(b + o_y); w.hid = (float*)(b + o_h);
  w.ties = (int*)(b + o_t);
  w.bytes = off;
  return w;
}

cudaError_t run_simt(tl_encoder* h, const void* x, int B, int L, const int32_t* vl, void* out,
                     void* ws, cudaStream_t s) {
  SimtWs w = simt_layout(h, B, L, ws);
  const int M = B * L, d = h->d;
  const size_t plane = (size_t)M * d;
  const void* cur = x;
  tl_dtype cur_t = h->dtype;
  cudaError_t e = cudaSuccess;
  for (int l = 0; l < h->n_layers && e == cudaSuccess; ++l) {
    const tl_layer_dev& P = h->layers[l];
    SimtGemmArgs g{};
    g.B = B; g.L = L; g.H = h->H; g.dh = h->dh; g.w_dtype = h->dtype;
    // a1: fused QKV projection, head-major epilogue.
    g.A = cur; g.a_dtype = cur_t; g.W = P.w_qkv; g.bias = P.b_qkv; g.out = w.qkv;
    g.M = M; g.N = 3 * d; g.K = d; g.epi = EPI_QKV_HEADMAJOR;
    { KernelTimer t(h, KC_SIMT_GEMM_QKV, s); e = simt_gemm(g, s); }
    if (e != cudaSuccess) break;
    // a2: masked attention, then the fp64 fix-up of near-tie rows.
    NearTieList ties{w.ties, w.ties + 1, M * h->H};
    if ((e = cudaMemsetAsync(w.ties, 0, sizeof(int), s)) != cudaSuccess) break;
    { KernelTimer t(h, KC_SIMT_ATTENTION, s);
      e = simt_attention(w.qkv, w.qkv + plane, w.qkv + 2 * plane, vl, w.ctx, B, h->H, L, h->dh,
                         h->status, ties, s); }
    if (e != cudaSuccess) break;
    {
      FixupArgs fa{};
      fa.ties = ties;
      fa.x = Plane{cur, nullptr, cur_t == TL_F32 ? 0 : (cur_t == TL_F16 ? 1 : 2)};
      fa.w_qkv = P.w_qkv; fa.w_kind = (int)h->dtype; fa.b_qkv = P.b_qkv;
      fa.q = Plane{w.qkv, nullptr, 0}; fa.k = Plane{w.qkv + plane, nullptr, 0};
      fa.v = Plane{w.qkv + 2 * plane, nullptr, 0};
      fa.v_transposed = 0; fa.Lp = L;
      fa.ctx_hi = w.ctx; fa.ctx_kind = 0; fa.valid_len = vl;
      fa.B = B; fa.H = h->H; fa.L = L; fa.dh = h->dh; fa.d = d;
      KernelTimer t(h, KC_AUX, s);
      if ((e = neartie_fixup(fa, s)) != cudaSuccess) break;
    }
    // a3: out-projection + bias + residual, then LayerNorm 1.
    g.A = w.ctx; g.a_dtype = TL_F32; g.W = P.w_o; g.bias = P.b_o; g.resid = cur; g.r_dtype = cur_t;
    g.out = w.r; g.N = d; g.K = d; g.epi = EPI_BIAS_RESID;
    { KernelTimer t(h, KC_SIMT_GEMM_OUT, s); e = simt_gemm(g, s); }
    if (e != cudaSuccess) break;
    { KernelTimer t(h, KC_SIMT_LAYERNORM, s); e = simt_layernorm(w.r, P.ln1_g, P.ln1_b, w.y, nullptr, TL_F32, M, d, s); }
    if (e != cudaSuccess) break;
    // a4: FFN1 + bias + exact GELU.
    g.A = w.y; g.W = P.w_1; g.bias = P.b_1; g.out = w.hid; g.N = h->dff; g.K = d; g.epi = EPI_BIAS_GELU;
    { KernelTimer t(h, KC_SIMT_GEMM_FFN1, s); e = simt_gemm(g, s); }
    if (e != cudaSuccess) break;
    // a5: FFN2 + bias + residual, then LayerNorm 2.
    g.A = w.hid; g.W = P.w_2; g.bias = P.b_2; g.resid = w.y; g.r_dtype = TL_F32; g.out = w.r;
    g.N = d; g.K = h->dff; g.epi = EPI_BIAS_RESID;
    { KernelTimer t(h, KC_SIMT_GEMM_FFN2, s); e = simt_gemm(g, s); }
    if (e != cudaSuccess) break;
    const bool last = l == h->n_layers - 1;
    KernelTimer t(h, KC_SIMT_LAYERNORM, s);
    e = simt_layernorm(w.r, P.ln2_g, P.ln2_b, last ? nullptr : w.resid, last ? out : nullptr,
                       h->dtype, M, d, s);
    cur = w.resid;
    cur_t = TL_F32;
  }
  return e;
}

}  // namespace

size_t packed_extra_bytes(const tl_encoder*) { return 0; }
cudaError_t pack_extra(tl_encoder*, void*, size_t) { return cudaSuccess; }

tl_path choose_path(const tl_encoder* h, int B, int L) {
  (void)B; (void)L;
  switch (h->path) {
    case TL_PATH_SIMT:
    case TL_PATH_AUTO:
      return TL_PATH_SIMT;
    default:
      return TL_PATH_AUTO;  // not built for this shape
  }
}

size_t path_workspace_bytes(const tl_encoder* h, tl_path p, int B, int L) {
  if (p == TL_PATH_SIMT) return simt_layout(h, B, L, nullptr).bytes;
  return 0;
}

cudaError_t run_path(tl_encoder* h, tl_path p, const void* x, int B, int L, const int32_t* vl,
                     void* out, void* ws, cudaStream_t s) {
  if (p == TL_PATH_SIMT) return run_simt(h, x, B, L, vl, out, ws, s);
  return cudaErrorInvalidValue;
}

}  // namespace tl
