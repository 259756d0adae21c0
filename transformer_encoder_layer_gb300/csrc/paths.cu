// Shape dispatch (the frozen plan table) and the launch sequence of each path.
#include "common.cuh"
#include "internal.h"
#include "paths.h"

#include <algorithm>
#include <vector>
#include "dag.h"
#include "mega.h"
#include "mega_simt.h"
#include "tc_attention.h"
#include "ln_apply.h"
#include "tc_gemm.h"

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
      AttnIO io{w.qkv, nullptr, w.qkv + plane, nullptr, w.qkv + 2 * plane, nullptr, 0, L,
                w.ctx, nullptr};
      e = simt_attention(io, 0, vl, B, h->H, L, h->dh, h->status, ties, s); }
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

// ---------------------------------------------------------------- LAYERED
// tcgen05 GEMMs with fused epilogues; activations between steps are (hi, lo)
// 16-bit planes so every GEMM operand keeps about fp32 accuracy.
// Largest N tile (a multiple of 32 and of `unit`, at most 256) dividing n.
int pick_bn(int n, int unit = 32) {
  for (int bn = 256; bn >= 32; bn -= 32)
    if (n % bn == 0 && bn % unit == 0) return bn;
  return 0;
}

bool layered_supported(const tl_encoder* h) {
  if (h->dtype == TL_F32) return false;
  const int d = h->d, dh = h->dh;
  // K of every GEMM a multiple of the 64-wide TMA box; N tiles of 32 columns.
  if (d % 64 || h->dff % 64) return false;
  if (!(dh % 32 == 0 || 32 % dh == 0)) return false;
  return pick_bn(3 * d, dh > 32 ? dh : 32) > 0;
}


struct LayeredWs {
  void *xh, *xl, *qh, *ql, *kh, *kl, *vth, *vtl, *ch, *cl, *yh, *yl, *hh, *hl;
  float* rs;
  float2* stats;  // per-row (mean, rstd) of the LN GEMMs when d spans several N tiles
  int* ties;
  int* kmax;
  void* att_part;  // split-K attention: partial states and arrival counters
  void* att_cnt;
  int Lp;
  size_t bytes;
};

LayeredWs layered_layout(const tl_encoder* h, int B, int L, void* base) {
  const size_t T = (size_t)B * L, d = h->d;
  const int Lp = (L + 7) / 8 * 8;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t at = off; off = align256(off + bytes); return at; };
  char* b = (char*)base;
  LayeredWs w;
  w.Lp = Lp;
  const size_t e = 2;
  size_t o[17];
  o[0] = take(T * d * e); o[1] = take(T * d * e);                          // x hi/lo
  o[2] = take(T * d * e); o[3] = take(T * d * e);                          // q
  o[4] = take(T * d * e); o[5] = take(T * d * e);                          // k
  o[6] = take((size_t)B * d * Lp * e); o[7] = take((size_t)B * d * Lp * e);  // v^T
  o[8] = take(T * d * e); o[9] = take(T * d * e);                          // ctx
  o[10] = take(T * d * e); o[11] = take(T * d * e);                        // y
  o[12] = take(T * h->dff * e); o[13] = take(T * h->dff * e);              // ffn hidden
  o[16] = take(d > 256 ? T * d * 4 : 4);                                   // LN scratch
  const size_t ost = take(d > 256 ? T * 8 : 8);                            // LN row stats
  size_t ot = take((1 + T * h->H) * 4);
  size_t ok_ = take((size_t)B * h->H * 4);
  const TcAttnSplit sp = tc_attention_supported(h->dh) && !h->simt_attention
                             ? tc_attention_split_plan(B, h->H, L, h->dh, h->num_sms, h->attn_split)
                             : TcAttnSplit{};
  size_t oap = take(sp.part_bytes ? sp.part_bytes : 4);
  size_t oac = take(sp.cnt_bytes ? sp.cnt_bytes : 4);
  void** p[14] = {&w.xh, &w.xl, &w.qh, &w.ql, &w.kh, &w.kl, &w.vth, &w.vtl, &w.ch, &w.cl,
                  &w.yh, &w.yl, &w.hh, &w.hl};
  for (int i = 0; i < 14; ++i) *p[i] = b + o[i];
  w.rs = (float*)(b + o[16]);
  w.stats = (float2*)(b + ost);
  w.ties = (int*)(b + ot);
  w.kmax = (int*)(b + ok_);
  w.att_part = b + oap;
  w.att_cnt = b + oac;
  w.bytes = off;
  return w;
}

cudaError_t run_layered(tl_encoder* h, const void* x, int B, int L, const int32_t* vl, void* out,
                        void* ws, cudaStream_t s) {
  LayeredWs w = layered_layout(h, B, L, ws);
  const int M = B * L, d = h->d, dff = h->dff, H = h->H, dh = h->dh;
  const bool bf = h->dtype == TL_BF16;
  const int pk = bf ? 4 : 3;  // (hi, lo) plane kind for the fix-up
  cudaError_t e = cudaSuccess;
  CUtensorMap ma0, ma1, mw;
  auto amaps = [&](const void* p0, const void* p1, int rows, int K) {
    bool ok = make_tmap_2d(&ma0, p0, bf, rows, K, K, 64, 128, 128);
    ok = ok && make_tmap_2d(&ma1, p1 ? p1 : p0, bf, rows, K, K, 64, 128, 128);
    return ok;
  };
  // Rows wider than one N tile: the LN GEMM left pre-normalised rows and
  // their statistics; normalise them into the GEMM's output buffers.
  auto apply_ln = [&](const TcGemmArgs& g) -> cudaError_t {
    if (!g.row_stats) return cudaSuccess;
    LnApplyArgs la{w.rs, w.stats, g.gamma, g.beta, M, d, g.o32, g.o_hi, g.o_lo, g.o_final};
    KernelTimer t(h, KC_LN_APPLY, s);
    return ln_apply(la, bf, h->num_sms, s);
  };
  for (int l = 0; l < h->n_layers; ++l) {
    const tl_layer_dev& P = h->layers[l];
    const bool first = l == 0, last = l == h->n_layers - 1;
    // a1: fused QKV projection, head-major (hi, lo) epilogue.
    {
      TcGemmArgs g{};
      g.M = M; g.N = 3 * d; g.K = d; g.BN = pick_bn(3 * d, dh > 32 ? dh : 32); g.n_parts = first ? 1 : 2;
      g.bias = P.b_qkv;
      g.q_hi = w.qh; g.q_lo = w.ql; g.k_hi = w.kh; g.k_lo = w.kl; g.vt_hi = w.vth; g.vt_lo = w.vtl;
      g.B = B; g.L = L; g.H = H; g.dh = dh; g.Lp = w.Lp; g.status = h->status;
      g.kmax = w.kmax;
      if ((e = cudaMemsetAsync(w.kmax, 0, (size_t)B * H * 4, s)) != cudaSuccess) return e;
      if (!amaps(first ? x : w.xh, first ? nullptr : w.xl, M, d) ||
          !make_tmap_2d(&mw, P.w_qkv, bf, 3 * d, d, d, 64, g.BN, 128))
        return cudaErrorInvalidValue;
      KernelTimer t(h, KC_TC_GEMM_QKV, s);
      if ((e = tc_gemm(ma0, ma1, mw, g, bf, TC_EPI_QKV, h->num_sms, s)) != cudaSuccess) return e;
    }
    // a2: masked attention (ctx as (hi, lo) planes), then the near-tie fix-up.
    NearTieList ties{w.ties, w.ties + 1, M * H};
    if ((e = cudaMemsetAsync(w.ties, 0, sizeof(int), s)) != cudaSuccess) return e;
    if (tc_attention_supported(dh) && !h->simt_attention) {
      TcAttnArgs ta{w.qh, w.ql, w.kh, w.kl, w.vth, w.vtl, w.ch, w.cl, vl, w.kmax, ties,
                    B, H, L, w.Lp, dh, d, h->status};
      KernelTimer t(h, KC_TC_ATTENTION, s);
      if ((e = tc_attention(ta, bf, h->num_sms, h->attn_split, w.att_part, w.att_cnt, s)) != cudaSuccess)
        return e;
    } else {
      AttnIO io{w.qh, w.ql, w.kh, w.kl, w.vth, w.vtl, 1, w.Lp, w.ch, w.cl};
      KernelTimer t(h, KC_SIMT_ATTENTION, s);
      if ((e = simt_attention(io, bf ? 2 : 1, vl, B, H, L, dh, h->status, ties, s)) != cudaSuccess) return e;
    }
    {
      FixupArgs fa{};
      fa.ties = ties;
      fa.x = first ? Plane{x, nullptr, bf ? 2 : 1} : Plane{w.xh, w.xl, pk};
      fa.w_qkv = P.w_qkv; fa.w_kind = (int)h->dtype; fa.b_qkv = P.b_qkv;
      fa.q = Plane{w.qh, w.ql, pk}; fa.k = Plane{w.kh, w.kl, pk}; fa.v = Plane{w.vth, w.vtl, pk};
      fa.v_transposed = 1; fa.Lp = w.Lp;
      fa.ctx_hi = w.ch; fa.ctx_lo = w.cl; fa.ctx_kind = pk; fa.valid_len = vl;
      fa.B = B; fa.H = H; fa.L = L; fa.dh = dh; fa.d = d;
      KernelTimer t(h, KC_AUX, s);
      if ((e = neartie_fixup(fa, s)) != cudaSuccess) return e;
    }
    // a3: out-projection + bias + residual + LayerNorm 1.
    {
      TcGemmArgs g{};
      g.M = M; g.N = d; g.K = d; g.BN = pick_bn(d); g.n_parts = 2; g.bias = P.b_o;
      // residual: the stack input, then the previous layer's (hi, lo) output
      g.resid = first ? x : (const void*)w.xh; g.resid_lo = first ? nullptr : w.xl;
      g.resid_kind = first ? 1 : 2;
      g.gamma = P.ln1_g; g.beta = P.ln1_b; g.o_hi = w.yh; g.o_lo = w.yl;
      g.rscratch = w.rs; g.status = h->status;
      if (d > g.BN) g.row_stats = w.stats;
      if (!amaps(w.ch, w.cl, M, d) || !make_tmap_2d(&mw, P.w_o, bf, d, d, d, 64, g.BN, 128))
        return cudaErrorInvalidValue;
      {
        KernelTimer t(h, KC_TC_GEMM_OUT_LN, s);
        if ((e = tc_gemm(ma0, ma1, mw, g, bf, TC_EPI_LN, h->num_sms, s)) != cudaSuccess) return e;
      }
      if ((e = apply_ln(g)) != cudaSuccess) return e;
    }
    // a4: FFN1 + bias + exact GELU.
    {
      TcGemmArgs g{};
      g.M = M; g.N = dff; g.K = d; g.BN = pick_bn(dff); g.n_parts = 2; g.bias = P.b_1;
      g.o_hi = w.hh; g.o_lo = w.hl; g.status = h->status;
      if (!amaps(w.yh, w.yl, M, d) || !make_tmap_2d(&mw, P.w_1, bf, dff, d, d, 64, g.BN, 128))
        return cudaErrorInvalidValue;
      KernelTimer t(h, KC_TC_GEMM_FFN1, s);
      if ((e = tc_gemm(ma0, ma1, mw, g, bf, TC_EPI_GELU, h->num_sms, s)) != cudaSuccess) return e;
    }
    // a5: FFN2 + bias + residual + LayerNorm 2.
    {
      TcGemmArgs g{};
      g.M = M; g.N = d; g.K = dff; g.BN = pick_bn(d); g.n_parts = 2; g.bias = P.b_2;
      g.resid = w.yh; g.resid_lo = w.yl; g.resid_kind = 2; g.gamma = P.ln2_g; g.beta = P.ln2_b;
      if (last) {
        g.o_final = out;
      } else {
        g.o_hi = w.xh; g.o_lo = w.xl;
      }
      g.rscratch = w.rs; g.status = h->status;
      if (d > g.BN) g.row_stats = w.stats;
      if (!amaps(w.hh, w.hl, M, dff) || !make_tmap_2d(&mw, P.w_2, bf, d, dff, dff, 64, g.BN, 128))
        return cudaErrorInvalidValue;
      {
        KernelTimer t(h, KC_TC_GEMM_FFN2_LN, s);
        if ((e = tc_gemm(ma0, ma1, mw, g, bf, TC_EPI_LN, h->num_sms, s)) != cudaSuccess) return e;
      }
      if ((e = apply_ln(g)) != cudaSuccess) return e;
    }
  }
  return e;
}


// ------------------------------------------------------------------- DAG
// fp32 workspace of the task-graph kernel; the counters come first so one
// small memset per forward resets them.
struct DagWs {
  int* cnt;
  float *xs0, *xs1, *q, *k, *v, *ctx, *y, *hb, *part;
  int RB;
  size_t cnt_bytes, bytes;
};

DagWs dag_layout(const tl_encoder* h, int B, int L, void* base) {
  const size_t T = (size_t)B * L, d = h->d;
  DagWs w;
  w.RB = (int)((T + kDagRows - 1) / kDagRows);
  const int kc_max = (int)((std::max(h->d, h->dff) + kDagKChunk - 1) / kDagKChunk);
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t at = off; off = align256(off + bytes); return at; };
  char* b = (char*)base;
  w.cnt_bytes = (size_t)dag_counter_ints(h->n_layers, w.RB) * 4;
  size_t oc = take(w.cnt_bytes);
  size_t o[10];
  for (int i = 0; i < 8; ++i) o[i] = take(T * d * 4);  // xs0 xs1 q k v ctx y (+1 spare slot)
  o[8] = take(T * h->dff * 4);
  o[9] = take((size_t)kc_max * T * d * 4);
  w.cnt = (int*)(b + oc);
  w.xs0 = (float*)(b + o[0]); w.xs1 = (float*)(b + o[1]); w.q = (float*)(b + o[2]);
  w.k = (float*)(b + o[3]); w.v = (float*)(b + o[4]); w.ctx = (float*)(b + o[5]);
  w.y = (float*)(b + o[6]); w.hb = (float*)(b + o[8]); w.part = (float*)(b + o[9]);
  w.bytes = off;
  return w;
}

bool dag_ok(const tl_encoder* h) { return dag_supported(h->d, h->H, h->dff, h->n_layers, h->dtype); }

cudaError_t run_dag(tl_encoder* h, const void* x, int B, int L, const int32_t* vl, void* out,
                    void* ws, cudaStream_t s) {
  DagWs w = dag_layout(h, B, L, ws);
  DagArgs a{};
  for (int l = 0; l < h->n_layers; ++l) a.layers[l] = h->layers[l];
  a.n_layers = h->n_layers;
  a.x = (const float*)x; a.out = (float*)out; a.vl = vl;
  a.xs0 = w.xs0; a.xs1 = w.xs1; a.q = w.q; a.k = w.k; a.v = w.v; a.ctx = w.ctx; a.y = w.y;
  a.hb = w.hb; a.part = w.part;
  a.cnt = w.cnt;
  const int nc = dag_counter_ints(h->n_layers, w.RB);
  a.head = w.cnt + nc - 2;
  a.abort = w.cnt + nc - 1;
  a.status = h->status;
  a.B = B; a.L = L; a.T = B * L; a.RB = w.RB; a.d = h->d; a.H = h->H; a.dh = h->dh; a.dff = h->dff;
  a.inject_stall = h->dag_inject_stall ? 1 : 0;
  cudaError_t e = cudaMemsetAsync(w.cnt, 0, w.cnt_bytes, s);
  if (e != cudaSuccess) return e;
  KernelTimer t(h, KC_DAG, s);
  return dag_forward(a, h->num_sms, s);
}

}  // namespace

// Packed extras: per layer four weight tensor maps (for the megakernel's TMA
// loads, which need them in device memory) followed by the MegaLayer array.
// For the megakernel: per layer four weight tensor maps and a MegaLayer,
// then a copy of W_qkv with its rows regrouped head by head (q_h, k_h, v_h
// of head h are rows [96h, 96h + 96)), so that each head's projections land
// in adjacent TMEM columns.
size_t packed_extra_bytes(const tl_encoder* h) {
  if (h->dtype == TL_F32 || h->d != 128) return 0;
  return (size_t)h->n_layers * (4 * sizeof(CUtensorMap) + sizeof(MegaLayer) + 3 * 128 * 128 * 2) + 2048;
}

cudaError_t pack_extra(tl_encoder* h, void* dst, size_t bytes) {
  if (bytes == 0) return cudaSuccess;
  const bool bf = h->dtype == TL_BF16;
  const int d = h->d, dff = h->dff, nl = h->n_layers;
  char* base = (char*)(((uintptr_t)dst + 63) & ~(uintptr_t)63);
  CUtensorMap* maps_dev = (CUtensorMap*)base;
  MegaLayer* layers_dev = (MegaLayer*)(base + (size_t)nl * 4 * sizeof(CUtensorMap));
  char* wperm = (char*)(((uintptr_t)(layers_dev + nl) + 1023) & ~(uintptr_t)1023);
  const size_t wq_bytes = (size_t)3 * d * d * 2;
  std::vector<CUtensorMap> maps(4 * (size_t)nl);
  std::vector<MegaLayer> ml(nl);
  const int H = h->H, dh = h->dh;
  for (int l = 0; l < nl; ++l) {
    const tl_layer_dev& P = h->layers[l];
    char* wq = wperm + (size_t)l * wq_bytes;
    for (int hh = 0; hh < H; ++hh)
      for (int part = 0; part < 3; ++part) {
        const size_t rows = dh, row_bytes = (size_t)d * 2;
        cudaError_t e = cudaMemcpy(wq + (size_t)(3 * dh * hh + dh * part) * row_bytes,
                                   (const char*)P.w_qkv + (size_t)(part * d + dh * hh) * row_bytes,
                                   rows * row_bytes, cudaMemcpyDeviceToDevice);
        if (e != cudaSuccess) return e;
      }
    bool ok = make_tmap_2d(&maps[4 * l + 0], wq, bf, 3 * d, d, d, 64, 128, 128) &&
              make_tmap_2d(&maps[4 * l + 1], P.w_o, bf, d, d, d, 64, 128, 128) &&
              make_tmap_2d(&maps[4 * l + 2], P.w_1, bf, dff, d, d, 64, 128, 128) &&
              make_tmap_2d(&maps[4 * l + 3], P.w_2, bf, d, dff, dff, 64, 128, 128);
    if (!ok) return cudaSuccess;  // the megakernel path stays unavailable
    MegaLayer& m = ml[l];
    m.map_qkv = maps_dev + 4 * l + 0; m.map_o = maps_dev + 4 * l + 1;
    m.map_1 = maps_dev + 4 * l + 2; m.map_2 = maps_dev + 4 * l + 3;
    m.w_qkv = P.w_qkv; m.b_qkv = P.b_qkv; m.b_o = P.b_o; m.ln1_g = P.ln1_g; m.ln1_b = P.ln1_b;
    m.b_1 = P.b_1; m.b_2 = P.b_2; m.ln2_g = P.ln2_g; m.ln2_b = P.ln2_b;
  }
  cudaError_t e = cudaMemcpy(maps_dev, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(layers_dev, ml.data(), ml.size() * sizeof(MegaLayer), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) h->mega_layers = layers_dev;
  return e;
}

bool mega_ok(const tl_encoder* h, int L) {
  if (h->dtype == TL_F32) return mega_simt_supported(h->d, h->H, h->dff, L, h->n_layers, h->dtype);
  return h->mega_layers != nullptr && mega_supported(h->d, h->H, h->dff, L, h->dtype);
}

tl_path choose_path(const tl_encoder* h, int B, int L) {
  // Row counts (B * L) and row-by-head counts are int in the kernels and
  // their launch arithmetic; refuse token counts that could overflow them.
  if ((long long)B * L > (1LL << 30) || (long long)B * L * h->H > (1LL << 31) - 1)
    return TL_PATH_AUTO;
  switch (h->path) {
    case TL_PATH_SIMT:
      return TL_PATH_SIMT;
    case TL_PATH_LAYERED:
      return layered_supported(h) ? TL_PATH_LAYERED : TL_PATH_AUTO;
    case TL_PATH_MEGA:
      return mega_ok(h, L) ? TL_PATH_MEGA : TL_PATH_AUTO;
    case TL_PATH_DAG:
      return dag_ok(h) ? TL_PATH_DAG : TL_PATH_AUTO;
    case TL_PATH_AUTO:
      // The frozen plan table: short sequences of the d_model = 128 family
      // (16-bit, tensor cores) and of small fp32 models (d_model <= 64, CUDA
      // cores) stay resident in one CTA for the whole stack; other 16-bit shapes
      // run the layered tensor-core path; fp32 I/O keeps fp32 weights, which
      // the 16-bit MMAs cannot hold exactly, and runs on the CUDA cores: in
      // one task-graph launch while the tokens fill a few waves of 64-row
      // tiles, else layer by layer.
      if (mega_ok(h, L)) return TL_PATH_MEGA;
      if (dag_ok(h) && (long long)B * L <= kDagAutoMaxTokens) return TL_PATH_DAG;
      return layered_supported(h) ? TL_PATH_LAYERED : TL_PATH_SIMT;
    default:
      return TL_PATH_AUTO;  // not built for this shape
  }
}

size_t path_workspace_bytes(const tl_encoder* h, tl_path p, int B, int L) {
  if (p == TL_PATH_SIMT) return simt_layout(h, B, L, nullptr).bytes;
  if (p == TL_PATH_LAYERED) return layered_layout(h, B, L, nullptr).bytes;
  if (p == TL_PATH_DAG) return dag_layout(h, B, L, nullptr).bytes;
  return 0;  // the megakernel needs no scratch memory
}

cudaError_t run_path(tl_encoder* h, tl_path p, const void* x, int B, int L, const int32_t* vl,
                     void* out, void* ws, cudaStream_t s) {
  if (p == TL_PATH_SIMT) return run_simt(h, x, B, L, vl, out, ws, s);
  if (p == TL_PATH_LAYERED) return run_layered(h, x, B, L, vl, out, ws, s);
  if (p == TL_PATH_DAG) return run_dag(h, x, B, L, vl, out, ws, s);
  if (p == TL_PATH_MEGA && h->dtype == TL_F32) {
    MegaSimtArgs a{};
    for (int l = 0; l < h->n_layers; ++l) a.layers[l] = h->layers[l];
    a.n_layers = h->n_layers;
    a.x = (const float*)x; a.out = (float*)out; a.vl = vl; a.status = h->status;
    a.B = B; a.L = L; a.d = h->d; a.H = h->H; a.dh = h->dh; a.dff = h->dff;
    KernelTimer t(h, KC_MEGA_SIMT, s);
    return mega_simt_forward(a, s);
  }
  if (p == TL_PATH_MEGA) {
    MegaArgs a{(const MegaLayer*)h->mega_layers, h->n_layers, B, h->dff, vl, out, h->status};
    KernelTimer t(h, KC_MEGA, s);
    return mega_forward(x, a, L, h->dtype == TL_BF16, h->num_sms, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace tl
