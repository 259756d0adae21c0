// The C ABI (include/tl_encoder.h): handle creation and weight packing,
// workspace sizing, shape dispatch and the per-layer launch sequence.
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "paths.h"
#include "mega.h"
#include "tc_attention.h"

using namespace tl;

namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

float host_half_to_float(uint16_t h) {
  uint32_t sign = (uint32_t)(h >> 15) << 31, exp = (h >> 10) & 0x1f, man = h & 0x3ff;
  uint32_t bits;
  if (exp == 0) {
    if (man == 0) {
      bits = sign;
    } else {  // subnormal: renormalise
      int e = -1;
      do { ++e; man <<= 1; } while ((man & 0x400) == 0);
      bits = sign | (uint32_t)(127 - 15 - e) << 23 | (man & 0x3ff) << 13;
    }
  } else if (exp == 31) {
    bits = sign | 0x7f800000u | man << 13;
  } else {
    bits = sign | (exp - 15 + 127) << 23 | man << 13;
  }
  float f;
  std::memcpy(&f, &bits, 4);
  return f;
}

float host_to_float(const void* p, size_t i, tl_dtype t) {
  if (t == TL_F32) return reinterpret_cast<const float*>(p)[i];
  uint16_t u = reinterpret_cast<const uint16_t*>(p)[i];
  if (t == TL_F16) return host_half_to_float(u);
  uint32_t bits = (uint32_t)u << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return f;
}

// Byte offsets of one layer's parameters inside the packed buffer.
struct LayerOffsets {
  size_t w_qkv, w_o, w_1, w_2, b_qkv, b_o, ln1_g, ln1_b, b_1, b_2, ln2_g, ln2_b, end;
};

LayerOffsets layer_offsets(size_t start, int d, int dff, size_t es) {
  LayerOffsets o;
  size_t p = start;
  auto take = [&](size_t bytes) { size_t at = p; p = align_up(p + bytes, 256); return at; };
  o.w_qkv = take((size_t)3 * d * d * es);
  o.w_o = take((size_t)d * d * es);
  o.w_1 = take((size_t)dff * d * es);
  o.w_2 = take((size_t)d * dff * es);
  o.b_qkv = take((size_t)3 * d * 4);
  o.b_o = take((size_t)d * 4);
  o.ln1_g = take((size_t)d * 4);
  o.ln1_b = take((size_t)d * 4);
  o.b_1 = take((size_t)dff * 4);
  o.b_2 = take((size_t)d * 4);
  o.ln2_g = take((size_t)d * 4);
  o.ln2_b = take((size_t)d * 4);
  o.end = p;
  return o;
}

// Copy n elements of a caller array (host or device) to host memory.
bool fetch(const void* src, size_t bytes, std::vector<unsigned char>& dst) {
  dst.resize(bytes);
  return cudaMemcpy(dst.data(), src, bytes, cudaMemcpyDefault) == cudaSuccess;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

constexpr int kMaxHostChunks = 64;

// How the host-buffer forward splits the batch.  Every path computes each
// sequence from its own tokens only, so a slice of sequences yields the same
// bits as the whole batch; slices alternate between two streams so that one
// slice's upload, another's kernels and a third's download overlap.  The
// path is the one chosen for the whole batch and every slice runs it.
struct HostPlan {
  tl_path p;
  int chunks, bc;  // slices, and the most sequences in one slice
  int start[kMaxHostChunks + 3];  // slice c holds sequences [start[c], start[c + 1])
  size_t row;      // bytes of one sequence of x or out
  size_t io;       // bytes of the device copy of x (and of out), padded
  size_t fw;       // forward workspace of one slice, padded
  size_t total;    // device workspace of the whole call
};

tl_status host_plan(const tl_encoder* h, int B, int L, HostPlan* hp) {
  const tl_path p = choose_path(h, B, L);
  if (p == TL_PATH_AUTO) return TL_ERR_UNSUPPORTED_SHAPE;
  const size_t row = (size_t)L * h->d * dtype_size(h->dtype);
  int n = h->host_chunks;
  if (n == 0) {
    // Automatic: slices of 8 MiB or more, at most 8; the layered path keeps
    // at least half the batch per slice so that its per-kernel grids stay
    // full; the task-graph path is sized for one launch over the batch.
    n = (int)std::min<size_t>(8, (size_t)B * row / ((size_t)8 << 20));
    if (p == TL_PATH_LAYERED) n = std::min(n, 2);
    if (p == TL_PATH_DAG) n = 1;
  }
  if (row % 16) n = 1;  // every slice of x and out must stay 16-byte aligned
  n = std::max(1, std::min(n, B));
  const int bc = (B + n - 1) / n;
  hp->p = p;
  hp->chunks = (B + bc - 1) / bc;  // no empty slice
  hp->bc = bc;
  int k = 0;
  for (int c = 0; c <= hp->chunks; ++c) hp->start[k++] = std::min(c * bc, B);
  if (h->host_chunks == 0 && hp->chunks >= 4 && bc >= 4) {
    // Automatic plans also cut a quarter slice off each end: the first
    // upload and the last download, which nothing overlaps, shrink 4x.
    const int first = bc / 4, last = (B - hp->start[hp->chunks - 1]) / 4;
    int s2[kMaxHostChunks + 3], m = 0;
    s2[m++] = 0;
    s2[m++] = first;
    for (int c = 1; c < hp->chunks; ++c) s2[m++] = hp->start[c];
    if (last >= 1) s2[m++] = B - last;
    s2[m++] = B;
    for (int i = 0; i < m; ++i) hp->start[i] = s2[i];
    k = m;
  }
  hp->chunks = k - 1;
  hp->row = row;
  hp->io = align_up((size_t)B * row, 256);
  hp->fw = align_up(path_workspace_bytes(h, p, bc, L), 256);
  hp->total = 2 * hp->io + align_up((size_t)B * 4, 256) + (hp->chunks > 1 ? 2 : 1) * hp->fw;
  return TL_OK;
}

// The pipeline's streams and events, made on first use on the current device.
bool host_streams(tl_encoder* h) {
  for (cudaStream_t& x : h->host_stream)
    if (!x && cudaStreamCreateWithFlags(&x, cudaStreamNonBlocking) != cudaSuccess) {
      x = nullptr;
      return false;
    }
  for (cudaEvent_t& x : h->host_event)
    if (!x && cudaEventCreateWithFlags(&x, cudaEventDisableTiming) != cudaSuccess) {
      x = nullptr;
      return false;
    }
  return true;
}

void drop_graph(tl_encoder* h) {
  if (h->graph_exec) cudaGraphExecDestroy(h->graph_exec);
  h->graph_exec = nullptr;
  h->graph_key = tl_encoder::GraphKey{};
}

// Record the path's launch sequence for these buffers into a CUDA graph on
// the handle's own stream (thread-local capture, so other threads' CUDA
// calls are unaffected) and keep its executable instance in the handle.
cudaError_t capture_graph(tl_encoder* h, tl_path p, const void* x, int B, int L, const int32_t* vl,
                          void* out, void* ws) {
  drop_graph(h);
  cudaError_t e = cudaSuccess;
  if (!h->capture_stream &&
      (e = cudaStreamCreateWithFlags(&h->capture_stream, cudaStreamNonBlocking)) != cudaSuccess) {
    h->capture_stream = nullptr;
    return e;
  }
  if ((e = cudaStreamBeginCapture(h->capture_stream, cudaStreamCaptureModeThreadLocal)) != cudaSuccess)
    return e;
  const cudaError_t er = run_path(h, p, x, B, L, vl, out, ws, h->capture_stream);
  cudaGraph_t g = nullptr;
  e = cudaStreamEndCapture(h->capture_stream, &g);
  if (er != cudaSuccess || e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return er != cudaSuccess ? er : e;
  }
  e = cudaGraphInstantiateWithFlags(&h->graph_exec, g, 0);
  cudaGraphDestroy(g);
  if (e != cudaSuccess) {
    h->graph_exec = nullptr;
    cudaGetLastError();
    return e;
  }
  ++h->graph_captures;
  return cudaSuccess;
}

}  // namespace

extern "C" {

const char* tl_status_string(tl_status s) {
  switch (s) {
    case TL_OK: return "ok";
    case TL_ERR_INVALID_ARG: return "invalid argument";
    case TL_ERR_UNSUPPORTED_SHAPE: return "unsupported shape for this path";
    case TL_ERR_CUDA: return "CUDA runtime error";
    case TL_ERR_OUT_OF_MEMORY: return "out of device memory";
    case TL_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case TL_ERR_BAD_VALID_LEN: return "valid_len outside [1, L] (clamped)";
    case TL_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

tl_status tl_encoder_create(const tl_layer_weights* weights, int n_layers, int d_model,
                            int n_heads, int d_ff, tl_dtype dtype, tl_encoder** out) {
  if (!out) return TL_ERR_INVALID_ARG;
  *out = nullptr;
  if (!weights || n_layers < 1 || d_model < 16 || n_heads < 1 || d_ff < 16)
    return TL_ERR_INVALID_ARG;
  if (dtype != TL_F32 && dtype != TL_F16 && dtype != TL_BF16) return TL_ERR_INVALID_ARG;
  if (d_model % 16 || d_ff % 16 || d_model % n_heads || d_model > 1024 || d_ff > 16384)
    return TL_ERR_UNSUPPORTED_SHAPE;
  const int dh = d_model / n_heads;
  if (dh > 128) return TL_ERR_UNSUPPORTED_SHAPE;
  for (int l = 0; l < n_layers; ++l) {
    const tl_layer_weights& w = weights[l];
    const void* ps[] = {w.w_qkv, w.b_qkv, w.w_o, w.b_o, w.ln1_g, w.ln1_b,
                        w.w_1, w.b_1, w.w_2, w.b_2, w.ln2_g, w.ln2_b};
    for (const void* p : ps)
      if (!p) return TL_ERR_INVALID_ARG;
  }

  tl_encoder* h = new (std::nothrow) tl_encoder();
  if (!h) return TL_ERR_OUT_OF_MEMORY;
  h->n_layers = n_layers; h->d = d_model; h->H = n_heads; h->dh = dh; h->dff = d_ff;
  h->dtype = dtype;
  // Debug switch: CUDA-core attention inside the layered path (cross-checks).
  if (const char* e = getenv("TL_SIMT_ATTENTION")) h->simt_attention = e[0] == '1';
  // Test hook for the bounded waits of the task-graph path: its first task
  // waits on a counter target no task reaches, so the forward must end with
  // TL_ERR_DEVICE_TIMEOUT after the wait's deadline.
  if (const char* e = getenv("TL_DAG_INJECT_STALL")) h->dag_inject_stall = e[0] == '1';
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
    delete h;
    return TL_ERR_CUDA;
  }
  // The static scratch array's address in this device's context, for
  // tl_encoder_forward_static (null if the lookup fails; that entry point
  // then returns TL_ERR_CUDA and every other call is unaffected).
  h->static_scratch = static_scratch_address();
  const size_t es = dtype_size(dtype);
  std::vector<LayerOffsets> offs;
  size_t total = 0;
  for (int l = 0; l < n_layers; ++l) {
    offs.push_back(layer_offsets(total, d_model, d_ff, es));
    total = offs.back().end;
  }
  size_t extra = packed_extra_bytes(h);
  size_t extra_off = total;
  total += extra;
  std::vector<unsigned char> stage(total, 0), tmp;
  const int d = d_model;
  for (int l = 0; l < n_layers; ++l) {
    const tl_layer_weights& w = weights[l];
    const LayerOffsets& o = offs[l];
    struct { const void* src; size_t off; size_t n; } mats[] = {
        {w.w_qkv, o.w_qkv, (size_t)3 * d * d}, {w.w_o, o.w_o, (size_t)d * d},
        {w.w_1, o.w_1, (size_t)d_ff * d}, {w.w_2, o.w_2, (size_t)d * d_ff}};
    for (auto& m : mats) {
      if (!fetch(m.src, m.n * es, tmp)) { delete h; return TL_ERR_INVALID_ARG; }
      std::memcpy(stage.data() + m.off, tmp.data(), m.n * es);
    }
    struct { const void* src; size_t off; size_t n; } vecs[] = {
        {w.b_qkv, o.b_qkv, (size_t)3 * d}, {w.b_o, o.b_o, (size_t)d},
        {w.ln1_g, o.ln1_g, (size_t)d}, {w.ln1_b, o.ln1_b, (size_t)d},
        {w.b_1, o.b_1, (size_t)d_ff}, {w.b_2, o.b_2, (size_t)d},
        {w.ln2_g, o.ln2_g, (size_t)d}, {w.ln2_b, o.ln2_b, (size_t)d}};
    for (auto& v : vecs) {
      if (!fetch(v.src, v.n * es, tmp)) { delete h; return TL_ERR_INVALID_ARG; }
      float* dst = reinterpret_cast<float*>(stage.data() + v.off);
      for (size_t i = 0; i < v.n; ++i) dst[i] = host_to_float(tmp.data(), i, dtype);
    }
  }
  if (cudaMalloc(&h->wbuf, total) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return TL_ERR_OUT_OF_MEMORY;
  }
  if (cudaMalloc((void**)&h->status, 256) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->wbuf);
    delete h;
    return TL_ERR_OUT_OF_MEMORY;
  }
  h->wbuf_bytes = total;
  h->layers = new (std::nothrow) tl_layer_dev[n_layers];
  unsigned char* base = reinterpret_cast<unsigned char*>(h->wbuf);
  for (int l = 0; l < n_layers && h->layers; ++l) {
    const LayerOffsets& o = offs[l];
    tl_layer_dev& L = h->layers[l];
    L.w_qkv = base + o.w_qkv; L.w_o = base + o.w_o; L.w_1 = base + o.w_1; L.w_2 = base + o.w_2;
    L.b_qkv = (const float*)(base + o.b_qkv); L.b_o = (const float*)(base + o.b_o);
    L.ln1_g = (const float*)(base + o.ln1_g); L.ln1_b = (const float*)(base + o.ln1_b);
    L.b_1 = (const float*)(base + o.b_1); L.b_2 = (const float*)(base + o.b_2);
    L.ln2_g = (const float*)(base + o.ln2_g); L.ln2_b = (const float*)(base + o.ln2_b);
  }
  bool ok = h->layers != nullptr &&
            cudaMemcpy(h->wbuf, stage.data(), total - extra, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemset(h->status, 0, 256) == cudaSuccess &&
            pack_extra(h, base + extra_off, extra) == cudaSuccess &&
            cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    tl_encoder_destroy(h);
    return TL_ERR_CUDA;
  }
  *out = h;
  return TL_OK;
}

tl_status tl_encoder_set_path(tl_encoder* h, tl_path path) {
  if (!h || path < TL_PATH_AUTO || path > TL_PATH_DAG) return TL_ERR_INVALID_ARG;
  h->path = path;
  return TL_OK;
}

tl_status tl_encoder_set_attention_split(tl_encoder* h, int key_tiles) {
  if (!h || key_tiles < -1 || key_tiles > 4096) return TL_ERR_INVALID_ARG;
  h->attn_split = key_tiles;
  return TL_OK;
}

tl_status tl_encoder_set_gemm_pairs(tl_encoder* h, int enable) {
  if (!h || enable < -1 || enable > 1) return TL_ERR_INVALID_ARG;
  h->gemm_pairs = enable;
  return TL_OK;
}

tl_status tl_encoder_set_mega_assist(tl_encoder* h, int enable) {
  if (!h || enable < -1 || enable > 1) return TL_ERR_INVALID_ARG;
  h->mega_assist = enable;
  return TL_OK;
}

tl_status tl_encoder_mega_assisted(const tl_encoder* h, int B, int L, int* assisted) {
  if (!h || !assisted || B < 1 || L < 1) return TL_ERR_INVALID_ARG;
  tl_path p = choose_path(h, B, L);
  if (p == TL_PATH_AUTO) return TL_ERR_UNSUPPORTED_SHAPE;
  *assisted = p == TL_PATH_MEGA && h->dtype != TL_F32 &&
              mega_assisted(B, L, h->dff, h->num_sms, h->mega_assist);
  return TL_OK;
}

tl_status tl_encoder_attention_split(const tl_encoder* h, int B, int L, int* key_tiles) {
  if (!h || !key_tiles || B < 1 || L < 1) return TL_ERR_INVALID_ARG;
  tl_path p = choose_path(h, B, L);
  if (p == TL_PATH_AUTO) return TL_ERR_UNSUPPORTED_SHAPE;
  *key_tiles = 0;
  if (p == TL_PATH_LAYERED && tc_attention_supported(h->dh) && !h->simt_attention)
    *key_tiles =
        tc_attention_split_plan(B, h->H, L, h->dh, h->num_sms, attention_split_setting(h, B, L)).kc;
  return TL_OK;
}

tl_status tl_encoder_plan(const tl_encoder* h, int B, int L, tl_path* path) {
  if (!h || !path || B < 1 || L < 1) return TL_ERR_INVALID_ARG;
  tl_path p = choose_path(h, B, L);
  if (p == TL_PATH_AUTO) return TL_ERR_UNSUPPORTED_SHAPE;
  *path = p;
  return TL_OK;
}

tl_status tl_encoder_workspace_size(const tl_encoder* h, int B, int L, size_t* bytes) {
  if (!h || !bytes || B < 1 || L < 1) return TL_ERR_INVALID_ARG;
  tl_path p = choose_path(h, B, L);
  if (p == TL_PATH_AUTO) return TL_ERR_UNSUPPORTED_SHAPE;
  *bytes = path_workspace_bytes(h, p, B, L);
  return TL_OK;
}

tl_status tl_encoder_forward(tl_encoder* h, const void* x, int B, int L, const int32_t* valid_len,
                             void* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (!h || !x || !out || !valid_len || B < 1 || L < 1) return TL_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(valid_len, 4)) return TL_ERR_INVALID_ARG;
  const size_t io_bytes = (size_t)B * L * h->d * dtype_size(h->dtype);
  const char* xb = (const char*)x; const char* ob = (const char*)out;
  if (xb < ob + io_bytes && ob < xb + io_bytes) return TL_ERR_INVALID_ARG;  // overlap
  tl_path p = choose_path(h, B, L);
  if (p == TL_PATH_AUTO) return TL_ERR_UNSUPPORTED_SHAPE;
  size_t need = path_workspace_bytes(h, p, B, L);
  if (workspace_bytes < need) return TL_ERR_WORKSPACE_TOO_SMALL;
  if (need > 0 && (!workspace || !aligned(workspace, 256))) return TL_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (h->graphs && p == TL_PATH_LAYERED && !h->timing) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return TL_ERR_CUDA;
    if (cs == cudaStreamCaptureStatusNone) {
      const tl_encoder::GraphKey key{(int)p, B, L, h->attn_split * 4 + h->gemm_pairs + 1, x, valid_len, out,
                                     workspace};
      if (h->graph_exec && h->graph_key == key) {
        ++h->graph_replays;
        return cudaGraphLaunch(h->graph_exec, st) == cudaSuccess ? TL_OK : TL_ERR_CUDA;
      }
      // A new (shape, buffers): run it as usual, and record the same launch
      // sequence on the handle's capture stream for the next call.
      cudaError_t e = run_path(h, p, x, B, L, valid_len, out, workspace, st);
      if (e != cudaSuccess) return TL_ERR_CUDA;
      if (capture_graph(h, p, x, B, L, valid_len, out, workspace) == cudaSuccess) h->graph_key = key;
      return TL_OK;
    }
  }
  cudaError_t e = run_path(h, p, x, B, L, valid_len, out, workspace, st);
  return e == cudaSuccess ? TL_OK : TL_ERR_CUDA;
}

tl_status tl_encoder_set_graphs(tl_encoder* h, int enable) {
  if (!h || enable < 0 || enable > 1) return TL_ERR_INVALID_ARG;
  h->graphs = enable != 0;
  if (!h->graphs) drop_graph(h);
  return TL_OK;
}

tl_status tl_encoder_graph_stats(const tl_encoder* h, long long* captures, long long* replays) {
  if (!h || !captures || !replays) return TL_ERR_INVALID_ARG;
  *captures = h->graph_captures;
  *replays = h->graph_replays;
  return TL_OK;
}

tl_status tl_encoder_set_host_chunks(tl_encoder* h, int chunks) {
  if (!h || chunks < 0 || chunks > kMaxHostChunks) return TL_ERR_INVALID_ARG;
  h->host_chunks = chunks;
  return TL_OK;
}

tl_status tl_encoder_host_workspace_size(const tl_encoder* h, int B, int L, size_t* bytes) {
  if (!h || !bytes || B < 1 || L < 1) return TL_ERR_INVALID_ARG;
  HostPlan hp;
  tl_status s = host_plan(h, B, L, &hp);
  if (s != TL_OK) return s;
  *bytes = hp.total;
  return TL_OK;
}

tl_status tl_encoder_forward_host(tl_encoder* h, const void* x_host, int B, int L,
                                  const int32_t* valid_len_host, void* out_host, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (!h || !x_host || !valid_len_host || !out_host || !workspace || B < 1 || L < 1)
    return TL_ERR_INVALID_ARG;
  HostPlan hp;
  tl_status s = host_plan(h, B, L, &hp);
  if (s != TL_OK) return s;
  if (workspace_bytes < hp.total) return TL_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(workspace, 256)) return TL_ERR_INVALID_ARG;
  char* w = (char*)workspace;
  char* xd = w;
  char* od = w + hp.io;
  int32_t* vld = (int32_t*)(w + 2 * hp.io);
  char* fw[2] = {w + 2 * hp.io + align_up((size_t)B * 4, 256), nullptr};
  fw[1] = fw[0] + hp.fw;
  const char* xh = (const char*)x_host;
  char* oh = (char*)out_host;
  cudaStream_t st = (cudaStream_t)stream;
  cudaStream_t ss[2] = {st, st};
  cudaError_t e = cudaSuccess;
  if (hp.chunks > 1) {
    if (!host_streams(h)) return TL_ERR_CUDA;
    ss[0] = h->host_stream[0];
    ss[1] = h->host_stream[1];
    // Fork: both pipeline streams start after the caller's earlier work.
    if ((e = cudaEventRecord(h->host_event[0], st)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(ss[0], h->host_event[0], 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(ss[1], h->host_event[0], 0)) != cudaSuccess)
      return TL_ERR_CUDA;
  }
  // Slice c: upload, forward and download on stream c % 2.  The download of
  // slice c - 1 is enqueued after slice c's forward, so that with pageable
  // buffers (whose downloads return only when done) slice c still computes
  // while slice c - 1 is copied back.
  auto down = [&](int c) {
    const size_t off = (size_t)hp.start[c] * hp.row;
    const size_t bytes = (size_t)(hp.start[c + 1] - hp.start[c]) * hp.row;
    return cudaMemcpyAsync(oh + off, od + off, bytes, cudaMemcpyDeviceToHost, ss[c & 1]);
  };
  for (int c = 0; c < hp.chunks && e == cudaSuccess; ++c) {
    const int b0 = hp.start[c], bn = hp.start[c + 1] - b0;
    const size_t off = (size_t)b0 * hp.row, bytes = (size_t)bn * hp.row;
    cudaStream_t sc = ss[c & 1];
    if ((e = cudaMemcpyAsync(xd + off, xh + off, bytes, cudaMemcpyHostToDevice, sc)) != cudaSuccess ||
        (e = cudaMemcpyAsync(vld + b0, valid_len_host + b0, (size_t)bn * 4, cudaMemcpyHostToDevice,
                             sc)) != cudaSuccess ||
        (e = run_path(h, hp.p, xd + off, bn, L, vld + b0, od + off, fw[c & 1], sc)) != cudaSuccess)
      break;
    if (c > 0) e = down(c - 1);
  }
  if (e == cudaSuccess) e = down(hp.chunks - 1);
  if (hp.chunks > 1) {
    // Join: the caller's stream waits for both pipeline streams; both are also
    // drained below, so no copy touches the caller's buffers after return.
    for (int i = 0; i < 2; ++i)
      if (cudaEventRecord(h->host_event[1 + i], ss[i]) == cudaSuccess)
        cudaStreamWaitEvent(st, h->host_event[1 + i], 0);
    cudaError_t e0 = cudaStreamSynchronize(ss[0]), e1 = cudaStreamSynchronize(ss[1]);
    if (e == cudaSuccess) e = e0 != cudaSuccess ? e0 : e1;
  }
  const cudaError_t es = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = es;
  return e == cudaSuccess ? TL_OK : TL_ERR_CUDA;
}

tl_status tl_encoder_get_status(tl_encoder* h, void* stream) {
  if (!h) return TL_ERR_INVALID_ARG;
  int v = 0;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return TL_ERR_CUDA;
  if (cudaMemcpy(&v, h->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(h->status, 0, sizeof(int)) != cudaSuccess)
    return TL_ERR_CUDA;
  return (tl_status)v;
}

tl_status tl_encoder_destroy(tl_encoder* h) {
  if (!h) return TL_OK;
  cudaDeviceSynchronize();
  timing_destroy(h);
  for (cudaStream_t& x : h->host_stream)
    if (x) cudaStreamDestroy(x);
  for (cudaEvent_t& x : h->host_event)
    if (x) cudaEventDestroy(x);
  drop_graph(h);
  if (h->capture_stream) cudaStreamDestroy(h->capture_stream);
  if (h->wbuf) cudaFree(h->wbuf);
  if (h->status) cudaFree(h->status);
  delete[] h->layers;
  delete h;
  return TL_OK;
}

}  // extern "C"
