// tl_encoder_forward_static: the forward pass with its scratch memory in a
// fixed array that the library itself holds on every device it is loaded on,
// for callers that may not allocate device memory at the point of the call.
//
// The array is TL_STATIC_SCRATCH_BYTES (32 MiB) of file-scope __device__
// memory, created when the library's module loads in a device's context and
// held until the process exits.  Host code cannot hand the array's name to a
// kernel (on the host it is only a stand-in symbol), so tl_encoder_create
// looks up its device address with cudaGetSymbolAddress, with the handle's
// device current, and keeps it in the handle.  The address then belongs to
// the same context as the handle's packed weights: a context that is torn
// down and re-created (cudaDeviceReset) invalidates both together, and a
// handle created afterwards looks the address up afresh.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"
#include "paths.h"

namespace {

constexpr size_t kStaticScratchBytes = (size_t)32 << 20;
static_assert(kStaticScratchBytes == TL_STATIC_SCRATCH_BYTES, "header and library agree");

static __device__ __align__(256) unsigned char tl_static_scratch[kStaticScratchBytes];

}  // namespace

namespace tl {

// Device address of the static array in the current context, or null if the
// lookup fails (the error is cleared).
void* static_scratch_address() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, tl_static_scratch) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return p;
}

}  // namespace tl

extern "C" tl_status tl_encoder_forward_static(tl_encoder* h, const void* x, int B, int L,
                                               const int32_t* valid_len, void* out, void* stream) {
  if (!h || !x || !out || !valid_len || B < 1 || L < 1) return TL_ERR_INVALID_ARG;
  size_t need = 0;
  tl_status st = tl_encoder_workspace_size(h, B, L, &need);
  if (st != TL_OK) return st;
  if (need > kStaticScratchBytes) return TL_ERR_WORKSPACE_TOO_SMALL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TL_ERR_CUDA;
  if (dev != h->device) return TL_ERR_INVALID_ARG;
  void* ws = h->static_scratch;  // looked up by tl_encoder_create
  if (!ws) return TL_ERR_CUDA;
  return tl_encoder_forward(h, x, B, L, valid_len, out, need ? ws : nullptr, need, stream);
}
