// tl_eval_gelu: evaluates the library's two GELU forms on device arrays, so
// a test can pin the branch-free form against the erff form.
#include <cuda_runtime.h>

#include "common.cuh"

namespace {
__global__ void eval_gelu_kernel(const float* x, float* y_erf, float* y_fast, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    y_erf[i] = tl::gelu_erf(x[i]);
    y_fast[i] = tl::gelu_as7128(x[i]);
  }
}
}  // namespace

extern "C" tl_status tl_eval_gelu(const float* x, float* y_erf, float* y_fast, size_t n, void* stream) {
  if (!x || !y_erf || !y_fast) return TL_ERR_INVALID_ARG;
  if (n == 0) return TL_OK;
  eval_gelu_kernel<<<256, 256, 0, (cudaStream_t)stream>>>(x, y_erf, y_fast, n);
  return cudaGetLastError() == cudaSuccess ? TL_OK : TL_ERR_CUDA;
}
