// tl_eval_gelu: evaluates the library's two GELU forms on device arrays, so
// a test can pin the branch-free (paired) form against the erff form.
#include <cuda_runtime.h>

#include "common.cuh"

namespace {
// Thread i evaluates elements 2i and 2i + 1 (a pair, as the kernels do).
__global__ void eval_gelu_kernel(const float* x, float* y_erf, float* y_fast, size_t n) {
  const size_t pairs = (n + 1) / 2;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < pairs; i += (size_t)gridDim.x * blockDim.x) {
    const size_t j = 2 * i;
    const bool two = j + 1 < n;
    float a = x[j], b = two ? x[j + 1] : 0.f;
    y_erf[j] = tl::gelu_erf(a);
    if (two) y_erf[j + 1] = tl::gelu_erf(b);
    tl::gelu_as7128_x2(a, b);
    y_fast[j] = a;
    if (two) y_fast[j + 1] = b;
  }
}
}  // namespace

extern "C" tl_status tl_eval_gelu(const float* x, float* y_erf, float* y_fast, size_t n, void* stream) {
  if (!x || !y_erf || !y_fast) return TL_ERR_INVALID_ARG;
  if (n == 0) return TL_OK;
  eval_gelu_kernel<<<256, 256, 0, (cudaStream_t)stream>>>(x, y_erf, y_fast, n);
  return cudaGetLastError() == cudaSuccess ? TL_OK : TL_ERR_CUDA;
}
