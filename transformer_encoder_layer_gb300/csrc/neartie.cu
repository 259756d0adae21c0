// fp64 fix-up of near-tie attention rows (the method is described in
// neartie.cuh).  One warp per queued (row, head); the kernel exits at once
// when nothing was queued.
#include "common.cuh"
#include "neartie.cuh"
#include "neartie_entry.cuh"

namespace tl {
namespace {

constexpr int FW = 4;  // warps per block

__global__ void __launch_bounds__(FW * 32) neartie_fixup_kernel(FixupArgs a) {
  extern __shared__ double fix_smem[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  double* q64 = fix_smem + (size_t)warp * (a.dh + a.d);
  double* u = q64 + a.dh;
  const int n = min(*a.ties.count, a.ties.capacity);
  for (int e = blockIdx.x * FW + warp; e < n; e += gridDim.x * FW) ntie::neartie_fix_entry(a, a.ties.list[e], q64, u, lane);
}

}  // namespace

cudaError_t neartie_fixup(const FixupArgs& a, cudaStream_t s) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t smem = (size_t)FW * (a.dh + a.d) * sizeof(double);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(neartie_fixup_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  neartie_fixup_kernel<<<sms, FW * 32, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace tl
