// Head-dimension-64 instantiations of the sm_103a forward kernel.
#include "attn_launch.h"

namespace attn {
namespace {

template <bool kBF16>
cudaError_t launch(const CUtensorMap& q, const CUtensorMap& k,
                   const CUtensorMap& v, const FwdParams& p, int grid,
                   cudaStream_t stream) {
  auto kernel = attn_fwd_sm103_kernel<64, kBF16>;
  const int smem = Layout<64>::kSmemBytes;
  // The attribute is per device; setting it again is cheap and idempotent.
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (configured_device != dev) {
    err = cudaFuncSetAttribute(kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               smem);
    if (err != cudaSuccess) return err;
    configured_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kernel, q, k, v, p);
}

}  // namespace

cudaError_t launch_fwd_d64(bool bf16, const CUtensorMap& q,
                           const CUtensorMap& k, const CUtensorMap& v,
                           const FwdParams& p, int grid, cudaStream_t stream) {
  return bf16 ? launch<true>(q, k, v, p, grid, stream)
              : launch<false>(q, k, v, p, grid, stream);
}

}  // namespace attn
