// Launch of one instantiation of the forward kernel; included by the
// per-variant translation units (compiled in parallel).
#pragma once

#include "attn_launch.h"

namespace attn {
// Internal linkage: each translation unit (and each loaded copy of the
// library) keeps its own "attribute set" flag per kernel.
namespace {

template <int D, bool kBF16, bool kPack, bool kSplit, bool kWindow,
          bool kFp8>
cudaError_t launch_variant(const CUtensorMap& q, const CUtensorMap& k,
                           const CUtensorMap& v, const CUtensorMap& o,
                           const FwdParams& p, int grid, cudaStream_t stream) {
  auto kernel = attn_fwd_sm103_kernel<D, kBF16, kPack, kSplit, kWindow, kFp8>;
  const int smem = Layout<D, kPack, kFp8>::kSmemBytes;
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
    if constexpr (!kPack) {
      // These variants split the launch's registers with setmaxnreg, which
      // only adds up when every thread launches with cfg::kRegsLaunch: a
      // build that allocated fewer would leave the increase waiting
      // forever, so refuse to launch it.
      cudaFuncAttributes attr{};
      err = cudaFuncGetAttributes(&attr, kernel);
      if (err != cudaSuccess) return err;
      if (attr.numRegs != cfg::kRegsLaunch) return cudaErrorInvalidConfiguration;
    }
    configured_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  // The key ranges of one (batch, K/V head) as one thread-block cluster
  // (the grid holds every unit, num_splits consecutive CTAs per group).
  cudaLaunchAttribute attr[1];
  if (p.cluster_merge) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.num_splits);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, q, k, v, o, p);
}

// Dtype, split-KV and window dispatch of one (D, tile mode) variant:
// split-KV when the parameters carry partial-result buffers, the window
// variant when a window is set.  FP8 inputs always write bf16.
template <int D, bool kPack, bool kSplit, bool kWindow, bool kFp8>
cudaError_t launch_dtype(bool bf16, const CUtensorMap& q, const CUtensorMap& k,
                         const CUtensorMap& v, const CUtensorMap& o,
                         const FwdParams& p, int grid, cudaStream_t stream) {
  if constexpr (kFp8) {
    return launch_variant<D, true, kPack, kSplit, kWindow, true>(q, k, v, o, p,
                                                                 grid, stream);
  } else {
    return bf16 ? launch_variant<D, true, kPack, kSplit, kWindow, false>(
                      q, k, v, o, p, grid, stream)
                : launch_variant<D, false, kPack, kSplit, kWindow, false>(
                      q, k, v, o, p, grid, stream);
  }
}

template <int D, bool kPack, bool kFp8 = false>
cudaError_t launch_mode(bool bf16, const CUtensorMap& q, const CUtensorMap& k,
                        const CUtensorMap& v, const CUtensorMap& o,
                        const FwdParams& p, int grid, cudaStream_t stream) {
  const bool split = p.o_part != nullptr;
  const bool window = p.window > 0;
  if (split)
    return window ? launch_dtype<D, kPack, true, true, kFp8>(bf16, q, k, v, o, p,
                                                             grid, stream)
                  : launch_dtype<D, kPack, true, false, kFp8>(bf16, q, k, v, o, p,
                                                              grid, stream);
  return window ? launch_dtype<D, kPack, false, true, kFp8>(bf16, q, k, v, o, p,
                                                            grid, stream)
                : launch_dtype<D, kPack, false, false, kFp8>(bf16, q, k, v, o, p,
                                                             grid, stream);
}

}  // namespace
}  // namespace attn
