// Launch of the split-KV merge kernel (attn_merge_kernel): the key ranges'
// partial results of a split-KV forward launch merged into O and LSE by a
// grid over all query rows, queued behind the forward kernel on the same
// stream with programmatic serialization.
#include <algorithm>

#include "attn_launch.h"
#include "attn_merge_kernel.cuh"

namespace attn {
namespace {

template <int D, bool kBF16, bool kWindow, int kRowBatch>
cudaError_t launch_merge_rows(const FwdParams& p, int sms, long long ctas,
                              cudaStream_t stream) {
  // Grid-stride beyond 8 CTAs per SM.
  const int grid = static_cast<int>(std::max<long long>(
      1, std::min<long long>(ctas, 8LL * std::max(sms, 1))));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kMergeThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg,
                            attn_merge_kernel<D, kBF16, kWindow, kRowBatch>,
                            p);
}

// Two rows per thread when that still gives every SM two CTAs, else one.
template <int D, bool kBF16, bool kWindow>
cudaError_t launch_merge_variant(const FwdParams& p, int sms,
                                 cudaStream_t stream) {
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.Sq;
  constexpr int kRows2 = merge_rows_per_cta<D, 2>();
  constexpr int kRows1 = merge_rows_per_cta<D, 1>();
  const long long ctas2 = (rows + kRows2 - 1) / kRows2;
  if (ctas2 >= 2LL * std::max(sms, 1))
    return launch_merge_rows<D, kBF16, kWindow, 2>(p, sms, ctas2, stream);
  return launch_merge_rows<D, kBF16, kWindow, 1>(
      p, sms, (rows + kRows1 - 1) / kRows1, stream);
}

template <int D>
cudaError_t launch_merge_d(bool bf16, const FwdParams& p, int sms,
                           cudaStream_t stream) {
  const bool window = p.window > 0;
  if (bf16)
    return window ? launch_merge_variant<D, true, true>(p, sms, stream)
                  : launch_merge_variant<D, true, false>(p, sms, stream);
  return window ? launch_merge_variant<D, false, true>(p, sms, stream)
                : launch_merge_variant<D, false, false>(p, sms, stream);
}

}  // namespace

cudaError_t launch_merge(int D, bool bf16, const FwdParams& p, int sms,
                         cudaStream_t stream) {
  return D == 64 ? launch_merge_d<64>(bf16, p, sms, stream)
                 : launch_merge_d<128>(bf16, p, sms, stream);
}

}  // namespace attn
