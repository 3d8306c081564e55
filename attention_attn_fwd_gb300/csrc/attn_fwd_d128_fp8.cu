// Head-dimension-128 two-tile instantiations of the sm_103a forward kernel
// for E4M3 (FP8) inputs.
#include "attn_fwd_launch.cuh"

namespace attn {

cudaError_t launch_fwd_d128_fp8(const CUtensorMap& q, const CUtensorMap& k,
                                const CUtensorMap& v, const CUtensorMap& o,
                                const FwdParams& p, int grid,
                                cudaStream_t stream) {
  return launch_mode<128, false, true>(true, q, k, v, o, p, grid, stream);
}

}  // namespace attn
