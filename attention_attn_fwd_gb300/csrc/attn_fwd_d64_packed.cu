// Head-dimension-64 packed-GQA instantiations (few query rows: all query heads of
// a K/V head in one tile) of the sm_103a forward kernel.
#include "attn_fwd_launch.cuh"

namespace attn {

cudaError_t launch_fwd_d64_packed(bool bf16, const CUtensorMap& q,
                                  const CUtensorMap& k, const CUtensorMap& v,
                                  const CUtensorMap& o, const FwdParams& p,
                                  int grid, cudaStream_t stream) {
  return launch_mode<64, true>(bf16, q, k, v, o, p, grid, stream);
}

}  // namespace attn
