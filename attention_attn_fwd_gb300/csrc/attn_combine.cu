// Split-KV merge: combines the per-key-range partial outputs of the forward
// kernel into O and LSE.  Each key range c of a row contributes its
// normalised partial output O_c and its log-sum-exp lse_c; with
// M = max_c lse_c and w_c = exp(lse_c - M):
//   O   = sum_c w_c O_c / sum_c w_c,     LSE = M + ln(sum_c w_c),
// which is the softmax over the union of the ranges (the same online-softmax
// rescaling the forward kernel applies tile by tile, applied once more).
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "attn_launch.h"

namespace attn {
namespace {

template <bool kBF16>
__device__ __forceinline__ uint32_t pack_pair(float lo, float hi) {
  if constexpr (kBF16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  } else {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
}

// One warp per output row; each lane owns D/32 consecutive columns.
template <int D, bool kBF16>
__global__ void __launch_bounds__(256)
    splitkv_combine_kernel(const float* __restrict__ o_part,
                           const float* __restrict__ lse_part, void* O,
                           float* LSE, long long rows, int Sq, int num_splits,
                           int split_keys, int Skv, int causal, int input_pos) {
  constexpr int kPer = D / 32;
  const long long row =
      (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  const int i = static_cast<int>(row % Sq);
  // Key ranges wholly after the row's causal horizon were not computed for
  // it (their first key is not visible).
  const int vis_end = causal ? min(Skv, input_pos + i + 1) : Skv;
  const int ns = min(num_splits, (vis_end + split_keys - 1) / split_keys);

  float m = -INFINITY;
  for (int c = 0; c < ns; ++c) m = fmaxf(m, lse_part[c * rows + row]);
  float l = 0.f;
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  for (int c = 0; c < ns; ++c) {
    const float lc = lse_part[c * rows + row];
    if (lc == -INFINITY) continue;
    const float wgt = expf(lc - m);
    l += wgt;
    const float* src = o_part + (c * rows + row) * D + lane * kPer;
#pragma unroll
    for (int e = 0; e < kPer; e += 2) {
      const float2 v = *reinterpret_cast<const float2*>(src + e);
      acc[e] += wgt * v.x;
      acc[e + 1] += wgt * v.y;
    }
  }
  const float inv_l = 1.f / l;
  uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(O) +
                                              row * D + lane * kPer);
#pragma unroll
  for (int e = 0; e < kPer; e += 2)
    dst[e / 2] = pack_pair<kBF16>(acc[e] * inv_l, acc[e + 1] * inv_l);
  if (LSE != nullptr && lane == 0) LSE[row] = m + logf(l);
}

template <int D, bool kBF16>
cudaError_t launch(const float* o_part, const float* lse_part, void* O,
                   float* LSE, long long rows, int Sq, int num_splits,
                   int split_keys, int Skv, int causal, int input_pos,
                   cudaStream_t stream) {
  constexpr int kThreads = 256;
  const long long blocks = (rows * 32 + kThreads - 1) / kThreads;
  splitkv_combine_kernel<D, kBF16><<<static_cast<unsigned>(blocks), kThreads, 0,
                                     stream>>>(o_part, lse_part, O, LSE, rows,
                                               Sq, num_splits, split_keys, Skv,
                                               causal, input_pos);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_splitkv_combine(int D, bool bf16, const float* o_part,
                                   const float* lse_part, void* O, float* LSE,
                                   long long rows, int Sq, int num_splits,
                                   int split_keys, int Skv, int causal,
                                   int input_pos, cudaStream_t stream) {
  if (D == 64)
    return bf16 ? launch<64, true>(o_part, lse_part, O, LSE, rows, Sq,
                                   num_splits, split_keys, Skv, causal,
                                   input_pos, stream)
                : launch<64, false>(o_part, lse_part, O, LSE, rows, Sq,
                                    num_splits, split_keys, Skv, causal,
                                    input_pos, stream);
  return bf16 ? launch<128, true>(o_part, lse_part, O, LSE, rows, Sq,
                                  num_splits, split_keys, Skv, causal,
                                  input_pos, stream)
              : launch<128, false>(o_part, lse_part, O, LSE, rows, Sq,
                                   num_splits, split_keys, Skv, causal,
                                   input_pos, stream);
}

}  // namespace attn
