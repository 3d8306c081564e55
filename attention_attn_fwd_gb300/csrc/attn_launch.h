// Internal launch interface between the C ABI and the kernel translation
// units (one per head dimension, compiled in parallel).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_fwd_kernel.cuh"

namespace attn {

// Unique id of the CUDA context current on the calling thread (binding the
// current device's primary context first if the thread has none).  Ids are
// never reused within a process, so a device reset, which replaces the
// context, also changes the id: caches of device addresses key on it.
bool current_context_id(unsigned long long* id);

// Dynamic shared memory one CTA of the (D, packed, FP8) variant needs.
int fwd_smem_bytes(int D, bool pack, bool fp8 = false);
// K/V stages (pairs of ring slots) of the (D, packed, FP8) variant.
int fwd_stages(int D, bool pack, bool fp8 = false);

// One entry per kernel translation unit: head dimension x tile mode (two
// 128-row Q tiles, or the query heads of a GQA group packed into one).
// `o` maps the 16-bit output O (used by the two-tile one-pass variants,
// which store O with TMA from shared memory).
cudaError_t launch_fwd_d64(bool bf16, const CUtensorMap& q,
                           const CUtensorMap& k, const CUtensorMap& v,
                           const CUtensorMap& o, const FwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_fwd_d128(bool bf16, const CUtensorMap& q,
                            const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& o, const FwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_fwd_d64_packed(bool bf16, const CUtensorMap& q,
                                  const CUtensorMap& k, const CUtensorMap& v,
                                  const CUtensorMap& o, const FwdParams& p, int grid,
                                  cudaStream_t stream);
cudaError_t launch_fwd_d128_packed(bool bf16, const CUtensorMap& q,
                                   const CUtensorMap& k, const CUtensorMap& v,
                                   const CUtensorMap& o, const FwdParams& p, int grid,
                                   cudaStream_t stream);
// E4M3 inputs, D = 128, bf16 output.
cudaError_t launch_fwd_d128_fp8(const CUtensorMap& q, const CUtensorMap& k,
                                const CUtensorMap& v, const CUtensorMap& o, const FwdParams& p,
                                int grid, cudaStream_t stream);
cudaError_t launch_fwd_d128_fp8_packed(const CUtensorMap& q,
                                       const CUtensorMap& k,
                                       const CUtensorMap& v,
                                       const CUtensorMap& o, const FwdParams& p, int grid,
                                       cudaStream_t stream);

// Split-KV merge launch (attn_merge.cu): merges p's key-range partials
// into p.o / p.lse for every query row; queued behind the forward kernel on
// `stream` as a programmatic dependent launch.  `bf16`: O's element type
// (bf16, else fp16).
cudaError_t launch_merge(int D, bool bf16, const FwdParams& p, int sms,
                         cudaStream_t stream);

// Backward pass: row pass (D, lse2 into p.lse2 / p.delta), dK/dV kernel,
// dQ kernel, in that order on `stream` (attn_bwd.cu).  `d` maps dO and `dq`
// maps dQ like `q` maps Q (dQ is stored through it by TMA).
struct BwdParams;
cudaError_t launch_bwd(int D, bool bf16, const CUtensorMap& q,
                       const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& d, const CUtensorMap& dq,
                       const void* O, const void* dO, const float* LSE,
                       const BwdParams& p, cudaStream_t stream);

}  // namespace attn
