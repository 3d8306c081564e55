// Launches of the backward kernels (row pass, dK/dV, dQ) for D = 64 / 128
// and fp16 / bf16.
#include "attn_bwd_kernel.cuh"
#include "attn_launch.h"

namespace attn {
namespace {

// The dK/dV and dQ kernels read the same inputs and write disjoint outputs,
// so they run concurrently: dQ goes to a side stream forked from the
// caller's stream after the row pass and joined back before the call
// returns.  The short dQ CTAs then fill the SMs that the long dK/dV CTAs
// (heaviest key tiles first) leave idle; on the GQA 8k workload a per-CTA
// timeline showed every SM busy for 99 % of the two kernels' span, against
// a 17 % longer critical path (the heaviest key tiles) when they ran one
// after the other.  One side stream and two events per host thread and
// device, created on first use and kept for the thread's lifetime.
constexpr int kMaxSideDevices = 64;

struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  ~SideStream() {
    if (join != nullptr) cudaEventDestroy(join);
    if (fork != nullptr) cudaEventDestroy(fork);
    if (stream != nullptr) cudaStreamDestroy(stream);
  }
};

cudaError_t side_stream(SideStream** out) {
  static thread_local SideStream side[kMaxSideDevices];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxSideDevices) return cudaErrorInvalidDevice;
  SideStream& s = side[dev];
  if (s.stream == nullptr) {
    err = cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming);
    if (err == cudaSuccess)
      err = cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming);
    if (err == cudaSuccess)
      err = cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking);
    if (err != cudaSuccess) return err;
  }
  *out = &s;
  return cudaSuccess;
}

template <class Kernel>
cudaError_t set_smem(Kernel kernel, int smem, int* configured,
                     int regs_required = 0) {
  // The attribute is per device; set it once per device and kernel.
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (*configured != dev) {
    err = cudaFuncSetAttribute(kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               smem);
    if (err != cudaSuccess) return err;
    if (regs_required > 0) {
      // A kernel that splits its registers with setmaxnreg needs exactly
      // the launch allocation the split adds up to.
      cudaFuncAttributes attr{};
      err = cudaFuncGetAttributes(&attr, kernel);
      if (err != cudaSuccess) return err;
      if (attr.numRegs != regs_required) return cudaErrorInvalidConfiguration;
    }
    *configured = dev;
  }
  return cudaSuccess;
}

template <class Kernel, class... Args>
cudaError_t launch(Kernel kernel, int smem, int grid, cudaStream_t stream,
                   const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(bwd::kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int D, bool kBF16>
cudaError_t run(const CUtensorMap& q, const CUtensorMap& k,
                const CUtensorMap& v, const CUtensorMap& d,
                const CUtensorMap& dqm, const void* O, const void* dO,
                const float* LSE, const BwdParams& p, cudaStream_t stream) {
  static thread_local int cfg_dkdv = -1, cfg_dq = -1;
  const long long planes = static_cast<long long>(p.B) * p.Hq;
  const long long rows = planes * p.Sq;
  const long long pad_rows = planes * (p.sq_pad - p.Sq);
  float* lse2 = const_cast<float*>(p.lse2);
  float* delta = const_cast<float*>(p.delta);
  // Warps: one per 8 rows, then one per 32 padding rows.
  const long long warps = (rows + 7) / 8 + (pad_rows + 31) / 32;
  const long long blocks = (warps * 32 + 255) / 256;
  attn_bwd_prep_kernel<D, kBF16><<<static_cast<unsigned>(blocks), 256, 0,
                                   stream>>>(O, dO, LSE, lse2, delta, rows,
                                             planes, p.Sq, p.sq_pad);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;

  auto dkdv = attn_bwd_dkdv_kernel<D, kBF16>;
  const int smem_kv = DkdvLayout<D>::kSmemBytes;
  err = set_smem(dkdv, smem_kv, &cfg_dkdv, 168);
  if (err != cudaSuccess) return err;
  auto dq = attn_bwd_dq_kernel<D, kBF16>;
  const int smem_q = DqLayout<D>::kSmemBytes;
  err = set_smem(dq, smem_q, &cfg_dq, 168);
  if (err != cudaSuccess) return err;
  SideStream* side = nullptr;
  err = side_stream(&side);
  if (err != cudaSuccess) return err;

  // Fork after the row pass, dK/dV first, dQ on the side stream, join.
  err = cudaEventRecord(side->fork, stream);
  if (err != cudaSuccess) return err;
  err = cudaStreamWaitEvent(side->stream, side->fork, 0);
  if (err != cudaSuccess) return err;
  err = launch(dkdv, smem_kv, p.B * p.Hkv * p.k_tiles, stream, q, k, v, d, p);
  if (err != cudaSuccess) return err;
  err = launch(dq, smem_q, p.B * p.Hq * p.q_tiles, side->stream, q, k, v, d,
               dqm, p);
  if (err != cudaSuccess) return err;
  err = cudaEventRecord(side->join, side->stream);
  if (err != cudaSuccess) return err;
  return cudaStreamWaitEvent(stream, side->join, 0);
}

}  // namespace

cudaError_t launch_bwd(int D, bool bf16, const CUtensorMap& q,
                       const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& d, const CUtensorMap& dq,
                       const void* O, const void* dO, const float* LSE,
                       const BwdParams& p, cudaStream_t stream) {
  if (D == 64)
    return bf16 ? run<64, true>(q, k, v, d, dq, O, dO, LSE, p, stream)
                : run<64, false>(q, k, v, d, dq, O, dO, LSE, p, stream);
  return bf16 ? run<128, true>(q, k, v, d, dq, O, dO, LSE, p, stream)
              : run<128, false>(q, k, v, d, dq, O, dO, LSE, p, stream);
}

}  // namespace attn
