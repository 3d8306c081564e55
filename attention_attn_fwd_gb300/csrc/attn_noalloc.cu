// Split-KV attention forward for callers that cannot allocate device memory.
//
// attn_fwd_splitkv needs a workspace for its per-key-range partial results.
// Some callers cannot provide one: code that runs where cudaMalloc is not
// allowed or not wanted (inside a memory-pool-less runtime, a plugin whose
// host owns every allocation, a real-time loop that must not enter the
// allocator).  This entry point uses a fixed scratch array compiled into
// the library instead, so the caller passes only its inputs and outputs.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/attn.h"
#include "attn_launch.h"

namespace {

// Fixed scratch for partial outputs and LSEs.  Every GPU that loads the
// library holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // context of the entry

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked
// up with that device current, once per device and context: a device reset
// replaces the context and loads the library's module (and the array) again,
// possibly at another address, so an entry of an earlier context is never
// used.
attn_status_t scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  unsigned long long ctx = 0;
  if (!attn::current_context_id(&ctx)) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess ||
        ptr == nullptr)
      return ATTN_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" {

size_t attn_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

attn_status_t attn_fwd_splitkv_noalloc(const void* Q, const void* K,
                                       const void* V, void* O, float* LSE,
                                       int B, int Hq, int Hkv, int Sq, int Skv,
                                       int D, float scale, int causal,
                                       int input_pos, attn_dtype_t dtype,
                                       int num_splits, attn_stream_t stream) {
  int splits = num_splits;
  size_t need = 0;
  attn_status_t st = attn_splitkv_plan(B, Hq, Hkv, Sq, Skv, D, causal,
                                       input_pos, dtype, &splits, &need);
  if (st != ATTN_OK) return st;
  if (B == 0 || Sq == 0) return ATTN_OK;
  // Like attn_fwd_splitkv: a positive count must be one the plan keeps.
  if (num_splits > 0 && splits != num_splits) return ATTN_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return ATTN_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != ATTN_OK) return st;
  // Every partial result the merge reads is written first by the forward
  // kernel of the same call, so the scratch needs no clearing between
  // calls.
  return attn_fwd_splitkv(Q, K, V, O, LSE, B, Hq, Hkv, Sq, Skv, D, scale,
                          causal, input_pos, dtype, splits, scratch,
                          kNoAllocScratchBytes, stream);
}

}  // extern "C"
