// C ABI of the attention-forward library: argument checks, tile dispatch,
// tensor-map construction and the kernel launch.  No device memory is
// allocated here; the caller owns every buffer.
#include <cmath>
#include <cstdint>
#include <algorithm>
#include <vector>
#include <cstddef>
#include <cstdlib>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/attn.h"
#include "attn_bwd_kernel.cuh"
#include "attn_launch.h"

// Device status word: bit 0 = a pipeline wait ran out, bits 8-15 = role.
__device__ unsigned int g_attn_status;

namespace {

constexpr int kVersion = 100;  // 0.1.0
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s
constexpr int kMaxDevices = 64;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

std::mutex g_status_mu;
unsigned int* g_status_ptr[kMaxDevices] = {};
unsigned long long g_status_ctx[kMaxDevices] = {};  // context of the entry
int g_num_sms[kMaxDevices] = {};

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    g_encode_err = cudaGetDriverEntryPointByVersion(
        "cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// Address of the status word on the current device, looked up once per
// device and context (a device reset replaces the context, and the module
// holding the word is loaded again, possibly elsewhere).
unsigned int* status_ptr(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned long long ctx = 0;
  if (!attn::current_context_id(&ctx)) return nullptr;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (g_status_ptr[dev] == nullptr || g_status_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned int*>(p);
    g_status_ctx[dev] = ctx;
  }
  return g_status_ptr[dev];
}

// Streaming multiprocessors of a device (looked up once).
int num_sms(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (g_num_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
        cudaSuccess)
      return 0;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

unsigned long long timeout_ns() {
  static const unsigned long long t = [] {
    const char* e = std::getenv("ATTN_WAIT_TIMEOUT_NS");
    if (e != nullptr) {
      const unsigned long long v = std::strtoull(e, nullptr, 10);
      if (v > 0) return v;
    }
    return kDefaultTimeoutNs;
  }();
  return t;
}

struct Shape {
  int B, Hq, Hkv, Sq, Skv, D, causal, input_pos;
  int window = 0;  // sliding window in keys (causal only), 0: none
};

// Tile dispatch.  Few query rows with grouped K/V heads (group * Sq <= 128):
// one Q tile packs the rows of all query heads of a K/V head.  Otherwise a
// CTA owns two 128-row Q tiles: two query heads of one K/V group at the
// same rows when the group size is even, else 256 consecutive rows of one
// head.
bool pack_gqa(const Shape& s) {
  const int g = s.Hq / s.Hkv;
  return g >= 2 && static_cast<long long>(g) * s.Sq <= attn::cfg::kTM;
}
bool pair_heads(const Shape& s) { return (s.Hq / s.Hkv) % 2 == 0; }

long long m_blocks(const Shape& s) {
  const int rows = pair_heads(s) ? attn::cfg::kTM : attn::cfg::kBlockM;
  return (static_cast<long long>(s.Sq) + rows - 1) / rows;
}

// Unit order of the two-tile modes.  Heaviest m-block first (a longest-
// processing-time order over the persistent CTAs) whenever a causal mask
// makes units differ in work; without a mask every unit is equal, and the
// m-blocks of one head run together so the K/V in flight stays in L2.  (A
// causal offset far past the rows also makes units nearly equal -- the
// prefill chunk's see 29 to 32 key tiles -- yet there the head-major order
// measured 2 % slower than the balanced one.)
bool head_major(const Shape& s) { return !s.causal; }

long long grid_size(const Shape& s) {
  if (pack_gqa(s)) return static_cast<long long>(s.B) * s.Hkv;
  const long long units = pair_heads(s) ? static_cast<long long>(s.B) * (s.Hq / 2)
                                        : static_cast<long long>(s.B) * s.Hq;
  return m_blocks(s) * units;
}

attn_status_t check_scalars(const Shape& s, float scale, attn_dtype_t dtype) {
  if (s.B < 0 || s.Hq <= 0 || s.Hkv <= 0 || s.Sq < 0 || s.Skv <= 0 ||
      s.D <= 0 || s.input_pos < 0)
    return ATTN_ERR_INVALID_ARG;
  if (s.Hq % s.Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16 && dtype != ATTN_E4M3)
    return ATTN_ERR_INVALID_ARG;
  // A window is defined for causal attention only, and every query row
  // must see a key: the last row (position input_pos + Sq - 1) sees keys
  // from input_pos + Sq - window on.
  if (s.window < 0 || (s.window > 0 && !s.causal)) return ATTN_ERR_INVALID_ARG;
  if (s.window > 0 && s.Sq > 0 &&
      static_cast<long long>(s.input_pos) + s.Sq - s.window >= s.Skv)
    return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  // Row positions of the last (partial) tile must stay within int32.
  if (static_cast<long long>(s.input_pos) + s.Sq + 2 * attn::cfg::kBlockM >
      0x7fffffffLL)
    return ATTN_ERR_INVALID_ARG;
  // Planes (B*H) index a 32-bit tensor-map dimension and kernel ints.
  if (static_cast<long long>(s.B) * s.Hq > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  if (s.D != 64 && s.D != 128) return ATTN_ERR_UNSUPPORTED;
  if (dtype == ATTN_E4M3 && s.D != 128) return ATTN_ERR_UNSUPPORTED;
  if (grid_size(s) > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// Dispatch table keyed on (D, causal, S, dtype, group): 2 x 128 query rows
// per CTA with 128-key K/V tiles, or group*Sq packed rows for short query
// blocks; the ring depth depends on D (shared-memory budget).
struct TileChoice {
  int block_m, block_n, stages, smem_bytes;
};

TileChoice choose_tiles(const Shape& s, attn_dtype_t dtype) {
  const bool pack = pack_gqa(s);
  const bool fp8 = dtype == ATTN_E4M3;
  const int block_m = pack ? (s.Hq / s.Hkv) * s.Sq : attn::cfg::kBlockM;
  return TileChoice{block_m, attn::cfg::kTN, attn::fwd_stages(s.D, pack, fp8),
                    attn::fwd_smem_bytes(s.D, pack, fp8)};
}

// Bytes of one element of Q, K, V (the output O is 16-bit throughout).
size_t elem_bytes(attn_dtype_t dtype) { return dtype == ATTN_E4M3 ? 1 : 2; }

bool is_device_ptr(const void* p, int dev) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error state
    return false;
  }
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
    return false;
  return a.device == dev;
}

// 3-D map (D, S, planes) of a [planes, S, D] tensor; boxes of one 128-byte
// row segment (64 16-bit or 128 8-bit elements) x box_rows x box_planes
// with 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, attn_dtype_t dtype, int D,
              int S, long long planes, int box_rows = 128,
              int box_planes = 1) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (enc == nullptr) return false;
  const cuuint64_t es = elem_bytes(dtype);
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D),
                              static_cast<cuuint64_t>(S),
                              static_cast<cuuint64_t>(planes)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * es,
                                 static_cast<cuuint64_t>(S) * D * es};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es),
                             static_cast<cuuint32_t>(box_rows),
                             static_cast<cuuint32_t>(box_planes)};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUtensorMapDataType type =
      dtype == ATTN_E4M3   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
      : dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = enc(
      m, type, 3, const_cast<void*>(base), dims, strides, box, estride,
      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a);
  const uintptr_t y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

namespace attn {
bool current_context_id(unsigned long long* id) {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
  if (g_ctx_current == nullptr || g_ctx_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return false;
  if (ctx == nullptr) {
    // No context bound to this thread yet: cudaSetDevice binds (and if
    // needed creates) the current device's primary context.
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess)
      return false;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  }
  return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

int fwd_smem_bytes(int D, bool pack, bool fp8) {
  if (fp8)
    return pack ? Layout<128, true, true>::kSmemBytes
                : Layout<128, false, true>::kSmemBytes;
  if (pack)
    return D == 64 ? Layout<64, true>::kSmemBytes : Layout<128, true>::kSmemBytes;
  return D == 64 ? Layout<64>::kSmemBytes : Layout<128>::kSmemBytes;
}
int fwd_stages(int D, bool pack, bool fp8) {
  // Each slot holds one K or one V tile; a stage is a K and a V tile.
  if (fp8)
    return (pack ? Layout<128, true, true>::kSlots
                 : Layout<128, false, true>::kSlots) / 2;
  if (pack) return (D == 64 ? Layout<64, true>::kSlots : Layout<128, true>::kSlots) / 2;
  return (D == 64 ? Layout<64>::kSlots : Layout<128>::kSlots) / 2;
}
}  // namespace attn

namespace {

constexpr int kMaxSplits = 128;
// Largest key-range count merged inside a thread-block cluster (the
// portable cluster size).
constexpr int kMaxClusterSplits = attn::cfg::kMaxClusterRanges;
constexpr size_t kWorkspaceAlign = 256;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bytes of the split-KV workspace: fp32 partial outputs, then partial
// LSEs.
size_t splitkv_bytes(const Shape& s, int splits) {
  const size_t rows = static_cast<size_t>(s.B) * s.Hq * s.Sq;
  return round_up(static_cast<size_t>(splits) * rows * s.D * 4, kWorkspaceAlign) +
         round_up(static_cast<size_t>(splits) * rows * 4, kWorkspaceAlign);
}

// Split count and K/V tiles per split.  `splits` <= 0 picks the count
// with the shortest estimated time, in half steps of one CTA (a step: one
// 128-key K/V tile for the unit's Q tiles, about 1.4 us with D = 128):
// waves of units over the SMs times (tiles per range + a fixed cost per
// unit), plus the merge launch, and never less than streaming every K/V
// byte once from HBM (about 7 MB per step of time).  Fixed costs, fitted to
// GB300 timings of one pass and of 2-32 ranges over seven shapes (B1-8,
// 8-32 query heads, 1-1024 query rows, 4k-128k keys): one pass 4 steps
// (Q load, pipeline fill, epilogue), a unit of a cluster-merged launch 4,
// any other split unit 9 (its fp32 partial rows written out) and its merge
// launch 3.5.  Ties go to fewer ranges (less partial traffic).
void splitkv_shape(const Shape& s, int splits, int sms, int elem,
                   int* out_splits, int* out_tiles) {
  const int tiles = (s.Skv + attn::cfg::kTN - 1) / attn::cfg::kTN;
  if (splits <= 0) {
    const long long units = grid_size(s);
    const double kv_bytes = 2.0 * s.B * s.Hkv * static_cast<double>(s.Skv) *
                            s.D * elem;
    const long long floor2 =
        static_cast<long long>(2.0 * kv_bytes / 7.0e6);
    long long best = -1;
    const int cap = std::max(1, std::min(tiles, kMaxSplits));
    for (int c = 1; c <= cap; ++c) {
      const int per = (tiles + c - 1) / c;
      if (c > 1 && (tiles + per - 1) / per != c) continue;  // not a count
      const long long waves = (units * c + sms - 1) / sms;
      const bool cluster = c > 1 && pack_gqa(s) && c <= kMaxClusterSplits &&
                           units * c <= sms;
      const int unit2 = (c == 1 || cluster) ? 8 : 18;
      const int merge2 = (c == 1 || cluster) ? 0 : 7;
      const long long cost =
          std::max(waves * (2LL * per + unit2) + merge2, floor2);
      if (best < 0 || cost < best) {
        best = cost;
        splits = c;
      }
    }
  }
  splits = std::max(1, std::min({splits, tiles, kMaxSplits}));
  const int per = (tiles + splits - 1) / splits;
  *out_tiles = per;
  *out_splits = (tiles + per - 1) / per;  // no empty trailing range
}

// Checks shared by the entry points; fills the device, status word and SMs.
attn_status_t check_call(const Shape& s, float scale, attn_dtype_t dtype,
                         const void* Q, const void* K, const void* V, void* O,
                         float* LSE, int* dev, unsigned int** status,
                         int* sms) {
  attn_status_t st = check_scalars(s, scale, dtype);
  if (st != ATTN_OK) return st;
  if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr)
    return ATTN_ERR_INVALID_ARG;
  auto misaligned = [](const void* p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) != 0;
  };
  if (misaligned(Q, 16) || misaligned(K, 16) || misaligned(V, 16) ||
      misaligned(O, 16) || (LSE != nullptr && misaligned(LSE, 4)))
    return ATTN_ERR_ALIGNMENT;
  const size_t es = elem_bytes(dtype);
  const size_t o_bytes = static_cast<size_t>(s.B) * s.Hq * s.Sq * s.D * 2;
  const size_t q_bytes = static_cast<size_t>(s.B) * s.Hq * s.Sq * s.D * es;
  const size_t kv_bytes = static_cast<size_t>(s.B) * s.Hkv * s.Skv * s.D * es;
  if (overlaps(O, o_bytes, Q, q_bytes) || overlaps(O, o_bytes, K, kv_bytes) ||
      overlaps(O, o_bytes, V, kv_bytes))
    return ATTN_ERR_INVALID_ARG;
  if (cudaGetDevice(dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (!is_device_ptr(Q, *dev) || !is_device_ptr(K, *dev) ||
      !is_device_ptr(V, *dev) || !is_device_ptr(O, *dev) ||
      (LSE != nullptr && !is_device_ptr(LSE, *dev)))
    return ATTN_ERR_INVALID_ARG;
  *status = status_ptr(*dev);
  if (*status == nullptr) return ATTN_ERR_CUDA;
  *sms = num_sms(*dev);
  if (*sms <= 0) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

// ---------------------------------------------------------------- unit plan
// Work (in K/V steps) of two-tile unit u of a one-pass launch: the key
// tiles its later Q tile sees, from the first tile its earlier one sees.
// The same arithmetic as the kernel's unit decode and tile_keys, for the
// host's balancing only (a different count would only unbalance, never
// drop or repeat a unit).
int unit_steps(const Shape& s, long long u) {
  const long long mbs = m_blocks(s);
  const long long per_m = pair_heads(s) ? static_cast<long long>(s.B) * (s.Hq / 2)
                                        : static_cast<long long>(s.B) * s.Hq;
  const long long mb = head_major(s) ? u % mbs : mbs - 1 - u / per_m;
  const int tm = attn::cfg::kTM, tn = attn::cfg::kTN;
  int lo = 0, n_kv = 0;
  for (int t = 0; t < 2; ++t) {
    const long long m0 = pair_heads(s) ? mb * tm : mb * attn::cfg::kBlockM + t * tm;
    if (m0 >= s.Sq) continue;
    const long long pos_first = s.input_pos + m0;
    const long long pos_last = s.input_pos + std::min<long long>(m0 + tm, s.Sq) - 1;
    const long long kend = s.causal ? std::min<long long>(pos_last + 1, s.Skv) : s.Skv;
    const int hi = static_cast<int>((kend + tn - 1) / tn);
    if (t == 0 && s.window > 0)
      lo = static_cast<int>(std::max<long long>(0, pos_first - s.window + 1) / tn);
    n_kv = std::max(n_kv, hi - lo);
  }
  return n_kv;
}

// Unit assignment of a causal two-tile one-pass launch of `units` units on
// `grid` CTAs.  The zigzag rounds leave the busiest CTA 2-4 % above the mean
// (unit granularity: 7 units against 6); packing the units heaviest first
// into the first CTA with room under a capacity, searched from the mean
// upwards (first-fit decreasing, as in the MULTIFIT method of Coffman,
// Garey and Johnson, 1978), leaves it within a fraction of a percent.  Each
// unit costs its K/V steps plus 1.5 (a unit boundary, measured).  Returns
// false (keep the zigzag rounds) when the plan would not be better.
struct UnitPlan {
  int units = 0;
  long long work_max = 0;     // busiest CTA, half K/V steps
  long long work_rounds = 0;  // the same under the zigzag rounds
  unsigned short start[attn::kMaxPlanCtas + 1];
  unsigned short unit[attn::kMaxPlanUnits];
};

// Plans the causal two-tile one-pass launches (other launches keep the
// rounds: their units are equal, or they take another path).
bool plannable(const Shape& s) {
  return s.causal && !pack_gqa(s);
}

bool make_plan(const Shape& s, int units, int grid, UnitPlan* plan) {
  plan->work_max = plan->work_rounds = 0;
  if (!plannable(s) || units <= grid || units > attn::kMaxPlanUnits ||
      grid > attn::kMaxPlanCtas)
    return false;
  std::vector<int> cost(units);  // in half steps
  long long total = 0;
  int cmax = 0;
  for (int u = 0; u < units; ++u) {
    const int n = unit_steps(s, u);
    cost[u] = n > 0 ? 2 * n + 3 : 0;
    total += cost[u];
    cmax = std::max(cmax, cost[u]);
  }
  // Makespan of the zigzag rounds.
  std::vector<long long> load(grid, 0);
  for (int u = 0; u < units; ++u) {
    const int k = u / grid, r = u % grid;
    load[(k & 1) ? grid - 1 - r : r] += cost[u];
  }
  const long long zigzag = *std::max_element(load.begin(), load.end());
  plan->work_max = plan->work_rounds = zigzag;
  // Heaviest first; equal costs keep the unit order (heads in turn).
  std::vector<int> order(units);
  for (int u = 0; u < units; ++u) order[u] = u;
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return cost[a] > cost[b]; });
  std::vector<int> bin(units);
  auto pack = [&](long long cap) {
    std::fill(load.begin(), load.end(), 0);
    for (int u : order) {
      int c = 0;
      while (c < grid && load[c] + cost[u] > cap) ++c;
      if (c == grid) return false;
      load[c] += cost[u];
      bin[u] = c;
    }
    return true;
  };
  long long lo = std::max<long long>((total + grid - 1) / grid, cmax);
  long long hi = zigzag - 1;  // a plan must beat the rounds
  if (lo > hi || !pack(hi)) return false;
  while (lo < hi) {  // smallest capacity that packs
    const long long mid = (lo + hi) / 2;
    if (pack(mid)) hi = mid; else lo = mid + 1;
  }
  pack(hi);
  plan->work_max = *std::max_element(load.begin(), load.end());
  // CTA c's units, heaviest first (the order they were packed in).
  std::vector<int> count(grid, 0);
  for (int u = 0; u < units; ++u) ++count[bin[u]];
  plan->start[0] = 0;
  for (int c = 0; c < grid; ++c)
    plan->start[c + 1] = static_cast<unsigned short>(plan->start[c] + count[c]);
  std::vector<int> fill(plan->start, plan->start + grid);
  for (int u : order) plan->unit[fill[bin[u]]++] = static_cast<unsigned short>(u);
  plan->units = units;
  return true;
}

// Plans are computed once per launch shape and kept (a few dozen bytes of
// key and 2.4 KB of plan each, the most recent kPlanCache shapes).
constexpr int kPlanCache = 16;
struct PlanEntry {
  long long key[10];
  bool used = false, valid = false;
  UnitPlan plan;
};
std::mutex g_plan_mu;
PlanEntry g_plans[kPlanCache];
int g_plan_next = 0;

// Copies the plan of this launch shape into `p` (computing it on first
// use); leaves p.plan_units at 0 when the zigzag rounds stay.
void apply_plan(const Shape& s, int units, int grid, attn::FwdParams* p) {
  const long long key[10] = {s.B, s.Hq, s.Hkv, s.Sq, s.Skv, s.causal,
                             s.input_pos, s.window, units, grid};
  std::lock_guard<std::mutex> lock(g_plan_mu);
  PlanEntry* e = nullptr;
  for (PlanEntry& c : g_plans)
    if (c.used && std::equal(key, key + 10, c.key)) e = &c;
  if (e == nullptr) {
    e = &g_plans[g_plan_next];
    g_plan_next = (g_plan_next + 1) % kPlanCache;
    std::copy(key, key + 10, e->key);
    e->used = true;
    e->valid = make_plan(s, units, grid, &e->plan);
  }
  if (!e->valid) return;
  p->plan_units = e->plan.units;
  std::copy(e->plan.start, e->plan.start + grid + 1, p->plan_start);
  std::copy(e->plan.unit, e->plan.unit + units, p->plan_unit);
}

// Builds the tensor maps and parameters and launches the forward kernel.
// `scale` is the score factor (FP8: times the Q and K descales), `o_scale`
// multiplies O (FP8: the V descale; else 1).
attn_status_t launch_forward(const Shape& s, const void* Q, const void* K,
                             const void* V, void* O, float* LSE, float scale,
                             attn_dtype_t dtype, unsigned int* status, int sms,
                             int splits, int split_tiles, float* o_part,
                             float* lse_part,
                             cudaStream_t stream, float o_scale = 1.f,
                             unsigned long long timeout = 0,
                             int withhold_first_load = 0) {
  CUtensorMap tq, tk, tv, to;
  const long long q_planes = static_cast<long long>(s.B) * s.Hq;
  const long long kv_planes = static_cast<long long>(s.B) * s.Hkv;
  const bool pack = pack_gqa(s);
  const int group = s.Hq / s.Hkv;
  const bool q_ok = pack ? make_map(&tq, Q, dtype, s.D, s.Sq, q_planes, s.Sq,
                                    group)
                         : make_map(&tq, Q, dtype, s.D, s.Sq, q_planes);
  if (!q_ok || !make_map(&tk, K, dtype, s.D, s.Skv, kv_planes) ||
      !make_map(&tv, V, dtype, s.D, s.Skv, kv_planes))
    return ATTN_ERR_CUDA;
  // O (16-bit; bf16 for E4M3 inputs), stored by TMA in 64-column boxes by
  // the two-tile one-pass variants.  The packed and split-KV variants store
  // per thread and never read this map.
  if (!pack && o_part == nullptr) {
    if (!make_map(&to, O, dtype == ATTN_E4M3 ? ATTN_BF16 : dtype, s.D, s.Sq,
                  q_planes))
      return ATTN_ERR_CUDA;
  } else {
    to = tq;
  }

  attn::FwdParams p{};
  p.B = s.B;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.Sq = s.Sq;
  p.Skv = s.Skv;
  p.causal = s.causal != 0;
  p.input_pos = s.causal != 0 ? s.input_pos : 0;
  p.window = s.causal != 0 ? s.window : 0;
  p.num_m_blocks = static_cast<int>(m_blocks(s));
  p.pair_heads = pair_heads(s);
  p.head_major = !pack && head_major(s);
  p.pack_gqa = pack;
  p.group = group;
  // D * element-size bytes per row: 128 rows per tile, or group*Sq packed.
  p.q_tile_bytes = static_cast<int>(s.D * elem_bytes(dtype)) *
                   (pack ? group * s.Sq : attn::cfg::kTM);
  p.scale_log2 = std::fabs(scale) * 1.4426950408889634f;
  p.negate_scores = scale < 0.f;
  p.o_scale = o_scale;
  p.o = O;
  p.lse = LSE;
  p.num_splits = splits;
  p.split_tiles = split_tiles;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.num_units = static_cast<int>(grid_size(s) * splits);
  p.fd_splits = attn::make_fast_div(splits);
  p.fd_m_blocks = attn::make_fast_div(p.num_m_blocks);
  p.fd_heads = attn::make_fast_div(p.pair_heads ? s.Hq / 2 : s.Hq);
  p.fd_per_m = attn::make_fast_div(s.B * p.fd_heads.d);
  p.fd_group = attn::make_fast_div(group);
  p.fd_hkv = attn::make_fast_div(s.Hkv);
  // Packed split-KV whose units all fit in one wave: the key ranges of a
  // (batch, K/V head) run as one cluster and merge over distributed shared
  // memory.  (The workspace still has to be valid: it is the fallback.)
  // Otherwise the merge is a second launch over the whole GPU.
  p.cluster_merge = pack && splits > 1 && splits <= kMaxClusterSplits &&
                    p.num_units <= sms && o_part != nullptr;
  p.status = status;
  p.timeout_ns = timeout != 0 ? timeout : timeout_ns();
  p.withhold_first_load = withhold_first_load;

  // Persistent launch: at most one CTA per SM, each walking its units.
  const int grid = static_cast<int>(std::min<long long>(p.num_units, sms));
  // Causal one-pass two-tile launches: units differ in work, so pack them
  // onto the CTAs on the host.
  if (plannable(s) && o_part == nullptr && withhold_first_load == 0)
    apply_plan(s, p.num_units, grid, &p);
  const bool bf16 = dtype == ATTN_BF16;
  auto launch = [&]() {
    return dtype == ATTN_E4M3
          ? (pack ? attn::launch_fwd_d128_fp8_packed(tq, tk, tv, to, p, grid,
                                                   stream)
                  : attn::launch_fwd_d128_fp8(tq, tk, tv, to, p, grid, stream))
      : s.D == 64
          ? (pack ? attn::launch_fwd_d64_packed(bf16, tq, tk, tv, to, p, grid,
                                              stream)
                  : attn::launch_fwd_d64(bf16, tq, tk, tv, to, p, grid, stream))
          : (pack ? attn::launch_fwd_d128_packed(bf16, tq, tk, tv, to, p, grid,
                                               stream)
                  : attn::launch_fwd_d128(bf16, tq, tk, tv, to, p, grid, stream));
  };
  cudaError_t err = launch();
  if (err != cudaSuccess && p.cluster_merge) {
    // No cluster of that size could be placed: merge through the
    // workspace instead.
    cudaGetLastError();
    p.cluster_merge = 0;
    err = launch();
  }
  if (err == cudaSuccess && o_part != nullptr && !p.cluster_merge)
    err = attn::launch_merge(s.D, dtype != ATTN_F16, p, sms, stream);
  return err == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// attn_fwd / attn_fwd_window.
attn_status_t fwd_impl(const Shape& s, const void* Q, const void* K,
                       const void* V, void* O, float* LSE, float scale,
                       attn_dtype_t dtype, attn_stream_t stream,
                       unsigned long long timeout = 0,
                       int withhold_first_load = 0) {
  // E4M3 inputs need their descale factors: attn_fwd_fp8 only.
  if (dtype == ATTN_E4M3) return ATTN_ERR_INVALID_ARG;
  attn_status_t st = check_scalars(s, scale, dtype);
  if (st != ATTN_OK) return st;
  if (s.B == 0 || s.Sq == 0) return ATTN_OK;
  int dev = 0, sms = 0;
  unsigned int* status = nullptr;
  st = check_call(s, scale, dtype, Q, K, V, O, LSE, &dev, &status, &sms);
  if (st != ATTN_OK) return st;
  const int tiles = (s.Skv + attn::cfg::kTN - 1) / attn::cfg::kTN;
  return launch_forward(s, Q, K, V, O, LSE, scale, dtype, status, sms, 1,
                        tiles, nullptr, nullptr,
                        reinterpret_cast<cudaStream_t>(stream), 1.f, timeout,
                        withhold_first_load);
}

// Clears the status bits a status query has reported (bits set since, by
// kernels on other streams, stay).
__global__ void clear_status_bits(unsigned int* status, unsigned int bits) {
  atomicAnd(status, ~bits);
}

// attn_fwd_splitkv / attn_fwd_splitkv_window.
attn_status_t splitkv_impl(const Shape& s, const void* Q, const void* K,
                           const void* V, void* O, float* LSE, float scale,
                           attn_dtype_t dtype, int num_splits, void* workspace,
                           size_t workspace_bytes, attn_stream_t stream,
                           float o_scale = 1.f) {
  attn_status_t st = check_scalars(s, scale, dtype);
  if (st != ATTN_OK) return st;
  if (s.B == 0 || s.Sq == 0) return ATTN_OK;
  if (num_splits < 1 || num_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  unsigned int* status = nullptr;
  st = check_call(s, scale, dtype, Q, K, V, O, LSE, &dev, &status, &sms);
  if (st != ATTN_OK) return st;
  int splits = 0, tiles = 0;
  splitkv_shape(s, num_splits, sms, elem_bytes(dtype), &splits, &tiles);
  if (splits != num_splits) return ATTN_ERR_INVALID_ARG;  // not a planned count
  if (workspace == nullptr ||
      reinterpret_cast<uintptr_t>(workspace) % kWorkspaceAlign != 0)
    return ATTN_ERR_ALIGNMENT;
  if (workspace_bytes < splitkv_bytes(s, splits)) return ATTN_ERR_INVALID_ARG;
  if (!is_device_ptr(workspace, dev)) return ATTN_ERR_INVALID_ARG;
  const size_t rows = static_cast<size_t>(s.B) * s.Hq * s.Sq;
  const size_t o_bytes =
      round_up(static_cast<size_t>(splits) * rows * s.D * 4, kWorkspaceAlign);
  char* ws = static_cast<char*>(workspace);
  // The forward launch, then (unless its key ranges merge in clusters) the
  // merge launch.
  return launch_forward(
      s, Q, K, V, O, LSE, scale, dtype, status, sms, splits, tiles,
      reinterpret_cast<float*>(ws), reinterpret_cast<float*>(ws + o_bytes),
      reinterpret_cast<cudaStream_t>(stream), o_scale);
}

// attn_fwd_fp8: the descales fold into the score factor (Q, K) and into
// the output factor (V); num_splits == 0 is the single-pass forward.
attn_status_t fp8_impl(const Shape& s, const void* Q, const void* K,
                       const void* V, void* O, float* LSE, float scale,
                       float q_descale, float k_descale, float v_descale,
                       int num_splits, void* workspace,
                       size_t workspace_bytes, attn_stream_t stream) {
  if (!std::isfinite(scale) || !std::isfinite(q_descale) ||
      !std::isfinite(k_descale) || !std::isfinite(v_descale))
    return ATTN_ERR_INVALID_ARG;
  const double eff = static_cast<double>(scale) * q_descale * k_descale;
  if (!(std::fabs(eff) <= 3.4e38)) return ATTN_ERR_INVALID_ARG;
  const float s_eff = static_cast<float>(eff);
  if (num_splits < 0) return ATTN_ERR_INVALID_ARG;
  if (num_splits > 0)
    return splitkv_impl(s, Q, K, V, O, LSE, s_eff, ATTN_E4M3, num_splits,
                        workspace, workspace_bytes, stream, v_descale);
  attn_status_t st = check_scalars(s, s_eff, ATTN_E4M3);
  if (st != ATTN_OK) return st;
  if (s.B == 0 || s.Sq == 0) return ATTN_OK;
  int dev = 0, sms = 0;
  unsigned int* status = nullptr;
  st = check_call(s, s_eff, ATTN_E4M3, Q, K, V, O, LSE, &dev, &status, &sms);
  if (st != ATTN_OK) return st;
  const int tiles = (s.Skv + attn::cfg::kTN - 1) / attn::cfg::kTN;
  return launch_forward(s, Q, K, V, O, LSE, s_eff, ATTN_E4M3, status, sms, 1,
                        tiles, nullptr, nullptr,
                        reinterpret_cast<cudaStream_t>(stream), v_descale);
}

// Rows per (batch, query head) plane of the backward's per-row arrays:
// Sq padded to whole 128-row tiles.
size_t bwd_sq_pad(const Shape& s) {
  return (static_cast<size_t>(s.Sq) + attn::bwd::kT - 1) / attn::bwd::kT *
         attn::bwd::kT;
}

// Bytes of the backward workspace: lse2 and D, fp32 per padded query row.
size_t bwd_workspace_bytes(const Shape& s) {
  const size_t rows = static_cast<size_t>(s.B) * s.Hq * bwd_sq_pad(s);
  return 2 * round_up(rows * 4, kWorkspaceAlign);
}

attn_status_t bwd_impl(const Shape& s, const void* Q, const void* K,
                       const void* V, const void* O, const float* LSE,
                       const void* dO, void* dQ, void* dK, void* dV,
                       float scale, attn_dtype_t dtype, void* workspace,
                       size_t workspace_bytes, attn_stream_t stream) {
  if (dtype == ATTN_E4M3) return ATTN_ERR_UNSUPPORTED;  // 16-bit only
  attn_status_t st = check_scalars(s, scale, dtype);
  if (st != ATTN_OK) return st;
  if (s.B == 0) return ATTN_OK;
  const void* in16[] = {Q, K, V, O, dO};
  void* out16[] = {dQ, dK, dV};
  for (const void* ptr : in16)
    if (ptr == nullptr) return ATTN_ERR_INVALID_ARG;
  for (void* ptr : out16)
    if (ptr == nullptr) return ATTN_ERR_INVALID_ARG;
  if (LSE == nullptr) return ATTN_ERR_INVALID_ARG;
  auto misaligned = [](const void* ptr, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(ptr) % a) != 0;
  };
  for (const void* ptr : in16)
    if (misaligned(ptr, 16)) return ATTN_ERR_ALIGNMENT;
  for (void* ptr : out16)
    if (misaligned(ptr, 16)) return ATTN_ERR_ALIGNMENT;
  if (misaligned(LSE, 4)) return ATTN_ERR_ALIGNMENT;
  const size_t q_bytes = static_cast<size_t>(s.B) * s.Hq * s.Sq * s.D * 2;
  const size_t kv_bytes = static_cast<size_t>(s.B) * s.Hkv * s.Skv * s.D * 2;
  const size_t lse_bytes = static_cast<size_t>(s.B) * s.Hq * s.Sq * 4;
  // Outputs must not overlap any input or each other.
  const void* ins[] = {Q, K, V, O, dO, LSE};
  const size_t in_bytes[] = {q_bytes, kv_bytes, kv_bytes, q_bytes, q_bytes,
                             lse_bytes};
  const size_t out_bytes[] = {q_bytes, kv_bytes, kv_bytes};
  for (int o = 0; o < 3; ++o) {
    for (int i = 0; i < 6; ++i)
      if (overlaps(out16[o], out_bytes[o], ins[i], in_bytes[i]))
        return ATTN_ERR_INVALID_ARG;
    for (int o2 = o + 1; o2 < 3; ++o2)
      if (overlaps(out16[o], out_bytes[o], out16[o2], out_bytes[o2]))
        return ATTN_ERR_INVALID_ARG;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  for (const void* ptr : ins)
    if (!is_device_ptr(ptr, dev)) return ATTN_ERR_INVALID_ARG;
  for (void* ptr : out16)
    if (!is_device_ptr(ptr, dev)) return ATTN_ERR_INVALID_ARG;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (s.Sq == 0) {
    // No query: the gradients of K and V are zero.
    if (cudaMemsetAsync(dK, 0, kv_bytes, cs) != cudaSuccess ||
        cudaMemsetAsync(dV, 0, kv_bytes, cs) != cudaSuccess)
      return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  if (workspace == nullptr ||
      reinterpret_cast<uintptr_t>(workspace) % kWorkspaceAlign != 0)
    return ATTN_ERR_ALIGNMENT;
  if (workspace_bytes < bwd_workspace_bytes(s)) return ATTN_ERR_INVALID_ARG;
  if (!is_device_ptr(workspace, dev)) return ATTN_ERR_INVALID_ARG;
  for (int i = 0; i < 6; ++i)
    if (overlaps(workspace, workspace_bytes, ins[i], in_bytes[i]))
      return ATTN_ERR_INVALID_ARG;
  for (int o = 0; o < 3; ++o)
    if (overlaps(workspace, workspace_bytes, out16[o], out_bytes[o]))
      return ATTN_ERR_INVALID_ARG;
  unsigned int* status = status_ptr(dev);
  if (status == nullptr) return ATTN_ERR_CUDA;

  const long long q_planes = static_cast<long long>(s.B) * s.Hq;
  const long long kv_planes = static_cast<long long>(s.B) * s.Hkv;
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!make_map(&tq, Q, dtype, s.D, s.Sq, q_planes) ||
      !make_map(&tk, K, dtype, s.D, s.Skv, kv_planes) ||
      !make_map(&tv, V, dtype, s.D, s.Skv, kv_planes) ||
      !make_map(&tdo, dO, dtype, s.D, s.Sq, q_planes) ||
      !make_map(&tdq, dQ, dtype, s.D, s.Sq, q_planes))
    return ATTN_ERR_CUDA;
  const size_t rows = static_cast<size_t>(s.B) * s.Hq * bwd_sq_pad(s);
  float* lse2 = static_cast<float*>(workspace);
  float* delta = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                          round_up(rows * 4, kWorkspaceAlign));
  attn::BwdParams p{};
  p.B = s.B;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.Sq = s.Sq;
  p.Skv = s.Skv;
  p.causal = s.causal != 0;
  p.input_pos = s.causal != 0 ? s.input_pos : 0;
  p.window = s.causal != 0 ? s.window : 0;
  p.group = s.Hq / s.Hkv;
  p.q_tiles = (s.Sq + attn::bwd::kT - 1) / attn::bwd::kT;
  p.k_tiles = (s.Skv + attn::bwd::kT - 1) / attn::bwd::kT;
  p.sq_pad = static_cast<int>(bwd_sq_pad(s));
  p.scale_log2 = std::fabs(scale) * 1.4426950408889634f;
  p.negate_scores = scale < 0.f;
  p.scale = scale;
  p.lse2 = lse2;
  p.delta = delta;
  p.dq = dQ;
  p.dk = dK;
  p.dv = dV;
  p.status = status;
  p.timeout_ns = timeout_ns();
  const cudaError_t err = attn::launch_bwd(s.D, dtype == ATTN_BF16, tq, tk,
                                           tv, tdo, tdq, O, dO, LSE, p, cs);
  return err == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

attn_status_t attn_fwd(const void* Q, const void* K, const void* V, void* O,
                       float* LSE, int B, int Hq, int Hkv, int Sq, int Skv,
                       int D, float scale, int causal, int input_pos,
                       attn_dtype_t dtype, attn_stream_t stream) {
  const Shape s{B, Hq, Hkv, Sq, Skv, D, causal != 0, input_pos};
  return fwd_impl(s, Q, K, V, O, LSE, scale, dtype, stream);
}

attn_status_t attn_fwd_window(const void* Q, const void* K, const void* V,
                              void* O, float* LSE, int B, int Hq, int Hkv,
                              int Sq, int Skv, int D, float scale, int causal,
                              int input_pos, int window, attn_dtype_t dtype,
                              attn_stream_t stream) {
  const Shape s{B, Hq, Hkv, Sq, Skv, D, causal != 0, input_pos, window};
  return fwd_impl(s, Q, K, V, O, LSE, scale, dtype, stream);
}

attn_status_t attn_splitkv_plan(int B, int Hq, int Hkv, int Sq, int Skv, int D,
                                int causal, int input_pos, attn_dtype_t dtype,
                                int* num_splits, size_t* workspace_bytes) {
  const Shape s{B, Hq, Hkv, Sq, Skv, D, causal != 0, input_pos};
  const attn_status_t st = check_scalars(s, 1.0f, dtype);
  if (st != ATTN_OK) return st;
  if (num_splits == nullptr) return ATTN_ERR_INVALID_ARG;
  int sms = 0;
  if (*num_splits <= 0) {
    // The current device's SM count (the GB300's 152 without a device).
    int dev = -1;
    if (cudaGetDevice(&dev) == cudaSuccess) sms = num_sms(dev);
    cudaGetLastError();  // no device: not an error of the caller's
    if (sms <= 0) sms = 152;
  }
  int splits = 0, tiles = 0;
  splitkv_shape(s, *num_splits, sms, elem_bytes(dtype), &splits, &tiles);
  *num_splits = splits;
  if (workspace_bytes != nullptr) *workspace_bytes = splitkv_bytes(s, splits);
  return ATTN_OK;
}

attn_status_t attn_fwd_splitkv(const void* Q, const void* K, const void* V,
                               void* O, float* LSE, int B, int Hq, int Hkv,
                               int Sq, int Skv, int D, float scale, int causal,
                               int input_pos, attn_dtype_t dtype,
                               int num_splits, void* workspace,
                               size_t workspace_bytes, attn_stream_t stream) {
  const Shape s{B, Hq, Hkv, Sq, Skv, D, causal != 0, input_pos};
  if (dtype == ATTN_E4M3) return ATTN_ERR_INVALID_ARG;  // attn_fwd_fp8
  return splitkv_impl(s, Q, K, V, O, LSE, scale, dtype, num_splits,
                      workspace, workspace_bytes, stream);
}

attn_status_t attn_fwd_splitkv_window(const void* Q, const void* K,
                                      const void* V, void* O, float* LSE,
                                      int B, int Hq, int Hkv, int Sq, int Skv,
                                      int D, float scale, int causal,
                                      int input_pos, int window,
                                      attn_dtype_t dtype, int num_splits,
                                      void* workspace, size_t workspace_bytes,
                                      attn_stream_t stream) {
  const Shape s{B, Hq, Hkv, Sq, Skv, D, causal != 0, input_pos, window};
  if (dtype == ATTN_E4M3) return ATTN_ERR_INVALID_ARG;  // attn_fwd_fp8
  return splitkv_impl(s, Q, K, V, O, LSE, scale, dtype, num_splits,
                      workspace, workspace_bytes, stream);
}

attn_status_t attn_fwd_fp8(const void* Q, const void* K, const void* V,
                           void* O, float* LSE, int B, int Hq, int Hkv,
                           int Sq, int Skv, int D, float scale,
                           float q_descale, float k_descale, float v_descale,
                           int causal, int input_pos, int window,
                           int num_splits, void* workspace,
                           size_t workspace_bytes, attn_stream_t stream) {
  const Shape s{B, Hq, Hkv, Sq, Skv, D, causal != 0, input_pos, window};
  return fp8_impl(s, Q, K, V, O, LSE, scale, q_descale, k_descale, v_descale,
                  num_splits, workspace, workspace_bytes, stream);
}

size_t attn_bwd_workspace_bytes(int B, int Hq, int Sq) {
  if (B < 0 || Hq < 0 || Sq < 0) return 0;
  const Shape s{B, Hq, 1, Sq, 1, 64, 0, 0};
  return bwd_workspace_bytes(s);
}

attn_status_t attn_bwd(const void* Q, const void* K, const void* V,
                       const void* O, const float* LSE, const void* dO,
                       void* dQ, void* dK, void* dV, int B, int Hq, int Hkv,
                       int Sq, int Skv, int D, float scale, int causal,
                       int input_pos, int window, attn_dtype_t dtype,
                       void* workspace, size_t workspace_bytes,
                       attn_stream_t stream) {
  const Shape s{B, Hq, Hkv, Sq, Skv, D, causal != 0, input_pos, window};
  return bwd_impl(s, Q, K, V, O, LSE, dO, dQ, dK, dV, scale, dtype,
                  workspace, workspace_bytes, stream);
}

const char* attn_status_string(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_ALIGNMENT: return "misaligned pointer";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device pipeline wait timed out";
  }
  return "unknown status";
}

attn_status_t attn_device_status(unsigned int* code) {
  if (code != nullptr) *code = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_attn_status, sizeof(v)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (v != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(zero)) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  if (code != nullptr) *code = v;
  return v != 0 ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

attn_status_t attn_stream_status(attn_stream_t stream, unsigned int* code) {
  if (code != nullptr) *code = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned int* status = status_ptr(dev);
  if (status == nullptr) return ATTN_ERR_CUDA;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // Ordered after the work already on `stream`; other streams keep running.
  unsigned int v = 0;
  if (cudaMemcpyAsync(&v, status, sizeof(v), cudaMemcpyDeviceToHost, cs) !=
          cudaSuccess ||
      cudaStreamSynchronize(cs) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (v != 0) {
    clear_status_bits<<<1, 1, 0, cs>>>(status, v);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  }
  if (code != nullptr) *code = v;
  return v != 0 ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

attn_status_t attn_selftest_wait_timeout(const void* Q, const void* K,
                                         const void* V, void* O, float* LSE,
                                         int B, int Hq, int Hkv, int Sq,
                                         int Skv, int D, float scale,
                                         int causal, int input_pos,
                                         attn_dtype_t dtype,
                                         unsigned long long timeout_ns,
                                         attn_stream_t stream) {
  if (timeout_ns == 0) return ATTN_ERR_INVALID_ARG;
  const Shape s{B, Hq, Hkv, Sq, Skv, D, causal != 0, input_pos};
  return fwd_impl(s, Q, K, V, O, LSE, scale, dtype, stream, timeout_ns, 1);
}

attn_status_t attn_tile_config(int B, int Hq, int Hkv, int Sq, int Skv, int D,
                               int causal, int input_pos, attn_dtype_t dtype,
                               int* block_m, int* block_n, int* stages,
                               int* grid, int* smem_bytes) {
  const Shape s{B, Hq, Hkv, Sq, Skv, D, causal != 0, input_pos};
  const attn_status_t st = check_scalars(s, 1.0f, dtype);
  if (st != ATTN_OK) return st;
  const TileChoice t = choose_tiles(s, dtype);
  if (block_m) *block_m = t.block_m;
  if (block_n) *block_n = t.block_n;
  if (stages) *stages = t.stages;
  if (grid) *grid = static_cast<int>(grid_size(s));
  if (smem_bytes) *smem_bytes = t.smem_bytes;
  return ATTN_OK;
}

attn_status_t attn_dispatch(int B, int Hq, int Hkv, int Sq, int Skv, int D,
                            int causal, int input_pos, int window,
                            attn_dtype_t dtype, int num_splits,
                            attn_dispatch_t* out) {
  if (out == nullptr) return ATTN_ERR_INVALID_ARG;
  const Shape s{B, Hq, Hkv, Sq, Skv, D, causal != 0, input_pos, window};
  const attn_status_t st = check_scalars(s, 1.0f, dtype);
  if (st != ATTN_OK) return st;
  if (num_splits < 0 || num_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  const TileChoice t = choose_tiles(s, dtype);
  const bool pack = pack_gqa(s);
  int splits = 1, tiles = 0;
  if (num_splits > 0)
    splitkv_shape(s, num_splits, 1, elem_bytes(dtype), &splits, &tiles);
  const bool split = num_splits > 0;
  attn_dispatch_t d{};
  d.block_m = t.block_m;
  d.block_n = t.block_n;
  d.q_tiles = pack ? 1 : 2;
  d.paired = !pack && pair_heads(s);
  d.s_buffers = (!pack && s.D == 64) ? 3 : 2;
  d.stages = t.stages;
  d.order = (!pack && head_major(s)) ? 1 : 0;
  // The current device's SM count (the GB300's 152 without a device).
  int dev = -1, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) sms = num_sms(dev);
  cudaGetLastError();  // no device: not an error of the caller's
  if (sms <= 0) sms = 152;
  if (!split && plannable(s)) {
    // The launch assigns causal units by a host-packed plan when one beats
    // the zigzag rounds; the grid is the SM count.
    const int units = static_cast<int>(grid_size(s));
    UnitPlan* plan = new UnitPlan;
    if (make_plan(s, units, std::min(units, sms), plan)) d.order = 2;
    delete plan;
  }
  d.o_store = (!pack && !split) ? 1 : 0;
  d.hold_scores = pack ? 0 : 1;
  d.num_splits = split ? splits : 0;
  d.units = static_cast<int>(grid_size(s) * splits);
  d.smem_bytes = t.smem_bytes;
  d.merge = !split ? 0
            : (pack && splits > 1 && splits <= kMaxClusterSplits &&
               d.units <= sms)
                ? 1
                : 2;
  // Static names: D x element type x tile mode x order x O store.
  static const char* const kNames[2][3][3][3][2] = {
#define ATTN_N(d, e, m, o, st) "d" d "." e "." m "." o "." st
#define ATTN_O(d, e, m)                                          \
  {{ATTN_N(d, e, m, "lpt", "rows"), ATTN_N(d, e, m, "lpt", "tma")}, \
   {ATTN_N(d, e, m, "head-major", "rows"),                       \
    ATTN_N(d, e, m, "head-major", "tma")},                       \
   {ATTN_N(d, e, m, "plan", "rows"), ATTN_N(d, e, m, "plan", "tma")}}
#define ATTN_M(d, e)                                                \
  {ATTN_O(d, e, "paired-heads"), ATTN_O(d, e, "256-rows"),           \
   ATTN_O(d, e, "gqa-packed")}
      {ATTN_M("64", "f16"), ATTN_M("64", "bf16"), ATTN_M("64", "e4m3")},
      {ATTN_M("128", "f16"), ATTN_M("128", "bf16"), ATTN_M("128", "e4m3")}};
#undef ATTN_M
#undef ATTN_O
#undef ATTN_N
  const int mode = pack ? 2 : (d.paired ? 0 : 1);
  d.name =
      kNames[s.D == 128][static_cast<int>(dtype)][mode][d.order][d.o_store];
  *out = d;
  return ATTN_OK;
}

attn_status_t attn_unit_plan(int B, int Hq, int Hkv, int Sq, int Skv, int D,
                             int causal, int input_pos, int window, int grid,
                             int* planned, long long* work_max,
                             long long* work_rounds, int* unit_order,
                             int* cta_start) {
  if (planned == nullptr || work_max == nullptr || work_rounds == nullptr ||
      grid < 1)
    return ATTN_ERR_INVALID_ARG;
  const Shape s{B, Hq, Hkv, Sq, Skv, D, causal != 0, input_pos, window};
  const attn_status_t st = check_scalars(s, 1.0f, ATTN_BF16);
  if (st != ATTN_OK) return st;
  const long long units = grid_size(s);
  const int g = static_cast<int>(std::min<long long>(units, grid));
  UnitPlan* plan = new UnitPlan;
  const bool ok = units > 0 && units <= 0x7fffffffLL &&
                  make_plan(s, static_cast<int>(units), g, plan);
  *planned = ok ? 1 : 0;
  if (ok) {
    *work_max = plan->work_max;
    *work_rounds = plan->work_rounds;
    if (unit_order != nullptr)
      for (int i = 0; i < plan->units; ++i) unit_order[i] = plan->unit[i];
    if (cta_start != nullptr)
      for (int c = 0; c <= g; ++c) cta_start[c] = plan->start[c];
  } else {
    // The rounds: busiest CTA of the zigzag order (when the plan had a say).
    *work_max = *work_rounds = plan->work_rounds;
  }
  delete plan;
  return ATTN_OK;
}

int attn_version(void) { return kVersion; }

}  // extern "C"
