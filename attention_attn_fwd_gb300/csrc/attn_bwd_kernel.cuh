// Backward pass of the attention forward on sm_103a: dQ, dK, dV for an
// upstream gradient dO.
//
// "Flash Attention from Scratch" lists the backward pass as future work
// (section "What's Next") and gives no design; this is the recomputation
// scheme of the flash method -- nothing of size Sq x Skv is stored, P is
// rebuilt tile by tile from the forward's log-sum-exp -- built from the
// forward kernel's tcgen05 / TMA pieces.  With lse2_i = LSE_i log2(e),
// c = |scale| log2(e) and D_i = sum_d dO_id O_id:
//   P_ij  = 2^(s_ij c - lse2_i)          (s_ij = +-q_i.k_j, sign of scale)
//   dV_j  = sum_i P_ij dO_i
//   dP_ij = dO_i . V_j,   dS_ij = P_ij (dP_ij - D_i)
//   dQ_i  = scale sum_j dS_ij K_j,       dK_j = scale sum_i dS_ij Q_i
// Three launches: a row pass computing D and lse2; the dK/dV kernel (one
// CTA per (batch, K/V head, 128-key tile), looping over the group's query
// heads and the query tiles that see those keys, dK and dV accumulating in
// TMEM); the dQ kernel (one CTA per (batch, query head, 128-row tile),
// looping over the key tiles it sees, dQ accumulating in TMEM).  S and dP
// are computed in both kernels (7 tile products where one pass with dQ
// atomics would need 5), so every output has a single writer and the result
// is deterministic.
//
// Roles (384 threads): warp 0 TMEM allocator and tcgen05.mma issuer, warp 1
// TMA producer, warp 2 (dK/dV kernel) per-step vector staging, warps 4-11
// the element-wise work and the epilogue -- two warpgroups on the same TMEM
// rows (one row per thread), each taking 64 of a tile's 128 columns, so
// that two warps per scheduler hide each other's latencies.  Warps 0-3 give
// up registers with setmaxnreg (72 each) so that the element-wise warps get
// 216: the launch allocation of 168 per thread, split.  Every mbarrier wait
// is bounded as in the forward kernel.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_sync.cuh"
#include "sm103_ptx.cuh"

namespace attn {

struct BwdParams {
  int B, Hq, Hkv, Sq, Skv;
  int causal;
  int input_pos;
  int window;              // sliding window in keys (causal only), 0: none
  int group;               // Hq / Hkv
  int q_tiles, k_tiles;    // 128-row query / key tiles per head
  int sq_pad;              // q_tiles * 128: rows per plane of lse2 / delta
  float scale_log2;        // |scale| * log2(e)
  int negate_scores;       // scale < 0: S is computed as -(Q K^T)
  float scale;             // signed; dQ and dK carry this factor
  const float* lse2;       // [B*Hq, sq_pad] LSE * log2(e), +inf past Sq
  const float* delta;      // [B*Hq, sq_pad] rowsum(dO * O), 0 past Sq
  void* dq;                // [B, Hq, Sq, D]
  void* dk;                // [B, Hkv, Skv, D]
  void* dv;                // [B, Hkv, Skv, D]
  unsigned int* status;
  unsigned long long timeout_ns;
};

namespace bwd {
constexpr int kT = 128;        // rows per query / key tile
constexpr int kThreads = 384;
constexpr int kMmaWarp = 0;
constexpr int kLoadWarp = 1;
constexpr int kVecWarp = 2;    // dK/dV kernel: stages the per-step vectors
constexpr int kWorkWarp0 = 4;  // warps 4-11: two warpgroups
constexpr int kWork = 256;     // element-wise threads
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
}  // namespace bwd

// Any valid query row of tile m sees a key of tile n.
__device__ __forceinline__ bool pair_visible(const BwdParams& p, int m,
                                             int n) {
  if (!p.causal) return true;
  const int pos_first = p.input_pos + m * bwd::kT;
  const int pos_last = p.input_pos + min(m * bwd::kT + bwd::kT, p.Sq) - 1;
  const int key_first = n * bwd::kT;
  const int key_last = min(n * bwd::kT + bwd::kT, p.Skv) - 1;
  if (key_first > pos_last) return false;
  if (p.window > 0 && key_last <= pos_first - p.window) return false;
  return true;
}

// Every valid query row of tile m sees every valid key of tile n.
__device__ __forceinline__ bool pair_full(const BwdParams& p, int m, int n) {
  if (!p.causal) return true;
  const int pos_first = p.input_pos + m * bwd::kT;
  const int pos_last = p.input_pos + min(m * bwd::kT + bwd::kT, p.Sq) - 1;
  const int key_first = n * bwd::kT;
  const int key_last = min(n * bwd::kT + bwd::kT, p.Skv) - 1;
  if (key_last > pos_first) return false;
  if (p.window > 0 && key_first <= pos_last - p.window) return false;
  return true;
}

// (y0, y1) = (x0, x1) * m + (a0, a1) as one packed f32x2 FMA.
__device__ __forceinline__ void ffma2v(float& y0, float& y1, float x0,
                                       float x1, float m, float a0, float a1) {
  asm("{\n\t.reg .b64 x, mm, aa, y;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 mm, {%4, %4};\n\t"
      "mov.b64 aa, {%5, %6};\n\t"
      "fma.rn.ftz.f32x2 y, x, mm, aa;\n\t"
      "mov.b64 {%0, %1}, y;\n\t}"
      : "=f"(y0), "=f"(y1)
      : "f"(x0), "f"(x1), "f"(m), "f"(a0), "f"(a1));
}

// ((a0, a1) - (b0, b1)) * (p0, p1) as two packed f32x2 instructions (four
// scalar ones would take the FMA pipe's issue slots twice).
__device__ __forceinline__ void sub_mul2(float& y0, float& y1, float a0,
                                         float a1, float b0, float b1,
                                         float p0, float p1) {
  asm("{\n\t.reg .b64 a, b, pp, y;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mov.b64 pp, {%6, %7};\n\t"
      "sub.rn.ftz.f32x2 y, a, b;\n\t"
      "mul.rn.ftz.f32x2 y, y, pp;\n\t"
      "mov.b64 {%0, %1}, y;\n\t}"
      : "=f"(y0), "=f"(y1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(p0), "f"(p1));
}

// 16-bit pair (as packed by ptx::pack2) back to two floats.
template <bool kBF16>
__device__ __forceinline__ float2 unpack2(uint32_t v) {
  if constexpr (kBF16) {
    return make_float2(__uint_as_float(v << 16),
                       __uint_as_float(v & 0xffff0000u));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(&v));
  }
}

// First (query head, query tile) index hm >= from whose tile sees key tile
// n (dK/dV steps), or `end`.
__device__ __forceinline__ int next_pair_hm(const BwdParams& p, int n,
                                            int from, int end) {
  int hm = from;
  while (hm < end && !pair_visible(p, hm % p.q_tiles, n)) ++hm;
  return hm;
}

// First key tile index >= from that query tile m sees (dQ steps), or
// k_tiles.
__device__ __forceinline__ int next_key_tile(const BwdParams& p, int m,
                                             int from) {
  int n = from;
  while (n < p.k_tiles && !pair_visible(p, m, n)) ++n;
  return n;
}

// ------------------------------------------------------------- row pass
// D_i = sum_d dO_id O_id and lse2_i = LSE_i log2(e) into the padded
// [planes, sq_pad] arrays; rows past Sq get lse2 = +inf (so P = 0 there) and
// D = 0, and the tile loops read whole tiles unchecked.  The first warps
// take kRows consecutive rows each of the flat [planes * Sq] row space
// (contiguous in O and dO): lane l reads the 16-byte chunks l, l + 32, ...
// of that block, so each load instruction of the warp covers 512
// contiguous bytes and every lane has 2 * kRows * D / 256 loads in flight;
// the lanes holding pieces of one row then reduce among themselves.  The
// warps after them fill the padding rows, 32 per warp.
template <int D, bool kBF16>
__global__ void __launch_bounds__(256)
    attn_bwd_prep_kernel(const void* __restrict__ O,
                         const void* __restrict__ dO,
                         const float* __restrict__ LSE,
                         float* __restrict__ lse2, float* __restrict__ delta,
                         long long rows, long long planes, int Sq,
                         int sq_pad) {
  constexpr int kRows = 8;                       // rows per warp
  constexpr int kRowChunks = D * 2 / 16;         // 16-byte chunks per row
  constexpr int kPerLane = kRows * kRowChunks / 32;
  static_assert(kRowChunks <= 32 && kPerLane >= 1, "row pass layout");
  const long long warp =
      (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  const long long row_warps = (rows + kRows - 1) / kRows;
  if (warp >= row_warps) {
    const int pad = sq_pad - Sq;
    const long long i = (warp - row_warps) * 32 + lane;
    if (pad > 0 && i < planes * pad) {
      const long long prow = (i / pad) * sq_pad + Sq + i % pad;
      delta[prow] = 0.f;
      lse2[prow] = INFINITY;
    }
    return;
  }
  const long long row0 = warp * kRows;
  const uint4* o = reinterpret_cast<const uint4*>(
      static_cast<const uint16_t*>(O) + row0 * D);
  const uint4* g = reinterpret_cast<const uint4*>(
      static_cast<const uint16_t*>(dO) + row0 * D);
  uint4 ov[kPerLane], gv[kPerLane];
#pragma unroll
  for (int k = 0; k < kPerLane; ++k) {
    const int c = lane + 32 * k;
    if (row0 + c / kRowChunks < rows) {
      ov[k] = __ldg(o + c);
      gv[k] = __ldg(g + c);
    } else {
      ov[k] = make_uint4(0u, 0u, 0u, 0u);
      gv[k] = ov[k];
    }
  }
  float acc[kPerLane];
#pragma unroll
  for (int k = 0; k < kPerLane; ++k) {
    const uint32_t* a = reinterpret_cast<const uint32_t*>(&ov[k]);
    const uint32_t* b = reinterpret_cast<const uint32_t*>(&gv[k]);
    acc[k] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 of, gf;
      if constexpr (kBF16) {
        of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a[e]));
        gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b[e]));
      } else {
        of = __half22float2(*reinterpret_cast<const __half2*>(&a[e]));
        gf = __half22float2(*reinterpret_cast<const __half2*>(&b[e]));
      }
      acc[k] = fmaf(of.x, gf.x, acc[k]);
      acc[k] = fmaf(of.y, gf.y, acc[k]);
    }
  }
  // Lanes l .. l + kRowChunks - 1 (aligned) hold the pieces of one row.
#pragma unroll
  for (int off = kRowChunks / 2; off > 0; off >>= 1) {
#pragma unroll
    for (int k = 0; k < kPerLane; ++k)
      acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], off);
  }
  if (lane % kRowChunks == 0) {
#pragma unroll
    for (int k = 0; k < kPerLane; ++k) {
      const long long row = row0 + (lane + 32 * k) / kRowChunks;
      if (row < rows) {
        const long long prow = (row / Sq) * sq_pad + row % Sq;
        delta[prow] = acc[k];
        lse2[prow] = LSE[row] * bwd::kLog2e;
      }
    }
  }
}

// ------------------------------------------------------ shared layouts
template <int D>
struct BwdTiles {
  static constexpr int kChunks = D / 64;
  static constexpr int kBoxBytes = 128 * 128;            // 128 rows x 128 B
  static constexpr int kTileBytes = kChunks * kBoxBytes; // one 128 x D tile
};

// dK/dV kernel: K and V tiles resident, separate rings of Q and dO tiles
// (Q is held until dK(s), dO only until dV(s), so the Q ring is the deeper
// one; 3 + 2 slots fill the 227 KB at D=128).
template <int D>
struct DkdvLayout : BwdTiles<D> {
  using T = BwdTiles<D>;
  static constexpr int kQSlots = (D == 128) ? 3 : 4;
  static constexpr int kDoSlots = (D == 128) ? 2 : 4;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = T::kTileBytes;
  static constexpr int kQOff = 2 * T::kTileBytes;
  static constexpr int kDoOff = kQOff + kQSlots * T::kTileBytes;
  // lse2 and D of the current step's 128 query rows (1 KB, staged one step
  // ahead by its own warp: read from L2 inside the element-wise passes their
  // latency sat on the critical path).
  static constexpr int kVecOff = kDoOff + kDoSlots * T::kTileBytes;
  static constexpr int kBarOff = kVecOff + 2 * bwd::kT * 4;
  // kv_full, q_full[QS], q_empty[QS], do_full[DS], do_empty[DS], s_ready,
  // dp_ready, p_ready, ds_ready, acc_done, drain, vec_full, vec_free
  static constexpr int kNumBars = 1 + 2 * kQSlots + 2 * kDoSlots + 8;
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

// dQ kernel: Q and dO resident, separate rings of K and V tiles.  K(s) is
// held from S(s) (issued two steps ahead) until dQ(s), V(s) only for dP(s);
// in one shared ring the late release of K(s-1) held back the copy of
// V(s+1).  At step s the MMA issuer wants V(s+1) and K(s+2): 3 K + 2 V
// slots (D=128) give both copies a step or more of lead.
template <int D>
struct DqLayout : BwdTiles<D> {
  using T = BwdTiles<D>;
  static constexpr int kKSlots = (D == 128) ? 3 : 4;
  static constexpr int kVSlots = (D == 128) ? 2 : 4;
  static constexpr int kQOff = 0;
  static constexpr int kDoOff = T::kTileBytes;
  static constexpr int kKOff = 2 * T::kTileBytes;
  static constexpr int kVOff = kKOff + kKSlots * T::kTileBytes;
  static constexpr int kBarOff = kVOff + kVSlots * T::kTileBytes;
  // q_full, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_ready[2],
  // dp_ready, ds_ready, acc_done, drain, box_full[2] (dQ output boxes)
  static constexpr int kNumBars = 1 + 2 * kKSlots + 2 * kVSlots + 6 + 2;
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

// Stores one 16-bit output row (D values, fp32 in TMEM at t_acc, times
// `mul`) from registers; `store` false reads TMEM only (every lane of the
// warp takes part in tcgen05.ld).
template <int D, bool kBF16>
__device__ __forceinline__ void store_row(uint32_t t_acc, float mul,
                                          uint16_t* dst, bool store) {
  uint4* out = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < D / 32; ++q) {
    uint32_t a[32];
    ptx::tmem_ld32(t_acc + 32 * q, a);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = ptx::pack2<kBF16>(__uint_as_float(a[8 * v + 2 * e]) * mul,
                                 __uint_as_float(a[8 * v + 2 * e + 1]) * mul);
      if (store) out[4 * q + v] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// Stores kCols columns (fp32 in TMEM at t_acc, times `mul`) of a 16-bit
// output row at dst; `store` false reads TMEM only (every lane of the warp
// takes part in tcgen05.ld).
template <int kCols, bool kBF16>
__device__ __forceinline__ void store_cols(uint32_t t_acc, float mul,
                                           uint16_t* dst, bool store) {
  uint4* out = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < kCols / 32; ++q) {
    uint32_t a[32];
    ptx::tmem_ld32(t_acc + 32 * q, a);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = ptx::pack2<kBF16>(__uint_as_float(a[8 * v + 2 * e]) * mul,
                                 __uint_as_float(a[8 * v + 2 * e + 1]) * mul);
      if (store) out[4 * q + v] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// ------------------------------------------------------- dK / dV kernel
// Unit u: key tile n = u / (B*Hkv) (under a causal mask the first key tiles
// see the most queries, so they start first), (b, K/V head) = u % (B*Hkv).
// Steps: the (query head of the group, query tile m) pairs that see tile
// n, in order.  TMEM: S^T [0,128), dP^T [128,256), dV [256,256+D),
// dK [256+D, 256+2D); P^T and dS^T (16-bit) overwrite columns 0-31 and
// 64-95 of S^T and dP^T and are the A operands of dV += P^T dO and
// dK += dS^T Q.
// Software pipeline: the element-wise pass is split at "P ready" and "dS
// ready" (P stays in registers, 16-bit, for the dS half), so the tensor
// pipe runs dV(s) and S^T(s+1) while dS(s) is computed, and dK(s) and
// dP^T(s+1) while P(s+1) is.
template <int D, bool kBF16>
__global__ void __launch_bounds__(bwd::kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do,
                         const BwdParams p) {
  using L = DkdvLayout<D>;
  using namespace bwd;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = ptx::smem_u32(smem);
  const uint32_t s_k = s_base + L::kKOff;
  const uint32_t s_v = s_base + L::kVOff;
  const uint32_t s_qr = s_base + L::kQOff;   // Q ring
  const uint32_t s_dor = s_base + L::kDoOff; // dO ring
  const uint32_t bar0 = s_base + L::kBarOff;
  const uint32_t bar_kv = bar0;
  const uint32_t bar_qf = bar0 + 8;                      // [kQSlots]
  const uint32_t bar_qe = bar_qf + 8 * L::kQSlots;       // [kQSlots]
  const uint32_t bar_df = bar_qe + 8 * L::kQSlots;       // [kDoSlots]
  const uint32_t bar_de = bar_df + 8 * L::kDoSlots;      // [kDoSlots]
  const uint32_t bar_s = bar_de + 8 * L::kDoSlots;
  const uint32_t bar_dp = bar_s + 8;
  const uint32_t bar_p = bar_dp + 8;
  const uint32_t bar_ds = bar_p + 8;
  const uint32_t bar_acc = bar_ds + 8;
  const uint32_t bar_drain = bar_acc + 8;
  const uint32_t bar_vf = bar_drain + 8;  // step vectors staged
  const uint32_t bar_ve = bar_vf + 8;     // step vectors consumed
  float* vec = reinterpret_cast<float*>(smem + L::kVecOff);  // lse2, D
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<int*>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int bkv = p.B * p.Hkv;
  const int n = static_cast<int>(blockIdx.x) / bkv;
  const int bk = static_cast<int>(blockIdx.x) % bkv;  // b * Hkv + kvh
  const int b = bk / p.Hkv;
  const int qplane0 = b * p.Hq + (bk % p.Hkv) * p.group;
  const int steps_all = p.group * p.q_tiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNumBars; ++i) {
      const uint32_t bar = bar0 + 8 * i;
      const bool work = bar == bar_p || bar == bar_ds || bar == bar_ve;
      ptx::mbar_init(bar, work ? kWork : 1);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < kWorkWarp0) {
  ptx::setmaxnreg_dec<72>();
  if (warp == kLoadWarp) {
    // -------------------------------------------------------- producer
    if (lane == 0) {
      ptx::prefetch_tensormap(&tm_q);
      ptx::prefetch_tensormap(&tm_k);
      ptx::prefetch_tensormap(&tm_v);
      ptx::prefetch_tensormap(&tm_do);
    }
    ptx::mbar_arrive_expect_tx_elect(bar_kv, 2 * L::kTileBytes);
    for (int c = 0; c < L::kChunks; ++c) {
      ptx::tma_load_3d_elect(s_k + c * L::kBoxBytes, &tm_k, bar_kv, c * 64,
                             n * kT, bk);
      ptx::tma_load_3d_elect(s_v + c * L::kBoxBytes, &tm_v, bar_kv, c * 64,
                             n * kT, bk);
    }
    bool ok = true;
    int s = 0;
    int nq = 0, nd = 0;  // Q / dO copies issued
    for (int hm = 0; hm < steps_all && ok; ++hm) {
      const int m = hm % p.q_tiles;
      if (!pair_visible(p, m, n)) continue;
      const int qplane = qplane0 + hm / p.q_tiles;
      const int qs = s % L::kQSlots, ds = s % L::kDoSlots;
      if (s >= L::kQSlots) {
        ok = __all_sync(0xffffffffu,
                        wait_bounded(bar_qe + 8 * qs,
                                     ((s / L::kQSlots) - 1) & 1, abort_flag,
                                     p, 1));
        if (!ok) break;
      }
      ptx::mbar_arrive_expect_tx_elect(bar_qf + 8 * qs, L::kTileBytes);
      for (int c = 0; c < L::kChunks; ++c)
        ptx::tma_load_3d_elect(s_qr + qs * L::kTileBytes + c * L::kBoxBytes,
                               &tm_q, bar_qf + 8 * qs, c * 64, m * kT, qplane);
      ++nq;
      if (s >= L::kDoSlots) {
        ok = __all_sync(0xffffffffu,
                        wait_bounded(bar_de + 8 * ds,
                                     ((s / L::kDoSlots) - 1) & 1, abort_flag,
                                     p, 1));
        if (!ok) break;
      }
      ptx::mbar_arrive_expect_tx_elect(bar_df + 8 * ds, L::kTileBytes);
      for (int c = 0; c < L::kChunks; ++c)
        ptx::tma_load_3d_elect(s_dor + ds * L::kTileBytes + c * L::kBoxBytes,
                               &tm_do, bar_df + 8 * ds, c * 64, m * kT,
                               qplane);
      ++nd;
      ++s;
    }
    if (!ok) {
      // Let every copy still in flight land before the CTA goes away.
      drain_wait(bar_kv, 0, p);
      for (int i = max(0, nq - L::kQSlots); i < nq; ++i)
        drain_wait(bar_qf + 8 * (i % L::kQSlots), (i / L::kQSlots) & 1, p);
      for (int i = max(0, nd - L::kDoSlots); i < nd; ++i)
        drain_wait(bar_df + 8 * (i % L::kDoSlots), (i / L::kDoSlots) & 1, p);
    }
    __syncwarp();
  } else if (warp == kVecWarp) {
    // ------------------------------------------- per-step vector staging
    // lse2 and D of step s's 128 query rows into shared memory, once the
    // element-wise warps are done with step s-1's (padded arrays: no
    // bounds checks).
    bool ok = true;
    int s = 0;
    for (int hm = 0; hm < steps_all && ok; ++hm) {
      const int m = hm % p.q_tiles;
      if (!pair_visible(p, m, n)) continue;
      if (s > 0) {
        ok = __all_sync(0xffffffffu,
                        wait_bounded(bar_ve, (s - 1) & 1, abort_flag, p, 5));
        if (!ok) break;
      }
      const long long vbase =
          static_cast<long long>(qplane0 + hm / p.q_tiles) * p.sq_pad + m * kT;
      float4 l4 = reinterpret_cast<const float4*>(p.lse2 + vbase)[lane];
      l4.x = -l4.x; l4.y = -l4.y; l4.z = -l4.z; l4.w = -l4.w;
      const float4 d4 = reinterpret_cast<const float4*>(p.delta + vbase)[lane];
      reinterpret_cast<float4*>(vec)[lane] = l4;
      reinterpret_cast<float4*>(vec + kT)[lane] = d4;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_vf);
      ++s;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------ MMA issuer
    constexpr uint32_t kHi = ptx::sdesc_hi_sw128(1024);
    const uint32_t idesc_s =
        ptx::idesc_f16(kBF16, kT, kT, false, p.negate_scores != 0);
    const uint32_t idesc_dp = ptx::idesc_f16(kBF16, kT, kT, false, false);
    const uint32_t idesc_acc = ptx::idesc_f16(kBF16, kT, D, true, false);
    const uint32_t t_st = tmem, t_dpt = tmem + kT;
    const uint32_t t_dv = tmem + 2 * kT, t_dk = tmem + 2 * kT + D;
    const uint32_t k_lo = ptx::sdesc_lo(s_k, 16);
    const uint32_t v_lo = ptx::sdesc_lo(s_v, 16);
    // Q / dO tiles of step s: K-major descriptors for S^T and dP^T,
    // MN-major ones for the B operands of dK and dV.
    auto q_tile = [&](int s) { return s_qr + (s % L::kQSlots) * L::kTileBytes; };
    auto do_tile = [&](int s) {
      return s_dor + (s % L::kDoSlots) * L::kTileBytes;
    };
    auto wait_q = [&](int s) {
      return __all_sync(0xffffffffu,
                        wait_bounded(bar_qf + 8 * (s % L::kQSlots),
                                     (s / L::kQSlots) & 1, abort_flag, p, 2));
    };
    auto wait_do = [&](int s) {
      return __all_sync(0xffffffffu,
                        wait_bounded(bar_df + 8 * (s % L::kDoSlots),
                                     (s / L::kDoSlots) & 1, abort_flag, p, 2));
    };
    // S^T = K Q^T or dP^T = V dO^T (M = keys, N = queries, K = D).
    auto issue_kq = [&](uint32_t d, uint32_t a_lo, uint32_t b_lo,
                        uint32_t idesc) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk / 4) * L::kBoxBytes + (kk % 4) * 32) >> 4;
        ptx::mma_ss_elect(d, a_lo + off, b_lo + off, kHi, idesc,
                          kk > 0 ? 1u : 0u);
      }
    };
    // dV += P^T dO or dK += dS^T Q (M = keys, N = D, K = queries).
    auto issue_acc = [&](uint32_t d, uint32_t a_tmem, uint32_t b_mn,
                         bool acc) {
#pragma unroll
      for (int kk = 0; kk < kT / 16; ++kk)
        ptx::mma_ts_elect(d, a_tmem + (kk / 4) * 64 + (kk % 4) * 8,
                          b_mn + ((kk * 16 * 128) >> 4),
                          kHi, idesc_acc, (acc || kk > 0) ? 1u : 0u);
    };
    bool ok = __all_sync(0xffffffffu,
                         wait_bounded(bar_kv, 0, abort_flag, p, 2));
    bool issued = false;
    int s = 0;
    int hm = next_pair_hm(p, n, 0, steps_all);
    if (ok && hm < steps_all) {
      ok = wait_q(0);
      if (ok) {
        ptx::tc_fence_after();
        issue_kq(t_st, k_lo, ptx::sdesc_lo(q_tile(0), 16), idesc_s);
        ptx::tc_commit_elect(bar_s);
        issued = true;
        ok = wait_do(0);
      }
      if (ok) {
        ptx::tc_fence_after();
        issue_kq(t_dpt, v_lo, ptx::sdesc_lo(do_tile(0), 16), idesc_dp);
        ptx::tc_commit_elect(bar_dp);
      }
    }
    while (ok && hm < steps_all) {
      const int hm_next = next_pair_hm(p, n, hm + 1, steps_all);
      const bool more = hm_next < steps_all;
      // dV(s) once P^T(s) is in TMEM (dO(s) free after it), then S^T(s+1)
      // (after dV in issue order, so P^T is read before it is overwritten).
      ok = __all_sync(0xffffffffu,
                      wait_bounded(bar_p, s & 1, abort_flag, p, 2));
      if (!ok) break;
      ptx::tc_fence_after();
      issue_acc(t_dv, t_st, ptx::sdesc_lo(do_tile(s), L::kBoxBytes), s > 0);
      ptx::tc_commit_elect(bar_de + 8 * (s % L::kDoSlots));
      if (more) {
        ok = wait_q(s + 1);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_kq(t_st, k_lo, ptx::sdesc_lo(q_tile(s + 1), 16), idesc_s);
        ptx::tc_commit_elect(bar_s);
      }
      // dK(s) once dS^T(s) is in TMEM (Q(s) free after it), then dP^T(s+1).
      ok = __all_sync(0xffffffffu,
                      wait_bounded(bar_ds, s & 1, abort_flag, p, 2));
      if (!ok) break;
      ptx::tc_fence_after();
      issue_acc(t_dk, t_dpt, ptx::sdesc_lo(q_tile(s), L::kBoxBytes), s > 0);
      ptx::tc_commit_elect(bar_qe + 8 * (s % L::kQSlots));
      if (more) {
        ok = wait_do(s + 1);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_kq(t_dpt, v_lo, ptx::sdesc_lo(do_tile(s + 1), 16), idesc_dp);
        ptx::tc_commit_elect(bar_dp);
      }
      ++s;
      hm = hm_next;
    }
    if (ok && s > 0) ptx::tc_commit_elect(bar_acc);
    if (!ok && issued) {
      ptx::tc_commit_elect(bar_drain);
      drain_wait(bar_drain, 0, p);
    }
    __syncwarp();
  }
  } else {
    ptx::setmaxnreg_inc<216>();
    // ----------------------------------------- P^T, dS^T and epilogue
    // Half h takes query columns [64h, 64h+64) of its key row.  Each pass
    // loads both of the half's 32-column chunks before one wait, then
    // stores its 16-bit results into the first 32 of those 64 columns,
    // which no other warp reads: the halves never wait for each other.
    // The dV / dK MMAs read P^T / dS^T from columns 0..31 and 64..95.
    const int h = (warp - kWorkWarp0) / 4;
    const int r = (warp % 4) * 32 + lane;  // key row in the tile
    const uint32_t lane_off = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t t_st = tmem + lane_off;
    const uint32_t t_dpt = tmem + lane_off + kT;
    const int key = n * kT + r;
    const float c = p.scale_log2;
    bool ok = true;
    int s = 0;
    for (int hm = 0; hm < steps_all && ok; ++hm) {
      const int m = hm % p.q_tiles;
      if (!pair_visible(p, m, n)) continue;
      // lse2 / D of the tile's 128 query rows, staged in shared memory.
      const float4* v_l = reinterpret_cast<const float4*>(vec);
      const float4* v_d = reinterpret_cast<const float4*>(vec + kT);
      // Query column j (position input_pos + m*128 + j) sees this key iff
      // j >= jlo and, with a window, j < jlo + window.
      const bool full = pair_full(p, m, n);
      const int jlo = key - (p.input_pos + m * kT);
      const unsigned span =
          p.window > 0 ? static_cast<unsigned>(p.window) : 0x40000000u;
      // P^T = 2^(S^T c - lse2), kept in registers (16-bit) for dS.
      ok = __all_sync(0xffffffffu,
                      wait_bounded(bar_s, s & 1, abort_flag, p, 3));
      if (ok)
        ok = __all_sync(0xffffffffu,
                        wait_bounded(bar_vf, s & 1, abort_flag, p, 3));
      if (!ok) break;
      ptx::tc_fence_after();
      uint32_t pk[32];
      uint32_t sv[2][32];
      ptx::tmem_ld32(t_st + 32 * (2 * h), sv[0]);
      ptx::tmem_ld32(t_st + 32 * (2 * h + 1), sv[1]);
      float lv0[32];  // -lse2 of the first chunk's query columns
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 t4 = v_l[8 * (2 * h) + i];
        lv0[4 * i] = t4.x;
        lv0[4 * i + 1] = t4.y;
        lv0[4 * i + 2] = t4.z;
        lv0[4 * i + 3] = t4.w;
      }
      ptx::tmem_wait_ld();
      auto p_pass = [&](auto mask_tag) {
        constexpr bool kMasked = decltype(mask_tag)::value;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int q = 2 * h + k;
          float lv[32];  // -lse2 of the query columns
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (k == 0) {
              lv[4 * i] = lv0[4 * i];
              lv[4 * i + 1] = lv0[4 * i + 1];
              lv[4 * i + 2] = lv0[4 * i + 2];
              lv[4 * i + 3] = lv0[4 * i + 3];
            } else {
              const float4 t4 = v_l[8 * q + i];
              lv[4 * i] = t4.x;
              lv[4 * i + 1] = t4.y;
              lv[4 * i + 2] = t4.z;
              lv[4 * i + 3] = t4.w;
            }
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = 32 * q + 2 * e;
            float x0, x1;
            ffma2v(x0, x1, __uint_as_float(sv[k][2 * e]),
                   __uint_as_float(sv[k][2 * e + 1]), c, lv[2 * e], lv[2 * e + 1]);
            if constexpr (kMasked) {
              if (static_cast<unsigned>(j - jlo) >= span) x0 = -INFINITY;
              if (static_cast<unsigned>(j + 1 - jlo) >= span) x1 = -INFINITY;
            }
            pk[16 * k + e] = ptx::pack2<kBF16>(ptx::ex2(x0), ptx::ex2(x1));
          }
        }
      };
      if (full)
        p_pass(BoolTag<false>{});
      else
        p_pass(BoolTag<true>{});
      // 16-bit P^T of query columns 64h.. into TMEM columns 64h..64h+31,
      // which only this half has read.
      ptx::tmem_st16(t_st + 64 * h, pk);
      ptx::tmem_st16(t_st + 64 * h + 16, pk + 16);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar_p);
      // dS^T = P^T (dP^T - D).
      ok = __all_sync(0xffffffffu,
                      wait_bounded(bar_dp, s & 1, abort_flag, p, 3));
      if (!ok) break;
      ptx::tc_fence_after();
      uint32_t dk[32];
      uint32_t dv[2][32];
      ptx::tmem_ld32(t_dpt + 32 * (2 * h), dv[0]);
      ptx::tmem_ld32(t_dpt + 32 * (2 * h + 1), dv[1]);
      float dl0[32];  // D of the first chunk's query columns
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 t4 = v_d[8 * (2 * h) + i];
        dl0[4 * i] = t4.x;
        dl0[4 * i + 1] = t4.y;
        dl0[4 * i + 2] = t4.z;
        dl0[4 * i + 3] = t4.w;
      }
      ptx::tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int q = 2 * h + k;
        float dl[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (k == 0) {
            dl[4 * i] = dl0[4 * i];
            dl[4 * i + 1] = dl0[4 * i + 1];
            dl[4 * i + 2] = dl0[4 * i + 2];
            dl[4 * i + 3] = dl0[4 * i + 3];
          } else {
            const float4 t4 = v_d[8 * q + i];
            dl[4 * i] = t4.x;
            dl[4 * i + 1] = t4.y;
            dl[4 * i + 2] = t4.z;
            dl[4 * i + 3] = t4.w;
          }
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 pp = unpack2<kBF16>(pk[16 * k + e]);
          float d0, d1;
          sub_mul2(d0, d1, __uint_as_float(dv[k][2 * e]),
                   __uint_as_float(dv[k][2 * e + 1]), dl[2 * e], dl[2 * e + 1],
                   pp.x, pp.y);
          dk[16 * k + e] = ptx::pack2<kBF16>(d0, d1);
        }
      }
      ptx::mbar_arrive(bar_ve);  // done with this step's vectors
      ptx::tmem_st16(t_dpt + 64 * h, dk);
      ptx::tmem_st16(t_dpt + 64 * h + 16, dk + 16);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar_ds);
      ++s;
    }
    if (ok) {
      // Epilogue: half 0 writes the dV row, half 1 the scale * dK row
      // (keys past Skv are not stored; a key tile no query sees gets zeros).
      const long long row = static_cast<long long>(bk) * p.Skv + key;
      const bool in = key < p.Skv;
      uint16_t* dst = static_cast<uint16_t*>(h ? p.dk : p.dv) + row * D;
      if (s > 0) {
        ok = __all_sync(0xffffffffu,
                        wait_bounded(bar_acc, 0, abort_flag, p, 4));
        if (ok) {
          ptx::tc_fence_after();
          store_cols<D, kBF16>(tmem + lane_off + 2 * kT + h * D,
                               h ? p.scale : 1.f, dst, in);
        }
      } else if (in) {
        uint4* z = reinterpret_cast<uint4*>(dst);
        for (int i = 0; i < D / 8; ++i) z[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------ dQ kernel
// Unit u: query tile m = q_tiles - 1 - u / (B*Hq) (under a causal mask the
// last rows see the most keys), plane (b, query head) = u % (B*Hq).  Steps:
// the key tiles n that tile m sees, in order.  TMEM: S double-buffered in
// [0,128) and [128,256), dP [256,384), dQ [384,384+D); dS (16-bit)
// overwrites columns 0-31 and 64-95 of dP and is the A operand of
// dQ += dS K.  Software pipeline: S(s+2) is issued as soon as step s's
// element-wise pass is done, so P(s+1) can be computed while the tensor
// pipe runs dQ(s) and dP(s+1).
template <int D, bool kBF16>
__global__ void __launch_bounds__(bwd::kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dq,
                       const BwdParams p) {
  using L = DqLayout<D>;
  using namespace bwd;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = ptx::smem_u32(smem);
  const uint32_t s_q = s_base + L::kQOff;
  const uint32_t s_do = s_base + L::kDoOff;
  const uint32_t s_kr = s_base + L::kKOff;  // K ring
  const uint32_t s_vr = s_base + L::kVOff;  // V ring
  const uint32_t bar0 = s_base + L::kBarOff;
  const uint32_t bar_q = bar0;
  const uint32_t bar_kf = bar0 + 8;                    // [kKSlots]
  const uint32_t bar_ke = bar_kf + 8 * L::kKSlots;     // [kKSlots]
  const uint32_t bar_vf = bar_ke + 8 * L::kKSlots;     // [kVSlots]
  const uint32_t bar_ve = bar_vf + 8 * L::kVSlots;     // [kVSlots]
  const uint32_t bar_s = bar_ve + 8 * L::kVSlots;  // [2], per S buffer
  const uint32_t bar_dp = bar_s + 16;
  const uint32_t bar_ds = bar_dp + 8;
  const uint32_t bar_acc = bar_ds + 8;
  const uint32_t bar_drain = bar_acc + 8;
  const uint32_t bar_box = bar_drain + 8;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<int*>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int bhq = p.B * p.Hq;
  const int m = p.q_tiles - 1 - static_cast<int>(blockIdx.x) / bhq;
  const int qplane = static_cast<int>(blockIdx.x) % bhq;  // b * Hq + h
  const int kvplane = (qplane / p.Hq) * p.Hkv + (qplane % p.Hq) / p.group;

  if (threadIdx.x == 0) {
    // dQ box b collects one arrival per thread that writes into it: both
    // halves at D = 64 (one 64-column box), one half each at D = 128.
    for (int i = 0; i < L::kNumBars; ++i) {
      const uint32_t bar = bar0 + 8 * i;
      const uint32_t count = bar == bar_ds                ? kWork
                             : bar == bar_box && D == 64 ? kWork
                             : (bar == bar_box || bar == bar_box + 8) ? kT
                                                                      : 1;
      ptx::mbar_init(bar, count);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < kWorkWarp0) {
  ptx::setmaxnreg_dec<72>();
  if (warp == kLoadWarp) {
    // -------------------------------------------------------- producer
    if (lane == 0) {
      ptx::prefetch_tensormap(&tm_q);
      ptx::prefetch_tensormap(&tm_k);
      ptx::prefetch_tensormap(&tm_v);
      ptx::prefetch_tensormap(&tm_do);
      ptx::prefetch_tensormap(&tm_dq);
    }
    ptx::mbar_arrive_expect_tx_elect(bar_q, 2 * L::kTileBytes);
    for (int c = 0; c < L::kChunks; ++c) {
      ptx::tma_load_3d_elect(s_q + c * L::kBoxBytes, &tm_q, bar_q, c * 64,
                             m * kT, qplane);
      ptx::tma_load_3d_elect(s_do + c * L::kBoxBytes, &tm_do, bar_q, c * 64,
                             m * kT, qplane);
    }
    bool ok = true;
    int nk = 0, nv = 0;  // K / V copies issued (step index of the next)
    for (int n = 0; n < p.k_tiles && ok; ++n) {
      if (!pair_visible(p, m, n)) continue;
      const int ks = nk % L::kKSlots;
      if (nk >= L::kKSlots) {
        ok = __all_sync(0xffffffffu,
                        wait_bounded(bar_ke + 8 * ks,
                                     ((nk / L::kKSlots) - 1) & 1, abort_flag,
                                     p, 1));
        if (!ok) break;
      }
      ptx::mbar_arrive_expect_tx_elect(bar_kf + 8 * ks, L::kTileBytes);
      for (int c = 0; c < L::kChunks; ++c)
        ptx::tma_load_3d_elect(s_kr + ks * L::kTileBytes + c * L::kBoxBytes,
                               &tm_k, bar_kf + 8 * ks, c * 64, n * kT,
                               kvplane);
      ++nk;
      const int vs = nv % L::kVSlots;
      if (nv >= L::kVSlots) {
        ok = __all_sync(0xffffffffu,
                        wait_bounded(bar_ve + 8 * vs,
                                     ((nv / L::kVSlots) - 1) & 1, abort_flag,
                                     p, 1));
        if (!ok) break;
      }
      ptx::mbar_arrive_expect_tx_elect(bar_vf + 8 * vs, L::kTileBytes);
      for (int c = 0; c < L::kChunks; ++c)
        ptx::tma_load_3d_elect(s_vr + vs * L::kTileBytes + c * L::kBoxBytes,
                               &tm_v, bar_vf + 8 * vs, c * 64, n * kT,
                               kvplane);
      ++nv;
    }
    if (!ok) {
      // Let every copy still in flight land before the CTA goes away.
      drain_wait(bar_q, 0, p);
      for (int i = max(0, nk - L::kKSlots); i < nk; ++i)
        drain_wait(bar_kf + 8 * (i % L::kKSlots), (i / L::kKSlots) & 1, p);
      for (int i = max(0, nv - L::kVSlots); i < nv; ++i)
        drain_wait(bar_vf + 8 * (i % L::kVSlots), (i / L::kVSlots) & 1, p);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------ MMA issuer
    constexpr uint32_t kHi = ptx::sdesc_hi_sw128(1024);
    const uint32_t idesc_s =
        ptx::idesc_f16(kBF16, kT, kT, false, p.negate_scores != 0);
    const uint32_t idesc_dp = ptx::idesc_f16(kBF16, kT, kT, false, false);
    const uint32_t idesc_acc = ptx::idesc_f16(kBF16, kT, D, true, false);
    const uint32_t t_dp = tmem + 2 * kT, t_dq = tmem + 3 * kT;
    const uint32_t q_lo = ptx::sdesc_lo(s_q, 16);
    const uint32_t do_lo = ptx::sdesc_lo(s_do, 16);
    // K(s) / V(s) landed, and their tiles.
    auto wait_k = [&](int s) {
      return __all_sync(0xffffffffu,
                        wait_bounded(bar_kf + 8 * (s % L::kKSlots),
                                     (s / L::kKSlots) & 1, abort_flag, p, 2));
    };
    auto wait_v = [&](int s) {
      return __all_sync(0xffffffffu,
                        wait_bounded(bar_vf + 8 * (s % L::kVSlots),
                                     (s / L::kVSlots) & 1, abort_flag, p, 2));
    };
    auto k_tile = [&](int s) {
      return s_kr + (s % L::kKSlots) * L::kTileBytes;
    };
    auto v_tile = [&](int s) {
      return s_vr + (s % L::kVSlots) * L::kTileBytes;
    };
    // d = A B^T with A, B K-major 128 x D tiles (S = Q K^T, dP = dO V^T).
    auto issue_nt = [&](uint32_t d, uint32_t a_lo, uint32_t b_lo,
                        uint32_t idesc) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk / 4) * L::kBoxBytes + (kk % 4) * 32) >> 4;
        ptx::mma_ss_elect(d, a_lo + off, b_lo + off, kHi, idesc,
                          kk > 0 ? 1u : 0u);
      }
    };
    bool ok = __all_sync(0xffffffffu,
                         wait_bounded(bar_q, 0, abort_flag, p, 2));
    bool issued = false;
    const int n0 = next_key_tile(p, m, 0);
    const int n1 = n0 < p.k_tiles ? next_key_tile(p, m, n0 + 1) : p.k_tiles;
    // Prologue: S(0), dP(0), S(1).
    if (ok && n0 < p.k_tiles) {
      ok = wait_k(0) && wait_v(0);
      if (ok) {
        ptx::tc_fence_after();
        issue_nt(tmem, q_lo, ptx::sdesc_lo(k_tile(0), 16), idesc_s);
        ptx::tc_commit_elect(bar_s);
        issue_nt(t_dp, do_lo, ptx::sdesc_lo(v_tile(0), 16), idesc_dp);
        ptx::tc_commit_elect(bar_dp);
        ptx::tc_commit_elect(bar_ve);  // V(0) slot
        issued = true;
      }
      if (ok && n1 < p.k_tiles) {
        ok = wait_k(1);
        if (ok) {
          ptx::tc_fence_after();
          issue_nt(tmem + kT, q_lo, ptx::sdesc_lo(k_tile(1), 16), idesc_s);
          ptx::tc_commit_elect(bar_s + 8);
        }
      }
    }
    int s = 0;
    int n_cur = n0, n_next = n1;
    while (ok && n_cur < p.k_tiles) {
      const int n_after =
          n_next < p.k_tiles ? next_key_tile(p, m, n_next + 1) : p.k_tiles;
      // dQ(s) += dS(s) K(s) once dS(s) is in TMEM.
      ok = __all_sync(0xffffffffu,
                      wait_bounded(bar_ds, s & 1, abort_flag, p, 2));
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t k_mn = ptx::sdesc_lo(k_tile(s), L::kBoxBytes);
#pragma unroll
      for (int kk = 0; kk < kT / 16; ++kk)
        ptx::mma_ts_elect(t_dq, t_dp + (kk / 4) * 64 + (kk % 4) * 8,
                          k_mn + ((kk * 16 * 128) >> 4),
                          kHi, idesc_acc, (s > 0 || kk > 0) ? 1u : 0u);
      ptx::tc_commit_elect(bar_ke + 8 * (s % L::kKSlots));
      // dP(s+1) into the dP region (after dQ(s) in issue order).
      if (n_next < p.k_tiles) {
        ok = wait_v(s + 1);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_nt(t_dp, do_lo, ptx::sdesc_lo(v_tile(s + 1), 16), idesc_dp);
        ptx::tc_commit_elect(bar_dp);
        ptx::tc_commit_elect(bar_ve + 8 * ((s + 1) % L::kVSlots));
      }
      // S(s+2) into S buffer s % 2, free since step s's pass is done.
      if (n_after < p.k_tiles) {
        ok = wait_k(s + 2);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_nt(tmem + (s & 1) * kT, q_lo, ptx::sdesc_lo(k_tile(s + 2), 16),
                 idesc_s);
        ptx::tc_commit_elect(bar_s + 8 * (s & 1));
      }
      ++s;
      n_cur = n_next;
      n_next = n_after;
    }
    if (ok && s > 0) ptx::tc_commit_elect(bar_acc);
    if (!ok && issued) {
      ptx::tc_commit_elect(bar_drain);
      drain_wait(bar_drain, 0, p);
    }
    __syncwarp();
  }
  } else {
    ptx::setmaxnreg_inc<216>();
    // -------------------------------------------- dS and the epilogue
    // Half h takes key columns [64h, 64h+64) of its query row; its 16-bit
    // dS goes into the first 32 of those dP columns, after both of its dP
    // chunks are loaded, so the halves never wait for each other.  The dQ
    // MMA reads dS from columns 0..31 and 64..95.
    const int h = (warp - kWorkWarp0) / 4;
    const int r = (warp % 4) * 32 + lane;  // query row in the tile
    const uint32_t lane_off = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t t_dp = tmem + lane_off + 2 * kT;
    const int q_row = m * kT + r;
    const long long vrow = static_cast<long long>(qplane) * p.sq_pad + q_row;
    const float lse2 = p.lse2[vrow];  // +inf past Sq: P = 0
    const float dlt = p.delta[vrow];
    const int pos = p.input_pos + q_row;
    const float c = p.scale_log2;
    const float neg_l = -lse2;
    bool ok = true;
    int s = 0;
    for (int n = 0; n < p.k_tiles && ok; ++n) {
      if (!pair_visible(p, m, n)) continue;
      // Key column k (key n*128 + k) is visible iff lo <= k < lo + span.
      const bool full = pair_full(p, m, n);
      const int kbase = n * kT;
      int lo = 0, lim = kT;
      if (!full) {
        lim = pos - kbase + 1;
        if (p.window > 0) lo = pos - p.window + 1 - kbase;
      }
      const unsigned span = static_cast<unsigned>(max(lim - lo, 0));
      // P = 2^(S c - lse2), kept in registers (16-bit) for dS.
      ok = __all_sync(0xffffffffu, wait_bounded(bar_s + 8 * (s & 1),
                                                (s >> 1) & 1, abort_flag, p,
                                                3));
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t t_s = tmem + lane_off + (s & 1) * kT;
      uint32_t pk[32];
      uint32_t sv[2][32];
      ptx::tmem_ld32(t_s + 32 * (2 * h), sv[0]);
      ptx::tmem_ld32(t_s + 32 * (2 * h + 1), sv[1]);
      ptx::tmem_wait_ld();
      auto p_pass = [&](auto mask_tag) {
        constexpr bool kMasked = decltype(mask_tag)::value;
#pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
          const int q = 2 * h + kh;
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int k = 32 * q + 2 * e;
            float x0, x1;
            ptx::ffma2(x0, x1, __uint_as_float(sv[kh][2 * e]),
                       __uint_as_float(sv[kh][2 * e + 1]), c, neg_l);
            if constexpr (kMasked) {
              if (static_cast<unsigned>(k - lo) >= span) x0 = -INFINITY;
              if (static_cast<unsigned>(k + 1 - lo) >= span) x1 = -INFINITY;
            }
            pk[16 * kh + e] = ptx::pack2<kBF16>(ptx::ex2(x0), ptx::ex2(x1));
          }
        }
      };
      if (full)
        p_pass(BoolTag<false>{});
      else
        p_pass(BoolTag<true>{});
      // dS = P (dP - D), 16-bit, over dP.
      ok = __all_sync(0xffffffffu,
                      wait_bounded(bar_dp, s & 1, abort_flag, p, 3));
      if (!ok) break;
      ptx::tc_fence_after();
      uint32_t dk[32];
      uint32_t dv[2][32];
      ptx::tmem_ld32(t_dp + 32 * (2 * h), dv[0]);
      ptx::tmem_ld32(t_dp + 32 * (2 * h + 1), dv[1]);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int kh = 0; kh < 2; ++kh) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 pp = unpack2<kBF16>(pk[16 * kh + e]);
          float d0, d1;
          sub_mul2(d0, d1, __uint_as_float(dv[kh][2 * e]),
                   __uint_as_float(dv[kh][2 * e + 1]), dlt, dlt, pp.x, pp.y);
          dk[16 * kh + e] = ptx::pack2<kBF16>(d0, d1);
        }
      }
      ptx::tmem_st16(t_dp + 64 * h, dk);
      ptx::tmem_st16(t_dp + 64 * h + 16, dk + 16);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar_ds);
      ++s;
    }
    if (ok && s > 0) {
      ok = __all_sync(0xffffffffu, wait_bounded(bar_acc, 0, abort_flag, p, 4));
      if (ok) {
        // scale * dQ in 16 bits through 128-row x 128-byte boxes in shared
        // memory (the K ring, idle now: every MMA has completed), stored by
        // TMA (rows >= Sq fall outside the tensor).  Half h writes columns
        // [h*D/2, (h+1)*D/2) of its row: at D = 128 one box per half, at
        // D = 64 half of one box each; chunk c of row r sits at c ^ (r % 8).
        // The storing thread waits (bounded) for every writer of its box;
        // nobody else waits, so an abort cannot strand a warp here.
        ptx::tc_fence_after();
        constexpr int kCols = D / 2;
        const int box = D == 64 ? 0 : h;
        const int chunk0 = D == 64 ? 4 * h : 0;
        const uint32_t row_base = s_kr + box * kT * 128 + r * 128;
        const uint32_t swz = r % 8;
#pragma unroll
        for (int q = 0; q < kCols / 32; ++q) {
          uint32_t a[32];
          ptx::tmem_ld32(tmem + lane_off + 3 * kT + h * kCols + 32 * q, a);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            uint32_t wv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              wv[e] = ptx::pack2<kBF16>(
                  __uint_as_float(a[8 * c8 + 2 * e]) * p.scale,
                  __uint_as_float(a[8 * c8 + 2 * e + 1]) * p.scale);
            ptx::st_shared_v4(row_base + (((chunk0 + 4 * q + c8) ^ swz) << 4),
                              wv[0], wv[1], wv[2], wv[3]);
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(bar_box + 8 * box);
        if (warp == kWorkWarp0 + 4 * box && (D == 128 || h == 0)) {
          const bool all_in = __all_sync(
              0xffffffffu,
              wait_bounded(bar_box + 8 * box, 0, abort_flag, p, 4));
          if (all_in && lane == 0) {
            ptx::tma_store_3d(&tm_dq, s_kr + box * kT * 128, 64 * box,
                              m * kT, qplane);
            ptx::bulk_commit_group();
            ptx::bulk_wait_group_all();
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace attn
