// Warp-specialised FlashAttention-style forward kernel for sm_103a.
//
// Method (from "Flash Attention in CUDA Tile (cuTile)", sections "How Flash
// Attention solves the memory bandwidth problem" and "Understanding online
// softmax"): tile Q, stream K/V tiles through on-chip memory, keep the
// running row maximum m, running sum l and accumulator O, rescale O and l by
// alpha = 2^(m_old - m_new) when the maximum moves, and divide O by l at the
// end.  Scores are taken in the log2 domain with scale*log2(e) folded into
// one multiply (the listing's INV_LOG_2 step).  Causal tiles that are fully
// masked are never visited and the mask is applied only to tiles that reach
// the diagonal or the key tail (same page, "K-loop split").  Query heads map
// to K/V heads by integer division (section "Grouped-query attention"), and
// query rows sit at absolute positions input_pos + i (the KV-cache offset).
//
// A persistent CTA per SM walks work units of two 128-row Q tiles.
// Roles (384 threads):
//   warp  0    TMEM allocator and single-thread tcgen05.mma issuer
//   warp  1    TMA producer: Q tiles once, then K_j, V_j into a slot ring
//   warps 2-3  idle
//   warps 4-7  softmax + correction + epilogue for Q tile 0 (TMEM lanes 0-127)
//   warps 8-11 the same for Q tile 1
// In the two-tile variants warps 0-3 give up registers (setmaxnreg) so that
// each softmax thread holds its row's 128 scores between the max and exp
// passes.
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 and O1 (D columns each)
// from 256.  P_t (16-bit) overwrites the first 64 columns of S_t and is the
// A operand of O_t += P_t V straight from TMEM.  At D = 64 the O tiles need
// only 128 columns, so three S buffers [0,384) rotate between the two Q
// tiles and O starts at 384: a tile's next S goes to the free buffer and is
// computed while its softmax still works on the current one.  With the
// query heads of a GQA group packed into tile 0 (few query rows), there is
// no tile 1: its S region double-buffers the scores of tile 0 and its
// shared memory goes to the K/V ring.
//
// Every mbarrier wait is bounded: on timeout the waiter raises a CTA-wide
// abort flag and a device status word, every role stops issuing work, waits
// (again bounded) for its own copies / MMAs in flight, and the CTA frees its
// TMEM and exits.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "attn_sync.cuh"
#include "fast_div.h"
#include "sm103_ptx.cuh"

namespace attn {

// Largest planned unit assignment (it travels in the kernel parameters).
constexpr int kMaxPlanUnits = 1024;
constexpr int kMaxPlanCtas = 160;

struct FwdParams {
  int B, Hq, Hkv, Sq, Skv;
  int causal;
  int input_pos;
  int window;              // sliding window in keys (causal only), 0: none
  int num_m_blocks;        // m-blocks per head (of 128 or 256 rows)
  int pair_heads;          // a unit = 2 heads x 128 rows (else 1 head x 256)
  // Unit order: 0 heaviest m-block first, the heads of an m-block in turn;
  // 1 (units of equal work) the m-blocks of a head (pair) in turn.
  int head_major;
  // GQA packing (few query rows): one Q tile holds the Sq rows of all
  // `group` query heads of a K/V head, row r = head (r / Sq), position
  // (r % Sq); the second tile is unused.
  int pack_gqa;
  int group;               // Hq / Hkv
  int q_tile_bytes;        // bytes one Q tile load brings in
  float scale_log2;        // |scale| * log2(e)
  int negate_scores;       // scale < 0: S is computed as -(Q K^T)
  float o_scale;           // multiplies O (FP8 inputs: the V descale; else 1)
  void* o;                 // [B, Hq, Sq, D] output (16-bit elements)
  float* lse;              // [B, Hq, Sq] or nullptr
  int num_units;           // work units (pairs of 128-row Q tiles x splits)
  // Split-KV: the keys are cut into num_splits ranges of split_tiles K/V
  // tiles; unit (tiles, split) writes normalised fp32 partial outputs and
  // natural-log LSEs of its key range to o_part / lse_part (num_splits == 1
  // and o_part == nullptr: the plain forward pass writing O and LSE).
  int num_splits;
  int split_tiles;
  float* o_part;           // [num_splits, B*Hq, Sq, D]
  float* lse_part;         // [num_splits, B*Hq, Sq]
  // Packed split-KV launch whose units all run at once, one per CTA, the
  // num_splits key ranges of a (batch, K/V head) forming one thread-block
  // cluster (rank = key range): each CTA keeps its partial results in its
  // own shared memory and rank 0 merges them over distributed shared
  // memory (no global partials, no counters).
  // (Otherwise the key ranges are merged by a second launch on the same
  // stream, attn_merge_kernel: this kernel only writes the partials.)
  int cluster_merge;
  // Divisors of the unit decode: num_splits, num_m_blocks, units per
  // m-block (B*Hq/2 paired, else B*Hq), heads per batch entry (Hq/2 paired,
  // else Hq), group, and Hkv (packed units).
  FastDiv fd_splits, fd_m_blocks, fd_per_m, fd_heads, fd_group, fd_hkv;
  // Planned unit assignment (plan_units > 0; two-tile one-pass launches of
  // at most kMaxPlanUnits units whose work differs): CTA c walks units
  // plan_unit[plan_start[c] .. plan_start[c + 1]) in that order.  Otherwise
  // the zigzag rounds of unit_index.
  int plan_units;
  unsigned short plan_start[kMaxPlanCtas + 1];
  unsigned short plan_unit[kMaxPlanUnits];
  unsigned int* status;    // device status word (timeouts)
  unsigned long long timeout_ns;
  // Self-test of the bounded waits (0 in every normal launch): CTA 0's
  // producer never loads its first K tile, so that CTA's MMA warp waits for
  // a tile that cannot arrive until the wait runs out and the CTA aborts.
  int withhold_first_load;
};

namespace cfg {
constexpr int kTM = 128;          // rows per Q tile (TMEM lanes)
constexpr int kTN = 128;          // keys per K/V tile
constexpr int kBlockM = 256;      // query rows per CTA (two Q tiles)
// The MMA issuer and the TMA producer take the lowest warp indices: warp
// schedulers favour older (lower-index) warps, and the single-thread MMA
// issue must not starve behind the instruction-dense softmax warps.
constexpr int kThreads = 384;
constexpr int kMmaWarp = 0;
constexpr int kLoadWarp = 1;
constexpr int kSoftmaxWarp0 = 4;  // warps 4-7: Q tile 0, warps 8-11: Q tile 1
constexpr int kTmemCols = 512;
// Key ranges merged in one thread-block cluster (the portable cluster size).
constexpr int kMaxClusterRanges = 8;
constexpr float kRescaleTau = 8.0f;  // lazy rescale threshold (log2 units)
// Register split of the variants that hold a whole S row (128 fp32) in
// registers from the max pass to the exp pass (all two-tile variants: 1-5 %
// faster than re-reading S from TMEM; the packed ones re-read): the launch
// gives every thread kRegsLaunch; warpgroup 0 (MMA issuer, producer, two
// idle warps) drops to kRegsControl and the two softmax warpgroups rise to
// kRegsSoftmax.  The shares must add up to the launch allocation exactly,
// or the increase would wait forever.
constexpr int kRegsLaunch = 168;
constexpr int kRegsControl = 72;
constexpr int kRegsSoftmax = 216;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <=
                  kThreads * kRegsLaunch,
              "register split exceeds the launch allocation");
constexpr float kLn2 = 0.6931471805599453f;
}  // namespace cfg

// Shared memory of one CTA: Q tiles, the K/V slot ring, mbarriers.  The
// packed variant has one Q tile and fills the rest of the 227 KB with ring
// slots (a decode step is bound by the K/V bytes in flight per SM).  Rows
// are cut into 128-byte boxes (64 16-bit or 128 8-bit elements): an FP8
// tile of D = 128 has the geometry of a 16-bit tile of D = 64.
template <int D, bool kPack = false, bool kFp8 = false>
struct Layout {
  static constexpr int kEs = kFp8 ? 1 : 2;               // element bytes
  static_assert((D * kEs) % 128 == 0, "rows of whole 128-byte boxes");
  static constexpr int kChunks = D * kEs / 128;          // 128-byte boxes/row
  static constexpr int kBoxElems = 128 / kEs;            // elements per box row
  static constexpr int kBoxBytes = 128 * 128;            // 128 rows x 128 B
  static constexpr int kTileBytes = kChunks * kBoxBytes; // one Q/K/V tile
  static constexpr int kQTiles = kPack ? 1 : 2;
  static constexpr int kSlots =                           // K/V ring slots
      kPack ? (kChunks == 2 ? 6 : 13) : (kChunks == 2 ? 4 : 8);
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = kQOff + kQTiles * kTileBytes;
  // Output staging of the two-tile variants: per Q tile one 128-row x
  // 128-byte box (64 16-bit columns of O, 128-byte swizzle), written by the
  // tile's softmax threads and stored to global memory by TMA.
  static constexpr int kStageTileBytes = kPack ? 0 : 128 * 128;
  static constexpr int kStageOff = kRingOff + kSlots * kTileBytes;
  static constexpr int kBarOff = kStageOff + 2 * kStageTileBytes;
  // barriers: q_full[2], full[S], empty[S], s_full[6] (two S regions, or
  // three shared S buffers with one barrier per tile and buffer),
  // p_full[2], o_full[2], drain[1], q_free[2], pv_done[2], epi[2]
  static constexpr int kNumBars = 2 + 2 * kSlots + 6 + 2 + 2 + 1 + 2 + 2 + 2;
  // misc: TMEM base, abort flag, per-tile "merge here" flags, per-tile
  // epilogue "saw O complete" flags (4 bytes per warp)
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
  static constexpr int kBytes = kMiscOff + 16 + 32;
  static constexpr int kSmemBytes = kBytes + 1024;  // slack for 1 KB alignment
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

// Key tiles of the Q tile whose first row is m0 (packed: the tile holding
// the Sq rows of every head of a GQA group, m0 = 0): tiles [lo, hi) hold
// every key its rows can see; tiles >= ms need the causal / key-tail mask
// and tiles < wl the sliding-window mask.  hi == 0: the tile has no rows.
struct TileKeys {
  int lo, hi, ms, wl;
};

template <bool kWindow>
__device__ __forceinline__ TileKeys tile_keys(const FwdParams& p, int m0) {
  TileKeys k{0, 0, 0, 0};
  if (m0 >= p.Sq) return k;
  // Absolute positions of the tile's first and last valid rows.
  const int pos_first = p.input_pos + m0;
  const int pos_last = p.input_pos + min(m0 + cfg::kTM, p.Sq) - 1;
  const int kend = p.causal ? min(pos_last + 1, p.Skv) : p.Skv;
  k.hi = (kend + cfg::kTN - 1) / cfg::kTN;
  const int full_tiles = p.Skv / cfg::kTN;
  k.ms = p.causal ? min((pos_first + 1) / cfg::kTN, full_tiles) : full_tiles;
  if constexpr (kWindow) {
    // Row at position r sees keys r - window + 1 .. r.
    k.lo = max(0, pos_first - p.window + 1) / cfg::kTN;
    k.wl = (max(0, pos_last - p.window + 1) + cfg::kTN - 1) / cfg::kTN;
  }
  return k;
}

// One work unit: two 128-row Q tiles.  With an even GQA group the tiles
// are two query heads of one K/V group at the same rows (identical causal
// extents and masks, shared K/V tiles); otherwise two consecutive row blocks
// of one head.  Unit 0 is the heaviest m-block (the page's reversed block
// order) and consecutive units are consecutive heads, so the heads of a K/V
// group run together and find K/V in L2; with units of equal work
// (p.head_major) consecutive units are the m-blocks of one head (pair).
struct Unit {
  int kb;        // first K/V tile the unit streams (tile j of the unit is
                 // key tile kb + j)
  int lo;        // first K/V tile any row of the unit can see (window)
  int split;     // key-range index (0 without split-KV)
  int plane[2];  // [B*Hq] plane of each Q tile
  int m0[2];     // first row of each Q tile
  int n[2];      // K/V tiles each Q tile visits (from kb)
  int hi[2];     // end of the key tiles each Q tile can see
  int ms[2];     // first K/V tile that needs the causal / tail mask
  int wl[2];     // K/V tiles below wl need the window mask
  int kv_plane;  // [B*Hkv] plane of the shared K/V head
  int n_kv;      // K/V tiles the unit streams
};

template <bool kPack, bool kWindow>
__device__ __forceinline__ Unit decode_unit(const FwdParams& p, int u) {
  Unit w;
  {
    const int us = fast_div(u, p.fd_splits);
    w.split = u - us * p.num_splits;
    u = us;
  }
  const int kt0 = w.split * p.split_tiles;  // key range of the unit
  const int kt1 = kt0 + p.split_tiles;
  TileKeys tk[2];
  if constexpr (kPack) {
    // Unit = one (batch, K/V head): tile 0 holds all its query rows.
    const int b = fast_div(u, p.fd_hkv);
    const int kvh = u - b * p.Hkv;
    w.kv_plane = b * p.Hkv + kvh;
    w.plane[0] = b * p.Hq + kvh * p.group;  // first head of the group
    w.plane[1] = w.plane[0];
    w.m0[0] = w.m0[1] = 0;
    tk[0] = tile_keys<kWindow>(p, 0);
    tk[1] = TileKeys{0, 0, 0, 0};
  } else {
    // Heaviest row block first, the heads of a row block in turn; or, when
    // every unit carries the same work (no mask), the row blocks of a head
    // in turn, so that the units in flight share a few heads' K/V (which
    // stay in L2) instead of each streaming its own head's.
    int mb, ub;
    if (p.head_major) {
      ub = fast_div(u, p.fd_m_blocks);
      mb = u - ub * p.num_m_blocks;
    } else {
      const int q = fast_div(u, p.fd_per_m);
      mb = p.num_m_blocks - 1 - q;
      ub = u - q * p.fd_per_m.d;
    }
    const int b = fast_div(ub, p.fd_heads);
    const int hh = ub - b * p.fd_heads.d;
    const int h0 = p.pair_heads ? 2 * hh : hh;
    w.kv_plane = b * p.Hkv + fast_div(h0, p.fd_group);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      w.plane[t] = b * p.Hq + h0 + (p.pair_heads ? t : 0);
      w.m0[t] = p.pair_heads ? mb * cfg::kTM : mb * cfg::kBlockM + t * cfg::kTM;
      tk[t] = tile_keys<kWindow>(p, w.m0[t]);
    }
  }
  // Both tiles share one K/V stream, from the first tile any of the unit's
  // rows can see (tile 0 holds the earliest rows); with a window, tile 1's
  // first tiles may then be fully masked for it.
  w.lo = tk[0].lo;
  w.kb = max(kt0, w.lo);
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    w.hi[t] = tk[t].hi;
    w.ms[t] = tk[t].ms;
    w.wl[t] = tk[t].wl;
    w.n[t] = max(0, min(tk[t].hi, kt1) - w.kb);
  }
  w.n_kv = max(w.n[0], w.n[1]);
  return w;
}


// The cluster form of merge_tile (packed tiles): the partial output rows of
// key range c live in cluster CTA c's shared memory, row r at
// part + r * D * 4 bytes, its LSE at part + kTM * D * 4 + r * 4.  Same
// weights as merge_tile; ranges past a row's causal horizon or before its
// window hold nothing for it and are not read.
template <int D, bool kBF16, bool kWindow>
__device__ __forceinline__ void merge_tile_cluster(const FwdParams& p,
                                                   int plane0, uint32_t part,
                                                   int tid) {
  constexpr float kLog2e = 1.4426950408889634f;
  constexpr int kGroups = D / 4;
  constexpr int kRowsPerPass = cfg::kTM / kGroups;
  const uint32_t lse_off = cfg::kTM * D * 4;
  const int split_keys = p.split_tiles * cfg::kTN;
  const int nrows = p.group * p.Sq;
  const int cg = tid % kGroups;
  for (int r = tid / kGroups; r < nrows; r += kRowsPerPass) {
    const int q_plane = plane0 + r / p.Sq;
    const int q_row = r % p.Sq;
    const long long row = static_cast<long long>(q_plane) * p.Sq + q_row;
    const int row_pos = p.input_pos + q_row;
    const int vis_end = p.causal ? min(p.Skv, row_pos + 1) : p.Skv;
    const int ns = min(p.num_splits, (vis_end + split_keys - 1) / split_keys);
    const int c0 =
        kWindow ? max(0, row_pos - p.window + 1) / split_keys : 0;
    const uint32_t lse_addr = part + lse_off + 4 * r;
    const uint32_t o_addr = part + (r * D + 4 * cg) * 4;
    // Every range's LSE and columns are requested before any is used: one
    // round trip over the cluster instead of one per range and pass.
    float lse_c[cfg::kMaxClusterRanges];
    float4 x_c[cfg::kMaxClusterRanges];
#pragma unroll
    for (int c = 0; c < cfg::kMaxClusterRanges; ++c) {
      lse_c[c] = -INFINITY;
      x_c[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c >= c0 && c < ns) {
        lse_c[c] = ptx::ld_shared_cluster_f32(ptx::mapa_shared(lse_addr, c));
        x_c[c] = ptx::ld_shared_cluster_v4(ptx::mapa_shared(o_addr, c));
      }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < cfg::kMaxClusterRanges; ++c) mx = fmaxf(mx, lse_c[c]);
    float wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < cfg::kMaxClusterRanges; ++c) {
      // Ranges outside [c0, ns) hold LSE -inf: weight 0.
      const float wc = ptx::ex2((lse_c[c] - mx) * kLog2e);
      wsum += wc;
      acc.x += wc * x_c[c].x;
      acc.y += wc * x_c[c].y;
      acc.z += wc * x_c[c].z;
      acc.w += wc * x_c[c].w;
    }
    const float inv = ptx::rcp(wsum);
    uint2 out;
    out.x = ptx::pack2<kBF16>(acc.x * inv, acc.y * inv);
    out.y = ptx::pack2<kBF16>(acc.z * inv, acc.w * inv);
    reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.o) + row * D)[cg] = out;
    if (cg == 0 && p.lse != nullptr)
      p.lse[row] = mx + ptx::lg2(wsum) * cfg::kLn2;
  }
}

// k-th unit of CTA `cta` among `ctas`: from the launch's plan, or rounds of
// `ctas` units with the CTA order reversed every other round.  With units
// sorted heaviest first the rounds keep the per-CTA totals within a few
// percent of the mean for causal masks (plain round-robin gives every
// CTA's first pick of each round to CTA 0); the plan, packed on the host,
// within a fraction of a percent.
__device__ __forceinline__ int unit_index(const FwdParams& p, int k, int cta,
                                          int ctas) {
  if (p.plan_units > 0) return p.plan_unit[p.plan_start[cta] + k];
  return k * ctas + ((k & 1) ? (ctas - 1 - cta) : cta);
}

// Units CTA `cta` walks (the loop bound of every role; under the zigzag
// rounds the last round's index may lie past num_units and is skipped).
__device__ __forceinline__ int units_of_cta(const FwdParams& p, int cta,
                                            int ctas) {
  if (p.plan_units > 0) return p.plan_start[cta + 1] - p.plan_start[cta];
  return (p.num_units + ctas - 1) / ctas;
}

// Persistent kernel: one CTA per SM walks its units (unit_index) in
// rounds.  Barrier phases, the K/V ring position and
// TMEM carry over from unit to unit, so the next unit's Q load and first
// MMAs overlap the current unit's last MMAs and epilogue.
// kPack: the query heads of a GQA group share tile 0 (few query rows).
// kSplit: split-KV launch (o_part set) -- each unit writes its key range's
// partial results: into its shared memory for the cluster merge (packed
// launches of one wave), else to o_part / lse_part for the merge launch.
// kWindow: causal sliding window (window > 0) -- compiles the lower mask.
// The variants keep each launch's softmax loop free of the others' code:
// in one kernel with run-time switches the two-tile loop ran out of
// registers and lost 5-11 %.
//
// kFp8: Q, K, V in E4M3 (O in bf16, kBF16 set): both products run as
// kind::f8f6f4 MMAs and P is rounded to E4M3 (four keys per TMEM column);
// p.scale_log2 carries the Q and K descales, p.o_scale the V descale.
template <int D, bool kBF16, bool kPack, bool kSplit, bool kWindow,
          bool kFp8 = false>
__global__ void __launch_bounds__(cfg::kThreads, 1)
    attn_fwd_sm103_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_o,
                          const FwdParams p) {
  static_assert(!kFp8 || kBF16, "FP8 inputs give a bf16 output");
  using L = Layout<D, kPack, kFp8>;
  constexpr bool kHoldS = !kPack;  // S row kept in registers (see cfg)
  // O leaves through shared memory and TMA stores (two-tile one-pass
  // variants); split-KV partials and packed tiles are stored per thread.
  constexpr bool kStageO = !kPack && !kSplit;
  // Three S buffers shared by the two Q tiles (D = 64: O needs 128 columns).
  constexpr bool kTriple = D == 64 && !kPack;
  constexpr int kOCol = kTriple ? 3 * cfg::kTN : 2 * cfg::kTN;  // first O column
  static_assert(kOCol + 2 * D <= cfg::kTmemCols, "TMEM columns");
  using namespace cfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = ptx::smem_u32(smem);
  const uint32_t s_q = s_base + L::kQOff;
  const uint32_t s_ring = s_base + L::kRingOff;
  const uint32_t bar0 = s_base + L::kBarOff;
  const uint32_t bar_q = bar0;                         // [2]
  const uint32_t bar_full = bar0 + 8 * 2;              // [kSlots]
  const uint32_t bar_empty = bar_full + 8 * L::kSlots; // [kSlots]
  const uint32_t bar_s = bar_empty + 8 * L::kSlots;    // [6]: [3 * t + buffer]
  const uint32_t bar_p = bar_s + 8 * 6;                // [2]
  const uint32_t bar_o = bar_p + 8 * 2;                // [2]
  const uint32_t bar_drain = bar_o + 8 * 2;            // [1]
  const uint32_t bar_qfree = bar_drain + 8;            // [2]
  const uint32_t bar_pvdone = bar_qfree + 8 * 2;       // [2] every PV but a unit's last
  const uint32_t bar_epi = bar_pvdone + 8 * 2;         // [2] epilogue entry, all warps
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<int*>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  constexpr int nslots = L::kSlots;
  const int u_first = static_cast<int>(blockIdx.x);
  const int u_step = static_cast<int>(gridDim.x);
  const int k_end = units_of_cta(p, u_first, u_step);  // units of this CTA

  // The merge launch queued behind a split-KV launch may be scheduled as
  // soon as every CTA has started (its CTAs only wait, for this grid's
  // completion).
  if constexpr (kSplit) {
    if (!p.cluster_merge) ptx::griddep_launch_dependents();
  }
  if constexpr (kPack) {
    // A packed Q load fills only group*Sq rows of the tile: keep the other
    // rows zero so their (discarded) scores stay finite.
    for (int i = threadIdx.x; i < L::kTileBytes / 16; i += kThreads)
      ptx::st_shared_v4(s_q + 16 * i, 0u, 0u, 0u, 0u);
    ptx::fence_proxy_async_smem();
  }
  if (warp == kLoadWarp && lane == 0 && k_end > 0) {
    // The first unit's Q tiles and first K/V tiles (as many as the ring
    // holds) start moving into L2 while the CTA initialises its barriers
    // and TMEM; the producer's loads of the same boxes follow.  Same-box
    // A/B: the split-KV decode step 2.7-3.1 % shorter, the one-pass
    // workloads unchanged.
    ptx::prefetch_tensormap(&tm_q);
    ptx::prefetch_tensormap(&tm_k);
    ptx::prefetch_tensormap(&tm_v);
    const int u0 = unit_index(p, 0, u_first, u_step);
    if (u0 < p.num_units) {
      const Unit w0 = decode_unit<kPack, kWindow>(p, u0);
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (w0.n[t] > 0)
          for (int c = 0; c < L::kChunks; ++c)
            ptx::tma_prefetch_3d(&tm_q, c * L::kBoxElems, w0.m0[t],
                                 w0.plane[t]);
      const int pre = min(w0.n_kv, nslots / 2);
      for (int j = 0; j < pre; ++j)
        for (int kv = 0; kv < 2; ++kv)
          for (int c = 0; c < L::kChunks; ++c)
            ptx::tma_prefetch_3d(kv ? &tm_v : &tm_k, c * L::kBoxElems,
                                 (w0.kb + j) * kTN, w0.kv_plane);
    }
  }
  if (threadIdx.x == 0) {
    // P-ready and epilogue-entry barriers collect one arrival per softmax
    // thread of the tile; the others one arrival (an expect-tx, a
    // tcgen05.commit).
    for (int i = 0; i < L::kNumBars; ++i) {
      const uint32_t bar = bar0 + 8 * i;
      const bool per_thread = bar == bar_p || bar == bar_p + 8 ||
                              bar == bar_epi || bar == bar_epi + 8;
      ptx::mbar_init(bar, per_thread ? kTM : 1);
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

  if (warp < kSoftmaxWarp0) {
  if constexpr (kHoldS) ptx::setmaxnreg_dec<kRegsControl>();
  if (warp == kLoadWarp) {
    // ------------------------------------------------------ TMA producer
    // The whole warp runs this loop (warp-uniform); one elected lane issues.
    // (Its tensor maps and first tiles were prefetched at kernel entry.)
    bool ok = true;
    int it = 0;               // ring items (K_0, V_0, K_1, ...) issued so far
    int q_loads[2] = {0, 0};  // Q tile loads issued so far, per tile
    const bool withhold = p.withhold_first_load != 0 && blockIdx.x == 0;
    for (int k = 0; k < k_end && ok; ++k) {
      const int u = unit_index(p, k, u_first, u_step);
      if (u >= p.num_units) continue;
      const Unit w = decode_unit<kPack, kWindow>(p, u);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (w.n[t] == 0 || !ok) continue;
        // The buffer is free once the previous unit's last S MMA on it is
        // done (committed by the MMA warp to q_free).
        if (q_loads[t] > 0)
          ok = __all_sync(0xffffffffu,
                          wait_bounded(bar_qfree + 8 * t, (q_loads[t] - 1) & 1,
                                       abort_flag, p, 1));
        if (!ok) break;
        const uint32_t dst = s_q + t * L::kTileBytes;
        ptx::mbar_arrive_expect_tx_elect(bar_q + 8 * t, p.q_tile_bytes);
        for (int c = 0; c < L::kChunks; ++c)
          ptx::tma_load_3d_elect(dst + c * L::kBoxBytes, &tm_q, bar_q + 8 * t,
                                 c * L::kBoxElems, w.m0[t], w.plane[t]);
        ++q_loads[t];
      }
      for (int j = 0; j < w.n_kv && ok; ++j) {
        for (int kv = 0; kv < 2; ++kv) {
          const int slot = it % nslots;
          if (it >= nslots) {
            ok = __all_sync(0xffffffffu,
                            wait_bounded(bar_empty + 8 * slot,
                                         ((it / nslots) - 1) & 1,
                                         abort_flag, p, 1));
            if (!ok) break;
          }
          if (withhold && it == 0) {  // self-test: item 0 never arrives
            ++it;
            continue;
          }
          const uint32_t dst = s_ring + slot * L::kTileBytes;
          ptx::mbar_arrive_expect_tx_elect(bar_full + 8 * slot, L::kTileBytes);
          for (int c = 0; c < L::kChunks; ++c)
            ptx::tma_load_3d_elect(dst + c * L::kBoxBytes, kv ? &tm_v : &tm_k,
                                   bar_full + 8 * slot, c * L::kBoxElems,
                                   (w.kb + j) * kTN, w.kv_plane);
          ++it;
        }
      }
    }
    if (!ok) {
      // Let every copy still in flight land before the CTA goes away.
      for (int t = 0; t < 2; ++t)
        if (q_loads[t] > 0) drain_wait(bar_q + 8 * t, (q_loads[t] - 1) & 1, p);
      for (int i = max(0, it - nslots); i < it; ++i)
        if (!(withhold && i == 0))
          drain_wait(bar_full + 8 * (i % nslots), (i / nslots) & 1, p);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (warp-uniform); one elected lane issues.
    const uint32_t idesc_qk =
        kFp8 ? ptx::idesc_e4m3(kTM, kTN, false, p.negate_scores != 0)
             : ptx::idesc_f16(kBF16, kTM, kTN, false, p.negate_scores != 0);
    const uint32_t idesc_pv = kFp8 ? ptx::idesc_e4m3(kTM, D, true, false)
                                   : ptx::idesc_f16(kBF16, kTM, D, true, false);
    bool ok = true;
    bool issued_any = false;

    // Descriptor low words, computed once; per MMA one add of a
    // compile-time offset.  K-major tiles: LBO unused (16), SBO = 1024
    // (8 rows of 128 B).  V (MN-major): LBO = 16 KB between the 128-byte
    // column boxes of D (16-bit D = 128 has two), SBO = 1024 between groups
    // of 8 keys.  One MMA consumes 32 bytes of K: 16 16-bit or 32 8-bit
    // elements.
    constexpr uint32_t kHi = ptx::sdesc_hi_sw128(1024);
    const uint32_t q_lo = ptx::sdesc_lo(s_q, 16);
    const uint32_t k_lo = ptx::sdesc_lo(s_ring, 16);
    const uint32_t v_lo = ptx::sdesc_lo(s_ring, L::kBoxBytes);
    constexpr uint32_t kTile16 = L::kTileBytes >> 4;

    // S = Q_t K_j^T into S region `sb`: A = Q tile (K-major), B = K tile
    // (K-major).
    auto issue_qk = [&](int t, int sb, int slot) {
      const uint32_t a0 = q_lo + t * kTile16;
      const uint32_t b0 = k_lo + slot * kTile16;
      const uint32_t d = tmem + sb * kTN;
#pragma unroll
      for (int kk = 0; kk < D * L::kEs / 32; ++kk) {
        const uint32_t off = ((kk / 4) * L::kBoxBytes + (kk % 4) * 32) >> 4;
        ptx::mma_ss_elect<kFp8>(d, a0 + off, b0 + off, kHi, idesc_qk,
                                kk > 0 ? 1u : 0u);
      }
    };
    // O_t (+)= P V_j : A = P in S region `sb` of TMEM, B = V tile
    // (MN-major).  Each MMA takes 32 / kEs keys: 8 TMEM columns of P and
    // that many 128-byte rows of V.
    auto issue_pv = [&](int t, int sb, int slot, bool acc) {
      constexpr int kKeys = 32 / L::kEs;
      const uint32_t b0 = v_lo + slot * kTile16;
      const uint32_t d = tmem + kOCol + t * D;
      const uint32_t a = tmem + sb * kTN;
#pragma unroll
      for (int kk = 0; kk < kTN / kKeys; ++kk) {
        ptx::mma_ts_elect<kFp8>(d, a + kk * 8,
                                b0 + ((kk * kKeys * 128) >> 4), kHi, idesc_pv,
                                (acc || kk > 0) ? 1u : 0u);
      }
    };

    int it = 0;               // ring items consumed so far
    int q_uses[2] = {0, 0};   // Q tile loads consumed, per tile
    int p_waits[2] = {0, 0};  // P-ready phases consumed, per tile
    int s_issued = 0;         // kTriple: S MMAs issued (buffer = count % 3)
    for (int k = 0; k < k_end && ok; ++k) {
      const int u = unit_index(p, k, u_first, u_step);
      if (u >= p.num_units) continue;
      const Unit w = decode_unit<kPack, kWindow>(p, u);
      // A key range wholly past the causal horizon of both tiles has no
      // work (split-KV only); the producer and softmax warps skip it too.
      if (w.n_kv == 0) continue;
      if constexpr (kPack) {
        // One Q tile whose scores alternate between the two S regions:
        // S(j+1) is computed while the softmax warps work on S(j), and
        // S(j+2) reuses region j%2 once PV(j) (issued just before it, and
        // executed in order) has read P(j).  Every PV but the unit's last
        // commits to o_full[1] so the softmax warps know when O may be
        // rescaled; the last commits to o_full[0] for the epilogue.
        const int n = w.n_kv;
        const int it0 = it;
        ok = __all_sync(0xffffffffu, wait_bounded(bar_q, q_uses[0] & 1,
                                                  abort_flag, p, 2));
        if (!ok) break;
        ++q_uses[0];
        for (int sb = 0; sb < 2 && sb < n && ok; ++sb) {
          const int it_k = it0 + 2 * sb;
          ok = __all_sync(0xffffffffu,
                          wait_bounded(bar_full + 8 * (it_k % nslots),
                                       (it_k / nslots) & 1, abort_flag, p,
                                       2));
          if (!ok) break;
          ptx::tc_fence_after();
          issue_qk(0, sb, it_k % nslots);
          ptx::tc_commit_elect(bar_s + 8 * sb);
          ptx::tc_commit_elect(bar_empty + 8 * (it_k % nslots));
          if (sb == n - 1) ptx::tc_commit_elect(bar_qfree);
          issued_any = true;
        }
        for (int j = 0; j < n && ok; ++j) {
          const int sb = j & 1;
          const int it_v = it0 + 2 * j + 1;
          ok = __all_sync(0xffffffffu,
                          wait_bounded(bar_full + 8 * (it_v % nslots),
                                       (it_v / nslots) & 1, abort_flag, p,
                                       2));
          if (!ok) break;
          const int pw = sb ? p_waits[1] : p_waits[0];
          ok = __all_sync(0xffffffffu, wait_bounded(bar_p + 8 * sb, pw & 1,
                                                    abort_flag, p, 2));
          if (!ok) break;
          if (sb) ++p_waits[1]; else ++p_waits[0];
          ptx::tc_fence_after();
          issue_pv(0, sb, it_v % nslots, j > 0);
          ptx::tc_commit_elect(j == n - 1 ? bar_o : bar_o + 8);
          ptx::tc_commit_elect(bar_empty + 8 * (it_v % nslots));
          if (j + 2 < n) {
            const int it_k = it0 + 2 * (j + 2);
            ok = __all_sync(0xffffffffu,
                            wait_bounded(bar_full + 8 * (it_k % nslots),
                                         (it_k / nslots) & 1, abort_flag,
                                         p, 2));
            if (!ok) break;
            issue_qk(0, sb, it_k % nslots);
            ptx::tc_commit_elect(bar_s + 8 * sb);
            ptx::tc_commit_elect(bar_empty + 8 * (it_k % nslots));
            if (j + 2 == n - 1) ptx::tc_commit_elect(bar_qfree);
          }
        }
        it = it0 + 2 * n;
        continue;
      }
      if constexpr (kTriple) {
        // Per K/V step j: S_0(j+1), PV_0(j), S_1(j+1), PV_1(j).  S MMA
        // number i goes to buffer i % 3; with two S issues between any S
        // and its own PV, the buffer an S overwrites was last read by a PV
        // issued (and, in issue order, executed) before it.  So a tile's
        // next S is computed while its softmax works on the current one.
        // Each PV but a unit's last commits to pv_done[t], which the softmax
        // waits on before it may rescale O.
        int pbuf[2] = {0, 0};  // buffer holding each tile's current S / P
        ok = __all_sync(0xffffffffu,
                        wait_bounded(bar_full + 8 * (it % nslots),
                                     (it / nslots) & 1, abort_flag, p, 2));
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok) break;
          if (w.n[t] == 0) continue;
          ok = __all_sync(0xffffffffu,
                          wait_bounded(bar_q + 8 * t, q_uses[t] & 1,
                                       abort_flag, p, 2));
          if (!ok) break;
          ++q_uses[t];
          ptx::tc_fence_after();
          const int b = s_issued % 3;
          issue_qk(t, b, it % nslots);
          ptx::tc_commit_elect(bar_s + 8 * (3 * t + b));
          pbuf[t] = b;
          ++s_issued;
          if (w.n[t] == 1) ptx::tc_commit_elect(bar_qfree + 8 * t);
          issued_any = true;
        }
        if (!ok) break;
        ptx::tc_commit_elect(bar_empty + 8 * (it % nslots));
        const int it0 = it;
        for (int j = 0; j < w.n_kv && ok; ++j) {
          const int it_v = it0 + 2 * j + 1;
          const int slot_v = it_v % nslots;
          const int it_k = it0 + 2 * j + 2;
          const int slot_k = it_k % nslots;
          ok = __all_sync(0xffffffffu,
                          wait_bounded(bar_full + 8 * slot_v,
                                       (it_v / nslots) & 1, abort_flag, p,
                                       2));
          if (!ok) break;
          bool k_ready = false;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (!ok) break;
            if (j >= w.n[t]) continue;
            int nb = -1;
            if (j + 1 < w.n[t]) {
              if (!k_ready) {
                ok = __all_sync(0xffffffffu,
                                wait_bounded(bar_full + 8 * slot_k,
                                             (it_k / nslots) & 1, abort_flag,
                                             p, 2));
                if (!ok) break;
                k_ready = true;
              }
              ptx::tc_fence_after();
              nb = s_issued % 3;
              issue_qk(t, nb, slot_k);
              ptx::tc_commit_elect(bar_s + 8 * (3 * t + nb));
              ++s_issued;
              if (j + 1 == w.n[t] - 1) ptx::tc_commit_elect(bar_qfree + 8 * t);
            }
            ok = __all_sync(0xffffffffu,
                            wait_bounded(bar_p + 8 * t, p_waits[t] & 1,
                                         abort_flag, p, 2));
            if (!ok) break;
            ++p_waits[t];
            ptx::tc_fence_after();
            issue_pv(t, pbuf[t], slot_v, j > 0);
            ptx::tc_commit_elect(j == w.n[t] - 1 ? bar_o + 8 * t
                                                 : bar_pvdone + 8 * t);
            if (nb >= 0) pbuf[t] = nb;
          }
          if (!ok) break;
          ptx::tc_commit_elect(bar_empty + 8 * slot_v);
          if (j + 1 < w.n_kv) ptx::tc_commit_elect(bar_empty + 8 * slot_k);
        }
        it = it0 + 2 * w.n_kv;
        continue;
      }
      // S_t = Q_t K_0^T for both tiles.
      ok = __all_sync(0xffffffffu,
                      wait_bounded(bar_full + 8 * (it % L::kSlots),
                                   (it / L::kSlots) & 1, abort_flag, p, 2));
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (!ok) break;
        if (w.n[t] == 0) continue;
        ok = __all_sync(0xffffffffu,
                        wait_bounded(bar_q + 8 * t, q_uses[t] & 1, abort_flag,
                                     p, 2));
        if (!ok) break;
        ++q_uses[t];
        ptx::tc_fence_after();
        issue_qk(t, t, it % L::kSlots);
        ptx::tc_commit_elect(bar_s + 8 * t);
        if (w.n[t] == 1) ptx::tc_commit_elect(bar_qfree + 8 * t);
        issued_any = true;
      }
      if (!ok) break;
      ptx::tc_commit_elect(bar_empty + 8 * (it % L::kSlots));
      const int it0 = it;
      for (int j = 0; j < w.n_kv && ok; ++j) {
        const int it_v = it0 + 2 * j + 1;
        const int slot_v = it_v % L::kSlots;
        const int it_k = it0 + 2 * j + 2;
        const int slot_k = it_k % L::kSlots;
        ok = __all_sync(0xffffffffu,
                        wait_bounded(bar_full + 8 * slot_v,
                                     (it_v / L::kSlots) & 1, abort_flag, p, 2));
        if (!ok) break;
        bool k_ready = false;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok) break;
          if (j >= w.n[t]) continue;
          ok = __all_sync(0xffffffffu,
                          wait_bounded(bar_p + 8 * t, p_waits[t] & 1,
                                       abort_flag, p, 2));
          if (!ok) break;
          ++p_waits[t];
          ptx::tc_fence_after();
          issue_pv(t, t, slot_v, j > 0);
          if (j == w.n[t] - 1) {
            ptx::tc_commit_elect(bar_o + 8 * t);
          } else {
            if (!k_ready) {
              ok = __all_sync(0xffffffffu,
                              wait_bounded(bar_full + 8 * slot_k,
                                           (it_k / L::kSlots) & 1, abort_flag,
                                           p, 2));
              if (!ok) break;
              k_ready = true;
            }
            issue_qk(t, t, slot_k);
            ptx::tc_commit_elect(bar_s + 8 * t);
            // After the tile's last S MMA, its Q buffer can be refilled.
            if (j + 1 == w.n[t] - 1) ptx::tc_commit_elect(bar_qfree + 8 * t);
          }
        }
        if (!ok) break;
        ptx::tc_commit_elect(bar_empty + 8 * slot_v);
        if (j + 1 < w.n_kv) ptx::tc_commit_elect(bar_empty + 8 * slot_k);
      }
      it = it0 + 2 * w.n_kv;
    }
    if (!ok && issued_any) {
      // Wait for the MMAs already issued before TMEM is released.
      ptx::tc_commit_elect(bar_drain);
      drain_wait(bar_drain, 0, p);
    }
    __syncwarp();
  }
  } else {
    if constexpr (kHoldS) ptx::setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------------- softmax / correction / epilogue
    const int t = warp / 4 - 1;             // Q tile of this warpgroup
    const int r = threadIdx.x % 128;        // row within the tile
    const uint32_t lane_off = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t t_o = tmem + lane_off + kOCol + t * D;
    // Score factor (log2 units).  A zero scale is replaced by 1e-30: the
    // weights stay uniform (every score times it is far below one ulp of
    // the exponent), and a masked -inf score times it stays -inf instead of
    // becoming NaN, so the exp pass needs no mask of its own once pass 1
    // has written -inf into the held scores.
    const float c = p.scale_log2 > 0.f ? p.scale_log2 : 1e-30f;
    // Packed query heads fill only group*Sq rows of the tile: a warp whose
    // 32 rows are all padding keeps in step (waits, arrivals) but computes
    // nothing.  Its P rows stay whatever S left there, which only reaches
    // the matching O rows (row i of P V is row i of P times V), and those
    // are never stored.
    const bool live = !kPack || (warp % 4) * 32 < p.group * p.Sq;
    bool ok = true;
    int s_waits = 0;   // S-ready phases consumed (packed: S region 0)
    int s_waits1 = 0;  // packed: S-ready phases of S region 1
    int o_waits = 0;   // O-done phases consumed
    int pv_waits = 0;  // packed, kTriple: per-step PV-done phases consumed
    int s_before = 0;           // kTriple: S MMAs of this CTA's earlier units
    int s_uses[3] = {0, 0, 0};  // kTriple: this tile's uses of each buffer

    for (int k = 0; k < k_end && ok; ++k) {
      const int u = unit_index(p, k, u_first, u_step);
      if (u >= p.num_units) continue;
      const Unit w = decode_unit<kPack, kWindow>(p, u);
      const int n = t ? w.n[1] : w.n[0];
      // kTriple: the MMA warp issues n[0] + n[1] S MMAs for this unit, in
      // the order S_0(0), S_1(0), then S_0(j+1), S_1(j+1) during step j.
      const int s_unit = s_before;
      s_before += w.n[0] + w.n[1];
      if (n == 0) continue;
      const int ms = t ? w.ms[1] : w.ms[0];
      const int wl = kWindow ? (t ? w.wl[1] : w.wl[0]) : 0;
      const int m0 = t ? w.m0[1] : w.m0[0];
      // This thread's query row: head plane and row index within the head.
      int q_plane = t ? w.plane[1] : w.plane[0];
      int q_row = m0 + r;
      bool row_ok = q_row < p.Sq;
      if constexpr (kPack) {
        q_plane += r / p.Sq;
        q_row = r % p.Sq;
        row_ok = r < p.group * p.Sq;
      }
      const int row_pos = p.input_pos + q_row;  // absolute query position
      float m_run = -INFINITY;  // running max of scaled scores (log2 units)
      float l_run = 0.f;        // running sum of 2^(s*c - m_run)

      for (int j = 0; j < n; ++j) {
        // S region of this step: the tile's own, (packed) alternating, or
        // (kTriple) the buffer of this tile's S MMA number s_unit + rel.
        int sb = kPack ? (j & 1) : t;
        if constexpr (kTriple) {
          const int n0 = w.n[0], n1 = w.n[1];
          int rel = 0;
          if (j > 0)
            rel = (n0 > 0) + (n1 > 0) + max(0, min(j - 1, n0 - 1)) +
                  max(0, min(j - 1, n1 - 1));
          if (t == 1 && j < n0) ++rel;
          sb = (s_unit + rel) % 3;
        }
        const uint32_t t_s = tmem + lane_off + sb * kTN;
        const bool odd = kPack && sb == 1;
        if constexpr (kTriple) {
          // One barrier per (tile, buffer): its phases are this tile's uses
          // of the buffer only, each awaited in turn.
          ok = __all_sync(0xffffffffu,
                          wait_bounded(bar_s + 8 * (3 * t + sb),
                                       s_uses[sb] & 1, abort_flag, p, 3));
          if (!ok) break;
          ++s_uses[sb];
        } else {
          ok = __all_sync(0xffffffffu,
                          wait_bounded(bar_s + 8 * sb,
                                       (odd ? s_waits1 : s_waits) & 1,
                                       abort_flag, p, 3));
          if (!ok) break;
          if (odd) ++s_waits1; else ++s_waits;
        }
        ptx::tc_fence_after();
        if (!live) {
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar_p + 8 * (kTriple ? t : sb));
          continue;
        }

        // Pass 1: row maximum of the scaled scores over the visible keys.
        // Visible keys of this row in the tile are the columns c with
        // lo <= c < lim: key < Skv, key <= row_pos when causal (only tiles
        // >= ms can cut), key > row_pos - window with a window (only tiles
        // < wl can cut; lo stays 0 without one).
        const int kt = w.kb + j;  // key tile index
        const bool masked = kt >= ms || (kWindow && kt < wl);
        int lim = kTN, lo = 0, span = kTN;
        if (masked) {
          const int kbase = kt * kTN;
          lim = min(kTN, p.Skv - kbase);
          if (p.causal) lim = min(lim, row_pos - kbase + 1);
          if constexpr (kWindow) {
            lo = row_pos - p.window + 1 - kbase;
            span = max(lim - lo, 0);
          }
        }
        // One unsigned compare tests both ends of [lo, lo + span); in a
        // same-box A/B it ran the window workload 11 % faster than two
        // signed compares.
        auto hidden = [&](int c) {
          if constexpr (kWindow)
            return static_cast<unsigned>(c - lo) >= static_cast<unsigned>(span);
          return c >= lim;
        };
        // kHoldS: the whole S row stays in registers for pass 2.
        uint32_t sr[kTN];
        float mx;
        {
#pragma unroll
          for (int q = 0; q < kTN / 32; ++q)
            ptx::tmem_ld32(t_s + 32 * q, sr + 32 * q);
          ptx::tmem_wait_ld();
          if (masked) {
#pragma unroll
            for (int q = 0; q < kTN; ++q)
              if (hidden(q)) sr[q] = __float_as_uint(-INFINITY);
          }
          // Four independent chains of 3-input max.
          float mc[4];
#pragma unroll
          for (int a = 0; a < 4; ++a)
            mc[a] = ptx::fmax3(__uint_as_float(sr[2 * a]),
                               __uint_as_float(sr[2 * a + 1]),
                               __uint_as_float(sr[8 + 2 * a]));
#pragma unroll
          for (int q = 16; q < kTN; q += 8) {
#pragma unroll
            for (int a = 0; a < 4; ++a)
              mc[a] = ptx::fmax3(mc[a], __uint_as_float(sr[q + 2 * a]),
                                 __uint_as_float(sr[q + 2 * a + 1]));
          }
          // Columns 9, 11, 13, 15 are not yet in any chain.
          const float h0 = ptx::fmax3(mc[0], mc[1],
                                      fmaxf(__uint_as_float(sr[9]),
                                            __uint_as_float(sr[11])));
          const float h1 = ptx::fmax3(mc[2], mc[3],
                                      fmaxf(__uint_as_float(sr[13]),
                                            __uint_as_float(sr[15])));
          const float raw = fmaxf(h0, h1);
          mx = (raw == -INFINITY) ? -INFINITY : raw * c;
        }

        // Lazy rescale: keep the stale maximum unless some row of the warp
        // grew by more than kRescaleTau (P stays <= 2^tau; exact either way,
        // since O and l share the same reference maximum).
        float m_new = m_run;
        if (__any_sync(0xffffffffu, mx > m_run + kRescaleTau))
          m_new = fmaxf(m_run, mx);
        const float alpha = (m_new == -INFINITY) ? 1.f : ptx::ex2(m_run - m_new);

        // Pass 2: P = 2^(s*c - m_new) and its row sum, packed to 16 bits into
        // TMEM over S_t (32 scores -> 16 columns, key 2e+1 | key 2e in column
        // e; FP8: E4M3, 32 scores -> 8 columns, key 4e in the low byte of
        // column e), 32 columns at a time: from the S row held in registers
        // since pass 1 (kHoldS), else re-read from TMEM with the next
        // chunk's load in flight while this one is computed (P chunk q only
        // overwrites S columns already consumed).  The row sum is taken from
        // the fp32 P.  P <= 2^tau = 256 stays inside E4M3's range (448).
        // Held scores (kHoldS) carry pass 1's -inf into the exp pass.
        // Re-read ones (packed) are masked again after the scaling, in a
        // second copy of the pass used only for masked tiles: left to the
        // compiler, the mask test inside the unrolled loop became a compare
        // and select on every score of every tile (about 2 ALU instructions
        // per score, 15 % of the step time).
        const float neg_m = (m_new == -INFINITY) ? 0.f : -m_new;
        float sm[4] = {0.f, 0.f, 0.f, 0.f};
        auto exp_pass = [&](auto mask_tag) {
          constexpr bool kMasked = decltype(mask_tag)::value;
          uint32_t buf[2][32];
          if constexpr (!kHoldS) {
            ptx::tmem_ld32(t_s, buf[0]);
            ptx::tmem_wait_ld();
          }
#pragma unroll
          for (int q = 0; q < kTN / 32; ++q) {
            const uint32_t* cur = sr + 32 * q;
            if constexpr (!kHoldS) {
              cur = buf[q & 1];
              if (q + 1 < kTN / 32)
                ptx::tmem_ld32(t_s + 32 * (q + 1), buf[(q + 1) & 1]);
            }
            if constexpr (kFp8) {
              uint32_t pk[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                float x[4];
                ptx::ffma2(x[0], x[1], __uint_as_float(cur[4 * e]),
                           __uint_as_float(cur[4 * e + 1]), c, neg_m);
                ptx::ffma2(x[2], x[3], __uint_as_float(cur[4 * e + 2]),
                           __uint_as_float(cur[4 * e + 3]), c, neg_m);
                if constexpr (kMasked) {
#pragma unroll
                  for (int a = 0; a < 4; ++a)
                    if (hidden(32 * q + 4 * e + a)) x[a] = -INFINITY;
                }
                float pe[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) pe[a] = ptx::ex2(x[a]);
                ptx::fadd2(sm[0], sm[1], pe[0], pe[1]);
                ptx::fadd2(sm[2], sm[3], pe[2], pe[3]);
                pk[e] = ptx::pack4_e4m3(pe[0], pe[1], pe[2], pe[3]);
              }
              ptx::tmem_st8(t_s + 8 * q, pk);
            } else {
              uint32_t pk[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                float x0, x1;
                ptx::ffma2(x0, x1, __uint_as_float(cur[2 * e]),
                           __uint_as_float(cur[2 * e + 1]), c, neg_m);
                if constexpr (kMasked) {
                  if (hidden(32 * q + 2 * e)) x0 = -INFINITY;
                  if (hidden(32 * q + 2 * e + 1)) x1 = -INFINITY;
                }
                const float p0 = ptx::ex2(x0);
                const float p1 = ptx::ex2(x1);
                if (e & 1)
                  ptx::fadd2(sm[2], sm[3], p0, p1);
                else
                  ptx::fadd2(sm[0], sm[1], p0, p1);
                pk[e] = ptx::pack2<kBF16>(p0, p1);
              }
              ptx::tmem_st16(t_s + 16 * q, pk);
            }
            if constexpr (!kHoldS) {
              if (q + 1 < kTN / 32) ptx::tmem_wait_ld();
            }
          }
        };
        if constexpr (kHoldS) {
          // Masked columns already hold -inf (pass 1).
          exp_pass(BoolTag<false>{});
        } else {
          if (masked)
            exp_pass(BoolTag<true>{});
          else
            exp_pass(BoolTag<false>{});
        }

        if ((kPack || kTriple) && j > 0) {
          // Packed / kTriple: S_j was issued before PV_{j-1}, so wait for
          // that PV's own commit before O may be touched (every step, to
          // keep the phases in step).
          ok = __all_sync(0xffffffffu,
                          wait_bounded(kTriple ? bar_pvdone + 8 * t : bar_o + 8,
                                       pv_waits & 1, abort_flag, p, 3));
          if (!ok) break;
          ++pv_waits;
          ptx::tc_fence_after();
        }
        if (j > 0 && __any_sync(0xffffffffu, m_new != m_run)) {
          // Correction: O_t *= alpha.  The previous PV into O_t is complete:
          // it was issued before this tile's S_t, whose commit we waited on
          // (packed, kTriple: its own commit, waited on just above).
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t o[32];
            ptx::tmem_ld32(t_o + 32 * q, o);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e)
              o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            ptx::tmem_st32(t_o + 32 * q, o);
          }
        }
        l_run *= alpha;
        ptx::tmem_wait_st();
        l_run += (sm[0] + sm[1]) + (sm[2] + sm[3]);
        m_run = m_new;
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_p + 8 * (kTriple ? t : sb));
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      // O / l in 16 bits straight from registers to global memory: each
      // thread owns one 2*D-byte row (rows >= Sq are not stored).  The next
      // unit's MMAs into S_t may already run; the next PV into O_t waits for
      // this warpgroup's next P, so the reads below come first.
      ok = __all_sync(0xffffffffu, wait_bounded(bar_o + 8 * t, o_waits & 1,
                                                abort_flag, p, 4));
      if (kStageO || (kSplit && !(kPack && p.cluster_merge))) {
        // The epilogue below meets at named barriers, which do not time out.
        // After an abort the tile's warps may have left the step loop at
        // different waits (a phase that completed for one had already been
        // given up by another), so they first meet on a bounded barrier and
        // go on only if all four came and all saw O complete; a warp that
        // never comes lets the others' wait run out.  With the staged store
        // this barrier is also the first box's "buffer free" signal: the
        // storing thread arrives once TMA has read the previous box out.
        // Split-KV tiles written to the workspace meet here too (the tile's
        // partial rows then go out together); no named barrier follows
        // them, but without the meeting the packed split variants compiled
        // with register spills and the decode step took 3 % longer
        // (same-box A/B).
        volatile int* in_ok = reinterpret_cast<volatile int*>(
            smem + L::kMiscOff + 16 + 16 * t);
        if (lane == 0) in_ok[warp % 4] = ok ? 1 : 0;
        if (kStageO && r == 0) ptx::bulk_wait_group_read_all();
        ptx::mbar_arrive(bar_epi + 8 * t);
        ok = __all_sync(0xffffffffu, wait_bounded(bar_epi + 8 * t, o_waits & 1,
                                                  abort_flag, p, 4));
        ok = ok && in_ok[0] && in_ok[1] && in_ok[2] && in_ok[3];
      }
      if (!ok) break;
      ++o_waits;
      ptx::tc_fence_after();

      if (!live) {
        // Padding rows only: nothing to store.
      } else if constexpr (kStageO) {
        // O / l in 16 bits through this tile's staging box: each thread
        // writes its row's 16-byte chunks at the 128-byte-swizzled places
        // (chunk c of row r at c ^ (r % 8): a warp's 32 rows cover every
        // bank once per 8 rows), then one thread stores the box with TMA
        // (rows >= Sq fall outside the tensor and are not written).  Per
        // thread row stores touched 32 lines per warp instruction and took
        // 4-5x longer.  D = 128 takes two boxes (columns 0-63, 64-127): the
        // second waits until TMA has read the first out of the buffer.
        const float inv_l =
            kFp8 ? ptx::rcp(l_run) * p.o_scale : ptx::rcp(l_run);
        const uint32_t stage = s_base + L::kStageOff + t * L::kStageTileBytes;
        const uint32_t row_base = stage + r * 128;
        const uint32_t sw = r % 8;
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          uint32_t o[64];
          ptx::tmem_ld32(t_o + 64 * h, o);
          ptx::tmem_ld32(t_o + 64 * h + 32, o + 32);
          ptx::tmem_wait_ld();
          // The buffer is free once TMA has read the previous box out of it
          // (for the first box: the entry barrier above).
          if (h > 0) {
            if (r == 0) ptx::bulk_wait_group_read_all();
            ptx::named_barrier_sync(1 + t, kTM);
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t wv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              wv[e] = ptx::pack2<kBF16>(
                  __uint_as_float(o[8 * c + 2 * e]) * inv_l,
                  __uint_as_float(o[8 * c + 2 * e + 1]) * inv_l);
            ptx::st_shared_v4(row_base + ((c ^ sw) << 4), wv[0], wv[1], wv[2],
                              wv[3]);
          }
          ptx::fence_proxy_async_smem();
          ptx::named_barrier_sync(1 + t, kTM);
          if (r == 0) {
            ptx::tma_store_3d(&tm_o, stage, 64 * h, m0, q_plane);
            ptx::bulk_commit_group();
          }
        }
        if (p.lse != nullptr && row_ok) {
          const long long row = static_cast<long long>(q_plane) * p.Sq + q_row;
          p.lse[row] = (m_run + ptx::lg2(l_run)) * kLn2;
        }
      } else if (p.o_part == nullptr) {
        const float inv_l =
            kFp8 ? ptx::rcp(l_run) * p.o_scale : ptx::rcp(l_run);
        const long long row = static_cast<long long>(q_plane) * p.Sq + q_row;
        uint4* orow =
            reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + row * D);
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          ptx::tmem_ld32(t_o + 32 * q, o);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t wv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              wv[e] = ptx::pack2<kBF16>(
                  __uint_as_float(o[8 * v + 2 * e]) * inv_l,
                  __uint_as_float(o[8 * v + 2 * e + 1]) * inv_l);
            if (row_ok) orow[4 * q + v] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
        }
        if (p.lse != nullptr && row_ok)
          p.lse[row] = (m_run + ptx::lg2(l_run)) * kLn2;
      } else {
        // Split-KV partial: O over this key range normalised by its own l,
        // in fp32, and the range's natural-log LSE; a row that sees no key
        // of the range gets O = 0 and LSE = -inf.
        const bool empty = !(l_run > 0.f);
        const float inv_l =
            empty ? 0.f : (kFp8 ? ptx::rcp(l_run) * p.o_scale : ptx::rcp(l_run));
        const float lse_row =
            empty ? -INFINITY : (m_run + ptx::lg2(l_run)) * kLn2;
        if (kPack && p.cluster_merge) {
          // Into this CTA's shared memory (the K/V ring, idle now: every
          // MMA of the unit is done), row r at r * D * 4 bytes; rank 0 of
          // the cluster reads it after the cluster barrier below.
          const uint32_t part = s_base + L::kRingOff;
          // 64 columns per TMEM wait.
#pragma unroll
          for (int q = 0; q < D / 64; ++q) {
            uint32_t o[64];
            ptx::tmem_ld32(t_o + 64 * q, o);
            ptx::tmem_ld32(t_o + 64 * q + 32, o + 32);
            ptx::tmem_wait_ld();
            if (row_ok) {
#pragma unroll
              for (int v = 0; v < 16; ++v)
                ptx::st_shared_v4(
                    part + (r * D + 64 * q + 4 * v) * 4,
                    __float_as_uint(__uint_as_float(o[4 * v]) * inv_l),
                    __float_as_uint(__uint_as_float(o[4 * v + 1]) * inv_l),
                    __float_as_uint(__uint_as_float(o[4 * v + 2]) * inv_l),
                    __float_as_uint(__uint_as_float(o[4 * v + 3]) * inv_l));
            }
          }
          if (row_ok) ptx::st_shared_f32(part + kTM * D * 4 + 4 * r, lse_row);
        } else if constexpr (!kPack) {
          // Through this warp's quarter of the tile's staging box: each
          // thread writes a 32-column slice of its row (128 bytes, chunk c
          // of row i at c ^ (i % 8), so 8 threads of a phase cover every
          // bank), then the warp stores 4 rows x 128 bytes per instruction
          // -- whole lines, where per-thread row stores touch 32 lines per
          // instruction.  Only this warp uses its quarter.
          const uint32_t wbuf = s_base + L::kStageOff +
                                t * L::kStageTileBytes + (warp % 4) * 4096;
          const long long plane_row0 =
              (static_cast<long long>(w.split) * p.B * p.Hq + q_plane) *
              p.Sq;
          const int wrow0 = m0 + 32 * (warp % 4);  // the warp's first row
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t o[32];
            ptx::tmem_ld32(t_o + 32 * q, o);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 8; ++c)
              ptx::st_shared_v4(
                  wbuf + lane * 128 + ((c ^ (lane % 8)) << 4),
                  __float_as_uint(__uint_as_float(o[4 * c]) * inv_l),
                  __float_as_uint(__uint_as_float(o[4 * c + 1]) * inv_l),
                  __float_as_uint(__uint_as_float(o[4 * c + 2]) * inv_l),
                  __float_as_uint(__uint_as_float(o[4 * c + 3]) * inv_l));
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int rr = 4 * i + lane / 8, c = lane % 8;
              const uint4 v =
                  ptx::ld_shared_v4(wbuf + rr * 128 + ((c ^ (rr % 8)) << 4));
              if (wrow0 + rr < p.Sq)
                *reinterpret_cast<uint4*>(
                    p.o_part + (plane_row0 + wrow0 + rr) * D + 32 * q +
                    4 * c) = v;
            }
            __syncwarp();
          }
          if (row_ok) p.lse_part[plane_row0 + q_row] = lse_row;
        } else {
          const long long prow =
              (static_cast<long long>(w.split) * p.B * p.Hq + q_plane) *
                  p.Sq +
              q_row;
          float4* orow = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t o[32];
            ptx::tmem_ld32(t_o + 32 * q, o);
            ptx::tmem_wait_ld();
            if (row_ok) {
#pragma unroll
              for (int v = 0; v < 8; ++v)
                orow[8 * q + v] =
                    make_float4(__uint_as_float(o[4 * v]) * inv_l,
                                __uint_as_float(o[4 * v + 1]) * inv_l,
                                __uint_as_float(o[4 * v + 2]) * inv_l,
                                __uint_as_float(o[4 * v + 3]) * inv_l);
            }
          }
          if (row_ok) p.lse_part[prow] = lse_row;
        }
      }
      ptx::tc_fence_before();
    }
    // Output boxes still being stored must be read out of shared memory
    // (and written) before the CTA exits.
    if constexpr (kStageO) {
      if (r == 0) ptx::bulk_wait_group_all();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (kPack && kSplit) {
    if (p.cluster_merge) {
      // Every thread of every CTA of the cluster takes part in both
      // barriers, on every path (an aborted CTA too), so neither can wait
      // for a thread that will not come.  After the first, rank 0's softmax
      // warps merge the key ranges (unless some CTA of the cluster gave up
      // a wait: then the status word already reports it); the second keeps
      // every CTA's shared memory alive until rank 0 has read it.
      ptx::cluster_arrive_release();
      ptx::cluster_wait_acquire();
      if (ptx::cluster_ctarank() == 0 && warp >= kSoftmaxWarp0 &&
          warp < kSoftmaxWarp0 + 4) {
        const uint32_t abort_addr = s_base + L::kMiscOff + 4;
        // Every CTA's abort flag in one round trip.
        int aborted = 0;
#pragma unroll
        for (int c = 0; c < cfg::kMaxClusterRanges; ++c)
          if (c < p.num_splits)
            aborted |= ptx::ld_shared_cluster_s32(ptx::mapa_shared(abort_addr, c));
        const bool all_ok = aborted == 0;
        if (all_ok) {
          const Unit w = decode_unit<kPack, kWindow>(p, u_first);
          merge_tile_cluster<D, kBF16, kWindow>(
              p, w.plane[0], s_base + L::kRingOff, threadIdx.x % 128);
        }
      }
      ptx::cluster_arrive_release();
      ptx::cluster_wait_acquire();
    }
  }
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace attn
