// Split-KV merge kernel: merges the key ranges' partial results of a
// split-KV forward launch (attn_fwd_sm103_kernel with o_part set) into O
// and the LSE.  Launched by attn_merge.cu.
#pragma once

#include "attn_fwd_kernel.cuh"

namespace attn {

// Split-KV merge of query rows.  Key range c of a row contributes its
// normalised partial output O_c and log-sum-exp lse_c; with
// M = max_c lse_c and w_c = e^(lse_c - M),  O = sum_c w_c O_c / sum_c w_c
// and LSE = M + ln(sum_c w_c) -- the online-softmax rescale applied once
// more, across ranges, here in its online form (a running maximum, the sums
// rescaled when it grows).  Ranges past a row's causal horizon or before
// its window hold nothing for it and are not read.  A thread takes 4
// columns (group cg) of kRowBatch rows (flat row index row[b] into
// [B*Hq, Sq], position q_row[b] in the chunk; q_row < 0: no row) and reads
// kRangeBatch ranges of them per round: the merge is bound by L2 latency,
// so every load of a round is issued before the first is used.
template <int D, bool kBF16, bool kWindow, int kRowBatch, int kRangeBatch>
__device__ __forceinline__ void merge_rows(const FwdParams& p,
                                           const long long (&row)[kRowBatch],
                                           const int (&q_row)[kRowBatch],
                                           int cg) {
  constexpr float kLog2e = 1.4426950408889634f;
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.Sq;
  const int split_keys = p.split_tiles * cfg::kTN;
  int c0[kRowBatch], ns[kRowBatch];
  int cmin = p.num_splits, cmax = 0;
#pragma unroll
  for (int b = 0; b < kRowBatch; ++b) {
    c0[b] = 0;
    ns[b] = 0;  // no range: not a row
    if (q_row[b] >= 0) {
      const int row_pos = p.input_pos + q_row[b];
      const int vis_end = p.causal ? min(p.Skv, row_pos + 1) : p.Skv;
      ns[b] = min(p.num_splits, (vis_end + split_keys - 1) / split_keys);
      c0[b] = kWindow ? max(0, row_pos - p.window + 1) / split_keys : 0;
      cmin = min(cmin, c0[b]);
      cmax = max(cmax, ns[b]);
    }
  }
  float mx[kRowBatch], wsum[kRowBatch];
  float4 acc[kRowBatch];
#pragma unroll
  for (int b = 0; b < kRowBatch; ++b) {
    mx[b] = -INFINITY;
    wsum[b] = 0.f;
    acc[b] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int cb = cmin; cb < cmax; cb += kRangeBatch) {
    float lc[kRangeBatch][kRowBatch];
    float4 xc[kRangeBatch][kRowBatch];
#pragma unroll
    for (int k = 0; k < kRangeBatch; ++k) {
      const int c = cb + k;
#pragma unroll
      for (int b = 0; b < kRowBatch; ++b) {
        lc[k][b] = -INFINITY;
        xc[k][b] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c >= c0[b] && c < ns[b]) {
          lc[k][b] = __ldcg(p.lse_part + c * rows + row[b]);
          xc[k][b] = __ldcg(reinterpret_cast<const float4*>(
                                p.o_part + (c * rows + row[b]) * D) +
                            cg);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kRangeBatch; ++k) {
#pragma unroll
      for (int b = 0; b < kRowBatch; ++b) {
        const float mn = fmaxf(mx[b], lc[k][b]);
        if (mn == -INFINITY) continue;  // nothing seen yet
        const float a = ptx::ex2((mx[b] - mn) * kLog2e);  // 0 while mx = -inf
        const float wc = ptx::ex2((lc[k][b] - mn) * kLog2e);
        wsum[b] = wsum[b] * a + wc;
        acc[b].x = acc[b].x * a + wc * xc[k][b].x;
        acc[b].y = acc[b].y * a + wc * xc[k][b].y;
        acc[b].z = acc[b].z * a + wc * xc[k][b].z;
        acc[b].w = acc[b].w * a + wc * xc[k][b].w;
        mx[b] = mn;
      }
    }
  }
#pragma unroll
  for (int b = 0; b < kRowBatch; ++b) {
    if (ns[b] == 0) continue;
    const float inv = ptx::rcp(wsum[b]);
    uint2 out;
    out.x = ptx::pack2<kBF16>(acc[b].x * inv, acc[b].y * inv);
    out.y = ptx::pack2<kBF16>(acc[b].z * inv, acc[b].w * inv);
    reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.o) + row[b] * D)[cg] =
        out;
    if (cg == 0 && p.lse != nullptr)
      p.lse[row[b]] = mx[b] + ptx::lg2(wsum[b]) * cfg::kLn2;
  }
}

// Split-KV merge as a launch of its own, after the forward kernel on the
// same stream (programmatic dependent launch: its CTAs wait in
// griddepcontrol.wait until the forward grid has completed).  The rows of
// all (batch, head) planes in one flat range, spread over the whole GPU:
// kMergeThreads threads take kRowBatch rows of kMergeThreads / (D/4) at a
// time per CTA, grid-stride, reading 8 / kRowBatch ranges of them per
// round.  The launch takes 2 rows per thread when that still gives every
// SM two CTAs, else 1 (launches of few rows over many ranges: more CTAs and
// fewer dependent rounds).  (Merging inside the forward kernel, by the unit
// whose arrival on a per-tile counter completed the set, put that CTA's
// latency-bound reads of every range -- about 4.6 us per range of a
// two-tile unit -- on each wave's critical path.)
constexpr int kMergeThreads = 256;
template <int D, int kRowBatch>
__host__ __device__ constexpr int merge_rows_per_cta() {
  return kMergeThreads / (D / 4) * kRowBatch;
}

template <int D, bool kBF16, bool kWindow, int kRowBatch>
__global__ void __launch_bounds__(kMergeThreads)
    attn_merge_kernel(const __grid_constant__ FwdParams p) {
  ptx::griddep_wait();
  constexpr int kGroups = D / 4;
  constexpr int kRowsPerPass = kMergeThreads / kGroups;
  constexpr int kRows = merge_rows_per_cta<D, kRowBatch>();
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.Sq;
  const int tid = threadIdx.x;
  for (long long r0 = static_cast<long long>(blockIdx.x) * kRows +
                      tid / kGroups;
       r0 < rows; r0 += static_cast<long long>(gridDim.x) * kRows) {
    long long row[kRowBatch];
    int q_row[kRowBatch];
#pragma unroll
    for (int b = 0; b < kRowBatch; ++b) {
      row[b] = r0 + b * kRowsPerPass;
      q_row[b] = row[b] < rows ? static_cast<int>(row[b] % p.Sq) : -1;
      if (q_row[b] < 0) row[b] = 0;
    }
    merge_rows<D, kBF16, kWindow, kRowBatch, 8 / kRowBatch>(p, row, q_row,
                                                             tid % kGroups);
  }
}

}  // namespace attn
