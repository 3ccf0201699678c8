// prefill_split.cuh -- key-range split of a prefill's last round of work units,
// shared by the CTA-pair and the single-CTA causal prefill kernels.
//
// What it computes: the design record's split-and-reduce ("ADR-0060: AHBM GQA
// Fused Attention Kernel (Llama3-70B)", section 2.2's contiguous key ranges and
// section 4's combination of partial softmax states) applied to prefill.  Work
// units (128 query rows of a few heads) are dealt in rounds over the resident
// workers, longest first; when the last round is partial, its units are each
// cut into pieces of contiguous key tiles so the round fills the workers.  A
// piece writes its partial state per query row -- O before division by l
// (fp32), the reference max m (log2 units) and l -- and the merge kernel
// combines the pieces of a unit:
//   M = max_i m_i,  L = sum_i 2^(m_i - M) l_i,
//   O = sum_i 2^(m_i - M) O_i / L,  lse = M ln 2 + ln L.
#pragma once

#include <math.h>
#include <stddef.h>
#include <stdint.h>

#include "device_common.cuh"
#include "kernels.h"

namespace gqa {
namespace prefill_split {

constexpr int kRows = 128;          // query rows per unit slot
constexpr int kD = 128;             // head dimension
constexpr int kMaxPieces = 32;      // pieces per unit (one lane each in the merge)
constexpr int kMinPieceTiles = 8;   // key tiles per piece at least
constexpr int kMergeThreads = 256;  // one warp per (split unit, head, row)

// Bytes of one piece's partial state for a unit of `heads` slots of 128 rows.
__host__ __device__ constexpr size_t piece_bytes(int heads) {
  return (size_t)heads * kRows * (kD + 2) * sizeof(float);
}

// Key tile where piece i of s of an n-tile range starts.  A unit's key range
// ends at most two tiles past the tile of its first query row (one more for a
// second slot on the query tile below), and every piece has at least
// kMinPieceTiles tiles, so every piece after the first starts at or before the
// tile of each slot's first row: its first tile has a visible key in every row.
__host__ __device__ __forceinline__ int piece_start(int i, int s, int n) {
  return (int)((long long)i * n / s);
}

// Paged K/V ([num_pages, H_kv, page_size, d], page_size a multiple of 128): keys
// [i*page_size, (i+1)*page_size) of sequence b are in page block_table[b *
// max_pages + i].  Empty for a dense kernel, whose parameters (and register
// allocation) it leaves untouched.
template <bool kPaged>
struct PageArgs {
  const int32_t *block_table;
  int page_size, max_pages, num_pages;
};
template <>
struct PageArgs<false> {};

using Plan = PrefillPlan;
constexpr int kMaxPieceRounds = 4;     // pieces never exceed this many rounds of workers
constexpr int kPieceOverheadTiles = 2;  // a piece's start and partial store, in key tiles

// `units` units on `workers` resident workers; `n_kv_min` key tiles of the
// shortest unit; a workspace of `ws_bytes` (none if `ws` is null).  The
// r = units mod workers units of the last round (all of them when there are
// fewer units than workers) may each be cut into s pieces of contiguous key
// tiles, dealt after the whole units like any other item, so the pieces of the
// last round can take several rounds of their own.  The s chosen minimises the
// modelled span of those rounds, ceil(r s / workers) * (n_kv_min / s +
// kPieceOverheadTiles + 1), against n_kv_min for the units run whole; at most
// kMaxPieces pieces per unit, at least kMinPieceTiles tiles each, at most
// kMaxPieceRounds rounds of pieces, and only pieces whose partials fit the
// workspace.
inline Plan make_plan(long long units, int workers, int n_kv_min, int heads, const void *ws,
                      size_t ws_bytes) {
  Plan pl;
  if (units <= 0 || units > 0x7fffffffLL || workers <= 0) return pl;
  const int U = (int)units;
  pl.units = U;
  pl.n_full = U;
  const int r = U % workers;
  if (ws != nullptr && r > 0) {
    int s_max = n_kv_min / kMinPieceTiles;
    if (s_max > kMaxPieces) s_max = kMaxPieces;
    double best = (double)n_kv_min;  // the last round's units run whole
    int best_s = 1;
    for (int sp = 2; sp <= s_max; ++sp) {
      const long long pieces = (long long)r * sp;
      const long long rounds = (pieces + workers - 1) / workers;
      if (rounds > kMaxPieceRounds || (size_t)pieces * piece_bytes(heads) > ws_bytes) break;
      const double span =
          (double)rounds * ((double)n_kv_min / sp + kPieceOverheadTiles + 1);
      if (span < best) {
        best = span;
        best_s = sp;
      }
    }
    if (best_s >= 2) {
      pl.n_full = U - r;
      pl.split_s = best_s;
    }
  }
  pl.pieces = (U - pl.n_full) * pl.split_s;
  pl.n_items = pl.n_full + pl.pieces;
  pl.workers = pl.n_items < workers ? pl.n_items : workers;
  return pl;
}

// Workspace that lets any partial round split as far as make_plan may cut it:
// at most kMaxPieceRounds rounds of workers, nor more than kMaxPieces pieces
// per unit.
inline size_t workspace_bound(long long units, int workers, int heads) {
  const long long most = units * kMaxPieces;
  const long long cap = (long long)workers * kMaxPieceRounds;
  const long long pieces = most < cap ? most : cap;
  return pieces > 0 ? (size_t)pieces * piece_bytes(heads) : 0;
}

// Where the partial of (piece, head slot hl, row) lives: ws_o row
// ((piece * heads + hl) * 128 + row) of 128 floats; ws_ml the same index of
// float2 (m, l).
__device__ __forceinline__ size_t partial_row(int piece, int heads, int hl, int row) {
  return ((size_t)piece * heads + hl) * kRows + row;
}

// The merge.  P provides n_items, n_full, split_s, ws_o, ws_ml, o, lse, and
// piece_out_row(p, item, hl, row, &orow): the output row (b, head, query) of
// slot hl's row `row` of work item `item`, false if that row is not stored.
// Launched as a programmatic dependent of the prefill kernel: the partials are
// read through L2 after the grid-dependency wait.
template <int kHeads, class P>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const P p) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5);
  const int row = gw % kRows;
  const int hl = (gw / kRows) % kHeads;
  const int su = gw / (kHeads * kRows);  // split unit
  const int s = p.split_s;
  if (su >= (p.n_items - p.n_full) / s) return;
  size_t orow;
  if (!piece_out_row(p, p.n_full + su * s, hl, row, &orow)) return;
  if (!store_ok(orow, (size_t)p.B * p.H_q * p.T_q, p.wait.status)) return;
  float m = -INFINITY, l = 0.f;
  if (lane < s) {
    const float2 ml =
        __ldcg(reinterpret_cast<const float2 *>(p.ws_ml) + partial_row(su * s + lane, kHeads, hl, row));
    m = ml.x;
    l = ml.y;
  }
  float M = m;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float wgt = m > -INFINITY ? fast_exp2(m - M) : 0.f;
  float L = wgt * l;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int i = 0; i < s; ++i) {
    const float wi = __shfl_sync(0xffffffffu, wgt, i);
    const float4 x = __ldcg(reinterpret_cast<const float4 *>(
                                p.ws_o + partial_row(su * s + i, kHeads, hl, row) * kD) +
                            lane);
    acc.x = fmaf(wi, x.x, acc.x);
    acc.y = fmaf(wi, x.y, acc.y);
    acc.z = fmaf(wi, x.z, acc.z);
    acc.w = fmaf(wi, x.w, acc.w);
  }
  const float inv_l = L > 0.f ? 1.f / L : 0.f;
  uint2 pk;
  pk.x = pack_bf16x2(acc.x * inv_l, acc.y * inv_l);
  pk.y = pack_bf16x2(acc.z * inv_l, acc.w * inv_l);
  reinterpret_cast<uint2 *>(p.o + orow * kD)[lane] = pk;
  if (lane == 0) p.lse[orow] = L > 0.f ? M * 0.69314718055994531f + logf(L) : -INFINITY;
}

// Launches the merge of plan pl's split units (nothing if there are none).
template <int kHeads, class P>
cudaError_t launch_merge(const P &p, const Plan &pl, cudaStream_t stream) {
  if (pl.pieces == 0) return cudaSuccess;
  const long long warps = (long long)(pl.pieces / pl.split_s) * kHeads * kRows;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((warps + kMergeThreads / 32 - 1) / (kMergeThreads / 32)), 1, 1);
  cfg.blockDim = dim3(kMergeThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_kernel<kHeads, P>, p);
}

}  // namespace prefill_split
}  // namespace gqa
