// decode_split.cu -- split-KV GQA decode for sm_103a.
//
// What it computes (design record "ADR-0060: AHBM GQA Fused Attention Kernel
// (Llama3-70B)"): for one sequence b and one KV head, the G = H_q / H_kv query
// heads that share that KV head are stacked into one matrix product (the
// record's "M-fold", TL;DR "Kernel 1" and section 5.2), so each K/V tile is read
// from HBM once for all G heads.  The key range of the head is cut into
// contiguous chunks (section 2.1, contiguous-block placement); each CTA runs the
// per-tile online softmax of section 3 over its chunk and writes a partial
// (O_s / l_s, lse_s).  A second kernel merges the partials with the
// log-sum-exp merge of section 4.
//
// GB300 mapping
//   * grid (num_splits, H_kv, B); 5 warps: warp 4 issues TMA loads of 64-key
//     K/V tiles (128B-swizzled, 4D tensor maps so tiles never cross a head)
//     into a 3-stage shared-memory ring; warps 0..3 consume every tile.
//   * The fold puts the G (<= 8) heads in the N = 8 dimension of
//     mma.sync m16n8k16 (bf16 in, fp32 accumulate): S^T[16 keys x 8 heads] =
//     K[16 x 128] Q^T, so no MMA lane is wasted on padding; P^T is moved into
//     the B-operand layout with movmatrix and O^T[128 x 8] += V^T P^T reads V
//     with ldmatrix.trans.
//   * Warp w owns keys [16w, 16w+16) of every tile and keeps its own running
//     (m, l, O); the four warp states are merged once per CTA, so no
//     cross-warp synchronisation sits in the tile loop.
//   * Decode moves 8 flop per byte of K/V, far below the tensor-core ridge;
//     the kernel is HBM bound and everything else exists to keep enough bytes
//     in flight (two CTAs per SM x 3 stages x 32 KiB).
#include <cudaTypedefs.h>
#include <math.h>

#include "device_common.cuh"
#include "kernels.h"

namespace gqa {
namespace decode {

constexpr int kD = 128;
constexpr int kTileKeys = kDecodeTileKeys;          // 64
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // 160: one column group
constexpr int kMaxColGroups = 2;                     // multi-token decode: G * T_q <= 32
constexpr int kThreadsWide = (kConsumerWarps * kMaxColGroups + 1) * 32;  // 288
constexpr int kMaxCols = 16 * kMaxColGroups;         // 32 (head, token) columns
constexpr int kHalfBytes = kTileKeys * 128;          // 64 keys x 64 d x 2 B = 8 KiB
constexpr int kStageBytes = 4 * kHalfBytes;          // K lo/hi + V lo/hi = 32 KiB
// Ring depth: 3 stages (96 KiB) per CTA, two CTAs per SM for plans that run
// several waves (a finishing CTA's epilogue overlaps its neighbour's
// streaming).  Single-wave plans run one CTA per SM with kOneWaveStages (4)
// stages; deeper rings measured slower on GB300 (more bytes in flight only
// queue longer in the memory system).
#ifndef GQA_DECODE_ONE_WAVE_STAGES
#define GQA_DECODE_ONE_WAVE_STAGES 4
#endif
constexpr int kOneWaveStages = GQA_DECODE_ONE_WAVE_STAGES;
// K/V tiles of its chunk a CTA prefetches into L2 before the grid-dependency wait
#ifndef GQA_DECODE_L2_PREFETCH_TILES
#define GQA_DECODE_L2_PREFETCH_TILES 3
#endif
constexpr int kRedStride = kD + 4;  // padded row of the per-warp O reduction buffer
constexpr int kMaxFusedSplits = kDecodeMaxFusedSplits;  // largest cluster of the fused variant
// Cluster-merged variant: what a CTA receives from the cluster, one slot per
// (sender, column it finalises): at most 16 slots for at most 8 columns (a
// cluster of cs CTAs gives each ceil(8 / cs) columns, cs * ceil(8 / cs) <= 16).
constexpr int kRecvSlots = 16;
constexpr int kRecvBytes = 16 + kRecvSlots * (kD + 1) * 4;  // barrier (padded), O rows, lse
template <int kStages, bool kFused = false>
constexpr int smem_bytes() {  // ring + barriers (+ receive area) + alignment slack
  return kStages * kStageBytes + 2 * kStages * 8 + (kFused ? kRecvBytes : 0) + 1024;
}

struct Params {
  const uint16_t *q;
  const int32_t *seqlens;
  float *o_part;
  float *lse_part;
  uint16_t *o;  // fused variant: final outputs
  float *lse;
  const int32_t *block_table;  // paged variant: [B, max_pages]
  int page_size, max_pages, num_pages;
  int B, H_q, H_kv, G, S_max, num_splits, chunk;
  int num_sms;  // SMs the host plan counted on (the device-side chunk rule)
  int T_q, n_cols, cgroups;  // new tokens per sequence, G * T_q, column groups of 4 warps
  float scale_log2;  // scale * log2(e)
  int l2_prefetch_tiles;  // tiles of its chunk a CTA pulls into L2 before the dependency wait
  int direct_out;  // one split per (sequence, KV head): the partial is the output (o, lse)
  WaitCtl wait;
};

__device__ __forceinline__ uint32_t mask_pair(uint32_t x, bool lo_ok, bool hi_ok) {
  return (lo_ok ? 0x0000FFFFu : 0u) & x | ((hi_ok ? 0xFFFF0000u : 0u) & x);
}

// Byte offset of 16-byte chunk `chunk` (0..15 across d) of key row `r` inside one
// K or V tile as TMA writes it: two 64-column halves, each [64 rows x 128 B]
// with the 128B swizzle (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t tile_offset(int r, int chunk) {
  const int half = chunk >> 3, c = chunk & 7;
  return half * kHalfBytes + r * 128 + ((c ^ (r & 7)) << 4);
}

// kFused = false: each CTA writes its split partial to the workspace and the
// merge kernel combines them.  kFused = true: the num_splits CTAs of one
// (sequence, KV head) form a thread-block cluster; each sends the partial of
// column n to the shared memory of CTA n % num_splits (st.async, the bytes
// counted on that CTA's barrier), which merges the columns it received, so one
// launch produces o and lse and no workspace is touched.
// kPaged = true: K and V live in pages [num_pages, H_kv, page_size, d] and
// block_table[b][i] names the page that holds keys [i*page_size, (i+1)*page_size)
// of sequence b (page_size a multiple of the 64-key tile, so no tile straddles
// two pages).  An out-of-range page id addresses outside the tensor map, which
// TMA fills with zeros.
// kNT: 8-column MMA n-tiles per consumer warp.  The query rows of one KV head
// are (head g, new token t) pairs, column n = g * T_q + t, n < G * T_q; with
// kNT = 1 one group of four warps covers 8 columns (decode, T_q = 1, G <= 8);
// with kNT = 2 each group covers 16 and p.cgroups groups of four warps split the
// columns (multi-token decode, G * T_q <= 32).  New token t sits at position
// seqlen - T_q + t and sees keys up to it.
template <int kStages, int kMinBlocks, bool kFused, bool kPaged, int kNT>
__global__ void __launch_bounds__(kNT == 1 ? kThreads : kThreadsWide, kMinBlocks)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
  uint64_t *empty_bar = full_bar + kStages;
  // cluster-merged variant: barrier counting the bytes the cluster sends this CTA,
  // then the received partials (slot = sender * per_rank + column / cluster size)
  uint64_t *recv_bar = empty_bar + kStages;
  float *recv_o = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(recv_bar) + 16);
  float *recv_lse = recv_o + kRecvSlots * kD;

  // grid (H_kv, B, splits): the first splits of every (sequence, KV head) come
  // first in launch order, so a multi-wave grid puts the CTAs that hold keys on
  // distinct SMs before any empty one; the cluster-merged grid is (splits, H_kv,
  // B), a cluster along x
  const int split = kFused ? blockIdx.x : blockIdx.z;
  const int kv = kFused ? blockIdx.y : blockIdx.x;
  const int b = kFused ? blockIdx.z : blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_consumers = kConsumerWarps * p.cgroups;  // warps before the producer
  __shared__ int failed;
  // A cluster-merged grid that leaves at least half of the SMs idle lets the next
  // grid start its prologue there right away (tiny decode 5.13 -> 4.75 us per
  // call).  A larger one triggers at its end: dependents placed early double up
  // on the SMs that are free first (batch of 4 at 4K keys: 15.08 -> 15.42 us).
  if (kFused && 2u * gridDim.x * gridDim.y * gridDim.z <= (unsigned)p.num_sms)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Cluster-merged variant with cs > 1 CTAs: CTA r finalises columns r, r + cs, ...
  // (per_rank of them at most), each sent by every CTA of the cluster.
  const int cs = p.num_splits;
  const int per_rank = (p.n_cols + cs - 1) / cs;
  const int n_mine = split < p.n_cols ? (p.n_cols - split + cs - 1) / cs : 0;
  const bool cluster_merge = kFused && cs > 1 && cs * per_rank <= kRecvSlots;
  // prologue that reads no input: overlaps the previous kernel when this grid
  // was launched as its programmatic dependent
  if (threadIdx.x == 0) {
    failed = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), n_consumers);
    }
    if (cluster_merge) {
      mbar_init(smem_u32(recv_bar), 1);
      mbar_arrive_expect_tx(smem_u32(recv_bar), (uint32_t)(n_mine * cs * (kD + 1) * 4));
    }
    fence_mbar_init();
  }
  // every CTA's receive barrier exists before any CTA of the cluster sends to it
  if (cluster_merge) cluster_sync();
  int hint_page = 0;  // paged: the page of this split's first key, as the hints give it
  if (warp == n_consumers && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    // One-wave grid: pull the first tiles of this split's key range into L2
    // while the preceding grid finishes.  Only a grid that is resident all at
    // once can overlap the preceding grid; in a larger one, splits past their
    // sequence's end would only prefetch padding.  The sequence length and a
    // paged cache's table are read here ahead of the wait as hints only
    // (relaxed loads; the preceding grid may still write them): the length
    // gives this split's device-side chunk and where the sequence ends, and a
    // stale value costs at most a wasted L2 fill.  Everything that matters is
    // read again after the wait.
    int tiles = 0, key_first = 0;
    if (p.l2_prefetch_tiles > 0) {
      const int len = min(max(ld_relaxed_s32(p.seqlens + b), 0), p.S_max);
      const int c = device_chunk(len, p.B, p.S_max, p.chunk, p.num_splits, p.H_kv, p.num_sms,
                                 kTileKeys);
      key_first = split * c;
      const int n = min(key_first + c, len) - key_first;
      tiles = n > 0 ? min(p.l2_prefetch_tiles, (n + kTileKeys - 1) / kTileKeys) : 0;
    } else {
      key_first = split * p.chunk;  // the host's chunk: exact for full-length sequences
    }
    if constexpr (kPaged) hint_page = key_first / p.page_size;
    int last_page = -1, page_id = -1;  // paged: one table read per page, not per tile
    for (int i = 0; i < tiles; ++i) {
      const int key0 = key_first + i * kTileKeys;
      int c2 = key0, c3 = b * p.H_kv + kv;
      if (kPaged) {
        const int page = key0 / p.page_size;
        if (page >= p.max_pages) break;
        if (page != last_page) {
          page_id = ld_relaxed_s32(p.block_table + (size_t)b * p.max_pages + page);
          last_page = page;
        }
        if (page_id < 0 || page_id >= p.num_pages) continue;
        c2 = key0 - page * p.page_size;
        c3 = page_id * p.H_kv + kv;
      }
      for (int half = 0; half < 2; ++half) {
        tma_prefetch_l2_4d(&tm_k, 0, half, c2, c3);
        tma_prefetch_l2_4d(&tm_v, 0, half, c2, c3);
      }
    }
  }
  // Inputs written by earlier grids are visible after this wait; they are read
  // with coherent loads (ld.global.ca), never the non-coherent read-only path.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // Paged: the producer warp loads the 32 block-table entries from the hinted
  // page on, alongside the length, so the first copy does not wait for two
  // dependent loads in a row; the entries are read after the wait (only which
  // window to load came from the hints), and a window that misses the split's
  // pages is simply loaded again.
  int page_base = -1 << 30, page_reg = 0;
  if (kPaged && warp == n_consumers) {
    page_base = __shfl_sync(0xffffffffu, hint_page, 0);
    const int idx = page_base + lane;
    page_reg = idx < p.max_pages ? __ldca(p.block_table + (size_t)b * p.max_pages + idx) : 0;
  }
  const int seqlen_in = __ldca(p.seqlens + b);
  const int seqlen = min(max(seqlen_in, 0), p.S_max);
  // the chunk for the batch's actual lengths (the host's chunk when they are S_max)
  const int chunk =
      device_chunk(seqlen, p.B, p.S_max, p.chunk, p.num_splits, p.H_kv, p.num_sms, kTileKeys);
  // out-of-range lengths are clamped and reported through the status word
  if ((seqlen_in < 0 || seqlen_in > p.S_max) && threadIdx.x == 0 && split == 0)
    atomicExch(p.wait.status, kStatusInvalidArg);
  const int key_begin = split * chunk;
  const int key_end = min(key_begin + chunk, seqlen);
  // an empty split: the merge never reads it (a fused CTA with no keys still takes
  // part in the cluster merge, and a direct-output CTA writes O = 0, lse = -inf)
  if (!kFused && !p.direct_out && key_begin >= key_end) return;
  const int n_tiles = max(0, (key_end - key_begin + kTileKeys - 1) / kTileKeys);
  // keys every column may see in this split (token 0 is the most restricted)
  const int key_all = min(key_end, seqlen - p.T_q + 1);
  __syncthreads();

  constexpr int kCols = 8 * kNT;  // columns per consumer warp
  float m_run[kNT][2], l_run[kNT][2], o_acc[8][kNT][4];

  if (warp == n_consumers) {
    // ---------------- producer: lane 0 issues all TMA loads ----------------
    // (paged: the whole warp keeps 32 block-table entries in registers, so the
    // page lookup is a shuffle, never a dependent global load per tile)
    const uint64_t pol = l2_policy_evict_first();
    const int row = b * p.H_kv + kv;
    int issued = 0;
    int page = 0, page_off = 0, page_c3 = 0;  // the tile's page, its first key there, its block
    for (int i = 0; i < n_tiles; ++i) {
      const int key0 = key_begin + i * kTileKeys;
      int c2 = key0, c3 = row;  // tensor-map coordinates of the tile's first key
      if (kPaged) {
        // pages advance by whole tiles: the page and the offset in it are
        // stepped, and the page's block is looked up only when a page begins
        if (i == 0) {
          page = key0 / p.page_size;
          page_off = key0 - page * p.page_size;
        } else if ((page_off += kTileKeys) == p.page_size) {
          ++page;
          page_off = 0;
        }
        if (i == 0 || page_off == 0) {  // warp-uniform
          if (page - page_base >= 32 || page < page_base) {
            page_base = page;
            const int idx = page_base + lane;
            page_reg = idx < p.max_pages ? __ldca(p.block_table + (size_t)b * p.max_pages + idx) : 0;
          }
          const int page_id = __shfl_sync(0xffffffffu, page_reg, page - page_base);
          // a page id outside the pool reads zeros (TMA out-of-bounds fill); report it
          const bool bad = page_id < 0 || page_id >= p.num_pages;
          if (bad && lane == 0) atomicExch(p.wait.status, kStatusInvalidArg);
          page_c3 = bad ? p.num_pages * p.H_kv : page_id * p.H_kv + kv;  // bad: past the map
        }
        c2 = page_off;
        c3 = page_c3;
      }
      bool ok = true;
      if (lane == 0) {
        const int s = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        ok = mbar_wait(smem_u32(&empty_bar[s]), ph ^ 1, p.wait);
        if (ok) {
          const uint32_t fb = smem_u32(&full_bar[s]);
          mbar_arrive_expect_tx(fb, kStageBytes);
          const uint32_t dst = smem_u32(smem + s * kStageBytes);
          tma_load_4d(dst + 0 * kHalfBytes, &tm_k, fb, 0, 0, c2, c3, pol);
          tma_load_4d(dst + 1 * kHalfBytes, &tm_k, fb, 0, 1, c2, c3, pol);
          tma_load_4d(dst + 2 * kHalfBytes, &tm_v, fb, 0, 0, c2, c3, pol);
          tma_load_4d(dst + 3 * kHalfBytes, &tm_v, fb, 0, 1, c2, c3, pol);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      ++issued;
    }
    if (lane == 0) {
      // Never leave the CTA with a copy in flight: wait for the last loads.
      for (int i = max(0, issued - kStages); i < issued; ++i)
        mbar_wait(smem_u32(&full_bar[i % kStages]), (i / kStages) & 1, p.wait);
      if (issued < n_tiles) atomicExch(&failed, 1);
    }
  } else if (warp < n_consumers) {
    // ---------------- consumers: key slice ks of column group cg ----------------
    const int ks = warp & 3, cg = warp >> 2;
    const int g = lane >> 2, t = lane & 3;
    const int col0 = cg * kCols;  // first column of this warp's group
    // Q^T as the B operand of n-tile j: b0 = Q[column col0 + 8j + g][16kk + 2t .. +1],
    // b1 = the same + 8; columns past G * T_q are zero.
    uint32_t qf[8][kNT][2];
#pragma unroll
    for (int j = 0; j < kNT; ++j) {
      const int n = col0 + 8 * j + g;
      const bool col_ok = n < p.n_cols;
      const int gh = col_ok ? n / p.T_q : 0, tq = col_ok ? n % p.T_q : 0;
      const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
          p.q + (((size_t)b * p.H_q + (size_t)kv * p.G + gh) * p.T_q + tq) * kD);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qf[kk][j][0] = col_ok ? __ldca(qrow + kk * 8 + t) : 0u;
        qf[kk][j][1] = col_ok ? __ldca(qrow + kk * 8 + 4 + t) : 0u;
      }
    }
    // keys each of this thread's columns may see (split end and causal limit)
    int lim[kNT][2];
#pragma unroll
    for (int j = 0; j < kNT; ++j)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int n = col0 + 8 * j + 2 * t + c;
        lim[j][c] = min(key_end, seqlen - p.T_q + (n % p.T_q) + 1);
        m_run[j][c] = -INFINITY;
        l_run[j][c] = 0.f;
      }
#pragma unroll
    for (int md = 0; md < 8; ++md)
#pragma unroll
      for (int j = 0; j < kNT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) o_acc[md][j][e] = 0.f;

    const int key_w0 = 16 * ks;  // this warp's keys inside a tile
    // ldmatrix lane roles (see the fragment layouts of mma.m16n8k16)
    const int k_row = key_w0 + (lane & 15), k_chunk_hi = lane >> 4;
    const int v_row = key_w0 + (lane & 7) + ((lane >> 4) << 3), v_chunk_hi = (lane >> 3) & 1;
    const float sl2 = p.scale_log2;

    for (int i = 0; i < n_tiles; ++i) {
      const int s = i % kStages;
      // every lane waits (acquiring the TMA data); the outcome is made warp-uniform
      const bool ready = mbar_wait(smem_u32(&full_bar[s]), (i / kStages) & 1, p.wait);
      if (!__all_sync(0xffffffffu, ready)) {
        if (lane == 0) atomicExch(&failed, 1);
        break;
      }
      const uint32_t kbase = smem_u32(smem + s * kStageBytes);
      const uint32_t vbase = kbase + 2 * kHalfBytes;
      const int tile_key0 = key_begin + i * kTileKeys;

      // S^T[16 keys x 8 columns] = K[16 x 128] * Q^T[128 x 8], per n-tile
      float sc[kNT][4];
#pragma unroll
      for (int j = 0; j < kNT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[j][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kbase + tile_offset(k_row, 2 * kk + k_chunk_hi), a0, a1, a2, a3);
#pragma unroll
        for (int j = 0; j < kNT; ++j)
          mma_bf16_16816(sc[j], a0, a1, a2, a3, qf[kk][j][0], qf[kk][j][1]);
      }
      // scale into the log2 domain; keys a column may not see are -inf
      const bool tail = tile_key0 + kTileKeys > key_all;
      const int k_lo = tile_key0 + key_w0 + g, k_hi = k_lo + 8;
      float pr[kNT][4], corr[kNT][2];
#pragma unroll
      for (int j = 0; j < kNT; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[j][e] *= sl2;
        if (tail) {
          if (k_lo >= lim[j][0]) sc[j][0] = -INFINITY;
          if (k_lo >= lim[j][1]) sc[j][1] = -INFINITY;
          if (k_hi >= lim[j][0]) sc[j][2] = -INFINITY;
          if (k_hi >= lim[j][1]) sc[j][3] = -INFINITY;
        }
        // online softmax; thread holds columns 2t (c = 0) and 2t+1 (c = 1)
        float mx0 = fmaxf(sc[j][0], sc[j][2]), mx1 = fmaxf(sc[j][1], sc[j][3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m_run[j][0], mx0), mn1 = fmaxf(m_run[j][1], mx1);
        const float ref0 = (mn0 == -INFINITY) ? 0.f : mn0;
        const float ref1 = (mn1 == -INFINITY) ? 0.f : mn1;
        pr[j][0] = fast_exp2(sc[j][0] - ref0);
        pr[j][1] = fast_exp2(sc[j][1] - ref1);
        pr[j][2] = fast_exp2(sc[j][2] - ref0);
        pr[j][3] = fast_exp2(sc[j][3] - ref1);
        corr[j][0] = fast_exp2(m_run[j][0] - ref0);
        corr[j][1] = fast_exp2(m_run[j][1] - ref1);
        l_run[j][0] = l_run[j][0] * corr[j][0] + pr[j][0] + pr[j][2];
        l_run[j][1] = l_run[j][1] * corr[j][1] + pr[j][1] + pr[j][3];
        m_run[j][0] = mn0;
        m_run[j][1] = mn1;
      }
      uint32_t pb[kNT][2];
#pragma unroll
      for (int j = 0; j < kNT; ++j) {
#pragma unroll
        for (int md = 0; md < 8; ++md) {
          o_acc[md][j][0] *= corr[j][0]; o_acc[md][j][1] *= corr[j][1];
          o_acc[md][j][2] *= corr[j][0]; o_acc[md][j][3] *= corr[j][1];
        }
        // P^T in the B-operand layout: rows (keys g, g+8) x cols (2t, 2t+1)
        // transposed to keys (2t, 2t+1) [+8] x column g.
        pb[j][0] = movmatrix_trans(pack_bf16x2(pr[j][0], pr[j][1]));
        pb[j][1] = movmatrix_trans(pack_bf16x2(pr[j][2], pr[j][3]));
      }
      // rows of V past the split end are zeroed so stale or NaN cache bytes never
      // meet a zero probability
      bool lo0 = true, lo1 = true, hi0 = true, hi1 = true;
      if (tile_key0 + kTileKeys > key_end) {
        const int kb = tile_key0 + key_w0 + 2 * t;
        lo0 = kb < key_end; lo1 = kb + 1 < key_end;
        hi0 = kb + 8 < key_end; hi1 = kb + 9 < key_end;
      }
      // O^T[128 x 8] += V^T[128 x 16 keys] * P^T[16 keys x 8], per n-tile
#pragma unroll
      for (int md = 0; md < 8; ++md) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(vbase + tile_offset(v_row, 2 * md + v_chunk_hi), a0, a1, a2, a3);
        if (tile_key0 + kTileKeys > key_end) {
          a0 = mask_pair(a0, lo0, lo1); a1 = mask_pair(a1, lo0, lo1);
          a2 = mask_pair(a2, hi0, hi1); a3 = mask_pair(a3, hi0, hi1);
        }
#pragma unroll
        for (int j = 0; j < kNT; ++j)
          mma_bf16_16816(o_acc[md][j], a0, a1, a2, a3, pb[j][0], pb[j][1]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
    }
    // per-thread partial sums over the 8 lanes that share columns 2t, 2t+1
#pragma unroll
    for (int j = 0; j < kNT; ++j)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l_run[j][0] += __shfl_xor_sync(0xffffffffu, l_run[j][0], off);
        l_run[j][1] += __shfl_xor_sync(0xffffffffu, l_run[j][1], off);
      }
  }
  __syncthreads();
  if (!kFused && failed) return;

  // ---------------- merge the four key slices, write the split partial ----------------
  // All loads have landed and been consumed; the stage ring is free.
  const int n_cols_pad = kCols * p.cgroups;                  // <= kMaxCols
  float *red_m = reinterpret_cast<float *>(smem);              // [4][n_cols_pad]
  float *red_l = red_m + kConsumerWarps * kMaxCols;            // [4][n_cols_pad]
  float *red_o = red_l + kConsumerWarps * kMaxCols;            // [4][n_cols_pad][kRedStride]
  if (warp < n_consumers) {
    const int ks = warp & 3, cg = warp >> 2;
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int j = 0; j < kNT; ++j) {
      const int n0 = cg * kCols + 8 * j + 2 * t;
      if (g == 0) {
        red_m[ks * kMaxCols + n0] = m_run[j][0];
        red_m[ks * kMaxCols + n0 + 1] = m_run[j][1];
        red_l[ks * kMaxCols + n0] = l_run[j][0];
        red_l[ks * kMaxCols + n0 + 1] = l_run[j][1];
      }
      float *ow = red_o + (size_t)ks * kMaxCols * kRedStride;
#pragma unroll
      for (int md = 0; md < 8; ++md) {
        ow[n0 * kRedStride + 16 * md + g] = o_acc[md][j][0];
        ow[(n0 + 1) * kRedStride + 16 * md + g] = o_acc[md][j][1];
        ow[n0 * kRedStride + 16 * md + g + 8] = o_acc[md][j][2];
        ow[(n0 + 1) * kRedStride + 16 * md + g + 8] = o_acc[md][j][3];
      }
    }
  }
  __syncthreads();
  // Weights of the four key slices of column n: reference max, weight
  // 2^(m_w - max) / l (0 for slices without keys, and for every slice of a
  // column that saw no key or of a failed CTA), lse_s = max ln 2 + ln l.
  const bool failed_cta = failed;
  auto slice_weights = [&](int n, float (&wt)[kConsumerWarps]) {
    float mw[kConsumerWarps], lw[kConsumerWarps];
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      mw[w] = red_m[w * kMaxCols + n];
      lw[w] = red_l[w * kMaxCols + n];
    }
    const float mmax = fmaxf(fmaxf(mw[0], mw[1]), fmaxf(mw[2], mw[3]));
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      wt[w] = mmax == -INFINITY ? 0.f : fast_exp2(mw[w] - mmax);
      lsum = fmaf(lw[w], wt[w], lsum);
    }
    const bool empty = failed_cta || !(lsum > 0.f);
    const float inv = empty ? 0.f : fast_rcp(lsum);  // lsum >= 1 when not empty
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) wt[w] *= inv;
    return empty ? -INFINITY : (mmax + fast_log2(lsum)) * 0.69314718055994531f;
  };
  auto out_row = [&](int n) {  // (sequence, query head, new token) row of column n
    const int gh = p.T_q == 1 ? n : n / p.T_q, tq = p.T_q == 1 ? 0 : n % p.T_q;
    return ((size_t)b * p.H_q + (size_t)kv * p.G + gh) * p.T_q + tq;
  };
  if constexpr (kNT == 2 && !kFused) {
    // many columns: one thread per column weighs its slices, then O_s = sum of
    // weight * O_slice per (column, four d values)
    float *wts = red_o + kConsumerWarps * kMaxCols * kRedStride;  // [4][kMaxCols]
    size_t *col_prow = reinterpret_cast<size_t *>(wts + kConsumerWarps * kMaxCols);  // [kMaxCols]
    if (threadIdx.x < p.n_cols) {
      const int n = threadIdx.x;
      float wt[kConsumerWarps];
      const float lse_s = slice_weights(n, wt);
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) wts[w * kMaxCols + n] = wt[w];
      const size_t prow = out_row(n) * p.num_splits + split;
      col_prow[n] = prow;
      if (store_ok(prow, (size_t)p.B * p.H_q * p.T_q * p.num_splits, p.wait.status))
        (p.direct_out ? p.lse : p.lse_part)[prow] = lse_s;  // one split: prow is the row
    }
    __syncthreads();
    for (int item = threadIdx.x; item < n_cols_pad * (kD / 4); item += blockDim.x) {
      const int n = item / (kD / 4), d4 = item % (kD / 4);
      if (n >= p.n_cols) continue;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float wt = wts[w * kMaxCols + n];
        const float4 x =
            reinterpret_cast<const float4 *>(red_o + ((size_t)w * kMaxCols + n) * kRedStride)[d4];
        acc.x = fmaf(wt, x.x, acc.x);
        acc.y = fmaf(wt, x.y, acc.y);
        acc.z = fmaf(wt, x.z, acc.z);
        acc.w = fmaf(wt, x.w, acc.w);
      }
      const size_t prow = col_prow[n];
      if (!store_ok(prow, (size_t)p.B * p.H_q * p.T_q * p.num_splits, p.wait.status)) continue;
      if (p.direct_out) {
        uint2 pk;
        pk.x = pack_bf16x2(acc.x, acc.y);
        pk.y = pack_bf16x2(acc.z, acc.w);
        reinterpret_cast<uint2 *>(p.o + prow * kD)[d4] = pk;
      } else {
        reinterpret_cast<float4 *>(p.o_part + prow * kD)[d4] = acc;
      }
    }
  } else {
    // at most 8 columns: each item = (column n, four d values) weighs its
    // column's slices itself (no second barrier).  The split's partial goes to
    // the workspace, or (cluster-merged) to the output when the cluster is one
    // CTA, else to the CTA that finalises the column.
    for (int item = threadIdx.x; item < n_cols_pad * (kD / 4); item += blockDim.x) {
      const int n = item / (kD / 4), d4 = item % (kD / 4);
      if (n >= p.n_cols) continue;  // padding columns (warp-uniform: 32 items per column)
      float4 xw[kConsumerWarps];
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w)
        xw[w] =
            reinterpret_cast<const float4 *>(red_o + ((size_t)w * kMaxCols + n) * kRedStride)[d4];
      float wt[kConsumerWarps];
      const float lse_s = slice_weights(n, wt);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        acc.x = fmaf(wt[w], xw[w].x, acc.x);
        acc.y = fmaf(wt[w], xw[w].y, acc.y);
        acc.z = fmaf(wt[w], xw[w].z, acc.z);
        acc.w = fmaf(wt[w], xw[w].w, acc.w);
      }
      const size_t row = out_row(n);
      if (!kFused && !p.direct_out) {
        const size_t prow = row * p.num_splits + split;
        if (!store_ok(prow, (size_t)p.B * p.H_q * p.T_q * p.num_splits, p.wait.status)) continue;
        if (d4 == 0) p.lse_part[prow] = lse_s;
        reinterpret_cast<float4 *>(p.o_part + prow * kD)[d4] = acc;
      } else if (!kFused || cs == 1) {  // one split (or a cluster of one): the whole sequence
        if (!store_ok(row, (size_t)p.B * p.H_q * p.T_q, p.wait.status)) continue;
        if (d4 == 0) p.lse[row] = lse_s;
        uint2 pk;
        pk.x = pack_bf16x2(acc.x, acc.y);
        pk.y = pack_bf16x2(acc.z, acc.w);
        reinterpret_cast<uint2 *>(p.o + row * kD)[d4] = pk;
      } else if (cluster_merge) {
        // to CTA n % cs, slot (this split, n / cs): bytes counted on its barrier
        // (n < 8 and cs >= 2: the quotient is at most 3)
        const int quo = (n >= cs) + (n >= 2 * cs) + (n >= 3 * cs);
        const uint32_t dst = (uint32_t)(n - quo * cs);
        const int slot = split * per_rank + quo;
        const uint32_t bar = dsmem_addr(smem_u32(recv_bar), dst);
        st_async_f32x4(dsmem_addr(smem_u32(recv_o + slot * kD + 4 * d4), dst), acc, bar);
        if (d4 == 0) st_async_f32(dsmem_addr(smem_u32(recv_lse + slot), dst), lse_s, bar);
      }
    }
  }
  if (kFused && cs > 1 && !cluster_merge && threadIdx.x == 0)
    atomicExch(p.wait.status, kStatusInvalidArg);  // more columns than the receive area holds
  if (cluster_merge && n_mine > 0) {
    // log-sum-exp merge of the cluster's partials of this CTA's columns, once every
    // CTA's bytes have landed here: lse = m + ln sum_c e^(lse_c - m),
    // O = sum_c e^(lse_c - lse) O_c.  No CTA reads another's shared memory, so
    // none waits for the others before it exits.
    // (a wait that runs out means a CTA of the cluster is stuck: the timeout is
    // recorded in the status word and this CTA's columns are not written)
    const bool landed = mbar_wait(smem_u32(recv_bar), 0, p.wait);
    constexpr float kLog2e = 1.4426950408889634f;
    for (int item = threadIdx.x; landed && item < n_mine * (kD / 4); item += blockDim.x) {
      const int nl = item / (kD / 4), d4 = item % (kD / 4);
      const int n = split + cs * nl;
      float ls[kMaxFusedSplits];
      float4 x[kMaxFusedSplits];
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kMaxFusedSplits; ++c) {
        ls[c] = -INFINITY;
        x[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < cs) {
          ls[c] = recv_lse[c * per_rank + nl];
          x[c] = reinterpret_cast<const float4 *>(recv_o + (c * per_rank + nl) * kD)[d4];
        }
        mx = fmaxf(mx, ls[c]);
      }
      float wsum = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (mx != -INFINITY) {
#pragma unroll
        for (int c = 0; c < kMaxFusedSplits; ++c) {
          const float w = fast_exp2((ls[c] - mx) * kLog2e);  // 0 for a split without keys
          wsum += w;
          acc.x = fmaf(w, x[c].x, acc.x);
          acc.y = fmaf(w, x[c].y, acc.y);
          acc.z = fmaf(w, x[c].z, acc.z);
          acc.w = fmaf(w, x[c].w, acc.w);
        }
      }
      const float inv = wsum > 0.f ? fast_rcp(wsum) : 0.f;
      const size_t row = out_row(n);
      if (!store_ok(row, (size_t)p.B * p.H_q * p.T_q, p.wait.status)) continue;
      uint2 pk;
      pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      reinterpret_cast<uint2 *>(p.o + row * kD)[d4] = pk;
      if (d4 == 0) p.lse[row] = wsum > 0.f ? mx + fast_log2(wsum) * 0.69314718055994531f : -INFINITY;
    }
  }
  // this CTA's partial is written: the merge grid may be scheduled (triggering
  // at the start instead measured 1 us slower per call: the waiting merge CTAs
  // slow the streaming ones; the cluster-merged grid has triggered at its start)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// One CTA per (query head, new token) row of a sequence, 128 threads: thread
// (g, lane) owns columns 4*lane .. 4*lane+3 and merges splits g, g+4, g+8, ...
// with an online log-sum-exp, kMergeRound splits per round whose lse and O
// loads are all issued before any is used (one L2 round trip for up to 32
// splits); the four group states are then combined once in shared memory.
// Used for merges of fewer than kMergeRowsMin rows (a layer's 64 heads of one
// token), where spreading each row over four warps shortens its load and
// accumulation chain; larger merges take decode_merge_rows_kernel below.
// lse = m + ln sum_s exp(lse_s - m); O = sum_s exp(lse_s - lse) O_s.
// Launched as a programmatic dependent of the split kernel; the partials are
// read through L2 (they were written by the split grid).
constexpr int kMergeThreads = 128;
constexpr int kMergeGroups = kMergeThreads / 32;
constexpr int kMergeRound = 8;

__global__ void __launch_bounds__(kMergeThreads)
    decode_merge_kernel(const float *__restrict__ o_part, const float *__restrict__ lse_part,
                        const int32_t *__restrict__ seqlens, uint16_t *__restrict__ o,
                        float *__restrict__ lse, int S_max, int num_splits, int chunk, int H_kv,
                        int num_sms, int tile) {
  __shared__ float4 red_o[kMergeGroups][32];
  __shared__ float red_w[kMergeGroups];
  __shared__ float red_m[kMergeGroups];
  // the next kernel (typically the next layer's split) may start its prologue
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int h = blockIdx.x, b = blockIdx.y;  // h: (query head, new token) row of sequence b
  const int t = threadIdx.x, grp = t >> 5, lane = t & 31;
  // The lengths are read ahead of the dependency wait: the merge takes the
  // lengths its split phase took, which the grids before that phase wrote (the
  // split kernel itself never writes them), so they are already visible here.
  const int seqlen = min(max(__ldcg(seqlens + b), 0), S_max);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the splits that hold keys of this row: the chunk the split kernel derived
  // from the same lengths
  const int dchunk = device_chunk(seqlen, gridDim.y, S_max, chunk, num_splits, H_kv, num_sms, tile);
  const int ns = min((seqlen + dchunk - 1) / dchunk, num_splits);
  const size_t row = (size_t)b * gridDim.x + h;
  const float *lp = lse_part + row * num_splits;
  const float4 *op = reinterpret_cast<const float4 *>(o_part + row * num_splits * kD) + lane;
  constexpr float kLog2e = 1.4426950408889634f;
  float m = -INFINITY, wsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = grp; s0 < ns; s0 += kMergeGroups * kMergeRound) {
    float ls[kMergeRound];
    float4 x[kMergeRound];
#pragma unroll
    for (int u = 0; u < kMergeRound; ++u) {
      const int s = s0 + u * kMergeGroups;
      ls[u] = s < ns ? __ldcg(lp + s) : -INFINITY;
      x[u] = s < ns ? __ldcg(op + (size_t)s * (kD / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kMergeRound; ++u) {
      if (ls[u] == -INFINITY) continue;  // a split that saw no key of this row
      const float m_new = fmaxf(m, ls[u]);
      const float c = fast_exp2((m - m_new) * kLog2e);  // 0 while m is -inf
      const float w = fast_exp2((ls[u] - m_new) * kLog2e);
      wsum = wsum * c + w;
      acc.x = fmaf(w, x[u].x, acc.x * c);
      acc.y = fmaf(w, x[u].y, acc.y * c);
      acc.z = fmaf(w, x[u].z, acc.z * c);
      acc.w = fmaf(w, x[u].w, acc.w * c);
      m = m_new;
    }
  }
  red_o[grp][lane] = acc;
  if (lane == 0) {
    red_w[grp] = wsum;
    red_m[grp] = m;
  }
  __syncthreads();
  if (grp == 0) {
    float mx = -INFINITY;
#pragma unroll
    for (int g = 0; g < kMergeGroups; ++g) mx = fmaxf(mx, red_m[g]);
    uint2 packed = make_uint2(0u, 0u);  // no visible key: O = 0, lse = -inf
    float lse_out = -INFINITY;
    if (mx != -INFINITY) {
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
      float W = 0.f;
#pragma unroll
      for (int g = 0; g < kMergeGroups; ++g) {
        const float f = fast_exp2((red_m[g] - mx) * kLog2e);  // empty groups: 0
        const float4 x = red_o[g][lane];
        sum.x = fmaf(f, x.x, sum.x);
        sum.y = fmaf(f, x.y, sum.y);
        sum.z = fmaf(f, x.z, sum.z);
        sum.w = fmaf(f, x.w, sum.w);
        W = fmaf(f, red_w[g], W);
      }
      const float inv = fast_rcp(W);  // W >= 1: the largest split weighs 1
      packed.x = pack_bf16x2(sum.x * inv, sum.y * inv);
      packed.y = pack_bf16x2(sum.z * inv, sum.w * inv);
      lse_out = mx + fast_log2(W) * 0.69314718055994531f;
    }
    reinterpret_cast<uint2 *>(o + row * kD)[lane] = packed;
    if (lane == 0) lse[row] = lse_out;
  }
}

// The same merge with one warp per row, four rows per CTA, for merges of many
// rows (16 new tokens of 64 heads: 1024 rows in 256 CTAs instead of 1024):
// lane l owns columns 4l .. 4l+3 and loads that float4 of up to 32 splits at
// once, lane s the lse of split s of the round (one L2 round trip per 32
// splits), then merges the round with an online log-sum-exp.  Measured against
// the CTA-per-row kernel: 16 new tokens 26.44 -> 25.92 us per call, 4 new
// tokens 24.61 -> 24.23; one token (64 rows) 21.28 -> 21.38, which keeps it.
constexpr int kMergeRowWarps = 4;
constexpr int kMergeRowRound = 32;
constexpr int kMergeRowsMin = 256;  // rows per launch from which this kernel is used

__global__ void __launch_bounds__(32 * kMergeRowWarps)
    decode_merge_rows_kernel(const float *__restrict__ o_part, const float *__restrict__ lse_part,
                             const int32_t *__restrict__ seqlens, uint16_t *__restrict__ o,
                             float *__restrict__ lse, int S_max, int num_splits, int chunk,
                             int H_kv, int num_sms, int tile, int rows_per_seq) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = blockIdx.y, lane = threadIdx.x & 31;
  const int h = blockIdx.x * kMergeRowWarps + (threadIdx.x >> 5);  // row of sequence b
  // lengths ahead of the dependency wait, as in decode_merge_kernel
  const int seqlen = min(max(__ldcg(seqlens + b), 0), S_max);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (h >= rows_per_seq) return;  // whole warps
  const int dchunk = device_chunk(seqlen, gridDim.y, S_max, chunk, num_splits, H_kv, num_sms, tile);
  const int ns = min((seqlen + dchunk - 1) / dchunk, num_splits);
  const size_t row = (size_t)b * rows_per_seq + h;
  const float *lp = lse_part + row * num_splits;
  const float4 *op = reinterpret_cast<const float4 *>(o_part + row * num_splits * kD) + lane;
  constexpr float kLog2e = 1.4426950408889634f;
  float m = -INFINITY, wsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < ns; s0 += kMergeRowRound) {
    const int n = min(kMergeRowRound, ns - s0);
    const float ls = lane < n ? __ldcg(lp + s0 + lane) : -INFINITY;
    float4 x[kMergeRowRound];
#pragma unroll
    for (int u = 0; u < kMergeRowRound; ++u)
      x[u] = u < n ? __ldcg(op + (size_t)(s0 + u) * (kD / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
    float mr = ls;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, off));
    if (mr == -INFINITY) continue;  // no split of the round saw a key of this row
    const float m_new = fmaxf(m, mr);
    const float c = fast_exp2((m - m_new) * kLog2e);  // 0 while m is -inf
    wsum *= c;
    acc.x *= c;
    acc.y *= c;
    acc.z *= c;
    acc.w *= c;
    const float wl = fast_exp2((ls - m_new) * kLog2e);  // lane u: weight of split s0 + u
#pragma unroll
    for (int u = 0; u < kMergeRowRound; ++u) {
      const float w = __shfl_sync(0xffffffffu, wl, u);  // 0 past the round and for empty splits
      wsum += w;
      acc.x = fmaf(w, x[u].x, acc.x);
      acc.y = fmaf(w, x[u].y, acc.y);
      acc.z = fmaf(w, x[u].z, acc.z);
      acc.w = fmaf(w, x[u].w, acc.w);
    }
    m = m_new;
  }
  uint2 packed = make_uint2(0u, 0u);  // no visible key: O = 0, lse = -inf
  float lse_out = -INFINITY;
  if (wsum > 0.f) {
    const float inv = fast_rcp(wsum);  // wsum >= 1: the largest split weighs 1
    packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    lse_out = m + fast_log2(wsum) * 0.69314718055994531f;
  }
  reinterpret_cast<uint2 *>(o + row * kD)[lane] = packed;
  if (lane == 0) lse[row] = lse_out;
}

// rows = keys per (sequence, KV head) block (S_max, or page_size for pages);
// blocks = B*H_kv (dense) or num_pages*H_kv (paged)
static CUresult make_kv_map(CUtensorMap *map, const uint16_t *base, long long blocks, int rows,
                            PFN_cuTensorMapEncodeTiled_v12000 encode) {
  // dims (innermost first): 64 columns, 2 column halves, rows, blocks
  const cuuint64_t dims[4] = {64, 2, (cuuint64_t)rows, (cuuint64_t)blocks};
  const cuuint64_t strides[3] = {128, 256, (cuuint64_t)rows * 256};  // bytes, dims 1..3
  const cuuint32_t box[4] = {64, 1, kTileKeys, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t *>(base), dims,
                strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace decode

template <int kStages, int kMinBlocks, bool kFused, int kNT>
static cudaError_t set_smem_attr() {
  using namespace decode;
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<kStages, kMinBlocks, kFused, false, kNT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_bytes<kStages, kFused>());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_split_kernel<kStages, kMinBlocks, kFused, true, kNT>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              smem_bytes<kStages, kFused>());
}

cudaError_t decode_prepare_device(int *fused_clusters) {
  using namespace decode;
  cudaError_t e;
  if ((e = set_smem_attr<3, 2, false, 1>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<kOneWaveStages, 1, false, 1>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<3, 2, true, 1>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<kOneWaveStages, 1, false, 2>()) != cudaSuccess) return e;
  // For each cluster size (splits per sequence and KV head) the number of
  // clusters of the fused kernel the device runs at once (the 3-stage variant,
  // which may pair two CTAs on an SM); 0 where it cannot.  Sizes above 8 need the
  // non-portable cluster size opt-in.
  const bool big = cudaFuncSetAttribute(decode_split_kernel<3, 2, true, false, 1>,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed,
                                        1) == cudaSuccess &&
                   cudaFuncSetAttribute(decode_split_kernel<3, 2, true, true, 1>,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed,
                                        1) == cudaSuccess;
  for (int cs = 1; cs <= kMaxFusedSplits; ++cs) {
    fused_clusters[cs] = 0;
    if (cs > 8 && !big) continue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, 1, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes<3, true>();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_split_kernel<3, 2, true, false, 1>, &cfg) ==
        cudaSuccess)
      fused_clusters[cs] = n;
  }
  cudaGetLastError();  // a refused opt-in or query is not an error for the caller
  return cudaSuccess;
}

static bool make_maps(const DecodeLaunch &a, PFN_cuTensorMapEncodeTiled_v12000 encode,
                      CUtensorMap *tm_k, CUtensorMap *tm_v) {
  using namespace decode;
  const bool paged = a.block_table != nullptr;
  const long long blocks = paged ? (long long)a.num_pages * a.H_kv : (long long)a.B * a.H_kv;
  const int rows = paged ? a.page_size : a.S_max;
  return make_kv_map(tm_k, a.k_cache, blocks, rows, encode) == CUDA_SUCCESS &&
         make_kv_map(tm_v, a.v_cache, blocks, rows, encode) == CUDA_SUCCESS;
}

// Launches decode_split_kernel<kStages, kMinBlocks, kFused, paged, kNT> for a's layout.
template <int kStages, int kMinBlocks, bool kFused, int kNT>
static cudaError_t launch_variant(cudaLaunchConfig_t *cfg, const CUtensorMap &tm_k,
                                  const CUtensorMap &tm_v, const decode::Params &p, bool paged) {
  using namespace decode;
  cfg->dynamicSmemBytes = smem_bytes<kStages, kFused>();
  cfg->blockDim = dim3(32 * (kConsumerWarps * p.cgroups + 1));
  if (paged)
    return cudaLaunchKernelEx(cfg, decode_split_kernel<kStages, kMinBlocks, kFused, true, kNT>,
                              tm_k, tm_v, p);
  return cudaLaunchKernelEx(cfg, decode_split_kernel<kStages, kMinBlocks, kFused, false, kNT>,
                            tm_k, tm_v, p);
}

static decode::Params make_params(const DecodeLaunch &a) {
  decode::Params p;
  p.q = a.q;
  p.seqlens = a.seqlens;
  p.o_part = a.o_part;
  p.lse_part = a.lse_part;
  p.o = a.o;
  p.lse = a.lse;
  p.B = a.B;
  p.H_q = a.H_q;
  p.H_kv = a.H_kv;
  p.G = a.H_q / a.H_kv;
  p.S_max = a.S_max;
  p.num_splits = a.num_splits;
  p.chunk = a.chunk;
  p.num_sms = a.num_sms;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.T_q = a.T_q > 0 ? a.T_q : 1;
  p.n_cols = p.G * p.T_q;
  p.cgroups = p.n_cols <= 8 ? 1 : (p.n_cols + 15) / 16;
  p.block_table = a.block_table;
  p.page_size = a.page_size;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.l2_prefetch_tiles = 0;
  p.direct_out = a.direct_out && a.num_splits == 1;
  p.wait = a.wait;
  return p;
}

bool decode_fused_eligible(const DecodeLaunch &a) {
  // one launch only when every (sequence, KV head) cluster runs in a single wave
  if (a.S_max <= 0 || a.num_splits < 1 || a.num_splits > decode::kMaxFusedSplits) return false;
  if ((long long)(a.H_q / a.H_kv) * (a.T_q > 0 ? a.T_q : 1) > 8) return false;  // one n-tile only
  return (long long)a.B * a.H_kv <= a.fused_clusters[a.num_splits];
}

cudaError_t decode_fused_launch(const DecodeLaunch &a, cudaStream_t stream,
                                PFN_cuTensorMapEncodeTiled_v12000 encode) {
  using namespace decode;
  if (!decode_fused_eligible(a)) return cudaErrorNotSupported;
  CUtensorMap tm_k, tm_v;
  if (!make_maps(a, encode, &tm_k, &tm_v)) return cudaErrorInvalidValue;
  const Params p = make_params(a);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_splits, a.H_kv, a.B);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = a.num_splits;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return launch_variant<3, 2, true, 1>(&cfg, tm_k, tm_v, p, a.block_table != nullptr);
}

cudaError_t decode_split_launch(const DecodeLaunch &a, cudaStream_t stream,
                                PFN_cuTensorMapEncodeTiled_v12000 encode) {
  using namespace decode;
  if (a.S_max <= 0) return cudaSuccess;
  CUtensorMap tm_k, tm_v;
  if (!make_maps(a, encode, &tm_k, &tm_v)) return cudaErrorInvalidValue;
  Params p = make_params(a);
  const long long ctas = (long long)a.num_splits * a.H_kv * a.B;
  if (ctas <= a.num_sms) p.l2_prefetch_tiles = GQA_DECODE_L2_PREFETCH_TILES;  // one wave
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.H_kv, a.B, a.num_splits);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool paged = a.block_table != nullptr;
  if (p.n_cols > 8)  // multi-token decode: two n-tiles per warp, one CTA per SM
    return launch_variant<kOneWaveStages, 1, false, 2>(&cfg, tm_k, tm_v, p, paged);
  if (ctas <= a.num_sms)  // one wave, one CTA per SM
    return launch_variant<kOneWaveStages, 1, false, 1>(&cfg, tm_k, tm_v, p, paged);
  return launch_variant<3, 2, false, 1>(&cfg, tm_k, tm_v, p, paged);
}

cudaError_t decode_merge_launch(const DecodeLaunch &a, cudaStream_t stream) {
  using namespace decode;
  const int rows_per_seq = a.H_q * (a.T_q > 0 ? a.T_q : 1);
  const int chunk = a.chunk > 0 ? a.chunk : 1;
  const int tile = a.chunk_tile > 0 ? a.chunk_tile : kTileKeys;
  cudaLaunchConfig_t cfg = {};
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((long long)rows_per_seq * a.B >= kMergeRowsMin) {
    cfg.gridDim = dim3((rows_per_seq + kMergeRowWarps - 1) / kMergeRowWarps, a.B);
    cfg.blockDim = dim3(32 * kMergeRowWarps);
    return cudaLaunchKernelEx(&cfg, decode_merge_rows_kernel, (const float *)a.o_part,
                              (const float *)a.lse_part, a.seqlens, a.o, a.lse, a.S_max,
                              a.num_splits, chunk, a.H_kv, a.num_sms, tile, rows_per_seq);
  }
  cfg.gridDim = dim3(rows_per_seq, a.B);
  cfg.blockDim = dim3(kMergeThreads);
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel, (const float *)a.o_part,
                            (const float *)a.lse_part, a.seqlens, a.o, a.lse, a.S_max,
                            a.num_splits, chunk, a.H_kv, a.num_sms, tile);
}

}  // namespace gqa
