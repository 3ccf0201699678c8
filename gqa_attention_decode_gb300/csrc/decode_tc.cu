// decode_tc.cu -- split-KV multi-token GQA decode on tcgen05 tensor cores (sm_103a).
//
// What it computes (design record "ADR-0060: AHBM GQA Fused Attention Kernel
// (Llama3-70B)"): decode with T_q new tokens per sequence, the record's T_q of
// section 0.5.2 with all G * T_q (head, token) rows of one KV head stacked into
// one matrix product (section 5.2's fold), so each K/V tile is read from HBM
// once for every row.  Token t of sequence b sits at position seqlen - T_q + t
// and sees keys up to it.  The key range is cut into contiguous chunks
// (section 2.1); each CTA runs the per-tile online softmax of section 3 over its
// chunk and writes one partial per row (O_s / l_s, lse_s), which the decode
// merge kernel combines (section 4).  Used for 32 < G * T_q <= 128, where the
// rows fill a 128-row tensor-core tile.
//
// GB300 mapping
//   * grid (splits, H_kv, B), 320 threads: warp 8 TMA producer (the row block
//     of Q once, then 128-key K and V tiles through a 5-stage ring), warp 9
//     TMEM allocation and the single thread issuing tcgen05.mma (M = 128 rows,
//     N = 128 keys or d, K = 16, bf16 in, fp32 accumulate), warps 0-3 / 4-7
//     softmax for two slots (one thread per row).  Slot s takes the key tiles
//     of parity s with its own S and O in tensor memory, so the tensor core
//     works on one slot's tile while the other slot's softmax runs; the two
//     slots' (m, l, O) are combined per row at the end.
//   * Rows past G * T_q in the 128-row tile (other heads' queries, or zeros
//     past the tensor) are computed and never stored.
//   * Decode moves 128 flop per byte of K/V here (128 rows): still below the
//     tensor ridge, so the kernel streams K/V at HBM rate like the T_q = 1 path.
#include <cudaTypedefs.h>
#include <math.h>

#include "device_common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace gqa {
namespace decode_tc {

constexpr int kD = 128;
constexpr int kRows = 128;                 // tensor-core rows: (head, token) pairs of one KV head
constexpr int kBN = 128;                   // keys per tile
constexpr int kStages = 5;                 // ring of 32 KiB stages (a K or a V tile)
constexpr int kWarpTma = 8, kWarpMma = 9;
constexpr int kThreads = 320;
constexpr int kTileBytes = kRows * kD * 2;  // 32 KiB
constexpr int kHalfBytes = kTileBytes / 2;  // one 64-column half: [128 rows x 128 B]
constexpr int kOffQ = 0;
constexpr int kOffStage = kTileBytes;
constexpr int kOffBar = kOffStage + kStages * kTileBytes;
// barriers: kv_full[S], kv_empty[S], q_full, s_full[2], p_full[2], o_final[2], tok[2],
// drain, V tail cleared
constexpr int kNumBars = 2 * kStages + 1 + 2 + 2 + 2 + 2 + 1 + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;        // tmem slot, abort flag
constexpr int kOffRed = kOffMisc + 16;                  // (m, l) of both slots per row
constexpr int kSmemBytes = kOffRed + 4 * kRows * 4 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kSumTrigger = 256.0f;      // 2^kRescaleThreshold
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Params {
  const int32_t *seqlens;
  const int32_t *block_table;  // paged cache: [B, max_pages]; nullptr: dense cache
  float *o_part;
  float *lse_part;
  uint16_t *o;     // the direct-output instantiation: [B, H_q, T_q, d] bf16
  float *lse;      // the direct-output instantiation: [B, H_q, T_q]
  int B, H_q, H_kv, G, T_q, S_max, num_splits, chunk;
  int page_size, max_pages, num_pages;
  int num_sms;  // SMs the host plan counted on (the device-side chunk rule)
  int l2_prefetch;  // one-wave grid: prefetch the first key tile before the wait
  float sl2;  // scale * log2(e)
  WaitCtl wait;
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const WaitCtl &ctl,
                                         volatile int *abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > ctl.timeout_ns) {
      atomicExch(ctl.status, kStatusTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

// Barrier over the 256 softmax threads (warps 0-7, named barrier 1) that also
// returns the AND of their flags.
__device__ __forceinline__ bool softmax_bar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Operand descriptors, built once per tile and advanced per k-step by a
// compile-time byte offset.  K-major 128-row tile stored as two 128B-swizzled
// 64-column halves (k-step kk = 16 columns); MN-major V tile (keys x d, d
// contiguous in two halves; k-step kk = 16 keys).
__device__ __forceinline__ uint64_t desc_kmajor_base(uint32_t tile) {
  return tc::smem_desc_sw128(tile, 16, 1024);
}
__device__ __forceinline__ constexpr uint32_t kmajor_step(int kk) {
  return (kk >> 2) * kHalfBytes + (kk & 3) * 32;
}
__device__ __forceinline__ uint64_t desc_mnmajor_base(uint32_t tile) {
  return tc::smem_desc_sw128(tile, kHalfBytes, 1024);
}
__device__ __forceinline__ constexpr uint32_t mnmajor_step(int kk) { return kk * 2048; }

// kDirect: one split per (sequence, KV head); the CTA writes o (bf16) and lse
// instead of a partial for the merge (a separate instantiation, so the
// partial-writing kernel's register allocation is untouched).
template <bool kDirect>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBar;
  auto kv_full = [&](int s) { return bar0 + 8u * s; };
  auto kv_empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  const uint32_t q_full = bar0 + 8u * (2 * kStages);
  auto s_full = [&](int i) { return bar0 + 8u * (2 * kStages + 1 + i); };
  auto p_full = [&](int i) { return bar0 + 8u * (2 * kStages + 3 + i); };
  auto o_final = [&](int i) { return bar0 + 8u * (2 * kStages + 5 + i); };
  auto tok = [&](int i) { return bar0 + 8u * (2 * kStages + 7 + i); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 9);
  const uint32_t v_tail = bar0 + 8u * (2 * kStages + 10);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
  float *red_m = reinterpret_cast<float *>(smem + kOffRed);  // [slot][row]
  float *red_l = red_m + 2 * kRows;

  // grid (H_kv, B, splits): the first splits of every (sequence, KV head) come
  // first in launch order (CTAs that hold keys before empty ones)
  const int split = blockIdx.z, kv = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  // One-wave grid: the first key tile of this split's chunk is pulled into L2
  // while the preceding grid finishes (L2 is the point of coherence, so this is
  // safe ahead of the wait).  The sequence length and a paged cache's
  // block-table entry are read here as hints only (relaxed loads): a preceding
  // grid may still write them, and the loads after the wait read them again,
  // so a stale value costs one wasted L2 fill; the length gives this split's
  // device-side chunk, and a split that starts past the sequence prefetches
  // nothing; an id outside the pool is skipped.
  int hint_page = 0;  // paged: the page of this split's first key, as the hints give it
  if (p.block_table != nullptr && warp == kWarpTma && lane == 0)
    hint_page = split * p.chunk / p.page_size;  // the host's chunk: exact for full lengths
  if (p.l2_prefetch && warp == kWarpTma && lane == 0 && p.chunk >= kBN) {
    const int len = min(max(ld_relaxed_s32(p.seqlens + b), 0), p.S_max);
    const int key0 =
        split * device_chunk(len, p.B, p.S_max, p.chunk, p.num_splits, p.H_kv, p.num_sms, kBN);
    int c2 = key0, c3 = b * p.H_kv + kv;
    bool go = key0 < len;
    if (p.block_table != nullptr) {
      const int page = key0 / p.page_size;
      hint_page = page;
      const int page_id =
          page < p.max_pages ? ld_relaxed_s32(p.block_table + (size_t)b * p.max_pages + page) : -1;
      go = go && page_id >= 0 && page_id < p.num_pages;
      c2 = key0 - page * p.page_size;
      c3 = page_id * p.H_kv + kv;
    }
    for (int half = 0; go && half < 2; ++half) {
      tma_prefetch_l2_4d(&tm_k, 0, half, c2, c3);
      tma_prefetch_l2_4d(&tm_v, 0, half, c2, c3);
    }
  }
  // Barriers and tensor memory are set up before the grid-dependency wait: none
  // of it reads another grid's output.
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full(i), 1);
      mbar_init(p_full(i), 128);
      mbar_init(o_final(i), 1);
      mbar_init(tok(i), 128);
    }
    mbar_init(drain_bar, 1);
    mbar_init(v_tail, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // inputs written by earlier grids are visible after this wait (coherent loads)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the row block of Q does not depend on the sequence length: its copy starts
  // before the length is read
  const uint64_t pol = l2_policy_evict_first();
  if (warp == kWarpTma && lane == 0) {
    const int q_row0 = (b * p.H_q + kv * p.G) * p.T_q;  // first (head, token) row of the group
    mbar_arrive_expect_tx(q_full, kTileBytes);
    for (int half = 0; half < 2; ++half)
      tma_load_4d(sbase + kOffQ + half * kHalfBytes, &tm_q, q_full, 0, half, q_row0, 0, pol);
  }
  // Paged: the producer warp loads the 32 block-table entries from the hinted
  // page on, alongside the length, so the first K/V copy does not wait for two
  // dependent loads in a row; the entries are read after the wait (only which
  // window to load came from the hints), and a window that misses the split's
  // pages is simply loaded again.
  int page_base = -(1 << 30), page_reg = 0;
  if (p.block_table != nullptr && warp == kWarpTma) {
    page_base = __shfl_sync(0xffffffffu, hint_page, 0);
    const int idx = page_base + lane;
    page_reg = idx < p.max_pages ? __ldca(p.block_table + (size_t)b * p.max_pages + idx) : 0;
  }
  const int seqlen_in = __ldca(p.seqlens + b);
  const int seqlen = min(max(seqlen_in, 0), p.S_max);
  // the chunk for the batch's actual lengths (the host's chunk when they are S_max)
  const int chunk =
      device_chunk(seqlen, p.B, p.S_max, p.chunk, p.num_splits, p.H_kv, p.num_sms, kBN);
  // out-of-range lengths are clamped and reported through the status word
  if ((seqlen_in < 0 || seqlen_in > p.S_max) && threadIdx.x == 0 && split == 0)
    atomicExch(p.wait.status, kStatusInvalidArg);
  const int key_begin = split * chunk;
  const int key_end = min(key_begin + chunk, seqlen);
  if (key_begin >= key_end) {  // empty split: the merge never reads it (CTA-uniform)
    if constexpr (kDirect) {  // the whole sequence is empty: O = 0, lse = -inf for its rows
      const size_t row0 = (size_t)(b * p.H_q + kv * p.G) * p.T_q;
      const int R = p.G * p.T_q;
      for (int i = threadIdx.x; i < R * (kD / 8); i += blockDim.x)
        if (store_ok(row0 + i / (kD / 8), (size_t)p.B * p.H_q * p.T_q, p.wait.status))
          reinterpret_cast<uint4 *>(p.o + (row0 + i / (kD / 8)) * kD)[i % (kD / 8)] =
              make_uint4(0u, 0u, 0u, 0u);
      for (int i = threadIdx.x; i < R; i += blockDim.x)
        if (store_ok(row0 + i, (size_t)p.B * p.H_q * p.T_q, p.wait.status))
          p.lse[row0 + i] = -INFINITY;
    }
    // no copy may still be in flight when the CTA exits
    if (warp == kWarpTma && lane == 0) wait_bar(q_full, 0, p.wait, abort_flag);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
      tc::fence_after_sync();
      tc::tmem_dealloc(tmem, kTmemCols);
    }
    return;
  }
  const int n_tiles = (key_end - key_begin + kBN - 1) / kBN;
  const int n_slot[2] = {(n_tiles + 1) / 2, n_tiles / 2};  // slot s: tiles j with j % 2 == s
  const int R = p.G * p.T_q;                                 // rows that are stored
  // the last tile may run past the sequence: its V rows there (cache rows that
  // may hold any bits) are cleared before P V reads them
  const int tail_keys = key_begin + n_tiles * kBN - seqlen;  // > 0: rows to clear

  if (warp == kWarpTma) {
    // ------------------------- TMA producer -------------------------
    // Lane 0 issues every copy.  With a paged cache the whole warp keeps 32
    // block-table entries in registers, so a tile's page is a shuffle away (a
    // 128-key tile never straddles pages: page sizes are multiples of 128).
    int ld = 0;
    bool ok = true;
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int key0 = key_begin + j * kBN;
      int c2 = key0, c3 = b * p.H_kv + kv;  // tensor-map coordinates of the tile's first key
      if (p.block_table != nullptr) {
        const int page = key0 / p.page_size;
        if (page - page_base >= 32 || page < page_base) {
          page_base = page;
          const int idx = page_base + lane;
          page_reg = idx < p.max_pages ? __ldca(p.block_table + (size_t)b * p.max_pages + idx) : 0;
        }
        const int page_id = __shfl_sync(0xffffffffu, page_reg, page - page_base);
        // a page id outside the pool reads zeros (a block past the tensor map:
        // TMA out-of-bounds fill); it is reported through the status word
        const bool bad = page_id < 0 || page_id >= p.num_pages;
        if (bad && lane == 0) atomicExch(p.wait.status, kStatusInvalidArg);
        c2 = key0 - page * p.page_size;
        c3 = bad ? p.num_pages * p.H_kv : page_id * p.H_kv + kv;
      }
      if (lane == 0) {
        for (int which = 0; which < 2; ++which, ++ld) {
          const int s = ld % kStages;
          if (!wait_bar(kv_empty(s), ((ld / kStages) & 1) ^ 1, p.wait, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t dst = sbase + kOffStage + s * kTileBytes;
          mbar_arrive_expect_tx(kv_full(s), kTileBytes);
          const CUtensorMap *map = which == 0 ? &tm_k : &tm_v;
          for (int half = 0; half < 2; ++half)
            tma_load_4d(dst + half * kHalfBytes, map, kv_full(s), 0, half, c2, c3, pol);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    ld = __shfl_sync(0xffffffffu, ld, 0);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok && tail_keys > 0) {
      // last V tile (load ld - 1): the warp zeroes rows [kBN - tail_keys, kBN) of
      // both halves once the copy has landed
      const int i = ld - 1;
      const bool landed = wait_bar(kv_full(i % kStages), (i / kStages) & 1, p.wait, abort_flag);
      if (__all_sync(0xffffffffu, landed)) {
        uint8_t *vt = smem + kOffStage + (i % kStages) * kTileBytes;
        const int first = kBN - tail_keys;
        for (int idx = lane; idx < tail_keys * 16; idx += 32) {  // 16 chunks of 16 B per row
          const int r = first + idx / 16, c = idx % 16;
          *reinterpret_cast<uint4 *>(vt + (c >> 3) * kHalfBytes + r * 128 + (c & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // the tensor core reads these rows
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(v_tail);
    }
    if (lane == 0) {
      for (int i = max(0, ld - kStages); i < ld; ++i)
        wait_bar(kv_full(i % kStages), (i / kStages) & 1, p.wait, abort_flag);
      wait_bar(q_full, 0, p.wait, abort_flag);
    }
  } else if (warp == kWarpMma) {
    // ------------------------- MMA issuer -------------------------
    // Step j: O_s += P_s(j-2) V(j-2), then S_s(j) = Q K(j)^T, with s = j % 2 (the
    // P V of a slot must precede the S that overwrites its P).
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kRows, kBN, 0);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(kRows, kD, 1);
      const uint32_t t_s[2] = {tmem + 0u, tmem + 128u};
      const uint32_t t_o[2] = {tmem + 256u, tmem + 384u};
      const uint64_t dq = desc_kmajor_base(sbase + kOffQ);
      bool ok = wait_bar(q_full, 0, p.wait, abort_flag);
      tc::fence_after_sync();
      for (int j = 0; ok && j < n_tiles + 2; ++j) {
        const int s = j & 1;
        if (j >= 2) {
          const int t = j - 2, ldV = 2 * t + 1;
          if (!wait_bar(kv_full(ldV % kStages), (ldV / kStages) & 1, p.wait, abort_flag) ||
              (t == n_tiles - 1 && tail_keys > 0 && !wait_bar(v_tail, 0, p.wait, abort_flag)) ||
              !wait_bar(p_full(s), (t >> 1) & 1, p.wait, abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint64_t dv = desc_mnmajor_base(sbase + kOffStage + (ldV % kStages) * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            tc::mma_ts(t_o[s], t_s[s] + kk * 8, tc::desc_advance(dv, mnmajor_step(kk)), idesc_pv,
                       (t >= 2 || kk > 0) ? 1u : 0u);
          tc::commit(kv_empty(ldV % kStages));
          if (t + 2 >= n_tiles) tc::commit(o_final(s));  // the slot's last tile
        }
        if (j < n_tiles) {
          const int ldK = 2 * j;
          if (!wait_bar(kv_full(ldK % kStages), (ldK / kStages) & 1, p.wait, abort_flag)) {
            ok = false;
            break;
          }
          const uint64_t dk = desc_kmajor_base(sbase + kOffStage + (ldK % kStages) * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            tc::mma_ss(t_s[s], tc::desc_advance(dq, kmajor_step(kk)),
                       tc::desc_advance(dk, kmajor_step(kk)), idesc_s, kk > 0 ? 1u : 0u);
          tc::commit(s_full(s));
          tc::commit(kv_empty(ldK % kStages));
        }
      }
      tc::commit(drain_bar);
      wait_bar(drain_bar, 0, p.wait, abort_flag);
    }
  } else {
    // ------------------------- softmax slots -------------------------
    const int s = warp >> 2;   // slot: key tiles of parity s
    const int wq = warp & 3;   // TMEM lane quarter
    const int row = 32 * wq + lane;
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    const uint32_t t_s = tmem + lane_off + 128u * s;
    const uint32_t t_o = tmem + lane_off + 256u + 128u * s;
    // keys this row may see: the causal limit of its token (rows past R see all)
    const int lim = row < R ? min(key_end, seqlen - p.T_q + row % p.T_q + 1) : key_end;
    const bool pos_scale = p.sl2 > 0.f;
    const float mul = pos_scale ? p.sl2 : 1.f;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int k = 0; ok && k < n_slot[s]; ++k) {
      const int key0 = key_begin + (2 * k + s) * kBN;
      bool ready = wait_bar(s_full(s), k & 1, p.wait, abort_flag);
      if (!__all_sync(0xffffffffu, ready)) { ok = false; break; }
      tc::fence_after_sync();
      uint32_t sv[kBN];
      // S row from tensor memory; keys the row may not see are -inf
      auto load_s = [&]() {
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::ld32(t_s + 32 * c, sv + 32 * c);
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::wait_ld32(sv + 32 * c);  // one wait; ties each chunk
        if (!pos_scale) {
#pragma unroll
          for (int e = 0; e < kBN; ++e) sv[e] = __float_as_uint(__uint_as_float(sv[e]) * p.sl2);
        }
        if (key0 + kBN > lim) {
#pragma unroll
          for (int e = 0; e < kBN; ++e)
            if (key0 + e >= lim) sv[e] = __float_as_uint(-INFINITY);
        }
      };
      load_s();
      auto row_max = [&]() {
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int e = 0; e < kBN; e += 8)
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            mx4[k4] = fmax3(mx4[k4], __uint_as_float(sv[e + 2 * k4]),
                            __uint_as_float(sv[e + 2 * k4 + 1]));
        const float mx = fmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
        return pos_scale ? mx * p.sl2 : mx;
      };
      // P = exp2(s * scale log2e - ref) as bf16 pairs, packed in place over the
      // scores (pair e goes to sv[e], whose score was already used); ref = 0 while
      // no key was seen
      auto exp_pass = [&]() {
        const float negm = m_ref == -INFINITY ? 0.f : -m_ref;
        const uint64_t mul2 = f32x2(mul, mul), negm2 = f32x2(negm, negm);
        uint64_t rs2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
        for (int e = 0; e < kBN / 2; ++e) {
          float x0, x1;
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])),
                                mul2, negm2),
                      x0, x1);
          const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
          rs2[e & 1] = add_f32x2(rs2[e & 1], f32x2(p0, p1));
          sv[e] = pack_bf16x2(p0, p1);
        }
        float a0, a1, a2, a3;
        f32x2_split(rs2[0], a0, a1);
        f32x2_split(rs2[1], a2, a3);
        return (a0 + a1) + (a2 + a3);
      };
      if (k == 0) m_ref = row_max();
      // exp turn: slot 0's tile k follows slot 1's tile k-1, slot 1's tile k follows
      // slot 0's tile k
      if (s == 0) {
        ready = k == 0 || wait_bar(tok(0), (k - 1) & 1, p.wait, abort_flag);
      } else {
        ready = wait_bar(tok(1), k & 1, p.wait, abort_flag);
      }
      if (!__all_sync(0xffffffffu, ready)) { ok = false; break; }
      float tsum = exp_pass();
      // the reference max moves only when a score exceeds it by more than the
      // threshold, which makes the tile's sum exceed 2^threshold (or not finite)
      if (k > 0 && __any_sync(0xffffffffu, !(tsum <= kSumTrigger))) {
        load_s();  // S is still in tensor memory (P not yet written over it)
        const float mt = row_max();
        if (__any_sync(0xffffffffu, mt > m_ref + kRescaleThreshold)) {
          const float m_new = fmaxf(m_ref, mt);
          const float corr = m_new == -INFINITY ? 1.f : fast_exp2(m_ref - m_new);  // 0 from -inf
          l *= corr;
          // O holds P V up to the slot's previous tile (complete: S was issued after it)
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            tc::ld32(t_o + 32 * c, r);
            tc::wait_ld32(r);
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * corr);
            tc::st32(t_o + 32 * c, r);
          }
          tc::wait_st();
          m_ref = m_new;
        }
        tsum = exp_pass();  // the scores were reloaded over P: P again (for m_ref)
      }
      // the other slot may use the exp unit now (slot 1 of an odd tile count has
      // no tile k = n_slot[0] - 1 to hand the token to: it is simply not awaited)
      mbar_arrive(tok(1 - s));
      tc::st32(t_s, sv);
      tc::st32(t_s + 32, sv + 32);
      tc::wait_st();
      l += tsum;
      tc::fence_before_sync();
      mbar_arrive(p_full(s));
    }
    // ---- epilogue: combine the two slots per row, write the split partial ----
    // Both slots' warps share it: after their (m, l) are exchanged through shared
    // memory, the warps of slot s combine and store columns [64 s, 64 s + 64) of
    // their 32 rows (eight warps storing instead of four).
    const bool has1 = n_slot[1] > 0;  // CTA-uniform: slot 1 holds a tile
    const bool live = ok && (s == 0 || has1);
    red_m[s * kRows + row] = live ? m_ref : -INFINITY;
    red_l[s * kRows + row] = live ? l : 0.f;
    ok = softmax_bar_and(ok);  // all 256 softmax threads; true only if every one is ok
    if (ok) {
      const bool ready = wait_bar(o_final(0), 0, p.wait, abort_flag) &&
                         (!has1 || wait_bar(o_final(1), 0, p.wait, abort_flag));
      ok = __all_sync(0xffffffffu, ready);
    }
    if (ok) {
      tc::fence_after_sync();
      const float m0 = red_m[row], l0 = red_l[row];
      const float m1 = red_m[kRows + row], l1 = red_l[kRows + row];
      const float mx = fmaxf(l0 > 0.f ? m0 : -INFINITY, l1 > 0.f ? m1 : -INFINITY);
      const float w0 = l0 > 0.f ? fast_exp2(m0 - mx) : 0.f;
      const float w1 = l1 > 0.f ? fast_exp2(m1 - mx) : 0.f;
      const float L = w0 * l0 + w1 * l1;
      const float inv = L > 0.f ? fast_rcp(L) : 0.f;  // L >= 1: the larger slot weighs 1
      const float c0 = w0 * inv, c1 = w1 * inv;  // 0 for a slot with no visible key
      // rows past G * T_q belong to other heads' queries: computed, never stored
      const size_t row0 = (size_t)(b * p.H_q + kv * p.G) * p.T_q;  // the group's first row
      const size_t n_part_rows = (size_t)p.B * p.H_q * p.T_q * p.num_splits;
      // (one split written directly: the partial row is the output row, o and lse)
      if (s == 0 && row < R && store_ok((row0 + row) * p.num_splits + split, n_part_rows,
                                        p.wait.status))
        (kDirect ? p.lse : p.lse_part)[(row0 + row) * p.num_splits + split] =
            L > 0.f ? (mx + fast_log2(L)) * 0.69314718055994531f : -INFINITY;
      // The combined rows go through shared memory so that the global stores are
      // contiguous 256-byte row halves: a thread holds one row, and storing it
      // directly would make every warp store touch 32 rows.  The ring is idle
      // here (both slots' last P V completed, so every copy has landed and every
      // MMA that read a stage is done).  Each warp stages its 32 rows x 64
      // columns (8 KiB), 16-byte chunk ch of row i at chunk slot ch ^ (i & 7)
      // (conflict-free both ways).
      uint8_t *stage = smem + kOffStage + (4 * s + wq) * (32 * 64 * 4);
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * s + cc;  // 32-column chunk of O
        uint32_t r0[32], r1[32];
        tc::ld32(t_o - 128u * s + 32 * c, r0);          // slot 0's O
        if (has1) tc::ld32(t_o - 128u * s + 128u + 32 * c, r1);  // slot 1's O
        tc::wait_ld32(r0);            // waits for both loads; ties r0's registers to it
        if (has1) tc::wait_ld32(r1);  // (already complete) ties r1's
        // both slots' O are finite (every slot with a tile wrote its O, and V
        // rows past the sequence were cleared); a slot with no tile is skipped
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float4 v;
          v.x = c0 * __uint_as_float(r0[4 * e + 0]);
          v.y = c0 * __uint_as_float(r0[4 * e + 1]);
          v.z = c0 * __uint_as_float(r0[4 * e + 2]);
          v.w = c0 * __uint_as_float(r0[4 * e + 3]);
          if (has1) {
            v.x = fmaf(c1, __uint_as_float(r1[4 * e + 0]), v.x);
            v.y = fmaf(c1, __uint_as_float(r1[4 * e + 1]), v.y);
            v.z = fmaf(c1, __uint_as_float(r1[4 * e + 2]), v.z);
            v.w = fmaf(c1, __uint_as_float(r1[4 * e + 3]), v.w);
          }
          const int ch = 8 * cc + e;  // 16-byte chunk of the warp's 64 columns
          *reinterpret_cast<float4 *>(stage + lane * 256 + ((ch ^ (lane & 7)) * 16)) = v;
        }
      }
      __syncwarp();
      // two rows per step: lanes 0-15 store row 2 it, lanes 16-31 row 2 it + 1,
      // lane l its 16-byte chunk l % 16 of the row's 256-byte half
#pragma unroll 4
      for (int it = 0; it < 16; ++it) {
        const int i = 2 * it + (lane >> 4), k = lane & 15;
        const int r = 32 * wq + i;
        const size_t prow = (row0 + r) * p.num_splits + split;
        if (r < R && store_ok(prow, n_part_rows, p.wait.status)) {
          const float4 x = *reinterpret_cast<const float4 *>(stage + i * 256 + ((k ^ (i & 7)) * 16));
          if constexpr (kDirect) {
            uint2 pk;
            pk.x = pack_bf16x2(x.x, x.y);
            pk.y = pack_bf16x2(x.z, x.w);
            reinterpret_cast<uint2 *>(p.o + prow * kD + 64 * s)[k] = pk;
          } else {
            reinterpret_cast<float4 *>(p.o_part + prow * kD + 64 * s)[k] = x;
          }
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  // this CTA's partials are written: the merge grid may be scheduled
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// dims (innermost first): 64 columns, 2 column halves, rows, blocks
CUresult make_map(CUtensorMap *map, const uint16_t *base, long long rows, long long blocks,
                  PFN_cuTensorMapEncodeTiled_v12000 encode) {
  const cuuint64_t dims[4] = {64, 2, (cuuint64_t)rows, (cuuint64_t)blocks};
  const cuuint64_t strides[3] = {128, 256, (cuuint64_t)rows * 256};
  const cuuint32_t box[4] = {64, 1, 128, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t *>(base), dims,
                strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace decode_tc

cudaError_t decode_tc_prepare_device() {
  const cudaError_t e = cudaFuncSetAttribute(decode_tc::decode_tc_kernel<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             decode_tc::kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_tc::decode_tc_kernel<true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, decode_tc::kSmemBytes);
}

cudaError_t decode_tc_split_launch(const DecodeLaunch &a, cudaStream_t stream,
                                   PFN_cuTensorMapEncodeTiled_v12000 encode) {
  using namespace decode_tc;
  if (a.S_max <= 0) return cudaSuccess;
  const bool paged = a.block_table != nullptr;
  if (a.chunk % kBN != 0 || (paged && (a.page_size <= 0 || a.page_size % kBN != 0)))
    return cudaErrorInvalidValue;
  // K/V blocks of rows: one per (sequence, KV head) of S_max keys, or one per
  // (page, KV head) of page_size keys
  const long long kv_blocks = paged ? (long long)a.num_pages * a.H_kv : (long long)a.B * a.H_kv;
  const int kv_rows = paged ? a.page_size : a.S_max;
  CUtensorMap tm_q, tm_k, tm_v;
  const long long q_rows = (long long)a.B * a.H_q * a.T_q;
  if (make_map(&tm_q, a.q, q_rows, 1, encode) != CUDA_SUCCESS ||
      make_map(&tm_k, a.k_cache, kv_rows, kv_blocks, encode) != CUDA_SUCCESS ||
      make_map(&tm_v, a.v_cache, kv_rows, kv_blocks, encode) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  Params p;
  p.seqlens = a.seqlens;
  p.block_table = a.block_table;
  p.page_size = a.page_size;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.l2_prefetch = (long long)a.num_splits * a.H_kv * a.B <= a.num_sms;
  p.o_part = a.o_part;
  p.lse_part = a.lse_part;
  p.o = a.o;
  p.lse = a.lse;
  p.B = a.B;
  p.H_q = a.H_q;
  p.H_kv = a.H_kv;
  p.G = a.H_q / a.H_kv;
  p.T_q = a.T_q;
  p.S_max = a.S_max;
  p.num_splits = a.num_splits;
  p.chunk = a.chunk;
  p.num_sms = a.num_sms;
  p.sl2 = a.scale * 1.4426950408889634f;
  p.wait = a.wait;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.H_kv, a.B, a.num_splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.direct_out && a.num_splits == 1)
    return cudaLaunchKernelEx(&cfg, decode_tc_kernel<true>, tm_q, tm_k, tm_v, p);
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel<false>, tm_q, tm_k, tm_v, p);
}

}  // namespace gqa
