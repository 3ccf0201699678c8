// prefill_pair.cu -- causal GQA prefill on CTA pairs (tcgen05 cta_group::2) for sm_103a.
//
// What it computes: exactly what prefill_causal.cu computes (design record
// "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", section 3's per-tile
// online softmax with section 5.4's tile classes: past key tiles unmasked, the
// boundary tiles masked, future tiles never loaded; query row i at absolute
// position q_offset + i).  Used when the group size G is a multiple of 4.
//
// GB300 mapping
//   * Clusters of two CTAs (one per SM) share every tensor-core instruction:
//     M = 256 rows, 128 from each CTA.  A work unit is one 128-row query tile of
//     FOUR query heads of one KV group; cluster rank r holds heads 4q + r
//     (slot 0) and 4q + 2 + r (slot 1).  One MMA computes S for slot s of both
//     CTAs at once: A = the two CTAs' Q tiles of that slot, B = the K tile,
//     whose 128 keys are split 64 / 64 between the CTAs; O += P V takes P from
//     each CTA's tensor memory and V split by columns (d 0..63 in rank 0,
//     64..127 in rank 1).  Per SM and key tile this moves half the K/V bytes of
//     the single-CTA kernel and runs the wider instruction, which sustains a
//     higher rate on this GPU (measured: S 6127 vs 5287, P V 5896 vs 4308
//     flop/clk/SM for back-to-back instructions).
//   * Each CTA: warps 0-3 and 4-7 softmax for slots 0 and 1 (one thread per
//     query row, the whole S row in registers), warp 8 TMA producer (its own halves of Q, K
//     and V; completion counted on rank 0's barriers), warp 9 TMEM allocation
//     (both CTAs) and, in rank 0 only, the single thread that issues every
//     tcgen05.mma and commit (completion multicast to both CTAs).
//   * TMEM per CTA: S0, S1, O0, O1 (128 columns each); P overwrites its S block
//     as bf16 and feeds P V from tensor memory.
//   * Ordering across the pair: rank 1's TMA loads complete on rank 0's "full"
//     barriers (rank 0 posts the byte count of both halves); each softmax warp
//     arrives once on rank 0's "P ready" barrier (remotely from rank 1), after
//     its lanes' tensor-memory stores have completed; everything the tensor core finishes is signalled to both CTAs by
//     multicast commits.  Every wait is bounded.
#include <cudaTypedefs.h>
#include <math.h>

#include "device_common.cuh"
#include "kernels.h"
#include "prefill_split.cuh"
#include "tcgen05.cuh"

namespace gqa {
namespace prefill_pair {

constexpr int kD = 128;
constexpr int kBM = 128;                  // query rows per tile (per CTA)
constexpr int kBN = 128;                  // keys per tile
constexpr int kHalfKeys = kBN / 2;        // keys of a K tile held by one CTA
constexpr int kStages = 6;                // ring of 16 KiB stages (a K half or a V half)
constexpr int kWarpTma = 8, kWarpMma = 9;
constexpr int kThreads = 320;
constexpr int kQBytes = kBM * kD * 2;     // 32 KiB per slot
constexpr int kQHalfBytes = kQBytes / 2;  // one 64-column half: [128 rows x 128 B]
constexpr int kStageBytes = 16384;        // K half: 2 x [64 rows x 128 B]; V half: [128 rows x 128 B]
constexpr int kKHalfColBytes = kHalfKeys * 128;  // 8 KiB: one 64-column half of the K half
constexpr int kOffQ = 0;
constexpr int kOffStage = 2 * kQBytes;
constexpr int kOffBar = kOffStage + kStages * kStageBytes;
// barriers: kv_full[S], kv_empty[S], q_full[2], q_empty, s_full[2], p_full[2], o_final[2],
// drain
constexpr int kNumBars = 2 * kStages + 2 + 1 + 2 + 2 + 2 + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base slot, abort flag
constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + 1024 alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units (a factor of 256)
constexpr float kSumTrigger = 256.0f;      // 2^kRescaleThreshold
constexpr uint16_t kBothCtas = 0x3;

static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Params {
  uint16_t *o;
  float *lse;
  int B, H_q, H_kv, G, T_q, S_kv, q_offset;
  int n_qtiles, n_quads, n_items, n_pairs;
  // Key-range split of the last round: items [0, n_full) are whole units; the
  // units after them are each cut into split_s pieces (items n_full + t, piece
  // t), whose partials go to ws_o / ws_ml and are combined by the merge kernel.
  int n_full, split_s;
  float *ws_o;   // [piece][4 heads][128 rows][128] fp32, O not yet divided by l
  float *ws_ml;  // [piece][4 heads][128 rows][2] fp32: m (log2 units), l
  float sl2;     // scale * log2(e)
  WaitCtl wait;
};

struct Unit {
  int b, kv, qt, quad, n_kv;
  int kv_lo, kv_hi;  // key tiles of this item: [kv_lo, kv_hi)
  int piece;         // -1: a whole unit, O and lse final; else its partial slot
};

// Item of round k for worker w of P: items are sorted longest first and dealt
// in snake order (left to right, then right to left), so no worker takes the
// longest item of every round; only the last round can be partial.
__device__ __forceinline__ int snake_unit(int k, int w, int P) {
  return k * P + ((k & 1) ? P - 1 - w : w);
}

__device__ __forceinline__ Unit unit_at(const Params &p, int item) {
  Unit w;
  int u = item;
  w.piece = -1;
  if (item >= p.n_full) {
    const int t = item - p.n_full;
    u = p.n_full + t / p.split_s;
    w.piece = t;
  }
  const int per_qt = p.B * p.H_kv * p.n_quads;
  w.qt = p.n_qtiles - 1 - u / per_qt;  // latest (longest) query tiles first
  int r = u % per_qt;
  w.quad = r % p.n_quads;
  r /= p.n_quads;
  w.kv = r % p.H_kv;
  w.b = r / p.H_kv;
  const int qe = min((w.qt + 1) * kBM, p.T_q);
  // key tiles up to the one of the tile's last query row (rows past the last key
  // see every key: no tile past the keys)
  w.n_kv = min((p.q_offset + qe - 1) / kBN + 1, (p.S_kv + kBN - 1) / kBN);
  w.kv_lo = 0;
  w.kv_hi = w.n_kv;
  if (w.piece >= 0) {
    const int i = w.piece % p.split_s;
    w.kv_lo = prefill_split::piece_start(i, p.split_s, w.n_kv);
    w.kv_hi = prefill_split::piece_start(i + 1, p.split_s, w.n_kv);
  }
  return w;
}

// Query head held by cluster rank `rank` in slot `slot` of unit w.
__device__ __forceinline__ int head_of(const Params &p, const Unit &w, int rank, int slot) {
  return w.kv * p.G + 4 * w.quad + 2 * slot + rank;
}

// Bounded wait with cluster-scope acquire; gives up when the CTA's abort flag is
// raised or the limit passes (recording the timeout).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const WaitCtl &ctl,
                                         volatile int *abort_flag) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > ctl.timeout_ns) {
      atomicExch(ctl.status, kStatusTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

// Operand descriptors: built once per tile, then advanced by the k-step's byte
// offset (a compile-time constant), which keeps the MMA thread's work between
// tensor-core instructions to a single add.
// Q tile: K-major, two 64-column halves of 128 rows; k-step kk = 16 columns of d.
__device__ __forceinline__ uint64_t desc_q_base(uint32_t tile) {
  return tc::smem_desc_sw128(tile, 16, 1024);
}
__device__ __forceinline__ constexpr uint32_t q_step(int kk) {
  return (kk >> 2) * kQHalfBytes + (kk & 3) * 32;
}
// K half (64 keys): K-major, two 64-column halves of 64 rows.
__device__ __forceinline__ uint64_t desc_k_base(uint32_t tile) {
  return tc::smem_desc_sw128(tile, 16, 1024);
}
__device__ __forceinline__ constexpr uint32_t k_step(int kk) {
  return (kk >> 2) * kKHalfColBytes + (kk & 3) * 32;
}
// V half: MN-major, 128 key rows of 64 d (one 64-element block); k-step kk = 16 keys.
__device__ __forceinline__ uint64_t desc_v_base(uint32_t tile) {
  return tc::smem_desc_sw128(tile, kStageBytes, 1024);
}
__device__ __forceinline__ constexpr uint32_t v_step(int kk) { return kk * 2048; }

using prefill_split::PageArgs;

// kPaged: K/V in pages through pg.block_table (a separate instantiation; the
// dense kernel's parameters are unchanged).  Used only when S_kv is a multiple
// of 128, so every key tile the pair loads holds keys of the sequence and no
// row of a page's unused tail is ever multiplied.
template <bool kPaged>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const Params p,
                        const PageArgs<kPaged> pg) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBar;
  auto kv_full = [&](int s) { return bar0 + 8u * s; };
  auto kv_empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto q_full = [&](int i) { return bar0 + 8u * (2 * kStages + i); };
  const uint32_t q_empty = bar0 + 8u * (2 * kStages + 2);
  auto s_full = [&](int i) { return bar0 + 8u * (2 * kStages + 3 + i); };
  auto p_full = [&](int i) { return bar0 + 8u * (2 * kStages + 5 + i); };
  auto o_final = [&](int i) { return bar0 + 8u * (2 * kStages + 7 + i); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 9);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();  // 0: issues the MMAs; 1: its peer
  const bool leader = rank == 0;
  const int pair_id = blockIdx.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full(i), 1);
      mbar_init(s_full(i), 1);
      mbar_init(p_full(i), 4 + 4);  // the slot's four softmax warps in each CTA
      mbar_init(o_final(i), 1);
    }
    mbar_init(q_empty, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tc::tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tc::tmem_relinquish_pair();
  }
  tc::fence_before_sync();
  cluster_sync();  // both CTAs' barriers and TMEM exist before any cross-CTA use
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTma) {
    // ------------------------- TMA producer (both CTAs) -------------------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      int ld = 0, it = 0;
      bool ok = true;
      for (int k = 0; ok; ++k, ++it) {
        const int u = snake_unit(k, pair_id, p.n_pairs);
        if (u >= p.n_items) break;
        const Unit w = unit_at(p, u);
        if (!wait_bar(q_empty, (it & 1) ^ 1, p.wait, abort_flag)) { ok = false; break; }
        for (int i = 0; i < 2; ++i) {
          const uint32_t full = dsmem_addr(q_full(i), 0);  // rank 0's barrier
          if (leader) mbar_arrive_expect_tx(q_full(i), 2 * kQBytes);
          const uint32_t dst = sbase + kOffQ + i * kQBytes;
          const int h = head_of(p, w, rank, i);
          for (int half = 0; half < 2; ++half)
            tma_load_4d_pair(dst + half * kQHalfBytes, &tm_q, full, 0, half, w.qt * kBM,
                             w.b * p.H_q + h, pol_q);
        }
        const int kv_row = w.b * p.H_kv + w.kv;
        // the next unit's Q is pulled into L2 a few key tiles before this unit
        // ends, so its copy at the unit change reads L2 rather than HBM
        const int u_next = snake_unit(k + 1, pair_id, p.n_pairs);
        const int j_pf = max(w.kv_lo, w.kv_hi - 4);
        for (int j = w.kv_lo; ok && j < w.kv_hi; ++j) {
          if (j == j_pf && u_next < p.n_items) {
            const Unit wn = unit_at(p, u_next);
            for (int i = 0; i < 2; ++i)
              for (int half = 0; half < 2; ++half)
                tma_prefetch_l2_4d(&tm_q, 0, half, wn.qt * kBM, wn.b * p.H_q + head_of(p, wn, rank, i));
          }
          for (int which = 0; which < 2; ++which, ++ld) {
            const int s = ld % kStages;
            if (!wait_bar(kv_empty(s), ((ld / kStages) & 1) ^ 1, p.wait, abort_flag)) {
              ok = false;
              break;
            }
            const uint32_t full = dsmem_addr(kv_full(s), 0);
            if (leader) mbar_arrive_expect_tx(kv_full(s), 2 * kStageBytes);
            const uint32_t dst = sbase + kOffStage + s * kStageBytes;
            int key0 = j * kBN, blk = kv_row;  // the tile's first key row and block
            if constexpr (kPaged) {
              // a 128-key tile lies in one page (page sizes are multiples of 128); a
              // page id outside the pool reads zeros (a block past the tensor map)
              // and is reported through the status word
              const int page = j * kBN / pg.page_size;
              const int page_id = __ldca(pg.block_table + (size_t)w.b * pg.max_pages + page);
              const bool bad = page_id < 0 || page_id >= pg.num_pages;
              if (bad) atomicExch(p.wait.status, kStatusInvalidArg);
              key0 = j * kBN - page * pg.page_size;
              blk = bad ? pg.num_pages * p.H_kv : page_id * p.H_kv + w.kv;
            }
            if (which == 0) {  // K: keys j*128 + 64*rank .. +63, all of d
              for (int half = 0; half < 2; ++half)
                tma_load_4d_pair(dst + half * kKHalfColBytes, &tm_k, full, 0, half,
                                 key0 + kHalfKeys * rank, blk, pol_kv);
            } else {  // V: keys j*128 .. +127, d 64*rank .. +63
              tma_load_4d_pair(dst, &tm_v, full, 0, rank, key0, blk, pol_kv);
            }
          }
        }
      }
      // No copy may still be in flight when the CTA exits: rank 0 sees its full
      // barriers complete; rank 1 sees the tensor core release each of its last
      // stages (a stage is released only after both halves were loaded and used).
      for (int i = max(0, ld - kStages); i < ld; ++i) {
        if (leader)
          wait_bar(kv_full(i % kStages), (i / kStages) & 1, p.wait, abort_flag);
        else
          wait_bar(kv_empty(i % kStages), (i / kStages) & 1, p.wait, abort_flag);
      }
      if (!leader && it > 0) wait_bar(q_empty, (it - 1) & 1, p.wait, abort_flag);
    }
  } else if (warp == kWarpMma) {
    // ------------------------- MMA issuer (rank 0, one thread) -------------------------
    if (leader && lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(2 * kBM, kBN, 0);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(2 * kBM, kD, 1);
      const uint32_t t_s[2] = {tmem + 0u, tmem + 128u};
      const uint32_t t_o[2] = {tmem + 256u, tmem + 384u};
      const uint64_t dq0 = desc_q_base(sbase + kOffQ), dq1 = desc_q_base(sbase + kOffQ + kQBytes);
      int ld_base = 0, tile_base = 0, it = 0;
      bool ok = true;
      for (int k = 0; ok; ++k, ++it) {
        const int u = snake_unit(k, pair_id, p.n_pairs);
        if (u >= p.n_items) break;
        const Unit w = unit_at(p, u);
        const int n = w.kv_hi - w.kv_lo;
        for (int i = 0; ok && i < 2; ++i)
          if (!wait_bar(q_full(i), it & 1, p.wait, abort_flag)) ok = false;
        tc::fence_after_sync();
        for (int j = 0; ok && j <= n; ++j) {
          const int ldK = ld_base + 2 * j, ldV = ld_base + 2 * (j - 1) + 1;
          const uint64_t dk = desc_k_base(sbase + kOffStage + (ldK % kStages) * kStageBytes);
          const uint64_t dv = desc_v_base(sbase + kOffStage + (ldV % kStages) * kStageBytes);
          if (j < n && !wait_bar(kv_full(ldK % kStages), (ldK / kStages) & 1, p.wait, abort_flag)) {
            ok = false;
            break;
          }
          if (j > 0 && !wait_bar(kv_full(ldV % kStages), (ldV / kStages) & 1, p.wait, abort_flag)) {
            ok = false;
            break;
          }
          for (int i = 0; i < 2; ++i) {
            if (j > 0) {  // O_i += P_i V_{j-1}, P_i read from each CTA's tensor memory
              if (!wait_bar(p_full(i), (tile_base + j - 1) & 1, p.wait, abort_flag)) {
                ok = false;
                break;
              }
              tc::fence_after_sync();
#pragma unroll
              for (int kk = 0; kk < kBN / 16; ++kk)
                tc::mma_ts_pair(t_o[i], t_s[i] + kk * 8, tc::desc_advance(dv, v_step(kk)), idesc_pv,
                                (j > 1 || kk > 0) ? 1u : 0u);
              if (i == 1) tc::commit_pair(kv_empty(ldV % kStages), kBothCtas);
              if (j == n) tc::commit_pair(o_final(i), kBothCtas);
            }
            if (j < n) {  // S_i = Q_i K_j^T
#pragma unroll
              for (int kk = 0; kk < kD / 16; ++kk)
                tc::mma_ss_pair(t_s[i], tc::desc_advance(i == 0 ? dq0 : dq1, q_step(kk)),
                                tc::desc_advance(dk, k_step(kk)), idesc_s, kk > 0 ? 1u : 0u);
              tc::commit_pair(s_full(i), kBothCtas);
              count_s_tiles(p.wait, 2);  // one query head in each CTA of the pair
              if (i == 1) {
                tc::commit_pair(kv_empty(ldK % kStages), kBothCtas);
                if (j == n - 1) tc::commit_pair(q_empty, kBothCtas);
              }
            }
          }
        }
        ld_base += 2 * n;
        tile_base += n;
      }
      // every issued MMA must finish before either CTA releases TMEM or exits
      tc::commit_pair(drain_bar, kBothCtas);
    }
    if (lane == 0) wait_bar(drain_bar, 0, p.wait, abort_flag);
  } else {
    // ------------------------- softmax warpgroups (both CTAs) -------------------------
    const int i = warp >> 2;  // slot
    const int wq = warp & 3;  // TMEM lane quarter of this warp
    const int row = 32 * wq + lane;
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    const uint32_t t_s = tmem + lane_off + 128u * i;
    const uint32_t t_o = tmem + lane_off + 256u + 128u * i;
    const uint32_t p_ready = dsmem_addr(p_full(i), 0);  // rank 0's barrier
    const bool pos_scale = p.sl2 > 0.f;
    const float mul = pos_scale ? p.sl2 : 1.f;  // multiplier still owed by the held scores
    int tile = 0, it = 0;
    bool ok = true;
    for (int k = 0; ok; ++k, ++it) {
      const int u = snake_unit(k, pair_id, p.n_pairs);
      if (u >= p.n_items) break;
      const Unit w = unit_at(p, u);
      const int q0 = p.q_offset + w.qt * kBM;  // absolute position of row 0 of the tile
      const int qpos = q0 + row;
      float m_ref = -INFINITY, l = 0.f;
      for (int j = w.kv_lo; j < w.kv_hi; ++j, ++tile) {
        bool ready = wait_bar(s_full(i), tile & 1, p.wait, abort_flag);
        if (!__all_sync(0xffffffffu, ready)) { ok = false; break; }
        tc::fence_after_sync();
        // The S row is streamed from tensor memory in four 32-column chunks (the
        // next chunk's load in flight while this one is used); keys the row may
        // not see are -inf.
        const bool masked = (j * kBN + kBN - 1 > q0) || (j * kBN + kBN > p.S_kv);
        const int lim = min(qpos + 1, p.S_kv) - j * kBN;  // keys [0, lim) of the tile visible
        auto prep = [&](uint32_t *v, int c) {
          tc::wait_ld32(v);
          if (!pos_scale) {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * p.sl2);
          }
          if (masked) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * c + e >= lim) v[e] = __float_as_uint(-INFINITY);
          }
        };
        // Row max over the 128 scores (three-input max), in the units of m_ref.
        auto row_max = [&]() {
          uint32_t va[32], vb[32];
          float mx = -INFINITY;
          tc::ld32(t_s, va);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t *v = (c & 1) ? vb : va;
            prep(v, c);
            if (c + 1 < 4) tc::ld32(t_s + 32 * (c + 1), (c & 1) ? va : vb);
            float m2[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int e = 0; e < 32; e += 4)
#pragma unroll
              for (int k = 0; k < 2; ++k)
                m2[k] = fmax3(m2[k], __uint_as_float(v[e + 2 * k]), __uint_as_float(v[e + 2 * k + 1]));
            mx = fmax3(mx, m2[0], m2[1]);
          }
          return pos_scale ? mx * p.sl2 : mx;
        };
        // P = exp2(s * scale log2e - m_ref) as bf16 pairs into pk for the 32 scores
        // of chunk c; returns their sum.  The argument and the sums use packed
        // fp32x2 instructions (two keys each).
        uint32_t pk[kBN / 2];
        auto exp_chunk = [&](const uint32_t *v, int c) {
          const float negm = -m_ref;
          const uint64_t mul2 = f32x2(mul, mul), negm2 = f32x2(negm, negm);
          uint64_t rs2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float x0, x1;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])),
                                  mul2, negm2),
                        x0, x1);
            const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
            rs2[e & 1] = add_f32x2(rs2[e & 1], f32x2(p0, p1));
            pk[16 * c + e] = pack_bf16x2(p0, p1);
          }
          float a, b, c2, d;
          f32x2_split(rs2[0], a, b);
          f32x2_split(rs2[1], c2, d);
          return (a + b) + (c2 + d);
        };
        // the same over the whole row, streamed from tensor memory chunk by chunk
        auto exp_streamed = [&]() {
          uint32_t va[32], vb[32];
          float sum = 0.f;
          tc::ld32(t_s, va);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t *v = (c & 1) ? vb : va;
            prep(v, c);
            if (c + 1 < 4) tc::ld32(t_s + 32 * (c + 1), (c & 1) ? va : vb);
            sum += exp_chunk(v, c);
          }
          return sum;
        };
        // common path: the whole row in registers (one load wait)
        uint32_t sv[kBN];
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::ld32(t_s + 32 * c, sv + 32 * c);
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::wait_ld32(sv + 32 * c);  // one wait; ties each chunk
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (!pos_scale) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              sv[32 * c + e] = __float_as_uint(__uint_as_float(sv[32 * c + e]) * p.sl2);
          }
          if (masked) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * c + e >= lim) sv[32 * c + e] = __float_as_uint(-INFINITY);
          }
        }
        if (j == w.kv_lo) {  // its first key is visible to every row: finite
          float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int e = 0; e < kBN; e += 8)
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
              mx4[k4] = fmax3(mx4[k4], __uint_as_float(sv[e + 2 * k4]),
                              __uint_as_float(sv[e + 2 * k4 + 1]));
          const float mx = fmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
          m_ref = pos_scale ? mx * p.sl2 : mx;
        }
        // The two slots' exp passes run whenever their scores are ready: handing
        // the exp unit from one slot to the other (a token barrier) measured
        // slower (8K causal 783 -> 804 us, chunked 1470 -> 1520 us).
        float tsum = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) tsum += exp_chunk(sv + 32 * c, c);
        // The reference max only moves when a score exceeds it by more than the
        // threshold; such a score alone makes the tile's sum exceed 2^threshold,
        // so the row max is computed only when a sum does (or is not finite).
        if (j > w.kv_lo && __any_sync(0xffffffffu, !(tsum <= kSumTrigger))) {
          const float mt = row_max();  // S is still in tensor memory (P not yet written)
          if (__any_sync(0xffffffffu, mt > m_ref + kRescaleThreshold)) {
            const float m_new = fmaxf(m_ref, mt);
            const float corr = fast_exp2(m_ref - m_new);
            l *= corr;
            // O_i holds P V up to tile j-1 (complete: S_i(j) was issued after it)
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
            tsum = exp_streamed();
          }
        }
        tc::st32(t_s, pk);
        tc::st32(t_s + 32, pk + 32);
        tc::wait_st();
        l += tsum;
        tc::fence_before_sync();
        __syncwarp();  // one arrival per warp, after all its lanes' P stores
        if (lane == 0) {
          if (leader)
            mbar_arrive(p_full(i));
          else
            mbar_arrive_remote(p_ready);
        }
      }
      if (!ok) break;
      // epilogue: O / l -> bf16, lse = m_ref ln2 + ln l
      const bool ready = wait_bar(o_final(i), it & 1, p.wait, abort_flag);
      if (!__all_sync(0xffffffffu, ready)) { ok = false; break; }
      tc::fence_after_sync();
      const int h = head_of(p, w, rank, i);
      const int qrow = w.qt * kBM + row;
      const size_t orow = ((size_t)w.b * p.H_q + h) * p.T_q + qrow;
      uint32_t ov[kD];
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) tc::ld32(t_o + 32 * c, ov + 32 * c);
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) tc::wait_ld32(ov + 32 * c);
      if (qrow < p.T_q && w.piece >= 0) {
        // a piece of a split unit: its partial (O not yet divided, m, l) for the merge
        const size_t prow = prefill_split::partial_row(w.piece, 4, 2 * i + rank, row);
        if (store_ok(prow, (size_t)(p.n_items - p.n_full) * 4 * kBM, p.wait.status)) {
          float4 *dst = reinterpret_cast<float4 *>(p.ws_o + prow * kD);
#pragma unroll
          for (int v4 = 0; v4 < kD / 4; ++v4)
            dst[v4] = make_float4(__uint_as_float(ov[4 * v4 + 0]), __uint_as_float(ov[4 * v4 + 1]),
                                  __uint_as_float(ov[4 * v4 + 2]), __uint_as_float(ov[4 * v4 + 3]));
          reinterpret_cast<float2 *>(p.ws_ml)[prow] = make_float2(m_ref, l);
        }
      } else if (qrow < p.T_q && store_ok(orow, (size_t)p.B * p.H_q * p.T_q, p.wait.status)) {
        const float inv_l = 1.f / l;
        uint4 *dst = reinterpret_cast<uint4 *>(p.o + orow * kD);
#pragma unroll
        for (int v8 = 0; v8 < kD / 8; ++v8) {
          uint4 pk4;
          pk4.x = pack_bf16x2(__uint_as_float(ov[8 * v8 + 0]) * inv_l,
                              __uint_as_float(ov[8 * v8 + 1]) * inv_l);
          pk4.y = pack_bf16x2(__uint_as_float(ov[8 * v8 + 2]) * inv_l,
                              __uint_as_float(ov[8 * v8 + 3]) * inv_l);
          pk4.z = pack_bf16x2(__uint_as_float(ov[8 * v8 + 4]) * inv_l,
                              __uint_as_float(ov[8 * v8 + 5]) * inv_l);
          pk4.w = pack_bf16x2(__uint_as_float(ov[8 * v8 + 6]) * inv_l,
                              __uint_as_float(ov[8 * v8 + 7]) * inv_l);
          dst[v8] = pk4;
        }
        p.lse[orow] = m_ref * 0.69314718055994531f + logf(l);
      }
      tc::fence_before_sync();  // O reads done before the next unit's first P signal
    }
  }

  tc::fence_before_sync();
  cluster_sync();  // neither CTA releases TMEM or leaves while the pair still works
  if (warp == kWarpMma) {
    tc::fence_after_sync();
    tc::tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// Output row of head slot hl (2 * slot + rank) of work item `item`, row `row`.
__device__ __forceinline__ bool piece_out_row(const Params &p, int item, int hl, int row,
                                              size_t *orow) {
  const Unit w = unit_at(p, item);
  const int qrow = w.qt * kBM + row;
  if (qrow >= p.T_q) return false;
  *orow = ((size_t)w.b * p.H_q + head_of(p, w, hl & 1, hl >> 1)) * p.T_q + qrow;
  return true;
}

// dims (innermost first): 64 columns, 2 column halves, rows, heads; box of
// `box_rows` rows of one 64-column half.
CUresult make_map(CUtensorMap *map, const uint16_t *base, int rows, int heads, int box_rows,
                  PFN_cuTensorMapEncodeTiled_v12000 encode) {
  const cuuint64_t dims[4] = {64, 2, (cuuint64_t)rows, (cuuint64_t)heads};
  const cuuint64_t strides[3] = {128, 256, (cuuint64_t)rows * 256};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t *>(base), dims,
                strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace prefill_pair

cudaError_t prefill_pair_prepare_device(int *max_pairs) {
  using namespace prefill_pair;
  *max_pairs = 0;
  cudaError_t e = cudaFuncSetAttribute(prefill_pair_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(prefill_pair_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  // clusters of two the device runs at once (each CTA takes a whole SM)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, prefill_pair_kernel<false>, &cfg) == cudaSuccess)
    *max_pairs = n;
  cudaGetLastError();  // a refused query only disables the pair kernel
  return cudaSuccess;
}

bool prefill_pair_eligible(const PrefillLaunch &a) {
  // a paged cache only when every key tile is whole (S_kv a multiple of 128);
  // otherwise it runs on the single-CTA kernel, which clears the V rows of a
  // page's unused tail before P V reads them
  return a.H_kv > 0 && (a.H_q / a.H_kv) % 4 == 0 && a.max_pairs > 0 &&
         (a.block_table == nullptr ||
          (a.S_kv % prefill_pair::kBN == 0 && a.page_size > 0 && a.page_size % prefill_pair::kBN == 0));
}

// Work plan: units of one 128-row query tile of four heads over the resident
// CTA pairs; with a workspace, the last round's units may be split by key range
// (the shortest unit is the one of query tile 0).
PrefillPlan prefill_pair_plan(const PrefillLaunch &a) {
  using namespace prefill_pair;
  const int G = a.H_q / a.H_kv;
  const int n_qtiles = (a.T_q + kBM - 1) / kBM;
  const long long units = (long long)n_qtiles * a.B * a.H_kv * (G / 4);
  const int n_kv_first = (a.q_offset + (a.T_q < kBM ? a.T_q : kBM) - 1) / kBN + 1;
  const int n_kv_all = (a.S_kv + kBN - 1) / kBN;
  const int n_kv_min = n_kv_first < n_kv_all ? n_kv_first : n_kv_all;
  return prefill_split::make_plan(units, a.max_pairs, n_kv_min, 4, a.ws, a.ws_bytes);
}

size_t prefill_pair_workspace_bound(long long units, int num_sms) {
  return prefill_split::workspace_bound(units, num_sms / 2, 4);
}

cudaError_t prefill_pair_launch(const PrefillLaunch &a, cudaStream_t stream,
                                PFN_cuTensorMapEncodeTiled_v12000 encode) {
  using namespace prefill_pair;
  if (!prefill_pair_eligible(a)) return cudaErrorNotSupported;
  const PrefillPlan pl = prefill_pair_plan(a);
  if (pl.units <= 0) return cudaErrorNotSupported;
  // K/V blocks of rows: one per (sequence, KV head) of S_kv keys, or one per
  // (page, KV head) of page_size keys
  const bool paged = a.block_table != nullptr;
  const int kv_rows = paged ? a.page_size : a.S_kv;
  const int kv_blocks = paged ? a.num_pages * a.H_kv : a.B * a.H_kv;
  CUtensorMap tm_q, tm_k, tm_v;
  if (make_map(&tm_q, a.q, a.T_q, a.B * a.H_q, kBM, encode) != CUDA_SUCCESS ||
      make_map(&tm_k, a.k, kv_rows, kv_blocks, kHalfKeys, encode) != CUDA_SUCCESS ||
      make_map(&tm_v, a.v, kv_rows, kv_blocks, kBN, encode) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  Params p;
  p.o = a.o;
  p.lse = a.lse;
  p.B = a.B;
  p.H_q = a.H_q;
  p.H_kv = a.H_kv;
  p.G = a.H_q / a.H_kv;
  p.T_q = a.T_q;
  p.S_kv = a.S_kv;
  p.q_offset = a.q_offset;
  p.n_qtiles = (a.T_q + kBM - 1) / kBM;
  p.n_quads = p.G / 4;
  p.n_items = pl.n_items;
  p.n_pairs = pl.workers;
  p.n_full = pl.n_full;
  p.split_s = pl.split_s;
  p.ws_o = pl.pieces > 0 ? static_cast<float *>(a.ws) : nullptr;
  p.ws_ml = pl.pieces > 0 ? p.ws_o + (size_t)pl.pieces * 4 * kBM * kD : nullptr;
  p.sl2 = a.scale * 1.4426950408889634f;
  p.wait = a.wait;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.n_pairs, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e =
      paged ? cudaLaunchKernelEx(&cfg, prefill_pair_kernel<true>, tm_q, tm_k, tm_v, p,
                                 PageArgs<true>{a.block_table, a.page_size, a.max_pages,
                                                a.num_pages})
            : cudaLaunchKernelEx(&cfg, prefill_pair_kernel<false>, tm_q, tm_k, tm_v, p,
                                 PageArgs<false>{});
  if (e != cudaSuccess) return e;
  // the pieces' merge, a programmatic dependent of the pair kernel
  return prefill_split::launch_merge<4>(p, pl, stream);
}

}  // namespace gqa
