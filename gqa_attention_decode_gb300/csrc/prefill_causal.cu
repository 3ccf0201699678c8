// prefill_causal.cu -- causal GQA prefill for sm_103a with tcgen05 tensor cores.
//
// What it computes (design record "ADR-0060: AHBM GQA Fused Attention Kernel
// (Llama3-70B)"): for each query tile, the per-tile online softmax of section 3
// (S = scale Q K^T, running max and sum, O = O corr + P V, normalise once) over
// the key tiles the tile can see; section 5.4's tile classes decide the work:
// key tiles wholly in the past run unmasked, the boundary tiles get the causal
// mask, and tiles wholly in the future are never loaded.  Query row i sits at
// absolute position q_offset + i (the record's q_block_meta), which makes the
// same kernel serve chunked prefill.
//
// GB300 mapping
//   * Persistent CTAs (one per SM, 320 threads).  A work unit is one 128-row
//     query tile of TWO query heads of the same KV group: both heads see exactly
//     the same key tiles, so every K/V tile loaded by TMA feeds two S = Q K^T and
//     two O += P V products (the record's GQA reuse, applied to prefill), and the
//     two softmax warpgroups ping-pong: a token passed between them lets only one
//     run its exp() phase at a time while the tensor core works on the other
//     head (the record's "GEMM idle during softmax" bubble, section 5.6 opt3,
//     removed by warp specialisation instead of software pipelining).  Units run
//     longest-first (latest query tile first).
//   * Warps 0-3 and 4-7: softmax for head 0 and head 1, one thread per query
//     row, the whole 128-column S row held in registers.  Warp 8: TMA producer
//     (Q tiles, then K_j, V_j through a 4-stage ring).  Warp 9: allocates the 512
//     TMEM columns and issues every tcgen05.mma from one thread (M = N = 128,
//     K = 16, bf16 in, fp32 accumulate).
//   * TMEM: S0, S1 (128 columns each) and O0, O1 (128 columns each).  P is
//     written back as bf16 over the first 64 columns of its S block and read by
//     the P V product straight from tensor memory (A operand in TMEM), so P never
//     touches shared memory.
//   * The running max is only moved (and O in TMEM rescaled) when a row's tile
//     max exceeds it by more than 8 in log2 units; the final O / l and
//     lse = m ln2 + ln l use the same reference max, so the result is exact.
#include <cudaTypedefs.h>
#include <math.h>

#include "device_common.cuh"
#include "kernels.h"
#include "prefill_split.cuh"
#include "tcgen05.cuh"

namespace gqa {
namespace prefill {

constexpr int kD = 128;
constexpr int kBM = 128;                     // query rows per tile
constexpr int kBN = 128;                     // keys per tile
constexpr int kStages = 4;                   // K/V ring depth (each stage holds one K or V tile)
constexpr int kWarpTma = 8, kWarpMma = 9;
constexpr int kThreads = 320;
constexpr int kTileBytes = kBM * kD * 2;     // 32 KiB
constexpr int kHalfBytes = kTileBytes / 2;   // one 64-column half: [128 rows x 128 B]
constexpr int kOffQ = 0;                     // Q0, Q1
constexpr int kOffStage = 2 * kTileBytes;    // K/V ring
constexpr int kOffBar = kOffStage + kStages * kTileBytes;
// barriers: kv_full[S], kv_empty[S], q_full[2], q_empty, s_full[2], p_full[2], o_final[2],
// exp-turn tokens[2], drain
constexpr int kNumBars = 2 * kStages + 2 + 1 + 2 + 2 + 2 + 2 + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base slot, abort flag
constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + 1024 alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;    // log2 units (a factor of 256)
constexpr float kSumTrigger = 256.0f;      // 2^kRescaleThreshold

struct Params {
  uint16_t *o;
  float *lse;
  int B, H_q, H_kv, G, T_q, S_kv, q_offset;
  int n_qtiles;
  int n_hp;         // head pairs of a KV group that share a query tile: G / 2
  int odd;          // G odd: the group's last head pairs two of its own query tiles
  // Items dealt to the CTAs: [0, n_full) whole units; the units after them
  // cut into split_s key-range pieces (item n_full + t is piece t), whose
  // partials go to ws_o / ws_ml and are combined by the merge kernel.
  int n_items, n_full, split_s;
  float *ws_o;   // [piece][2 slots][128 rows][128] fp32, O not yet divided by l
  float *ws_ml;  // [piece][2 slots][128 rows][2] fp32: m (log2 units), l
  float sl2;  // scale * log2(e)
  WaitCtl wait;
};

using prefill_split::PageArgs;

// Two slots of 128 query rows: slot i is query tile qt_i of head h_i.  Either
// two heads of a KV group on one query tile, or (G odd) the group's last head
// on query tiles qt and qt - 1, which read the same key tiles (the lower one
// has its last key tile wholly in the future: masked, a tile of zeros).
struct Unit {
  int b, kv, qt0, qt1, h0, h1, n_kv;
  bool second_valid;
  int kv_lo, kv_hi;  // key tiles of this item: [kv_lo, kv_hi)
  int piece;         // -1: a whole unit, O and lse final; else its partial slot
};

// Unit of round k for worker w of P: units are sorted longest first and dealt
// in snake order (left to right, then right to left), so no worker takes the
// longest unit of every round; only the last round can be partial.
__device__ __forceinline__ int snake_unit(int k, int w, int P) {
  return k * P + ((k & 1) ? P - 1 - w : w);
}

// Units, longest first.  Query tiles are taken in ranks r = 0, 1, ... (tile
// n_qtiles - 1 - r); rank r holds B * H_kv * n_hp head-pair units and, for even
// r when G is odd, B * H_kv last-head units (tiles of ranks r and r + 1).
__device__ __forceinline__ Unit unit_at(const Params &p, int item) {
  Unit w;
  int u = item;
  w.piece = -1;
  if (item >= p.n_full) {
    const int t = item - p.n_full;
    u = p.n_full + t / p.split_s;
    w.piece = t;
  }
  const int bh = p.B * p.H_kv;
  const int pn = bh * p.n_hp;                 // head-pair units per rank
  const int two = 2 * pn + (p.odd ? bh : 0);  // units of ranks 2t and 2t + 1
  const int t = u / two;
  int idx = u % two, rank = 2 * t;
  if (idx >= pn + (p.odd ? bh : 0)) {
    idx -= pn + (p.odd ? bh : 0);
    rank += 1;
  }
  w.qt0 = p.n_qtiles - 1 - rank;  // latest (longest) query tiles first
  if (idx < pn) {                 // heads 2 hp and 2 hp + 1 of a group, one query tile
    const int hp = idx % p.n_hp;
    const int r = idx / p.n_hp;
    w.kv = r % p.H_kv;
    w.b = r / p.H_kv;
    w.h0 = w.kv * p.G + 2 * hp;
    w.h1 = w.h0 + 1;
    w.qt1 = w.qt0;
    w.second_valid = true;
  } else {                        // the group's last head, query tiles qt0 and qt0 - 1
    const int r = idx - pn;
    w.kv = r % p.H_kv;
    w.b = r / p.H_kv;
    w.h0 = w.h1 = w.kv * p.G + p.G - 1;
    w.second_valid = w.qt0 > 0;
    w.qt1 = w.second_valid ? w.qt0 - 1 : w.qt0;
  }
  const int qe = min((w.qt0 + 1) * kBM, p.T_q);
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

// Output row of slot hl of work item `item`, row `row` (false: not stored).
__device__ __forceinline__ bool piece_out_row(const Params &p, int item, int hl, int row,
                                              size_t *orow) {
  const Unit w = unit_at(p, item);
  if (hl == 1 && !w.second_valid) return false;
  const int qrow = (hl == 0 ? w.qt0 : w.qt1) * kBM + row;
  if (qrow >= p.T_q) return false;
  *orow = ((size_t)w.b * p.H_q + (hl == 0 ? w.h0 : w.h1)) * p.T_q + qrow;
  return true;
}

__device__ __forceinline__ bool wait_abortable(uint32_t bar, uint32_t parity, const WaitCtl &ctl,
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

// Operand descriptors, built once per tile and advanced per k-step by a
// compile-time byte offset (one add between tensor-core instructions).
// K-major 128x128 bf16 tile stored as two 128B-swizzled 64-column halves; k-step
// kk = 16 consecutive K-columns.
__device__ __forceinline__ uint64_t desc_kmajor_base(uint32_t tile) {
  return tc::smem_desc_sw128(tile, 16, 1024);
}
__device__ __forceinline__ constexpr uint32_t kmajor_step(int kk) {
  return (kk >> 2) * kHalfBytes + (kk & 3) * 32;
}
// MN-major tile (V: keys x d, d contiguous); the two 64-column halves are the two
// MN blocks (lbo); k-step kk = 16 consecutive K-rows.
__device__ __forceinline__ uint64_t desc_mnmajor_base(uint32_t tile) {
  return tc::smem_desc_sw128(tile, kHalfBytes, 1024);
}
__device__ __forceinline__ constexpr uint32_t mnmajor_step(int kk) { return kk * 2048; }

static_assert(kSmemBytes <= 232448, "shared memory budget");

// kPaged: K/V in pages through pg.block_table (a separate instantiation, so the
// dense kernel carries none of the page handling)
template <bool kPaged>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_causal_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const Params p,
                          const PageArgs<kPaged> pg) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
  const uint32_t bar0 = smem_u32(bars);
  auto kv_full = [&](int s) { return bar0 + 8u * s; };
  auto kv_empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto q_full = [&](int i) { return bar0 + 8u * (2 * kStages + i); };
  const uint32_t q_empty = bar0 + 8u * (2 * kStages + 2);
  auto s_full = [&](int i) { return bar0 + 8u * (2 * kStages + 3 + i); };
  auto p_full = [&](int i) { return bar0 + 8u * (2 * kStages + 5 + i); };
  auto o_final = [&](int i) { return bar0 + 8u * (2 * kStages + 7 + i); };
  auto tok = [&](int i) { return bar0 + 8u * (2 * kStages + 9 + i); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 11);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full(i), 1);
      mbar_init(s_full(i), 1);
      mbar_init(p_full(i), 128);
      mbar_init(o_final(i), 1);
      mbar_init(tok(i), 128);
    }
    mbar_init(q_empty, 1);
    mbar_init(drain_bar, 1);
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

  if (warp == kWarpTma) {
    // ------------------------- TMA producer -------------------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      int ld = 0, it = 0;
      bool ok = true;
      for (int k = 0; ok; ++k, ++it) {
        const int u = snake_unit(k, blockIdx.x, gridDim.x);
        if (u >= p.n_items) break;
        const Unit w = unit_at(p, u);
        if (!wait_abortable(q_empty, (it & 1) ^ 1, p.wait, abort_flag)) { ok = false; break; }
        for (int i = 0; i < 2; ++i) {
          const int h = i == 0 ? w.h0 : w.h1;
          const uint32_t dst = sbase + kOffQ + i * kTileBytes;
          mbar_arrive_expect_tx(q_full(i), kTileBytes);
          for (int half = 0; half < 2; ++half)
            tma_load_4d(dst + half * kHalfBytes, &tm_q, q_full(i), 0, half,
                        (i == 0 ? w.qt0 : w.qt1) * kBM, w.b * p.H_q + h, pol_q);
        }
        for (int j = w.kv_lo; ok && j < w.kv_hi; ++j) {
          for (int which = 0; which < 2; ++which, ++ld) {
            const int s = ld % kStages;
            if (!wait_abortable(kv_empty(s), ((ld / kStages) & 1) ^ 1, p.wait, abort_flag)) {
              ok = false;
              break;
            }
            const uint32_t dst = sbase + kOffStage + s * kTileBytes;
            mbar_arrive_expect_tx(kv_full(s), kTileBytes);
            const CUtensorMap *map = which == 0 ? &tm_k : &tm_v;
            int c2 = j * kBN, c3 = w.b * p.H_kv + w.kv;  // the tile's first key row and block
            if constexpr (kPaged) {
              // a 128-key tile lies in one page (page sizes are multiples of 128); a
              // page id outside the pool reads zeros (a block past the tensor map)
              // and is reported through the status word
              const int page = j * kBN / pg.page_size;
              const int page_id = __ldca(pg.block_table + (size_t)w.b * pg.max_pages + page);
              const bool bad = page_id < 0 || page_id >= pg.num_pages;
              if (bad) atomicExch(p.wait.status, kStatusInvalidArg);
              c2 = j * kBN - page * pg.page_size;
              c3 = bad ? pg.num_pages * p.H_kv : page_id * p.H_kv + w.kv;
            }
            for (int half = 0; half < 2; ++half)
              tma_load_4d(dst + half * kHalfBytes, map, kv_full(s), 0, half, c2, c3, pol_kv);
          }
        }
      }
      // no copy may still be in flight when the CTA exits
      for (int i = max(0, ld - kStages); i < ld; ++i)
        wait_abortable(kv_full(i % kStages), (i / kStages) & 1, p.wait, abort_flag);
    }
  } else if (warp == kWarpMma) {
    // ------------------------- MMA issuer -------------------------
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kBM, kBN, 0);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(kBM, kD, 1);
      const uint32_t t_s[2] = {tmem + 0u, tmem + 128u};
      const uint32_t t_o[2] = {tmem + 256u, tmem + 384u};
      const uint64_t dq0 = desc_kmajor_base(sbase + kOffQ);
      const uint64_t dq1 = desc_kmajor_base(sbase + kOffQ + kTileBytes);
      int ld_base = 0, tile_base = 0, it = 0;
      bool ok = true;
      for (int k = 0; ok; ++k, ++it) {
        const int u = snake_unit(k, blockIdx.x, gridDim.x);
        if (u >= p.n_items) break;
        const Unit w = unit_at(p, u);
        const int n = w.kv_hi - w.kv_lo;
        for (int i = 0; ok && i < 2; ++i)
          if (!wait_abortable(q_full(i), it & 1, p.wait, abort_flag)) ok = false;
        tc::fence_after_sync();
        for (int j = 0; ok && j <= n; ++j) {
          const int ldK = ld_base + 2 * j, ldV = ld_base + 2 * (j - 1) + 1;
          const uint64_t dk = desc_kmajor_base(sbase + kOffStage + (ldK % kStages) * kTileBytes);
          const uint64_t dv = desc_mnmajor_base(sbase + kOffStage + (ldV % kStages) * kTileBytes);
          if (j < n) {
            if (!wait_abortable(kv_full(ldK % kStages), (ldK / kStages) & 1, p.wait, abort_flag)) {
              ok = false;
              break;
            }
          }
          if (j > 0) {
            if (!wait_abortable(kv_full(ldV % kStages), (ldV / kStages) & 1, p.wait, abort_flag)) {
              ok = false;
              break;
            }
          }
          for (int i = 0; i < 2; ++i) {
            if (j > 0) {  // O_i += P_i V_{j-1}, P_i read from tensor memory
              if (!wait_abortable(p_full(i), (tile_base + j - 1) & 1, p.wait, abort_flag)) {
                ok = false;
                break;
              }
              tc::fence_after_sync();
#pragma unroll
              for (int kk = 0; kk < kBN / 16; ++kk)
                tc::mma_ts(t_o[i], t_s[i] + kk * 8, tc::desc_advance(dv, mnmajor_step(kk)),
                           idesc_pv, (j > 1 || kk > 0) ? 1u : 0u);
              if (i == 1) tc::commit(kv_empty(ldV % kStages));
              if (j == n) tc::commit(o_final(i));
            }
            if (j < n) {  // S_i = Q_i K_j^T
#pragma unroll
              for (int kk = 0; kk < kD / 16; ++kk)
                tc::mma_ss(t_s[i], tc::desc_advance(i == 0 ? dq0 : dq1, kmajor_step(kk)),
                           tc::desc_advance(dk, kmajor_step(kk)), idesc_s, kk > 0 ? 1u : 0u);
              tc::commit(s_full(i));
              count_s_tiles(p.wait, 1);
              if (i == 1) {
                tc::commit(kv_empty(ldK % kStages));
                if (j == n - 1) tc::commit(q_empty);
              }
            }
          }
        }
        ld_base += 2 * n;
        tile_base += n;
      }
      // every issued MMA must finish before TMEM is released
      tc::commit(drain_bar);
      wait_abortable(drain_bar, 0, p.wait, abort_flag);
    }
  } else if (warp < kWarpTma) {
    // ------------------------- softmax warpgroups -------------------------
    const int i = warp >> 2;  // 0: head h0, 1: head h1
    const int wq = warp & 3;  // TMEM lane quarter of this warp
    const int row = 32 * wq + lane;
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    const uint32_t t_s = tmem + lane_off + 128u * i;
    const uint32_t t_o = tmem + lane_off + 256u + 128u * i;
    const bool pos_scale = p.sl2 > 0.f;
    const float mul = pos_scale ? p.sl2 : 1.f;  // multiplier still owed by the held scores
    int tile = 0, it = 0;
    bool ok = true;
    for (int k = 0; ok; ++k, ++it) {
      const int u = snake_unit(k, blockIdx.x, gridDim.x);
      if (u >= p.n_items) break;
      const Unit w = unit_at(p, u);
      const int qt = i == 0 ? w.qt0 : w.qt1;
      const int q0 = p.q_offset + qt * kBM;  // absolute position of row 0 of the tile
      const int qpos = q0 + row;
      float m_ref = -INFINITY, l = 0.f;
      for (int j = w.kv_lo; j < w.kv_hi; ++j, ++tile) {
        bool ready = wait_abortable(s_full(i), tile & 1, p.wait, abort_flag);
        if (!__all_sync(0xffffffffu, ready)) { ok = false; break; }
        tc::fence_after_sync();
        const bool masked = (j * kBN + kBN - 1 > q0) || (j * kBN + kBN > p.S_kv);
        const int lim = min(qpos + 1, p.S_kv) - j * kBN;  // keys [0, lim) of the tile visible
        // scores of chunk c (32 keys) as held: times sl2 unless that is still owed,
        // keys the row may not see set to -inf
        auto prep = [&](uint32_t *v, int c) {
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
        // row max over the 128 scores, re-read from tensor memory, in the units of m_ref
        auto row_max = [&]() {
          uint32_t va[32], vb[32];
          float mx = -INFINITY;
          tc::ld32(t_s, va);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t *v = (c & 1) ? vb : va;
            tc::wait_ld32(v);
            prep(v, c);
            if (c + 1 < 4) tc::ld32(t_s + 32 * (c + 1), (c & 1) ? va : vb);
            float m2[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int e = 0; e < 32; e += 4)
#pragma unroll
              for (int k2 = 0; k2 < 2; ++k2)
                m2[k2] = fmax3(m2[k2], __uint_as_float(v[e + 2 * k2]), __uint_as_float(v[e + 2 * k2 + 1]));
            mx = fmax3(mx, m2[0], m2[1]);
          }
          return pos_scale ? mx * p.sl2 : mx;
        };
        // P = exp2(s * mul - m_ref) as bf16 pairs for the 32 scores of chunk c, with
        // their sum; argument and sums in packed fp32x2 instructions (two keys each)
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
            tc::wait_ld32(v);
            prep(v, c);
            if (c + 1 < 4) tc::ld32(t_s + 32 * (c + 1), (c & 1) ? va : vb);
            sum += exp_chunk(v, c);
          }
          return sum;
        };
        // common path: the whole row in registers (one load wait), before the exp turn
        uint32_t sv[kBN];
        tc::ld128_wait(t_s, sv);
#pragma unroll
        for (int c = 0; c < 4; ++c) prep(sv + 32 * c, c);
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
        // exp turn: head 0's tile k follows head 1's tile k-1, head 1's tile k follows
        // head 0's tile k, so only one warpgroup feeds the exp unit at a time
        if (i == 0) {
          ready = tile == 0 || wait_abortable(tok(0), (tile - 1) & 1, p.wait, abort_flag);
        } else {
          ready = wait_abortable(tok(1), tile & 1, p.wait, abort_flag);
        }
        if (!__all_sync(0xffffffffu, ready)) { ok = false; break; }
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
        mbar_arrive(tok(1 - i));  // the exp unit is free: the other warpgroup may start
        tc::st64(t_s, pk);
        if constexpr (kPaged) if (i == 0 && (j + 1) * kBN > p.S_kv) {
          // Paged K/V: the rows of this tile past the sequence come from the page's
          // unused slots (any bits, NaN included), and P V multiplies them by zero:
          // clear them in the V stage (load 2 * tile + 1) before P V reads it.  Slot
          // 0's P V is the first to read the stage and waits for this signal.
          const int ldv = 2 * tile + 1;
          const bool landed = wait_abortable(kv_full(ldv % kStages), (ldv / kStages) & 1, p.wait,
                                             abort_flag);
          if (landed) {
            uint8_t *vt = smem + kOffStage + (ldv % kStages) * kTileBytes;
            const int first = p.S_kv - j * kBN;  // first row past the sequence
            for (int idx = threadIdx.x; idx < (kBN - first) * 16; idx += 128) {
              const int r = first + idx / 16, c = idx % 16;  // 16 chunks of 16 B per row
              *reinterpret_cast<uint4 *>(vt + (c >> 3) * kHalfBytes + r * 128 + (c & 7) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();  // the tensor core reads these rows
          }
        }
        tc::wait_st();
        l += tsum;
        tc::fence_before_sync();
        mbar_arrive(p_full(i));
      }
      if (!ok) break;
      // epilogue: O / l -> bf16, lse = m_ref ln2 + ln l
      const bool ready = wait_abortable(o_final(i), it & 1, p.wait, abort_flag);
      if (!__all_sync(0xffffffffu, ready)) { ok = false; break; }
      tc::fence_after_sync();
      const int h = i == 0 ? w.h0 : w.h1;
      const int qrow = qt * kBM + row;
      const bool store = (i == 0 || w.second_valid) && qrow < p.T_q;
      const size_t orow = ((size_t)w.b * p.H_q + h) * p.T_q + qrow;
      uint32_t ov[kD];
      tc::ld128_wait(t_o, ov);
      if (store && w.piece >= 0) {
        // a piece of a split unit: its partial (O not yet divided, m, l) for the merge
        const size_t prow = prefill_split::partial_row(w.piece, 2, i, row);
        if (store_ok(prow, (size_t)(p.n_items - p.n_full) * 2 * kBM, p.wait.status)) {
          float4 *dst = reinterpret_cast<float4 *>(p.ws_o + prow * kD);
#pragma unroll
          for (int v4 = 0; v4 < kD / 4; ++v4)
            dst[v4] = make_float4(__uint_as_float(ov[4 * v4 + 0]), __uint_as_float(ov[4 * v4 + 1]),
                                  __uint_as_float(ov[4 * v4 + 2]), __uint_as_float(ov[4 * v4 + 3]));
          reinterpret_cast<float2 *>(p.ws_ml)[prow] = make_float2(m_ref, l);
        }
      } else if (store && store_ok(orow, (size_t)p.B * p.H_q * p.T_q, p.wait.status)) {
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
  __syncthreads();
  if (warp == kWarpMma) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

CUresult make_map(CUtensorMap *map, const uint16_t *base, int rows, int heads,
                  PFN_cuTensorMapEncodeTiled_v12000 encode) {
  // dims (innermost first): 64 columns, 2 column halves, rows, heads
  const cuuint64_t dims[4] = {64, 2, (cuuint64_t)rows, (cuuint64_t)heads};
  const cuuint64_t strides[3] = {128, 256, (cuuint64_t)rows * 256};
  const cuuint32_t box[4] = {64, 1, 128, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t *>(base), dims,
                strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace prefill

cudaError_t prefill_prepare_device() {
  cudaError_t e = cudaFuncSetAttribute(prefill::prefill_causal_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       prefill::kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(prefill::prefill_causal_kernel<true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, prefill::kSmemBytes);
}

long long prefill_units(int B, int H_q, int H_kv, int T_q) {
  using namespace prefill;
  const int G = H_q / H_kv;
  const long long n_qtiles = (T_q + kBM - 1) / kBM;
  const long long bh = (long long)B * H_kv;
  return n_qtiles * bh * (G / 2) + ((G & 1) ? bh * ((n_qtiles + 1) / 2) : 0);
}

// Work plan: one CTA per SM; units longest first (the shortest are those of
// query tile 0); with a workspace, the last round's units may be split.
PrefillPlan prefill_plan(const PrefillLaunch &a) {
  using namespace prefill;
  const long long units = prefill_units(a.B, a.H_q, a.H_kv, a.T_q);
  const int n_kv_first = (a.q_offset + (a.T_q < kBM ? a.T_q : kBM) - 1) / kBN + 1;
  const int n_kv_all = (a.S_kv + kBN - 1) / kBN;
  const int n_kv_min = n_kv_first < n_kv_all ? n_kv_first : n_kv_all;
  return prefill_split::make_plan(units, a.num_sms, n_kv_min, 2, a.ws, a.ws_bytes);
}

size_t prefill_workspace_bound(long long units, int num_sms) {
  return prefill_split::workspace_bound(units, num_sms, 2);
}

cudaError_t prefill_launch(const PrefillLaunch &a, cudaStream_t stream,
                           PFN_cuTensorMapEncodeTiled_v12000 encode) {
  using namespace prefill;
  const PrefillPlan pl = prefill_plan(a);
  if (pl.units <= 0) return cudaErrorNotSupported;
  const bool paged = a.block_table != nullptr;
  if (paged && (a.page_size <= 0 || a.page_size % kBN != 0)) return cudaErrorInvalidValue;
  // K/V blocks of rows: one per (sequence, KV head) of S_kv keys, or one per
  // (page, KV head) of page_size keys
  const int kv_rows = paged ? a.page_size : a.S_kv;
  const int kv_blocks = paged ? a.num_pages * a.H_kv : a.B * a.H_kv;
  CUtensorMap tm_q, tm_k, tm_v;
  if (make_map(&tm_q, a.q, a.T_q, a.B * a.H_q, encode) != CUDA_SUCCESS ||
      make_map(&tm_k, a.k, kv_rows, kv_blocks, encode) != CUDA_SUCCESS ||
      make_map(&tm_v, a.v, kv_rows, kv_blocks, encode) != CUDA_SUCCESS)
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
  p.n_hp = p.G / 2;
  p.odd = p.G & 1;
  p.n_items = pl.n_items;
  p.n_full = pl.n_full;
  p.split_s = pl.split_s;
  p.ws_o = pl.pieces > 0 ? static_cast<float *>(a.ws) : nullptr;
  p.ws_ml = pl.pieces > 0 ? p.ws_o + (size_t)pl.pieces * 2 * kBM * kD : nullptr;
  p.sl2 = a.scale * 1.4426950408889634f;
  p.wait = a.wait;
  if (paged) {
    const PageArgs<true> pg{a.block_table, a.page_size, a.max_pages, a.num_pages};
    prefill_causal_kernel<true>
        <<<pl.workers, kThreads, kSmemBytes, stream>>>(tm_q, tm_k, tm_v, p, pg);
  } else {
    prefill_causal_kernel<false>
        <<<pl.workers, kThreads, kSmemBytes, stream>>>(tm_q, tm_k, tm_v, p, PageArgs<false>{});
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the pieces' merge, a programmatic dependent of the prefill kernel
  return prefill_split::launch_merge<2>(p, pl, stream);
}

}  // namespace gqa
