// kernels.h -- host-side launch interface between the C ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "device_common.cuh"

namespace gqa {

// ---- decode ----------------------------------------------------------------
struct DecodeLaunch {
  const uint16_t *q;        // [B, H_q, d]
  const uint16_t *k_cache;  // dense [B, H_kv, S_max, d], or pages [num_pages, H_kv, page_size, d]
  const uint16_t *v_cache;  // same layout as k_cache
  const int32_t *block_table;  // paged: [B, max_pages]; nullptr for the dense layout
  int num_pages, page_size, max_pages;  // paged layout (S_max = max_pages * page_size)
  const int32_t *seqlens;   // [B]
  int B, H_q, H_kv, S_max, num_splits, chunk;
  int chunk_tile;   // keys a chunk is a multiple of: 64 (split kernel) or 128 (tcgen05 kernel)
  int T_q;          // new tokens per sequence (1: plain decode); G * T_q <= kDecodeMaxCols
  float scale;
  uint16_t *o;      // [B, H_q, T_q, d]
  float *lse;       // [B, H_q, T_q]
  float *o_part;    // [B, H_q, T_q, num_splits, d]
  float *lse_part;  // [B, H_q, T_q, num_splits]
  int num_sms;
  const int *fused_clusters;  // [kDecodeMaxFusedSplits + 1]: co-resident clusters per size
  int direct_out;  // split kernel with num_splits == 1: write o and lse, no merge follows
  WaitCtl wait;
};

constexpr int kDecodeTileKeys = 64;  // keys per pipeline stage
constexpr int kDecodeMaxG = 8;       // query heads per KV head that fit the MMA N dimension
constexpr int kDecodeMaxFusedSplits = 16;  // largest cluster of the single-kernel decode
constexpr int kDecodeMaxCols = 32;         // (head, new token) rows per KV head: G * T_q

// One-time per-device kernel attributes (dynamic shared memory, cluster size
// opt-in); fills fused_clusters[1..kDecodeMaxFusedSplits] with the number of
// clusters of that size the single-kernel variant runs at once.
cudaError_t decode_prepare_device(int *fused_clusters);
// Single-kernel decode: the splits of one (sequence, KV head) form a cluster and
// merge through distributed shared memory.  Eligible when every cluster of the
// plan runs in one wave; cudaErrorNotSupported otherwise.
bool decode_fused_eligible(const DecodeLaunch &a);
cudaError_t decode_fused_launch(const DecodeLaunch &a, cudaStream_t stream,
                                PFN_cuTensorMapEncodeTiled_v12000 encode);
// Encodes the tensor maps and launches the split kernel (no-op when S_max == 0).
cudaError_t decode_split_launch(const DecodeLaunch &a, cudaStream_t stream,
                                PFN_cuTensorMapEncodeTiled_v12000 encode);
// Launches the log-sum-exp merge of the split partials.
cudaError_t decode_merge_launch(const DecodeLaunch &a, cudaStream_t stream);

// Split kernel on tcgen05 tensor cores for many (head, token) rows per KV head:
// 32 < G * T_q <= kDecodeTcRows, or G > kDecodeMaxG (dense cache, chunk a
// multiple of 128 keys).  Writes the same partials as decode_split_launch, for
// decode_merge_launch.
constexpr int kDecodeTcRows = 128;
constexpr int kDecodeTcTileKeys = 128;
cudaError_t decode_tc_prepare_device();
cudaError_t decode_tc_split_launch(const DecodeLaunch &a, cudaStream_t stream,
                                   PFN_cuTensorMapEncodeTiled_v12000 encode);

// ---- causal prefill ----------------------------------------------------------
struct PrefillLaunch {
  const uint16_t *q;  // [B, H_q, T_q, d]
  const uint16_t *k;  // [B, H_kv, S_kv, d]
  const uint16_t *v;  // [B, H_kv, S_kv, d]
  int B, H_q, H_kv, T_q, S_kv, q_offset;
  float scale;
  uint16_t *o;  // [B, H_q, T_q, d]
  float *lse;   // [B, H_q, T_q]
  int num_sms;
  int max_pairs;  // CTA-pair kernel: clusters of two resident at once (0: not available)
  void *ws;         // optional scratch for key-split pieces (nullptr: no split)
  size_t ws_bytes;
  // paged K/V (single-CTA kernel only): [num_pages, H_kv, page_size, d] pages,
  // block table [B, max_pages]; nullptr: dense K/V
  const int32_t *block_table;
  int page_size, max_pages, num_pages;
  WaitCtl wait;
};

// Work plan of a prefill launch (host only): units of 128 query rows dealt in
// rounds over the resident workers (CTAs or CTA pairs); the units of a partial
// last round may be cut into key-range pieces merged afterwards.
struct PrefillPlan {
  int units = 0;    // work units
  int n_full = 0;   // units run whole
  int split_s = 1;  // pieces per split unit
  int pieces = 0;   // (units - n_full) * split_s
  int n_items = 0;  // n_full + pieces
  int workers = 0;  // CTAs (or CTA pairs) launched
};
// Single-CTA kernel (any group size).
cudaError_t prefill_prepare_device();
PrefillPlan prefill_plan(const PrefillLaunch &a);
size_t prefill_workspace_bound(long long units, int num_sms);
long long prefill_units(int B, int H_q, int H_kv, int T_q);
cudaError_t prefill_launch(const PrefillLaunch &a, cudaStream_t stream,
                           PFN_cuTensorMapEncodeTiled_v12000 encode);
// CTA-pair kernel (tcgen05 cta_group::2), for group sizes that are multiples of 4.
cudaError_t prefill_pair_prepare_device(int *max_pairs);
bool prefill_pair_eligible(const PrefillLaunch &a);
PrefillPlan prefill_pair_plan(const PrefillLaunch &a);
// Workspace that lets every partial round split as far as the plan may cut it.
size_t prefill_pair_workspace_bound(long long units, int num_sms);
cudaError_t prefill_pair_launch(const PrefillLaunch &a, cudaStream_t stream,
                                PFN_cuTensorMapEncodeTiled_v12000 encode);

// ---- combination of attention states over key shards ---------------------------
// o_parts [n_parts][rows][128] bf16, lse_parts [n_parts][rows] fp32 (natural log).
cudaError_t merge_states_launch(const uint16_t *o_parts, const float *lse_parts, int n_parts,
                                long long rows, uint16_t *o, float *lse, cudaStream_t stream);

// ---- diagnostics --------------------------------------------------------------
cudaError_t selftest_bounded_wait_launch(WaitCtl wait, cudaStream_t stream);

}  // namespace gqa
