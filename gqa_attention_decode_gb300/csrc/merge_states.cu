// merge_states.cu -- combination of attention states computed over disjoint key
// shards, for sm_103a.
//
// What it computes (design record "ADR-0060: AHBM GQA Fused Attention Kernel
// (Llama3-70B)", section 4 "Reduction": the log-sum-exp merge of per-shard
// partials, associative and commutative): for each row r (a (sequence, query
// head[, token]) triple) with finalised shard states (O_i, lse_i),
//   M = max_i lse_i,  L = sum_i exp(lse_i - M),
//   lse = M + ln L,   O = sum_i exp(lse_i - M) O_i / L,
// a shard with lse_i = -inf (no visible key) contributing nothing and a row
// with no visible key in any shard giving O = 0, lse = -inf.  The shard states
// are the outputs of decode or prefill calls over key shards: on one GPU a
// shared prefix and per-sequence suffixes (cascade), across GPUs the KV shards
// of a sequence-parallel decode gathered to one rank (section 4's reduce).
//
// GB300 mapping: one warp per row; lane l owns columns 4l .. 4l+3 (d = 128);
// the shards' lse values are read lane-parallel for the max, then the warp
// walks the shards, each lane loading its 8 bytes of O_i.  Launched as a
// programmatic dependent: the inputs (written by the preceding grids) are read
// after the grid-dependency wait, through L2.
#include <math.h>

#include "device_common.cuh"
#include "kernels.h"

namespace gqa {
namespace merge_states {

constexpr int kD = 128;
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

__global__ void __launch_bounds__(kThreads)
    merge_states_kernel(const uint16_t *__restrict__ o_parts, const float *__restrict__ lse_parts,
                        int n_parts, long long rows, uint16_t *__restrict__ o,
                        float *__restrict__ lse) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (row >= rows) return;
  float M = -INFINITY;
  for (int i = lane; i < n_parts; i += 32) M = fmaxf(M, __ldcg(lse_parts + (size_t)i * rows + row));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  uint2 out = make_uint2(0u, 0u);
  float lse_out = -INFINITY;
  if (M > -INFINITY) {
    float L = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 4
    for (int i = 0; i < n_parts; ++i) {
      const float li = __ldcg(lse_parts + (size_t)i * rows + row);
      const float w = li > -INFINITY ? fast_exp2((li - M) * kLog2e) : 0.f;
      const uint2 x =
          __ldcg(reinterpret_cast<const uint2 *>(o_parts + ((size_t)i * rows + row) * kD) + lane);
      L += w;
      a0 = fmaf(w, bf16_lo(x.x), a0);
      a1 = fmaf(w, bf16_hi(x.x), a1);
      a2 = fmaf(w, bf16_lo(x.y), a2);
      a3 = fmaf(w, bf16_hi(x.y), a3);
    }
    const float inv = 1.f / L;  // L >= 1: the shard holding M has weight 1
    out.x = pack_bf16x2(a0 * inv, a1 * inv);
    out.y = pack_bf16x2(a2 * inv, a3 * inv);
    lse_out = M + logf(L);
  }
  reinterpret_cast<uint2 *>(o + (size_t)row * kD)[lane] = out;
  if (lane == 0) lse[row] = lse_out;
}

}  // namespace merge_states

cudaError_t merge_states_launch(const uint16_t *o_parts, const float *lse_parts, int n_parts,
                                long long rows, uint16_t *o, float *lse, cudaStream_t stream) {
  using namespace merge_states;
  if (rows <= 0) return cudaSuccess;
  const long long blocks = (rows + kThreads / 32 - 1) / (kThreads / 32);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_states_kernel, o_parts, lse_parts, n_parts, rows, o, lse);
}

}  // namespace gqa
