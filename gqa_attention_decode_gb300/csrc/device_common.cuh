// device_common.cuh -- sm_103a device primitives shared by the attention kernels:
// mbarriers with bounded waits, TMA tile loads, warp-level bf16 MMA fragments.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gqa {

// Status word values (mirrors gqa_status_t).
constexpr int kStatusInvalidArg = 1;  // a device-side input out of range (clamped)
constexpr int kStatusTimeout = 5;
constexpr int kStatusOutOfBounds = 6;  // debug builds: a store index past its extent

// Guard of a global store: whether element `idx` lies inside the `extent`
// elements the kernel derives from its own arguments.  Debug builds
// (GQA_DEBUG_BOUNDS) record a violation in the status word and skip the store;
// release builds compile the check away.
__device__ __forceinline__ bool store_ok(size_t idx, size_t extent, int *status) {
#ifdef GQA_DEBUG_BOUNDS
  if (idx < extent) return true;
  atomicExch(status, kStatusOutOfBounds);
  return false;
#else
  (void)idx;
  (void)extent;
  (void)status;
  return true;
#endif
}

// Bounded-wait control passed to every kernel: where to record a timeout and
// how long a single wait may take.
struct WaitCtl {
  int *status;          // device status word (never null)
  uint64_t timeout_ns;  // per-wait limit
#ifdef GQA_DEBUG_BOUNDS
  unsigned long long *s_tiles;  // S = Q K^T tile products issued (one per query head and key tile)
#endif
};

// Bounds-checked builds count every S = Q K^T product of one query head's
// 128-row tile with one 128-key tile that a prefill kernel issues, so a test can
// hold the total against the causal (lower-triangular) tile count; release
// builds compile this away.
__device__ __forceinline__ void count_s_tiles(const WaitCtl &w, unsigned n) {
#ifdef GQA_DEBUG_BOUNDS
  atomicAdd(w.s_tiles, (unsigned long long)n);
#else
  (void)w;
  (void)n;
#endif
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits until the phase with the given parity has completed.  Gives up after
// ctl.timeout_ns, records kStatusTimeout and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl &ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > ctl.timeout_ns) {
      atomicExch(ctl.status, kStatusTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) loads into shared memory, completion on an mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar),
      "l"(policy)
      : "memory");
}

// A relaxed (morally strong) load of a value another grid may be writing:
// either the old or the new value, for use as a hint only.
__device__ __forceinline__ int ld_relaxed_s32(const int32_t *p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Prefetch of a tile into L2 (no shared memory, no completion to wait for).
// Safe ahead of a grid-dependency wait: L2 is the point of coherence, so a later
// write by the preceding grid still reaches every load that follows the wait.
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap *map, int c0, int c1, int c2,
                                                   int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

// ceil(n / d) for n < 2^20, d >= 1: the approximate hardware reciprocal (a few
// ulp) puts n * (1/d) within one of n / d, and one integer correction each way
// makes the quotient exact (checked against exact division with the
// reciprocal perturbed by up to 4 ulp either way).
__device__ __forceinline__ unsigned ceil_div_small(unsigned n, unsigned d) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(__uint2float_rn(d)));
  unsigned q = __float2uint_rz(__uint2float_rn(n) * r);
  if (q * d > n) --q;
  else if ((q + 1) * d <= n) ++q;  // q = floor(n / d)
  return q + (q * d != n ? 1u : 0u);
}

// Keys per split for a sequence of `seqlen` keys (the decode's split planner,
// second half).  The host plan sized `chunk` (keys, a multiple of `tile`) for
// S_max, the only length it knows; the length itself lives on the device.  A
// shorter sequence is spread as if the batch held B like it: its key tiles t
// times B * H_kv, over the SMs, give ceil(t * B * H_kv / num_sms) tiles per
// chunk, never more than the host's chunk and never so few that the sequence
// needs more than `splits` chunks.  A sequence at S_max keeps the host's
// chunk.  The split kernels and the merge call it with the same arguments and
// get the same value.
__device__ __forceinline__ int device_chunk(int seqlen, int B, int S_max, int chunk, int splits,
                                            int H_kv, int num_sms, int tile) {
  if (seqlen >= S_max) return chunk;
  const unsigned t = (unsigned)(seqlen + tile - 1) / tile;
  const unsigned chunk_tiles = (unsigned)(chunk / tile);
  // totals of 2^20 tiles or more are far above any cap: the host's chunk
  const unsigned long long work = (unsigned long long)t * (unsigned)H_kv * (unsigned)B;
  unsigned c = work >= (1u << 20) ? chunk_tiles : ceil_div_small((unsigned)work, (unsigned)num_sms);
  c = min(c, chunk_tiles);
  // at least what fits the sequence into the splits (the host's chunk always does)
  c = max(c, t < (1u << 20) ? ceil_div_small(t, (unsigned)splits) : chunk_tiles);
  return (int)max(c, 1u) * tile;
}

// Tile load into this CTA's shared memory whose completion is counted on an
// mbarrier that may live in the peer CTA of a CTA pair (`bar` is a
// shared::cluster address, e.g. from dsmem_addr).
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                                 int c0, int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2.L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar),
      "l"(policy)
      : "memory");
}

// Arrive on an mbarrier in another CTA of the cluster (the default-semantics
// form of cluster barriers; an explicit .release.cluster arrive measured about
// 1.5k cycles per call on GB300).  Callers complete their own prior writes first
// (tcgen05.wait::st, fence.proxy.async) so the peer only ever acts on finished data.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// Packed fp32x2 arithmetic (sm_100 and later): two lanes of float in one 64-bit
// register, one instruction for both.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_split(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// max(a, b, c) in one instruction (three-input max, sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// try_wait with cluster-scope acquire: for barriers that receive arrivals or
// transaction bytes from the other CTA of a pair.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA / tensor core) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Thread-block clusters and distributed shared memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Asynchronous stores into another CTA's shared memory (shared::cluster addresses,
// from dsmem_addr): the bytes land in that CTA, whose mbarrier `bar` (also a
// shared::cluster address) counts them as completed transaction bytes.
__device__ __forceinline__ void st_async_f32x4(uint32_t addr, float4 v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::
          "r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(addr),
               "f"(v), "r"(bar)
               : "memory");
}

// Every thread of every CTA in the cluster; shared-memory writes before it are
// visible to DSMEM reads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Warp-level bf16 MMA (m16n8k16, fp32 accumulate) and fragment movement
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                              uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transposes an 8x8 b16 matrix held one row-pair per thread (ldmatrix layout).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Packs two fp32 into a bf16x2 register (round to nearest even); `lo` goes to
// the lower 16 bits (the lower column index of an MMA fragment).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Approximate reciprocal and base-2 logarithm (one special-function instruction
// each; relative errors near 2^-23 and 2^-22), for normalising a softmax row.
__device__ __forceinline__ float fast_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace gqa
