/*
 * gqa_attn.h -- C ABI of the GB300 (sm_103a) grouped-query attention library.
 *
 * Two operations, both defined by the design record "ADR-0060: AHBM GQA Fused
 * Attention Kernel (Llama3-70B)" (kernbench2):
 *
 *   gqa_attn_decode          split-KV decode (FlashDecoding).  The G query heads
 *                            that share one KV head are folded into one matrix
 *                            product so every K/V tile is read from HBM once
 *                            (record: TL;DR "Kernel 1", section 5.2 "DECODE, no
 *                            SP"); each KV chunk yields a partial that a
 *                            log-sum-exp merge combines (section 4 "Reduction").
 *   gqa_attn_prefill_causal  causal prefill with online softmax and fully masked
 *                            tiles skipped (section 3 "Per-tile op sequence",
 *                            section 5.4 "PREFILL, no SP"), with q_offset for
 *                            chunked prefill (section 0.5.3 "q_block_meta");
 *                            gqa_attn_prefill_causal_ws adds a workspace so
 *                            the last round of work can be split by key range
 *                            and merged like decode's chunks.
 *
 * Both compute, for query head h, KV head h / G (G = H_q / H_kv) and the keys
 * visible to the query,
 *     O   = softmax(scale * q K^T) V          (bf16 out, rounded to nearest even)
 *     lse = scale * max_j s_j + ln sum_j exp(scale * (s_j - max_j s_j))   (fp32)
 * i.e. lse is the natural-log log-sum-exp of the scaled scores.  A query that
 * sees no key (decode with seqlen 0) gets O = 0 and lse = -inf.
 *
 * Conventions common to every entry point
 *   - bf16 tensors are passed as uint16_t bit patterns (gqa_bf16_t).
 *   - Every tensor is dense, row-major (C order) with the shape given below;
 *     head dimension d is innermost.
 *   - Device pointers must point to device memory of the current CUDA device
 *     and be 16-byte aligned.  The caller owns every buffer; the library keeps
 *     no pointer after a call returns and allocates no device memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous and stream-ordered; they never synchronise except where a
 *     function says so.  Inputs must stay valid until the stream reaches the
 *     work.
 *   - On any return other than GQA_OK nothing has been launched, except
 *     GQA_ERR_CUDA, which reports a launch failure (the CUDA error is left for
 *     cudaGetLastError to read).
 *   - Waits inside the kernels are bounded (about two seconds).  A wait that
 *     runs out sets a device-side status word and the kernel returns early;
 *     gqa_attn_device_status reads it.  No kernel traps.
 *
 * Thread safety: all entry points may be called from several host threads; the
 * per-device set-up done on first use is guarded by a mutex.
 */
#ifndef GQA_ATTN_H_
#define GQA_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GQA_API __attribute__((visibility("default")))
#else
#define GQA_API
#endif

#define GQA_ATTN_ABI_VERSION 1

typedef uint16_t gqa_bf16_t; /* bf16 bit pattern */
typedef void *gqa_stream_t;  /* a cudaStream_t */

typedef enum {
  GQA_OK = 0,
  GQA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or shape       */
  GQA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. d != 128, G > 8)  */
  GQA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed                 */
  GQA_ERR_WORKSPACE = 4,   /* workspace smaller than the size function reports */
  GQA_ERR_TIMEOUT = 5,     /* a bounded device-side wait ran out               */
  GQA_ERR_OUT_OF_BOUNDS = 6 /* bounds-checked builds: a kernel store index past
                              its extent (the store is skipped)                 */
} gqa_status_t;

/* Human-readable name of a status code; never NULL, static storage. */
GQA_API const char *gqa_status_string(int status);

/* GQA_ATTN_ABI_VERSION of the loaded library. */
GQA_API int gqa_attn_abi_version(void);

/* ------------------------------------------------------------------------- */
/* Decode                                                                      */
/* ------------------------------------------------------------------------- */

/*
 * Split plan for decode (host only, no CUDA call).  The KV sequence of every
 * (batch, KV head) is cut into contiguous chunks; split s owns keys
 * [s*c, min((s+1)*c, seqlen)) -- the contiguous-block placement of the
 * record's section 2.1 ("KV cache allocation"), rank r owning [r*B, (r+1)*B).
 * The plan fixes the grid (out_num_splits) and the largest chunk (out_chunk),
 * sized for S_max, the only length the host knows.  On the device each call
 * takes c per sequence from the length it finds there: with t key tiles of
 * 64 keys (128 on the tensor-core path), c is ceil(t * B * H_kv / num_sms)
 * tiles, at most out_chunk and at least what fits the sequence into
 * out_num_splits chunks; a sequence that fills its cache uses out_chunk.
 * Short sequences in a long cache are thereby spread over the SMs rather than
 * over the first few splits.  A split whose range is empty does no work and
 * is skipped by the merge.  This is the plan of the warp-MMA split kernel
 * (G * T_q <= 32 rows per KV head); the tcgen05 kernel rounds chunks up to 128
 * keys and, for an automatic plan of several waves whose B*H_kv units fill
 * half to all of the SMs, takes one split.
 *
 *   B, H_kv, S_max  batch, KV heads, capacity of the KV cache in keys (>= 0)
 *   num_sms         streaming multiprocessors of the target device (> 0)
 *   num_splits      0: choose from S_max, B*H_kv and num_sms so one wave of CTAs
 *                   fills the GPU, with chunks no longer than 2048 keys;
 *                   > 0: use this many splits (clamped to the number of 64-key
 *                   tiles in S_max).
 *   out_num_splits  written: splits per sequence (grid width), >= 1 if S_max > 0
 *   out_chunk       written: keys per split at most, a multiple of 64
 * Returns GQA_OK or GQA_ERR_INVALID_ARG (negative sizes, num_sms <= 0, null
 * outputs).
 */
GQA_API int gqa_attn_decode_plan(int B, int H_kv, int S_max, int num_sms, int num_splits,
                                 int *out_num_splits, int *out_chunk);

/*
 * Bytes of device workspace gqa_attn_decode needs for these sizes (host only).
 * Same arguments as gqa_attn_decode_plan plus H_q and d.  The workspace holds
 * one fp32 partial (O_s [d] normalised by its own sum, and lse_s) per
 * (batch, query head, split): B*H_q*num_splits*(d+1)*4 bytes, rounded up to
 * 256.  Returns 0 for invalid arguments.
 */
GQA_API size_t gqa_attn_decode_workspace_size(int B, int H_q, int H_kv, int S_max, int d,
                                              int num_sms, int num_splits);

/*
 * Split-KV GQA decode, T_q = 1 (record: TL;DR "Kernel 1", sections 3, 4, 5.2,
 * 5.3).
 *
 *   q         device [B, H_q, d] bf16, post-RoPE queries (section 0.5.3).
 *   k_cache   device [B, H_kv, S_max, d] bf16, post-RoPE keys; read only.
 *   v_cache   device [B, H_kv, S_max, d] bf16; read only.
 *   seqlens   device [B] int32, 0 <= seqlens[b] <= S_max: sequence b sees keys
 *             0..seqlens[b]-1.  Cache rows at or past seqlens[b] are never
 *             used and may hold any bits (NaN included).  Values outside
 *             [0, S_max] are clamped on the device and reported as
 *             GQA_ERR_INVALID_ARG by gqa_attn_device_status.
 *   B, H_q, H_kv, S_max, d   sizes; d must be 128; H_q % H_kv == 0 and
 *             G = H_q / H_kv <= 128.  G <= 8: the G heads fill the 8-wide
 *             dimension of the warp-level MMA; 8 < G <= 128: the tcgen05 split
 *             kernel (one 128-row tensor-core tile per KV head): split +
 *             merge, or one kernel when the plan has one split.
 *   scale     softmax scale (the record uses 1/sqrt(d)); any finite value.
 *   num_splits 0 = automatic plan, else the requested split count (see
 *             gqa_attn_decode_plan; the plan uses this device's SM count).
 *   o         device [B, H_q, d] bf16 output.
 *   lse       device [B, H_q] fp32 output (natural log, scaled scores).
 *   workspace device scratch of at least gqa_attn_decode_workspace_size(...)
 *             bytes for this device's SM count, 16-byte aligned; its contents
 *             on entry do not matter; it is overwritten.
 *   ws_bytes  size of `workspace` in bytes.
 *   stream    cudaStream_t.
 * Kernels on `stream` (one CTA per (split, KV head, batch)):
 *   - plans of at most 16 splits whose B*H_kv clusters (one per sequence and
 *     KV head, one CTA per split) the device runs all at once: ONE kernel;
 *     the splits of a (sequence, KV head) form a thread-block cluster and
 *     merge their partials through distributed shared memory; `workspace` is
 *     not touched;
 *   - other plans of one split per (sequence, KV head): ONE kernel, the split
 *     kernel writing o and lse itself; `workspace` is not touched;
 *   - other plans: the split kernel, which writes one partial per split to
 *     `workspace`, then the log-sum-exp merge kernel (launched as a
 *     programmatic dependent, so its launch overlaps the split kernel).
 * gqa_attn_decode_kernel_count reports which.  Deterministic: the same inputs
 * give bit-identical outputs (fixed reduction order, no atomics).  B == 0
 * launches nothing and returns GQA_OK.
 */
GQA_API int gqa_attn_decode(const gqa_bf16_t *q, const gqa_bf16_t *k_cache,
                            const gqa_bf16_t *v_cache, const int32_t *seqlens, int B,
                            int H_q, int H_kv, int S_max, int d, float scale, int num_splits,
                            gqa_bf16_t *o, float *lse, void *workspace, size_t ws_bytes,
                            gqa_stream_t stream);

/*
 * Decode over a paged KV cache (block table): the next step beside the
 * record's per-rank dense buffers (section 2.1), where each sequence's keys
 * live in fixed-size pages drawn from a shared pool.
 *
 *   k_pages, v_pages   device [num_pages, H_kv, page_size, d] bf16: page p holds
 *                      page_size consecutive keys of one sequence for every KV
 *                      head; read only; pages may be shared between sequences.
 *   block_table        device [B, max_pages_per_seq] int32: keys
 *                      [i*page_size, (i+1)*page_size) of sequence b are in page
 *                      block_table[b*max_pages_per_seq + i]; entries past the
 *                      sequence's last key are never read.  An entry outside
 *                      [0, num_pages) reads zeros (wrong result, no fault)
 *                      and is reported as GQA_ERR_INVALID_ARG by
 *                      gqa_attn_device_status.
 *   seqlens            device [B] int32, 0 <= seqlens[b] <= max_pages_per_seq *
 *                      page_size (clamped on the device).
 *   page_size          a positive multiple of 64 (else GQA_ERR_UNSUPPORTED); a
 *                      multiple of 128 where the tcgen05 split kernel runs
 *                      (G > 8, or G * T_q > 32 rows in gqa_attn_decode_paged_multi),
 *                      whose 128-key tiles must not straddle pages.
 *   num_pages * H_kv   below 2^31 (else GQA_ERR_UNSUPPORTED).
 * Everything else, including the plan and the workspace size, is that of
 * gqa_attn_decode with S_max = max_pages_per_seq * page_size.
 */
GQA_API int gqa_attn_decode_paged(const gqa_bf16_t *q, const gqa_bf16_t *k_pages,
                                  const gqa_bf16_t *v_pages, const int32_t *block_table,
                                  const int32_t *seqlens, int B, int H_q, int H_kv,
                                  int num_pages, int page_size, int max_pages_per_seq, int d,
                                  float scale, int num_splits, gqa_bf16_t *o, float *lse,
                                  void *workspace, size_t ws_bytes, gqa_stream_t stream);

/*
 * Multi-token decode over a paged KV cache: the arguments of
 * gqa_attn_decode_paged plus T_q, with q, o, lse and the token positions of
 * gqa_attn_decode_multi (token t of sequence b at seqlens[b] - T_q + t).  The
 * workspace is gqa_attn_decode_multi_workspace_size(B, H_q, H_kv, T_q,
 * max_pages_per_seq * page_size, d, num_sms, num_splits) bytes.
 */
GQA_API int gqa_attn_decode_paged_multi(const gqa_bf16_t *q, const gqa_bf16_t *k_pages,
                                        const gqa_bf16_t *v_pages, const int32_t *block_table,
                                        const int32_t *seqlens, int B, int H_q, int H_kv,
                                        int T_q, int num_pages, int page_size,
                                        int max_pages_per_seq, int d, float scale,
                                        int num_splits, gqa_bf16_t *o, float *lse,
                                        void *workspace, size_t ws_bytes, gqa_stream_t stream);

/*
 * Multi-token decode: T_q new tokens per sequence (speculative decoding
 * verification, the record's T_q of section 0.5.2 with the G*T_q rows of one KV
 * head folded into one product, section 5.2).
 *
 *   q        device [B, H_q, T_q, d] bf16; token t of sequence b sits at
 *            absolute position seqlens[b] - T_q + t.
 *   k_cache, v_cache, seqlens   as gqa_attn_decode; seqlens[b] counts every
 *            cached key, the T_q new tokens' keys included.
 *   Token t sees keys 0..seqlens[b]-T_q+t (causal among the new tokens); a
 *   token whose position is negative sees nothing (O = 0, lse = -inf).
 *   o        device [B, H_q, T_q, d] bf16; lse device [B, H_q, T_q] fp32.
 *   Supported: d = 128 and G * T_q <= 128 (T_q <= 16 for G = 8), else
 *   GQA_ERR_UNSUPPORTED.  K and V are read once per KV head for all G*T_q rows:
 *   up to 32 rows with warp-level MMAs, 33..128 rows (or G > 8) as one 128-row
 *   tcgen05 tile per KV head, whose split plan uses chunks of whole 128-key
 *   tiles (gqa_attn_decode_multi_workspace_size accounts for it).
 *   workspace: gqa_attn_decode_multi_workspace_size(...) bytes
 *   (B*H_q*T_q*splits*(d+1)*4, rounded up to 256).  T_q = 1 is gqa_attn_decode.
 */
GQA_API size_t gqa_attn_decode_multi_workspace_size(int B, int H_q, int H_kv, int T_q, int S_max,
                                                    int d, int num_sms, int num_splits);
GQA_API int gqa_attn_decode_multi(const gqa_bf16_t *q, const gqa_bf16_t *k_cache,
                                  const gqa_bf16_t *v_cache, const int32_t *seqlens, int B,
                                  int H_q, int H_kv, int T_q, int S_max, int d, float scale,
                                  int num_splits, gqa_bf16_t *o, float *lse, void *workspace,
                                  size_t ws_bytes, gqa_stream_t stream);

/*
 * Number of kernels gqa_attn_decode launches for these arguments on the current
 * device: 1 (single-kernel cluster path, or one split per sequence and KV
 * head), 2 (split + merge), 0 when B == 0.
 * Host only except for the first call on a device, which performs the
 * per-device set-up.  Returns the status of the argument checks.
 */
GQA_API int gqa_attn_decode_kernel_count(int B, int H_q, int H_kv, int S_max, int d,
                                         int num_splits, int *out_kernels);

/*
 * The two phases of gqa_attn_decode as separate calls (same arguments, same
 * plan, same workspace).  gqa_attn_decode_split runs the split kernel and
 * leaves the per-split partials in `workspace`; gqa_attn_decode_merge reads
 * them and writes o and lse.  Calling split then merge on one stream is
 * the result of gqa_attn_decode (bit for bit when gqa_attn_decode also runs
 * split + merge); between the two the workspace must not be touched, and
 * seqlens must hold the lengths the split call read (the merge kernel may read
 * them before a kernel launched between the two calls has finished).
 * split needs q, k_cache, v_cache, seqlens; merge needs seqlens, o, lse (the
 * other pointers may be NULL for the phase that does not use them).
 */
GQA_API int gqa_attn_decode_split(const gqa_bf16_t *q, const gqa_bf16_t *k_cache,
                                  const gqa_bf16_t *v_cache, const int32_t *seqlens, int B,
                                  int H_q, int H_kv, int S_max, int d, float scale,
                                  int num_splits, void *workspace, size_t ws_bytes,
                                  gqa_stream_t stream);
GQA_API int gqa_attn_decode_merge(const int32_t *seqlens, int B, int H_q, int H_kv, int S_max,
                                  int d, int num_splits, gqa_bf16_t *o, float *lse,
                                  const void *workspace, size_t ws_bytes, gqa_stream_t stream);

/*
 * Decode without a workspace argument, for callers that cannot allocate device
 * memory where they run attention: code inside a custom allocator or memory
 * pool that must not re-enter it, runtimes that forbid allocation after
 * start-up, and hosts that have no allocator to hand.  The design record has
 * no counterpart to this entry point; it exists only for such callers.
 *
 * Arguments, outputs and errors are those of gqa_attn_decode minus `workspace`
 * and `ws_bytes`.  The per-split partials go to a scratch array of
 * GQA_NOALLOC_SCRATCH_BYTES (48 MiB) in the library's static device memory,
 * which every GPU that loads the library holds until the process exits.  The
 * call allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 *   - Size limit: a problem whose workspace (gqa_attn_decode_workspace_size for
 *     this device) exceeds GQA_NOALLOC_SCRATCH_BYTES is rejected with
 *     GQA_ERR_WORKSPACE and nothing is launched; pass a smaller num_splits or use
 *     gqa_attn_decode.  (One 32K-key Llama3-70B layer needs under 2 MiB; a batch
 *     of 16 sequences in a 128K-key cache needs about 33 MiB.)
 *   - Shared scratch: every call uses the same array, and it keeps the last
 *     call's contents.  Calls whose GPU work overlaps (other streams, other host
 *     threads on the same device) race on it; serialise them.  Nothing needs
 *     clearing between calls: each call writes every partial it reads.
 *   - Set-up: the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 */
#define GQA_NOALLOC_SCRATCH_BYTES (48u << 20)
GQA_API int gqa_attn_decode_noalloc(const gqa_bf16_t *q, const gqa_bf16_t *k_cache,
                                    const gqa_bf16_t *v_cache, const int32_t *seqlens, int B,
                                    int H_q, int H_kv, int S_max, int d, float scale,
                                    int num_splits, gqa_bf16_t *o, float *lse,
                                    gqa_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Causal prefill                                                              */
/* ------------------------------------------------------------------------- */

/*
 * Causal GQA prefill with online softmax (record: Kernel 2's math, sections 3
 * and 5.4; the ring of section 5.5 is not used on one GPU).
 *
 *   q        device [B, H_q, T_q, d] bf16; row i is the query at absolute
 *            position q_offset + i.
 *   k, v     device [B, H_kv, S_kv, d] bf16; read only.
 *   q_offset 0 <= q_offset.  Row i sees keys 0..min(q_offset+i, S_kv-1) (the
 *            diagonal included); q_offset = 0 with T_q = S_kv is the square
 *            causal mask, q_offset = S_kv - T_q is the last chunk of a chunked
 *            prefill, and rows at or past the last key (q_offset + i >= S_kv - 1)
 *            see every key -- a KV block wholly before the query block, as in
 *            the ring steps of section 5.5.  S_kv >= 1 when T_q > 0.
 *   scale    softmax scale.
 *   o        device [B, H_q, T_q, d] bf16 output.
 *   lse      device [B, H_q, T_q] fp32 output.
 *   d must be 128; H_q % H_kv == 0.  T_q == 0 or B == 0 launches nothing.
 * Key tiles wholly after a query tile are never loaded.  Deterministic.
 */
GQA_API int gqa_attn_prefill_causal(const gqa_bf16_t *q, const gqa_bf16_t *k,
                                    const gqa_bf16_t *v, int B, int H_q, int H_kv, int T_q,
                                    int S_kv, int d, int q_offset, float scale, gqa_bf16_t *o,
                                    float *lse, gqa_stream_t stream);

/*
 * Bytes of device workspace that let gqa_attn_prefill_causal_ws split key
 * ranges (host only, no CUDA call).  Work is dealt in rounds of units (128
 * query rows of four heads of a KV group on a CTA pair when G is a multiple of
 * 4, else of two 128-row slots on one CTA) over the device's resident workers;
 * when the last round is partial -- or there are fewer units than workers, as
 * for a short chunk after a long prefix -- its units may be cut into pieces of
 * contiguous key tiles (at least 8 tiles each, at most 32 per unit, at most
 * four rounds of pieces over the workers; the count chosen to shorten those
 * rounds most), each piece's partial softmax state (O before division, m, l)
 * goes to the workspace and a log-sum-exp merge kernel combines them: the
 * record's split-and-reduce (sections 2.2 and 4) applied to prefill.  The
 * bound is four pieces per worker: min(32 * units, 4 * (num_sms / 2)) *
 * 266240 bytes (CTA pairs) or min(32 * units, 4 * num_sms) * 133120 bytes
 * (single CTAs), rounded up to 256; with less workspace the plan takes fewer
 * pieces (or none).  Returns 0 for invalid arguments.
 */
GQA_API size_t gqa_attn_prefill_causal_workspace_size(int B, int H_q, int H_kv, int T_q,
                                                      int S_kv, int d, int q_offset,
                                                      int num_sms);

/*
 * The prefill work plan on a device of `num_sms` SMs (one CTA per SM: num_sms / 2
 * CTA pairs when G is a multiple of 4, else num_sms CTAs) with `ws_bytes` of
 * workspace (host only, no CUDA call): writes the number of units, how many of
 * them (the last round's) are split, and the pieces per split unit (1 if
 * none).  Piece i of s of a unit with n key tiles covers tiles
 * [i*n/s, (i+1)*n/s).  Units are dealt longest first, so the split ones are
 * the shortest.  Returns GQA_OK or GQA_ERR_INVALID_ARG.
 */
GQA_API int gqa_attn_prefill_causal_plan(int B, int H_q, int H_kv, int T_q, int S_kv, int d,
                                         int q_offset, int num_sms, size_t ws_bytes,
                                         int *out_units, int *out_split_units,
                                         int *out_pieces_per_unit);

/*
 * gqa_attn_prefill_causal with a workspace for key-range splitting.
 *   workspace  device scratch, 16-byte aligned, contents on entry irrelevant
 *              (overwritten); nullptr with ws_bytes == 0 is the plain call.
 *   ws_bytes   its size.  The plan splits only if the pieces it wants fit;
 *              otherwise it runs whole units (never an error for being small).
 * With a split, two kernels run on `stream`: the pair kernel and the merge
 * (a programmatic dependent).  Results agree with the plain call within
 * rounding (the split changes the fp32 summation order); repeated calls with
 * the same sizes and workspace size are bit-identical.
 */
GQA_API int gqa_attn_prefill_causal_ws(const gqa_bf16_t *q, const gqa_bf16_t *k,
                                       const gqa_bf16_t *v, int B, int H_q, int H_kv, int T_q,
                                       int S_kv, int d, int q_offset, float scale, gqa_bf16_t *o,
                                       float *lse, void *workspace, size_t ws_bytes,
                                       gqa_stream_t stream);

/*
 * Causal prefill over a paged KV cache (block table): the chunked prefill of a
 * serving engine, whose prefix (and, once appended, the chunk's own keys) live
 * in the same pages as decode reads (see gqa_attn_decode_paged).
 *
 *   k_pages, v_pages   device [num_pages, H_kv, page_size, d] bf16; read only.
 *   block_table        device [B, max_pages_per_seq] int32: keys
 *                      [i*page_size, (i+1)*page_size) of sequence b are in page
 *                      block_table[b*max_pages_per_seq + i]; entries past key
 *                      S_kv - 1 are never read.  An entry outside
 *                      [0, num_pages) reads zeros and is reported as
 *                      GQA_ERR_INVALID_ARG by gqa_attn_device_status.
 *   S_kv               keys of every sequence (<= max_pages_per_seq * page_size);
 *                      rows of the last page past it may hold any bits (they
 *                      are cleared before use).
 *   page_size          a positive multiple of 128 (else GQA_ERR_UNSUPPORTED).
 *   num_pages * H_kv   below 2^31.
 * Everything else is that of gqa_attn_prefill_causal_ws (the workspace size of
 * gqa_attn_prefill_causal_workspace_size serves).  Runs the CTA-pair kernel
 * when G is a multiple of 4 and S_kv a multiple of 128 (the results then equal
 * gqa_attn_prefill_causal_ws's on the same keys bit for bit), the
 * one-CTA-per-unit kernel otherwise.
 */
GQA_API int gqa_attn_prefill_causal_paged(
    const gqa_bf16_t *q, const gqa_bf16_t *k_pages, const gqa_bf16_t *v_pages,
    const int32_t *block_table, int B, int H_q, int H_kv, int T_q, int S_kv, int num_pages,
    int page_size, int max_pages_per_seq, int d, int q_offset, float scale, gqa_bf16_t *o,
    float *lse, void *workspace, size_t ws_bytes, gqa_stream_t stream);

/*
 * Kernels one gqa_attn_prefill_causal_ws call with `ws_bytes` of workspace
 * launches on the current device: 1, 2 (split + merge), 0 for an empty
 * problem.  Initialises the library's per-device state (a CUDA call).
 */
GQA_API int gqa_attn_prefill_causal_kernel_count(int B, int H_q, int H_kv, int T_q, int S_kv,
                                                 int d, int q_offset, size_t ws_bytes,
                                                 int *out_kernels);

/* ------------------------------------------------------------------------- */
/* Combination of attention states over key shards                            */
/* ------------------------------------------------------------------------- */

/*
 * Combines attention states computed over disjoint key shards (record:
 * section 4 "Reduction", the associative log-sum-exp merge, here of
 * finalised states).  For each row r and shards i = 0 .. n_parts-1:
 *     lse[r] = ln sum_i exp(lse_parts[i][r])
 *     o[r]   = sum_i exp(lse_parts[i][r] - lse[r]) * o_parts[i][r]
 * A shard with lse = -inf (no visible key) contributes nothing; a row with
 * -inf in every shard gets O = 0, lse = -inf.  The shard states are outputs
 * of this library's calls over key shards, e.g. decode over a shared prefix
 * and over each sequence's own suffix, or the KV shards of a
 * sequence-parallel decode gathered from several GPUs (section 4's reduce
 * across ranks; the gather itself is the caller's).
 *
 *   o_parts    device [n_parts, rows, d] bf16 (each shard's normalised O).
 *   lse_parts  device [n_parts, rows] fp32 (natural log, scaled scores).
 *   n_parts    >= 1; rows >= 0 (rows == 0 launches nothing); d must be 128.
 *   o          device [rows, d] bf16 output; lse device [rows] fp32 output.
 * One kernel on `stream`, launched as a programmatic dependent.  The result
 * differs from one call over all keys by the rounding of the bf16 shard
 * outputs (at most about 2^-9 relative per element of O).
 */
GQA_API int gqa_attn_merge_states(const gqa_bf16_t *o_parts, const float *lse_parts,
                                  int n_parts, long long rows, int d, gqa_bf16_t *o, float *lse,
                                  gqa_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Host-buffer variants (whole-call end-to-end path)                           */
/* ------------------------------------------------------------------------- */

/*
 * Device bytes gqa_attn_decode_from_host needs in `device_arena`: room for q,
 * k_cache, v_cache, seqlens, o, lse and the decode workspace, each 256-byte
 * aligned.  Host only; 0 for invalid arguments.
 */
GQA_API size_t gqa_attn_decode_from_host_arena_size(int B, int H_q, int H_kv, int S_max, int d,
                                                    int num_sms, int num_splits);

/*
 * gqa_attn_decode on HOST buffers: copies q, k_cache, v_cache and seqlens from
 * host memory into `device_arena` (cudaMemcpyAsync on `stream`), runs the
 * decode there, and copies o and lse back to host memory.  Host buffers should
 * be page-locked for the copies to be asynchronous.  The call returns once the
 * work is queued; the host outputs are valid after the stream synchronises.
 * Argument rules are those of gqa_attn_decode; `device_arena` must hold
 * gqa_attn_decode_from_host_arena_size(...) bytes and be 256-byte aligned.
 */
GQA_API int gqa_attn_decode_from_host(const gqa_bf16_t *q_host, const gqa_bf16_t *k_cache_host,
                                      const gqa_bf16_t *v_cache_host,
                                      const int32_t *seqlens_host, int B, int H_q, int H_kv,
                                      int S_max, int d, float scale, int num_splits,
                                      gqa_bf16_t *o_host, float *lse_host, void *device_arena,
                                      size_t arena_bytes, gqa_stream_t stream);

/* Device bytes gqa_attn_prefill_causal_from_host needs (q, k, v, o, lse). */
GQA_API size_t gqa_attn_prefill_causal_from_host_arena_size(int B, int H_q, int H_kv, int T_q,
                                                            int S_kv, int d);

/* gqa_attn_prefill_causal on host buffers, staged through `device_arena`. */
GQA_API int gqa_attn_prefill_causal_from_host(const gqa_bf16_t *q_host, const gqa_bf16_t *k_host,
                                              const gqa_bf16_t *v_host, int B, int H_q,
                                              int H_kv, int T_q, int S_kv, int d, int q_offset,
                                              float scale, gqa_bf16_t *o_host, float *lse_host,
                                              void *device_arena, size_t arena_bytes,
                                              gqa_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Diagnostics                                                                 */
/* ------------------------------------------------------------------------- */

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word.  Kernels set it when a bounded wait runs out (GQA_ERR_TIMEOUT) or when a
 * decode finds a device-side input out of range (GQA_ERR_INVALID_ARG): a seqlens
 * entry outside [0, S_max] (used clamped) or a block-table entry outside
 * [0, num_pages) (its keys read as zeros).  *out_status receives GQA_OK or that
 * code.  Returns GQA_ERR_CUDA if a CUDA call fails.
 */
GQA_API int gqa_attn_device_status(gqa_stream_t stream, int *out_status);

/*
 * Exercises the bounded wait: launches one CTA that waits on a shared-memory
 * barrier nobody arrives at, with a limit of `timeout_us` microseconds
 * (1 .. 1000000).  The kernel gives up, records GQA_ERR_TIMEOUT in the status
 * word read by gqa_attn_device_status, and returns; nothing traps or hangs.
 */
GQA_API int gqa_attn_selftest_bounded_wait(int timeout_us, gqa_stream_t stream);

/*
 * Bounds-checked builds (libgqa_attn_debug.so, compiled with GQA_DEBUG_BOUNDS)
 * check, in every kernel, the index of each global store against the extent
 * the kernel derives from its arguments; a store past it is skipped and
 * GQA_ERR_OUT_OF_BOUNDS is recorded in the status word read by
 * gqa_attn_device_status.  A stand-in for a memory checker: slower, same
 * results.  gqa_attn_bounds_checked returns 1 in such a build, else 0.
 * gqa_attn_selftest_bounds launches one store one element past its range, which
 * a bounds-checked build records (and skips); release builds return
 * GQA_ERR_UNSUPPORTED and launch nothing.
 */
GQA_API int gqa_attn_bounds_checked(void);
GQA_API int gqa_attn_selftest_bounds(gqa_stream_t stream);

/*
 * Causal tile count (ADR-0060, section 11 "Verification plan": the causal
 * prefill must issue the lower-triangular number of Q K^T tile products, never
 * a full square).  Bounds-checked builds count every S = Q K^T product of one
 * query head's 128-row tile with one 128-key tile that the prefill kernels
 * issue (key-range pieces of a split unit each count their own tiles).  This
 * call waits for `stream`, stores the count since the previous call in
 * *out_count and resets it to 0 (a device-wide counter: concurrent prefill
 * calls on other streams add to it).  Release builds return GQA_ERR_UNSUPPORTED.
 * Expected values: query tile t of a head (rows [128t, min(128t + 128, T_q)))
 * sees key tiles 0 .. min((q_offset + min(128t + 128, T_q) - 1) / 128,
 * (S_kv - 1) / 128), and the sum of those counts over every (sequence, query
 * head, query tile) is the causal count.  One known excess: for odd group sizes the group's last head runs query
 * tiles t and t - 1 in one unit over tile t's key range (one more key tile for
 * tile t - 1, wholly in its future and masked), and a lone tile 0 in such a unit
 * is paired with a discarded copy of itself.
 */
GQA_API int gqa_attn_debug_s_tile_count(gqa_stream_t stream, unsigned long long *out_count);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* GQA_ATTN_H_ */
