/*
 * compkv.h -- C ABI of the CompKV decode-step library (libcompkv.so).
 *
 * CompKV (onedev.kr/papers/157) is a compensation-aware block-sparse attention
 * for autoregressive decoding.  Per decode step, for every (sequence, KV head):
 *   1. the 16-token block that receives the new token gets its summary
 *      {|b|, kbar_b, Dbar_b, vbar_b} recomputed and the new K/V is packed into
 *      the cache  (section "어떻게 쓰나" / how it is used: the fused "update the
 *      current block's statistics and pack the new K/V" kernel; the summary is
 *      defined in section "무엇과 다른가" / how it differs);
 *   2. every block is scored from its summary (same section):
 *        zbar_{g,b}   = q_g . kbar_b / sqrt(d)
 *        sigma2_{g,b} = (1/d) sum_t (sum_{i in G_t} q_{g,i}^2) (Dbar_b)_t
 *        phat_{g,b}   = |b| exp(zbar + sigma2/2) / sum_c |c| exp(zbar_c + sigma2_c/2)
 *        S_b          = sum_g phat_{g,b} sigma2_{g,b}
 *   3. the sink block and the two most recent blocks are always selected and
 *      count against the K-block budget; the rest of the budget goes to the
 *      highest S_b, ties to the lower block index (same section);
 *   4. exact attention over the selected blocks' bf16 K/V, and
 *   5. Mean compensation: each unselected block adds |b| exp(zbar_{g,b}) vbar_b
 *      to the numerator and |b| exp(zbar_{g,b}) to the denominator; both parts
 *      share one normaliser (sections "무엇과 다른가" and "어떻게 동작하나").
 *
 * Everything (the bf16 cache, the fp32 summaries, the scratch) lives in the
 * memory of one GPU.  The library allocates no device memory: every device
 * buffer below is owned by the caller.  Every call is asynchronous on the
 * caller's CUDA stream (passed as `void*`, a cudaStream_t; NULL = legacy
 * default stream) and returns after enqueueing its kernels.
 *
 * Shapes.  B = batch (sequences), Hkv = KV heads, G = query heads per KV head
 * (query head j reads KV head j / G), d = head dim (64 or 128), r = variance
 * groups (r divides d; group t = coordinates [t*d/r, (t+1)*d/r)), block = 16
 * tokens, K = budget_tokens / 16 selected blocks, L = tokens of a sequence,
 * N = ceil(L / 16) blocks (the last may be partial).
 *
 * Cache layout ("rows").  One row = one 16-token block of one (layer,
 * sequence, KV head).  Row index of block b of (layer l, sequence s, head h):
 *     l * rows_per_layer + seq_row0[s] + h * cap_blocks[s] + b
 * where cap_blocks[s] = capacity_tokens[s] / 16 (or max_tokens / 16 for every
 * sequence), seq_row0[s] = Hkv * sum_{s' < s} cap_blocks[s'] and
 * rows_per_layer = Hkv * sum_s cap_blocks[s].  compkv_row_offset() returns the
 * first row of a (layer, sequence, head).  Per row:
 *     k, v   : bf16 [16][d]  (token j of block b at position 16 b + j)
 *     kbar   : fp32 [d]      mean key of the block's tokens
 *     vbar   : fp32 [d]      mean value
 *     dbar   : fp32 [r]      per group, mean over its coordinates of the
 *                            within-block population variance of the keys
 * |b| is implicit: 16 for every block but the last, L - 16 (N - 1) for it.
 * seq_len: int32 [num_layers][B], device memory, the tokens held by each
 * (layer, sequence); compkv_append and compkv_decode increment it.
 *
 * Queries q: fp32 [B][Hkv*G][d].  New tokens k_new, v_new: bf16 [B][Hkv][d].
 * Outputs out: fp32 [B][Hkv*G][d].  Selections sel: int32 [B][Hkv][K], the
 * selected block indices ascending, padded with -1 when N < K.
 *
 * Errors.  Argument and shape problems are detected on the host and returned
 * synchronously (nothing is enqueued); compkv_last_error() then describes the
 * problem.  Problems found by a kernel (a sequence at capacity, an invalid
 * selection passed to compkv_attend, a bounded wait that ran out) set a status
 * word in the scratch buffer; compkv_device_status() synchronises the stream,
 * reads it and clears it.  No call throws, aborts or falls back to the CPU.
 *
 * Threading: a compkv_ctx may be used from one host thread at a time; calls on
 * one context must be ordered on one stream (they share the scratch buffer).
 */
#ifndef COMPKV_H
#define COMPKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  COMPKV_OK = 0,
  COMPKV_ERR_INVALID_ARG = 1,      /* null pointer, bad layer index, bad size      */
  COMPKV_ERR_UNSUPPORTED_SHAPE = 2,/* d not 64/128, r does not divide d, G > 8 ... */
  COMPKV_ERR_CAPACITY = 3,         /* a sequence would exceed its capacity          */
  COMPKV_ERR_CUDA = 4,             /* a CUDA runtime call failed                    */
  COMPKV_ERR_TIMEOUT = 5,          /* a bounded device-side wait ran out            */
  COMPKV_ERR_BAD_SELECTION = 6,    /* compkv_attend got indices not ascending / out of range */
  COMPKV_ERR_INTERNAL = 7          /* a device-side consistency check failed (a bug)       */
} compkv_status;

typedef struct {
  int num_layers;               /* >= 1                                             */
  int batch;                    /* B, 1..64                                         */
  int num_kv_heads;             /* Hkv >= 1                                         */
  int group_size;               /* G, 1..8                                          */
  int head_dim;                 /* d, 64 or 128                                     */
  int block_size;               /* must be 16 (the page's block size)               */
  int r;                        /* variance groups, 1..d, divides d, power of two   */
  int budget_tokens;            /* multiple of 16, K = budget/16 >= 3               */
  int max_tokens;               /* per-sequence capacity (multiple of 16) when      */
                                /* capacity_tokens is NULL                          */
  const int *capacity_tokens;   /* optional host array [batch], each a multiple of  */
                                /* 16: ragged per-sequence capacities; copied       */
  int variant;                  /* 0 = CompKV as defined; or an OR of the           */
                                /* COMPKV_VARIANT_* ablation bits below             */
} compkv_config;

/* Ablations of the method, named in section "전제와 한계" (assumptions and
 * limits) of the CompKV page; each bit switches one term off in every call of
 * a context:
 *   FIRST_ORDER_MASS    phat uses |b| exp(zbar) instead of |b| exp(zbar + sigma2/2)
 *                       (no second-order mass correction);
 *   NO_VARIANCE_FACTOR  S_b = sum_g phat_{g,b} (no external variance factor);
 *   NO_COMPENSATION     unselected blocks are dropped: the output is softmax
 *                       attention over the selected blocks alone (with G = 1 the
 *                       selection is then Top-K by estimated mass, the appendix
 *                       case of section "어떻게 동작하나"). */
#define COMPKV_VARIANT_FIRST_ORDER_MASS 1
#define COMPKV_VARIANT_NO_VARIANCE_FACTOR 2
#define COMPKV_VARIANT_NO_COMPENSATION 4

/* Placement.  kbar, vbar, dbar, seq_len and scratch are device memory.  k and
 * v are both device memory, or both page-locked host memory mapped at the same
 * address on the device (cudaHostAlloc / cudaMallocHost): the host placement
 * is the GB300 form of the page's offloaded cache (section "어떻게 쓰나": KV in
 * pinned CPU memory), read by the GPU over its chip-to-chip link, while the
 * summaries stay in GPU memory.  compkv_init recognises the placement from the
 * pointers and rejects anything else (pageable or managed memory, or k and v
 * in different places).  In device memory the cache may hold at most 2^31
 * token slots (num_layers * rows_per_layer * 16): its blocks are read through
 * tensor maps. */
typedef struct {
  void  *k;                     /* bf16 [num_layers * rows_per_layer][16][d]         */
  void  *v;                     /* bf16, same shape                                 */
  float *kbar;                  /* fp32 [num_layers * rows_per_layer][d]            */
  float *vbar;                  /* fp32 [num_layers * rows_per_layer][d]            */
  float *dbar;                  /* fp32 [num_layers * rows_per_layer][r]            */
  int   *seq_len;               /* int32 [num_layers][batch]                        */
  void  *scratch;               /* compkv_scratch_bytes() bytes, 256-byte aligned,  */
                                /* zero-filled by compkv_init                       */
  size_t scratch_bytes;
} compkv_buffers;

typedef struct compkv_ctx compkv_ctx;

/* Rows of one layer (rows_per_layer, see "Cache layout"); 0 on a bad config. */
int64_t compkv_rows_per_layer(const compkv_config *cfg);

/* Bytes of device scratch a context of this configuration needs; 0 on a bad config. */
size_t compkv_scratch_bytes(const compkv_config *cfg);

/* Validate cfg and bufs, zero the scratch (synchronously) and create a context.
 * It also sets, on the current device, the decode kernels' dynamic
 * shared-memory limits (raised, never lowered) and permission for clusters of
 * more than 8 CTAs, so that calls launch without those driver calls.  The
 * library keeps the pointers; the caller keeps ownership of every buffer and
 * must keep them alive until compkv_destroy. */
compkv_status compkv_init(const compkv_config *cfg, const compkv_buffers *bufs, compkv_ctx **out);

/* First row of (layer, seq, head) and that sequence's capacity in blocks. */
compkv_status compkv_row_offset(const compkv_ctx *ctx, int layer, int seq, int head,
                                int64_t *first_row, int *capacity_blocks);

/* Bulk build: the caller has written tokens [0, lens[s]) of every sequence of
 * `layer` into k/v; compute the summaries of all their blocks and set
 * seq_len[layer][s] = lens[s].  lens: host int32 [batch], 0 <= lens[s] <= capacity.
 * (The page keeps the summaries up to date token by token; a bulk build over
 * whole blocks is the same definition applied to a prefilled cache.) */
compkv_status compkv_prefill(compkv_ctx *ctx, int layer, const int *lens, void *stream);

/* Step 1 alone: write token seq_len into every (sequence, head) of `layer`,
 * recompute the summary of the block that holds it from its tokens, and
 * increment seq_len.  k_new, v_new: device bf16 [B][Hkv][d].  A sequence at
 * capacity is left unchanged and raises COMPKV_ERR_CAPACITY in the device status. */
compkv_status compkv_append(compkv_ctx *ctx, int layer, const void *k_new, const void *v_new,
                            void *stream);

/* Steps 2-3: scores and selection for the current cache.  q: device fp32
 * [B][Hq][d].  sel: device int32 [B][Hkv][K] (required).  scores: optional
 * device fp32 [B][Hkv][max_cap_blocks] receiving S_b for b < N (NULL to skip);
 * max_cap_blocks = the largest capacity in blocks. */
compkv_status compkv_score_select(compkv_ctx *ctx, int layer, const float *q, int *sel,
                                  float *scores, void *stream);

/* Steps 4-5 for a given selection: exact attention over the listed blocks and
 * Mean compensation for every other block, jointly normalised.  sel: device
 * int32 [B][Hkv][K], ascending, entries in [0, N), padded with -1.  A
 * non-ascending or out-of-range entry is skipped and raises
 * COMPKV_ERR_BAD_SELECTION in the device status.  out: device fp32 [B][Hq][d]. */
compkv_status compkv_attend(compkv_ctx *ctx, int layer, const float *q, const int *sel,
                            float *out, void *stream);

/* Steps 1-5 fused: append (k_new, v_new), score, select and attend, reading
 * every block summary once.  sel: optional device int32 [B][Hkv][K] that
 * receives the selection (NULL to skip). */
compkv_status compkv_decode(compkv_ctx *ctx, int layer, const float *q, const void *k_new,
                            const void *v_new, float *out, int *sel, void *stream);

/* Steps 1-5 from host memory to host memory, for callers whose inputs and
 * outputs live on the host: q (fp32 [B][Hq][d]), k_new and v_new (bf16
 * [B][Hkv][d]) go into staging space inside the context's scratch, the decode
 * step of compkv_decode runs on them, out (fp32 [B][Hq][d]) and, when sel_host
 * is not NULL, the selection (int32 [B][Hkv][K]) come back, and `stream` is
 * synchronised: when it returns COMPKV_OK, out_host holds the result.  When
 * every buffer is page-locked host memory mapped at the same address on the
 * device (cudaHostAlloc) and 16-byte aligned, the inputs come in through one
 * small kernel and the kernels write out and the selection straight into host
 * memory; otherwise each buffer is copied with cudaMemcpyAsync.  Device-side
 * problems are reported by compkv_device_status as for compkv_decode. */
compkv_status compkv_decode_host(compkv_ctx *ctx, int layer, const float *q_host, const void *k_new_host,
                                 const void *v_new_host, float *out_host, int *sel_host, void *stream);

/* Scratch-free decode step.  The CompKV page has no counterpart to this call;
 * it exists for callers that cannot allocate device memory at the time they
 * decode (an engine that reserved the whole GPU for its cache pool at
 * start-up and hands plug-ins no allocator, code under a hard memory budget
 * where a new allocation would fail or synchronise the device, or a host
 * application that owns the CUDA context and forbids its plug-ins to
 * allocate).  It does exactly what compkv_decode does for `layer`, without a
 * context: `cfg` and `bufs` are as for compkv_init, except that bufs->scratch
 * and bufs->scratch_bytes are ignored.  The scratch is instead a device array
 * of COMPKV_STATIC_SCRATCH_BYTES (16 MiB) inside the library, which every GPU
 * that loads the library holds until the process exits.  A configuration
 * whose compkv_scratch_bytes() exceeds that size is rejected with
 * COMPKV_ERR_UNSUPPORTED_SHAPE and a message naming both sizes.  The call
 * allocates nothing; it enqueues a clear of the array's status word and
 * counters and the decode kernels on `stream`.  The first call on each device
 * (with that device current) looks up the array's device address once and
 * keeps it for the life of the process; make that first call before any
 * stream capture.  A cudaDeviceReset() destroys the array with the context,
 * and the kept address is then stale: do not call compkv_decode_static after
 * a reset of a device it has run on.  All calls share the one array, so
 * calls whose work overlaps on the GPU (different streams, or several host
 * threads) race and corrupt each other: order them on one stream.  None of
 * its device-side checks is reported back (a sequence at capacity, a bounded
 * wait that ran out): the status word is cleared by the next call and no call
 * reads it, so check capacities on the host.  Returns host-side errors like
 * compkv_decode. */
#define COMPKV_STATIC_SCRATCH_BYTES (16u << 20)
compkv_status compkv_decode_static(const compkv_config *cfg, const compkv_buffers *bufs, int layer,
                                   const float *q, const void *k_new, const void *v_new, float *out,
                                   int *sel, void *stream);

/* Synchronise `stream`, read and clear the device status word.  Returns
 * COMPKV_OK or the first device-side error since the last call. */
compkv_status compkv_device_status(compkv_ctx *ctx, void *stream);

/* Failure-path self-test: enqueues one kernel whose bounded wait on an
 * mbarrier that nothing completes runs out (after its poll cap; no trap, no
 * hang) and records COMPKV_ERR_TIMEOUT in the context's status word, which
 * compkv_device_status() then returns (and clears).  Touches nothing else. */
compkv_status compkv_selftest_wait_timeout(compkv_ctx *ctx, void *stream);

/* Kernel launches enqueued by this context since compkv_init (host counter). */
int64_t compkv_launch_count(const compkv_ctx *ctx);

/* Per-kernel timing (tracing aid, off by default).  enable = 1: every API
 * call that launches kernels is bracketed by two CUDA events on the launch
 * stream; enable = 2: in addition each kernel of a two-kernel chain is
 * bracketed on its own (the events between them stop the second kernel from
 * launching early behind the first, so chains run slower); 0 switches it
 * off; other values give COMPKV_ERR_INVALID_ARG.  compkv_profile_read()
 * synchronises on the recorded events and returns, for one kernel family, the
 * summed device time in milliseconds and the number of launches since the
 * last read (then resets them).  Families COMPKV_KERNEL_PREFILL, _APPEND,
 * _SCORE, _ATTEND and _DECODE time whole API calls (compkv_prefill,
 * compkv_append, compkv_score_select, compkv_attend, compkv_decode).  A
 * score/select, attend or decode call launches two kernels, each timed on its
 * own (enable = 2) under COMPKV_KERNEL_K_STREAM (append, and the stream over
 * every block summary: zbar, sigma2, the logsumexp parts and the compensation
 * sums) and COMPKV_KERNEL_K_POST (LSE, S_b, forced set + Top-K, attention,
 * compensation and the joint normalisation).  Events are host-side CUDA
 * objects; no device memory is allocated. */
enum {
  COMPKV_KERNEL_PREFILL = 0,
  COMPKV_KERNEL_APPEND = 1,
  COMPKV_KERNEL_SCORE = 2,
  COMPKV_KERNEL_SELECT = 3,   /* reserved (no call of its own) */
  COMPKV_KERNEL_ATTEND = 4,
  COMPKV_KERNEL_DECODE = 5,
  COMPKV_KERNEL_K_STREAM = 6,
  COMPKV_KERNEL_K_POST = 7,
  COMPKV_KERNEL_FAMILIES = 8
};
compkv_status compkv_profile_enable(compkv_ctx *ctx, int enable);

/* Work-item trace of the decode chain (tracing aid, off by default).  buf:
 * caller device memory, 8-byte aligned, `bytes` long, zeroed by the caller
 * before a traced call.  Word 0 is unused; record slot i occupies words
 * 1 + 8 i .. 8 + 8 i, for i < (bytes - 8) / 64 (slots beyond are not
 * written).  Times are %globaltimer nanoseconds.  With W CTAs in the stream
 * kernel's grid (in a call that appends, its first CTAs recompute the open
 * blocks and the rest stream the summaries) and X CTAs (C per unit) in the
 * second kernel:
 *   slot x < W, stream CTA x: (x << 32 | segments it processed), 0, t0 its
 *     start, t1 its plan known (after waiting for the previous work), t2 its
 *     first segment done, t3 its end;
 *   slot W + x, CTA x of the second kernel: (x << 32 | 1 << 24 | cluster
 *     rank), unit (= sequence * Hkv + head), t0 its start, t1 the end of its
 *     wait for the stream kernel, t2 = t3 its attention done, t4 its end, and
 *     the unit's selected block count;
 *   slots W + k X + x, k = 1 .. 5: (x << 32 | (k + 1) << 24 | ...) and seven
 *     phase times of CTA x each (0 for a phase it did not reach).
 * A slot a call does not use stays as the caller left it.  buf = NULL
 * switches tracing off. */
compkv_status compkv_trace(compkv_ctx *ctx, void *buf, size_t bytes);
compkv_status compkv_profile_read(compkv_ctx *ctx, int family, double *total_ms, int64_t *launches);

/* Description of the last error returned on this host thread ("" if none). */
const char *compkv_last_error(void);

/* Name of a status code. */
const char *compkv_status_string(compkv_status s);

/* Free the context (host memory only; caller buffers are untouched). */
void compkv_destroy(compkv_ctx *ctx);

#ifdef __cplusplus
}
#endif
#endif /* COMPKV_H */
