/*
 * flce.h — C ABI of the fused LM-head linear + softmax cross-entropy for GB300 (sm_103a).
 *
 * The operation (per token row i, vocabulary entry v, hidden index k):
 *   x_iv   = sum_k H[i,k] * W[v,k]                  logits Z = H W^T, never stored
 *            (ai-infra-kb M011 "模型最后一层为什么也能占很多内存", §01: W is the [V, D]
 *             output weight, Z = H W^T)
 *   z_iv   = softcap > 0 ? softcap * tanh(x_iv / softcap) : x_iv
 *            (Unsloth fused-CE notes, §4 forward: optional Gemma-2 softcap scaling)
 *   lse_i  = log sum_v exp(z_iv), computed as max + log sum exp(z - max)
 *            (ai-infra-kb M011, §03 stable per-row form; vocabulary tiles merged with
 *             the running (max, sum) rule of §05)
 *   loss_i = lse_i - z_{i,y_i} for valid rows, 0 for ignored rows
 *            (Liger-CCE blog, §三 "CCE": LSE term plus the indexed-matmul target term)
 *   mean   = sum_i loss_i / n_valid, divided once by the valid count
 *            (ai-infra-kb M011, §04 and §07; Unsloth notes, §4 "n_items")
 * Backward (ai-infra-kb M011, §06; Liger-CCE blog, §二 observation 1):
 *   dZ_iv  = (exp(z_iv - lse_i) - [v == y_i]) * scale_i * (softcap > 0 ? 1 - tanh^2(x_iv/softcap) : 1)
 *   dH     = dZ W   (summed over the vocabulary),   dW = dZ^T H   (summed over tokens)
 *   scale_i = grad/n_valid (mean), grad (sum), grad_i (none); 0 for ignored rows.
 *
 * Conventions shared by every entry point
 *   - Pointers marked (device) are CUDA device pointers on the current device; the
 *     library never allocates or frees memory.  The caller owns every buffer.
 *   - H is [N, Hd] and W is [V, Hd], bf16, row-major and dense (row pitch = Hd
 *     elements).  labels is [N] int64.  Base addresses must be 16-byte aligned and
 *     Hd a multiple of 8 (TMA needs 16-byte row pitches).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  All work is
 *     enqueued on it asynchronously and no call synchronises the host; argument
 *     errors are detected and returned before anything is enqueued.
 *   - A label equal to ignore_index is ignored.  A label outside [0, V) that is not
 *     ignore_index is "bad": it is counted in counts[1] and the row is treated as
 *     ignored (nothing traps on the device).
 *   - Mean with n_valid == 0 gives loss 0 and zero gradients; counts[0] == 0 tells
 *     the caller.  N == 0 is allowed (loss 0, counts 0, dW zeroed).
 *   - Results are deterministic: every reduction runs in a fixed order, so two calls
 *     on the same device with the same arguments give bitwise-identical outputs.
 *   - Device-side errors set bits in counts[2] (FLCE_DEVERR_*): a bounded wait that
 *     expires (the kernels then stop early instead of hanging) or an out-of-range
 *     vocabulary-order entry (the access is skipped).
 *   - Kernels are built for sm_103a only; other devices get FLCE_ERR_UNSUPPORTED.
 */
#ifndef FLCE_H_
#define FLCE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FLCE_API __attribute__((visibility("default")))
#else
#define FLCE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum flce_status {
  FLCE_OK = 0,
  FLCE_ERR_ARG = 1,          /* null pointer, negative size, unknown reduction, NaN    */
  FLCE_ERR_ALIGN = 2,        /* a base address is not 16-byte aligned, or Hd % 8 != 0 */
  FLCE_ERR_WORKSPACE = 3,    /* workspace smaller than the size query, or not 256-B aligned */
  FLCE_ERR_OVERFLOW = 4,     /* a size overflows 64-bit byte counts or the 2^31 TMA limits */
  FLCE_ERR_CUDA = 5,         /* a CUDA runtime call failed; see flce_last_cuda_error() */
  FLCE_ERR_UNSUPPORTED = 6   /* device is not sm_103                                    */
} flce_status;

typedef enum flce_reduction {
  FLCE_REDUCTION_MEAN = 0,   /* loss[0] = sum of valid losses / n_valid (0 if n_valid == 0) */
  FLCE_REDUCTION_SUM = 1,    /* loss[0] = sum of valid losses                               */
  FLCE_REDUCTION_NONE = 2    /* loss[i] = per-row loss, 0 for ignored rows                  */
} flce_reduction;

/* counts[2] bits */
#define FLCE_DEVERR_WAIT_TIMEOUT 1u  /* an mbarrier wait exceeded its limit */
#define FLCE_DEVERR_BAD_INDEX 2u     /* a vocabulary order entry outside [0, V) (never
                                        expected; the access it would index is skipped) */

/* Backward options (bit flags). */
#define FLCE_BWD_SORT_VOCAB 1u   /* process the vocabulary in sorted order (flce_vocab_order) */
#define FLCE_BWD_COMPENSATED 2u  /* carry dZ's bf16 rounding remainder into dH and dW */

/* Bytes of scratch that flce_forward needs for these sizes (0 when N == 0 is fine).
   Returns 0 and sets no error for invalid sizes; flce_forward reports those. */
FLCE_API size_t flce_forward_workspace_size(int64_t N, int64_t Hd, int64_t V);

/* Bytes of scratch that flce_backward needs.  The backward runs on the rows that carry
   a gradient only (a valid label and a non-zero upstream gradient; every other row's
   gradient is exactly zero): it gathers them, in order, into a compact bf16 copy of H
   (N rounded up to 256 rows) with their per-row data and a row map, and their count stays
   on the device.  It walks the vocabulary in
   chunks of Vc columns and keeps one bf16 [N, Vc] dZ chunk plus an fp32 [N, Hd] dH
   accumulator (the latter only when there is more than one chunk, or when dH is split),
   plus one byte per 64 x 64 block of the chunk for the filtered mode.  When the dH
   product has too few 256 x 256 output tiles to fill the GPU's SM pairs evenly (fewer
   than about 300: N x Hd below roughly 8192 x 4096), each tile's vocabulary range is
   split into up to 4 parts and parts 2..4 keep their fp32 [N, Hd] sums here until they
   are added to the accumulator.  With FLCE_BWD_SORT_VOCAB it also
   holds a bf16 [Vc, Hd] copy of the chunk's weight rows in sorted order and the order
   itself (about 28 bytes per vocabulary row); with FLCE_BWD_COMPENSATED a second bf16
   [N, Vc] chunk (the rounding remainder of dZ).
   chunk_budget_bytes bounds the dZ chunk(s) plus that weight copy (0 = default 512 MiB):
   at most budget / (2 N, 4 N when compensated, + 2 Hd when sorting) columns, rounded down
   to 256; the vocabulary's 256-column tiles are dealt out over the fewest chunks that
   bound allows, as evenly as whole tiles allow (widths differ by at most 256 columns), and
   the widest chunk Vc sets the size.  The same budget and options must be passed to
   flce_backward.  Unknown option bits: returns 0. */
FLCE_API size_t flce_backward_workspace_size(int64_t N, int64_t Hd, int64_t V, size_t chunk_budget_bytes,
                                             unsigned options);

/* Forward: loss, per-row LSE (saved for the backward), target logits and counts.
 *   H            (device) bf16 [N, Hd]
 *   W            (device) bf16 [V, Hd]
 *   labels       (device) int64 [N]
 *   ignore_index label value that marks an ignored row (PyTorch default -100)
 *   softcap      tanh logit softcap c; <= 0 turns it off
 *   reduction    flce_reduction
 *   loss         (device) fp32 [1] for MEAN/SUM, [N] for NONE
 *   lse          (device) fp32 [N], LSE of every row (ignored rows included)
 *   target_logit (device) fp32 [N] or NULL: z_{i,y_i} (capped), 0 for ignored rows
 *   counts       (device) int64 [3]: n_valid, n_bad, device error bits (written)
 *   workspace    (device) >= flce_forward_workspace_size() bytes, 256-byte aligned
 *   stream       cudaStream_t
 * Cites: Liger-CCE blog, §三 (indexed dot for the target, tiled linear-LSE for the
 * denominator); ai-infra-kb M011, §05 (tile merge). */
FLCE_API flce_status flce_forward(const void* H, const void* W, const int64_t* labels,
                         int64_t N, int64_t Hd, int64_t V, int64_t ignore_index,
                         float softcap, int reduction,
                         float* loss, float* lse, float* target_logit, int64_t* counts,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Backward: dH and dW from the saved LSE, recomputing the logits tile by tile.
 *   H, W, labels, N, Hd, V, ignore_index, softcap, reduction: as in the forward call
 *   lse          (device) fp32 [N] from flce_forward
 *   counts       (device) int64 [3] from flce_forward; counts[0] (n_valid) scales the
 *                mean; error bits are OR-ed into counts[2]
 *   grad_out     (device) fp32 [1] (MEAN/SUM) or [N] (NONE): upstream gradient
 *   filter_threshold  0: exact backward.  > 0: gradient filtering (Liger-CCE blog, §三
 *                "CCE": softmax entries below 2^-12 vanish in a bf16 gradient): entries with
 *                p < threshold other than a valid row's target are dropped from dZ, and
 *                every 64 x 64 (token x vocabulary) block of dZ left all zero is skipped
 *                by the dW and dH products.  An approximation; the exact path is the
 *                default.  Negative or NaN: FLCE_ERR_ARG.
 *   options      0, or FLCE_BWD_SORT_VOCAB: walk the vocabulary in the order of
 *                flce_vocab_order (mean logit descending) so that the entries that
 *                survive filtering gather in few blocks and more blocks are skipped
 *                (Liger-CCE blog, §三 "CCE", vocabulary sorting).  The gradients are the
 *                same sums taken in another order; dW rows are written back to their
 *                ids.
 *                FLCE_BWD_COMPENSATED: each dZ entry d is kept as its bf16 rounding
 *                hi = bf16(d) plus the rounded remainder lo = bf16(d - hi), and dH and dW
 *                accumulate both in fp32 (|d - hi - lo| <= 2^-18 |d| instead of 2^-9): the
 *                part of the gradient that the bf16 rounding would drop is carried along,
 *                as the compensation term is in Kahan summation (Liger-CCE blog, §三: CCE's
 *                kahan variants buy precision, and kahan_full_c also leaves the vocabulary
 *                side unfiltered, for pretraining).  Requires the unfiltered gradient: with
 *                filter_threshold > 0, FLCE_ERR_ARG.  Twice the dW and dH tensor work.
 *                Options combine.  Other bits: FLCE_ERR_ARG.
 *   dH           (device) bf16 [N, Hd] (written), or NULL: dH is not computed
 *   dW           (device) bf16 [V, Hd] (written, every row), or NULL: dW is not computed
 *                (a frozen head, or hidden states that need no gradient, skip a quarter of
 *                the step).  dH and dW both NULL: FLCE_ERR_ARG.
 *   workspace    (device) >= flce_backward_workspace_size(N, Hd, V, chunk_budget_bytes)
 *   chunk_budget_bytes  as passed to the size query (0 = default)
 * Cites: ai-infra-kb M011, §06 (recompute the logit tile, p = exp(z - lse),
 * dH summed over vocabulary tiles, dW over all valid tokens); Unsloth notes, §4
 * backward (softcap derivative 1 - tanh^2). */
FLCE_API flce_status flce_backward(const void* H, const void* W, const int64_t* labels,
                          const float* lse, int64_t* counts,
                          int64_t N, int64_t Hd, int64_t V, int64_t ignore_index,
                          float softcap, int reduction, const float* grad_out,
                          float filter_threshold, unsigned options, void* dH, void* dW,
                          void* workspace, size_t workspace_bytes, size_t chunk_budget_bytes,
                          void* stream);

/* Vocabulary order used by FLCE_BWD_SORT_VOCAB (Liger-CCE blog, §三 "CCE": the mean
 * logit of every word over the batch puts the frequent words next to each other).
 *   keys  (device) fp32 [V] or NULL: key_v = (1/N) sum_i h_i . w_v, the raw logit
 *         (before any softcap) averaged over all N rows, ignored rows included, computed
 *         as hbar . w_v with hbar the fp32 column mean of H; 0 when N == 0
 *   perm  (device) int32 [V]: perm[p] = the row placed at position p; keys descending,
 *         equal keys (as fp32, -0 == +0) by ascending row
 *   inv   (device) int32 [V] or NULL: inv[perm[p]] = p
 *   workspace >= flce_vocab_order_workspace_size(N, Hd, V) bytes, 256-byte aligned.
 * Deterministic (fixed summation and merge orders).  NaN keys sort in an unspecified
 * place.  Errors as in flce_forward. */
FLCE_API size_t flce_vocab_order_workspace_size(int64_t N, int64_t Hd, int64_t V);
FLCE_API flce_status flce_vocab_order(const void* H, const void* W, int64_t N, int64_t Hd, int64_t V,
                             float* keys, int32_t* perm, int32_t* inv,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Forward pass that allocates nothing and takes no workspace.  The pages have no
 * counterpart: this entry point exists for callers that cannot allocate device memory
 * where they compute the loss (a plug-in inside a runtime that owns all device memory
 * through its own pool, a process that reserves its memory once at start-up, a path
 * that cannot afford an allocation's implicit synchronisation).
 * Arguments and outputs are those of flce_forward without workspace/workspace_bytes.
 * The forward's scratch is one static device array inside the library of
 * flce_static_scratch_bytes() bytes (16 MiB); every GPU that loads the library holds it
 * until the process exits.
 *   - Returns FLCE_ERR_WORKSPACE, before enqueuing anything, when
 *     flce_forward_workspace_size(N, Hd, V) exceeds that size (N = 8192 fits V up to
 *     about 256K; larger problems must use flce_forward with their own workspace).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call before
 *     any stream capture.  Under CUDA's lazy module loading that lookup may also load
 *     the module on the device, reserving the 16 MiB and synchronising implicitly:
 *     callers that cannot accept that on their hot path make the first call at
 *     start-up.  A failed lookup is not remembered (the next call retries it) and
 *     returns FLCE_ERR_CUDA with its error in flce_last_cuda_error(); an unsupported
 *     device returns FLCE_ERR_UNSUPPORTED, as from flce_forward.
 *   - Every call shares the one array, which keeps the last call's contents.  Nothing
 *     in it has to start at zero: each call writes every scratch word before reading
 *     it.  Calls that overlap on the GPU (on two streams, or from two host threads)
 *     race on the array and must be serialised by the caller. */
FLCE_API size_t flce_static_scratch_bytes(void);
FLCE_API flce_status flce_forward_noalloc(const void* H, const void* W, const int64_t* labels,
                                 int64_t N, int64_t Hd, int64_t V, int64_t ignore_index,
                                 float softcap, int reduction,
                                 float* loss, float* lse, float* target_logit, int64_t* counts,
                                 void* stream);

/* ---------------------------------------------------------------- vocabulary sharding
 * Vocabulary-parallel use (ai-infra-kb M011, §07: with the vocabulary split across ranks,
 * the global max, the global sum of exponentials and the target logit must be combined,
 * and dH gets a contribution from every shard; GPU CE post, §4.3).  Each rank holds the
 * rows [v_offset, v_offset + V_shard) of a vocabulary of V_total and the same H and
 * labels (labels are global ids).
 *   1. flce_forward_shard: lse_shard[i] = log sum over this shard's rows of e^{z_iv};
 *      target_shard[i] = z_{i,y_i} when y_i is one of this shard's rows, else 0;
 *      counts as in flce_forward (validity against V_total).  Workspace:
 *      flce_forward_workspace_size(N, Hd, V_shard).
 *   2. gather lse_shard and target_shard of all shards, in shard order, into
 *      [n_shards][N] arrays (e.g. an all-gather), then flce_merge_shards: global lse,
 *      loss (reduction as in flce_forward) and counts, merged in a fixed shard order.
 *   3. flce_backward_shard with the global lse and counts: dW_shard (bf16 [V_shard, Hd],
 *      complete) and dH_partial (fp32 [N, Hd], this shard's sum over its rows); the
 *      caller sums dH_partial over the shards (e.g. an all-reduce) and rounds as needed.
 *      Either output may be NULL to skip it, as in flce_backward.
 *      A row whose label lives in another shard is still a valid row here.
 *      Workspace: flce_backward_workspace_size(N, Hd, V_shard, chunk_budget_bytes, options);
 *      FLCE_BWD_SORT_VOCAB sorts this shard's rows only.
 * v_offset < 0, V_shard <= 0 or v_offset + V_shard > V_total: FLCE_ERR_ARG. */
FLCE_API flce_status flce_forward_shard(const void* H, const void* W_shard, const int64_t* labels,
                               int64_t N, int64_t Hd, int64_t V_shard, int64_t v_offset,
                               int64_t V_total, int64_t ignore_index, float softcap,
                               float* lse_shard, float* target_shard, int64_t* counts,
                               void* workspace, size_t workspace_bytes, void* stream);
/* Bytes of scratch that flce_merge_shards needs. */
FLCE_API size_t flce_merge_shards_workspace_size(int64_t N);
/*   lse_parts, target_parts (device) fp32 [n_shards][N], shard order
 *   loss (device) fp32 [1] (MEAN/SUM) or [N] (NONE); lse (device) fp32 [N] global;
 *   counts (device) int64 [3] written as by flce_forward. */
FLCE_API flce_status flce_merge_shards(const float* lse_parts, const float* target_parts, int64_t n_shards,
                              const int64_t* labels, int64_t N, int64_t V_total, int64_t ignore_index,
                              int reduction, float* loss, float* lse, int64_t* counts,
                              void* workspace, size_t workspace_bytes, void* stream);
FLCE_API flce_status flce_backward_shard(const void* H, const void* W_shard, const int64_t* labels,
                                const float* lse, int64_t* counts, int64_t N, int64_t Hd,
                                int64_t V_shard, int64_t v_offset, int64_t V_total,
                                int64_t ignore_index, float softcap, int reduction,
                                const float* grad_out, float filter_threshold, unsigned options,
                                float* dH_partial, void* dW_shard, void* workspace,
                                size_t workspace_bytes, size_t chunk_budget_bytes, void* stream);

/* Host-to-device staging, for callers that feed the entry points from host buffers
 * (the pages' methods take their inputs already on the device; this is I/O around them).
 * Copies `bytes` from pinned host memory `src` (page-locked by cudaHostAlloc /
 * cudaMallocHost or cudaHostRegister, so it has a device mapping) to device memory `dst`,
 * enqueued on `stream` as one kernel whose threads read the host buffer through that
 * mapping over the CPU-GPU link and store 16-byte words (the last bytes % 16 one by one).
 * It is meant to run on a second stream beside the library's kernels, the next step's
 * inputs arriving while this step computes: it uses no shared memory and few registers,
 * so its blocks fit beside the tensor-core kernels' one block per SM.  On GB300 a
 * copy-engine transfer (cudaMemcpyAsync) of the same bytes from host memory slowed those
 * kernels several times more (a 1 GB copy per 20 ms step: +1.6-2.0 ms against +0.3 ms).
 * Both pointers 16-byte aligned, else FLCE_ERR_ALIGN.  FLCE_ERR_ARG, nothing enqueued: a
 * null pointer (with bytes > 0), a src that is not page-locked host memory (pageable
 * memory is refused even where the GPU could reach it through address translation), or a
 * dst that is not device memory of the current device.  bytes == 0: FLCE_OK, nothing
 * enqueued.  The host buffer must stay allocated, and unchanged, until
 * the copy has run (stream order). */
FLCE_API flce_status flce_stage_h2d(void* dst, const void* src, size_t bytes, void* stream);

/* Failure-detection self-test.  The pages have no counterpart: it checks the device-side
 * bounded waits that keep a broken pipeline from hanging the GPU.  Launches one kernel
 * whose thread waits, with the same bounded mbarrier wait the tensor-core kernels use
 * (limit 2 s), on a barrier nothing arrives on.  When the stream reaches it,
 * status_word[0] (device int64, zeroed first) holds FLCE_DEVERR_WAIT_TIMEOUT and the
 * kernel has returned normally; the context stays usable. */
FLCE_API flce_status flce_selftest_wait_timeout(int64_t* status_word, void* stream);

/* Human-readable text for a flce_status value. */
FLCE_API const char* flce_strerror(int status);

/* The cudaError_t value behind the last FLCE_ERR_CUDA returned on this thread. */
FLCE_API int flce_last_cuda_error(void);

/* Instrumentation (host side, per calling thread).
 * flce_launch_count: number of kernels this thread has launched through the library.
 * flce_set_event_sink: while capacity > 0, every kernel launch k (in launch order) is
 *   bracketed by cudaEventRecord(start_events[k]) / cudaEventRecord(end_events[k]) on
 *   the launch stream and kernel_ids[k] receives its FLCE_KERNEL_* id; launches past
 *   capacity are not recorded.  Events are cudaEvent_t created by the caller.
 *   capacity 0 turns the sink off.  Returns 0.
 * flce_event_sink_used: number of launches recorded since the last flce_set_event_sink. */
#define FLCE_KERNEL_LABEL_DOT 0   /* label scan + indexed dot (target logits)          */
#define FLCE_KERNEL_LINEAR_LSE 1  /* tensor-core H W^T tiles -> per-group (max, sum)   */
#define FLCE_KERNEL_LSE_MERGE 2   /* fixed-order merge -> lse, per-row loss, row sums  */
#define FLCE_KERNEL_REDUCE 3      /* fixed-order total, counts, mean                   */
#define FLCE_KERNEL_BWD_PREP 4    /* per-row scale / label / lse for the backward      */
#define FLCE_KERNEL_DZ 5          /* tensor-core recompute of Z -> bf16 dZ chunk       */
#define FLCE_KERNEL_DW 6          /* tensor-core dW chunk = dZ^T H                     */
#define FLCE_KERNEL_DH 7          /* tensor-core dH += dZ W_chunk                      */
#define FLCE_KERNEL_ZERO 8        /* zero fill (dW when N == 0)                        */
#define FLCE_KERNEL_BLOCK_MASK 9  /* filtered backward: live K steps per dW / dH tile   */
#define FLCE_KERNEL_SELFTEST 10   /* flce_selftest_wait_timeout                        */
#define FLCE_KERNEL_SHARD_MERGE 11 /* vocabulary shards: fixed-order LSE / loss merge  */
#define FLCE_KERNEL_VOCAB_KEYS 12  /* column mean of H, mean logit per vocabulary row     */
#define FLCE_KERNEL_VOCAB_SORT 13  /* run sort + merge passes -> perm / inv               */
#define FLCE_KERNEL_GATHER 14      /* sorted chunk's weight rows -> contiguous copy       */
#define FLCE_KERNEL_DH_COMBINE 15  /* dH split: fp32 part sums added in part order        */
#define FLCE_KERNEL_COMPACT 16     /* backward: rows with a gradient gathered to the front  */
#define FLCE_KERNEL_DH_ZERO 17     /* backward: zero dH rows that carry no gradient         */
#define FLCE_KERNEL_STAGE 18       /* flce_stage_h2d: pinned host buffer -> device memory   */
FLCE_API uint64_t flce_launch_count(void);
FLCE_API int flce_set_event_sink(void* const* start_events, void* const* end_events, int* kernel_ids,
                        int capacity);
FLCE_API int flce_event_sink_used(void);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H_ */
