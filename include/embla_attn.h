/*
 * embla_attn.h — C ABI for long-context single-token decode attention of the
 * Embla 1 layer types, on one NVIDIA GB300 (sm_103a) GPU.
 *
 * The operations follow "The Architecture of Embla 1" (Sevren blog):
 *   - full layer   : section "Sevren Sparse Attention learns to be sparse" and
 *                    "Skipping V" — ReLU^2 weights over RMS-normalised query and
 *                    key, value rows read only for keys some head of the KV
 *                    group weighs above zero;
 *   - selection    : section "Three kinds of attention" (Sparse) — the 1,024
 *                    keys the full layer scored highest plus the 128 newest;
 *   - sparse layer : same section — softmax over the selected rows of the full
 *                    layer's cache, no position encoding;
 *   - window layer : same section (Sliding window) — softmax over the newest
 *                    128 keys with rotary position embedding.
 *
 * The page's display equation for the full layer was lost in extraction, so
 * its score scale (alpha), the constant added to the normaliser (c) and the
 * RMS epsilon (eps) are arguments.  With s = alpha * qhat . khat and
 * w = max(s, 0)^2, the full layer returns sum_j w_j v_j / (c + sum_j w_j), and
 * 0 where c + sum_j w_j == 0.
 *
 * Conventions shared by every call
 *   - Layouts are dense row-major.  q: [B, Hq, D] bf16.  Caches: [B, Hkv,
 *     cache_stride, D] bf16 (row j of unit (b, g) at ((b*Hkv + g)*cache_stride
 *     + j)*D).  Query head h reads KV head h / G, G = Hq / Hkv.
 *   - Every pointer argument except `shape` and `workspace_bytes`-sized host
 *     values is a DEVICE pointer owned by the caller.  The library never
 *     allocates, frees or synchronises; work is enqueued on `stream` (a
 *     cudaStream_t; NULL means the legacy default stream).
 *   - Arguments are validated on the host before any launch; a failed check
 *     returns a status and enqueues nothing.  A launch failure returns
 *     EMBLA_ERR_CUDA.  No call throws, traps or aborts.
 *   - Device pointers must be 16-byte aligned.  head_dim must be 128;
 *     G must be 4 or 8.
 *   - `workspace` is caller-provided device scratch of at least the size the
 *     matching *_workspace_size call returns for the same shape on the
 *     current device (NULL when that size is 0).  Its contents need not be initialised and are not
 *     meaningful after the call.  Calls that share a workspace must be
 *     ordered on one stream.
 *   - A *_workspace_size call returns 0 both when the shape needs no
 *     workspace and when its arguments are invalid (the size functions have
 *     no error channel); the matching call checks the same arguments itself
 *     and returns the error status.
 */
#ifndef EMBLA_ATTN_H
#define EMBLA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  EMBLA_OK = 0,
  EMBLA_ERR_INVALID_ARG = 1,   /* a null pointer, bad size, misaligned pointer, bad scalar */
  EMBLA_ERR_UNSUPPORTED = 2,   /* valid but not built: head_dim != 128, G not in {4, 8} */
  EMBLA_ERR_WORKSPACE = 3,     /* workspace smaller than the *_workspace_size result */
  EMBLA_ERR_CUDA = 4,          /* a CUDA runtime/driver call or launch failed */
  EMBLA_ERR_DEVICE_CHECK = 5   /* a kernel recorded a failed device-side check */
} embla_status;

typedef struct {
  int32_t batch;         /* B >= 0 */
  int32_t n_q_heads;     /* Hq >= 1 */
  int32_t n_kv_heads;    /* Hkv >= 1, Hq % Hkv == 0 */
  int32_t head_dim;      /* D; 128 */
  int64_t ctx_len;       /* n: keys in the cache, the current token is key n-1; 0 <= n < 2^31 */
  int64_t cache_stride;  /* rows between consecutive (b, g) planes of K and V; >= n */
} embla_shape;

/* Text for a status code (static storage, never NULL). */
const char *embla_status_string(embla_status status);

/* Number of streaming multiprocessors the launches size their grids for (current device). */
int embla_device_sm_count(void);

/*
 * Full (ReLU^2) layer decode — "Sevren Sparse Attention learns to be sparse",
 * "Skipping V".
 *   q          bf16 [B, Hq, D]              raw query (normalised inside)
 *   k_cache    bf16 [B, Hkv, cache_stride, D]
 *   v_cache    bf16 [B, Hkv, cache_stride, D]; only rows of surviving keys are read
 *   alpha      score scale, finite and > 0
 *   c          normaliser constant, finite and >= 0
 *   eps        RMS epsilon, finite and >= 0 (eps == 0 with an all-zero row gives NaN)
 *   out        fp32 [B, Hq, D]
 *   n_surv     int32 [B, Hkv]: keys j < n with max over the group of s_hj > 0
 *   sel_scores fp32 [B, Hkv, cache_stride] or NULL: sigma_j = max over the
 *              group's heads of s_hj for j < n (the selection score); rows
 *              >= n are not written
 *   sel_hist   uint32 [B, Hkv, 2048], required iff sel_scores != NULL:
 *              per unit, how many keys j < n fall in each of 2048 bins of the
 *              order-preserving 32-bit form of sigma_j (its top 11 bits).
 *              Zeroed and filled by this call; embla_select_topk reads it.
 */
size_t embla_full_decode_workspace_size(const embla_shape *shape);
embla_status embla_full_decode(const embla_shape *shape, const void *q, const void *k_cache,
                               const void *v_cache, float alpha, float c, float eps, float *out,
                               int32_t *n_surv, float *sel_scores, uint32_t *sel_hist,
                               void *workspace, size_t workspace_bytes, void *stream);

/*
 * Full (ReLU^2) layer decode over 8-bit caches — the same operation as
 * embla_full_decode, on K and V kept in 8-bit precision ("KV bridge, KV reuse,
 * and prefill": the full caches grow by 2.6 KB per token at 8 bits).  The page
 * does not name the 8-bit format; this call takes OCP FP8 E4M3 codes (bias 7,
 * no infinities, S.1111.111 is NaN, largest finite 448) with one fp32 scale per
 * (token, KV head): row j of unit u stands for scale[u][j] * decode(code[u][j][:]).
 * Results are those of embla_full_decode on those decoded rows.
 *   k_codes, v_codes   uint8 [B, Hkv, cache_stride, D] E4M3 codes
 *   k_scales, v_scales fp32 [B, Hkv, cache_stride]; cache_stride % 4 == 0
 *   every other argument, the workspace size (embla_full_decode_workspace_size)
 *   and every result as for embla_full_decode.
 * The query enters the tensor cores as three E4M3 terms per element (q = 2^e
 * (t1 + t2/16 + t3/256), 2^e a power of two per head); the sum reproduces every
 * query element of magnitude at least 2^-14 times its head's largest exactly,
 * and every other one to within 2^-25 times that largest.  Rows j >= n are read (they share 128-key tiles with
 * rows < n) but nothing they hold reaches a result.
 */
embla_status embla_full_decode_e4m3(const embla_shape *shape, const void *q,
                                    const uint8_t *k_codes, const float *k_scales,
                                    const uint8_t *v_codes, const float *v_scales, float alpha,
                                    float c, float eps, float *out, int32_t *n_surv,
                                    float *sel_scores, uint32_t *sel_hist, void *workspace,
                                    size_t workspace_bytes, void *stream);

/*
 * Full (ReLU^2) layer decode on library-owned scratch.  The Embla pages have
 * no counterpart to this call: it computes exactly what embla_full_decode
 * computes, with the same arguments and results, but takes no workspace.  It
 * is meant for callers that cannot hand the library device memory for
 * scratch: an engine that lays out all of its device memory once at start-up
 * and must not allocate while it decodes (a cudaMalloc can stall the whole
 * device and breaks up a pooled allocator), or a C program with no device
 * allocator of its own.  Nothing is allocated, here or inside: the scratch is
 * one fixed array of EMBLA_FULL_DECODE_SCRATCH_BYTES (4 MiB) in the library's
 * device memory, one per device.
 *   Limit: the scratch holds the partial records of the work split.  Where
 *     embla_full_decode would cut each CTA's share of a long batch into several
 *     pieces and their records do not fit, this call takes fewer pieces (its
 *     partial sums are then grouped differently, so results can differ from
 *     embla_full_decode's in rounding); when even one piece per CTA does not fit, it returns
 *     EMBLA_ERR_WORKSPACE and launches nothing.  On a 152-SM device that is
 *     above about 1860 (b, g) units at G = 4 and about 860 at G = 8.
 *   Set-up: the first call on a device, made with that device current, looks
 *     up the array's device address and keeps it for later calls (a failed
 *     look-up returns EMBLA_ERR_CUDA).  Make that first call before beginning
 *     any stream capture.
 *   Zeroing: none needed; the scratch (the partial records) is written before
 *     it is read.
 *   Concurrency: all calls on one device share the one array.  Two calls that
 *     may run at the same time on the device (different streams or host
 *     threads with no ordering between them) race on it and give wrong
 *     results; calls ordered on one stream are safe.
 */
#define EMBLA_FULL_DECODE_SCRATCH_BYTES ((size_t)4 << 20)
embla_status embla_full_decode_static_scratch(const embla_shape *shape, const void *q,
                                              const void *k_cache, const void *v_cache,
                                              float alpha, float c, float eps, float *out,
                                              int32_t *n_surv, float *sel_scores,
                                              uint32_t *sel_hist, void *stream);

/*
 * Sparse-layer selection — "Three kinds of attention" (Sparse): the `topk`
 * keys with the highest sel_scores among j < n - recent (equal scores: the
 * smaller index first) together with the `recent` newest keys n-recent..n-1;
 * every key when n <= topk + recent.
 *   sel_scores, sel_hist  as written by embla_full_decode for the same shape
 *   topk, recent          >= 0 (1024 and 128 in Embla 1)
 *   idx        int32 [B, Hkv, idx_stride], idx_stride >= topk + recent:
 *              selected key indices in ascending order; entries at and past
 *              count[b, g] are not written
 *   count      int32 [B, Hkv] = min(n, topk + recent)
 *   workspace  embla_select_topk_workspace_size bytes (0 for contexts up to
 *              524,288 keys, which shared memory holds), 16-byte aligned
 */
size_t embla_select_topk_workspace_size(const embla_shape *shape, int32_t topk, int32_t recent);
embla_status embla_select_topk(const embla_shape *shape, const float *sel_scores,
                               const uint32_t *sel_hist, int32_t topk, int32_t recent,
                               int32_t *idx, int32_t idx_stride, int32_t *count, void *workspace,
                               size_t workspace_bytes, void *stream);

/*
 * Full-layer decode followed by the sparse layers' selection, in one call —
 * "Three kinds of attention": the full layer's scores choose the keys its
 * block's sparse layers read.  The results are exactly those of
 * embla_full_decode (or embla_full_decode_e4m3) with sel_scores and sel_hist,
 * then embla_select_topk on them: out, n_surv, sel_scores, sel_hist, idx and
 * count as documented there (sel_scores and sel_hist are required).  The
 * selection starts as soon as the scores are complete; the full layer's
 * output is finished beside it, so the pair takes less time than the two
 * calls.  Everything is ordered on `stream` as for the two calls.
 *   workspace  embla_full_decode_select_workspace_size(shape, topk, recent)
 *              bytes, 16-byte aligned
 */
size_t embla_full_decode_select_workspace_size(const embla_shape *shape, int32_t topk,
                                               int32_t recent);
embla_status embla_full_decode_select(const embla_shape *shape, const void *q, const void *k_cache,
                                      const void *v_cache, float alpha, float c, float eps,
                                      float *out, int32_t *n_surv, float *sel_scores,
                                      uint32_t *sel_hist, int32_t topk, int32_t recent,
                                      int32_t *idx, int32_t idx_stride, int32_t *count,
                                      void *workspace, size_t workspace_bytes, void *stream);
embla_status embla_full_decode_e4m3_select(const embla_shape *shape, const void *q,
                                           const uint8_t *k_codes, const float *k_scales,
                                           const uint8_t *v_codes, const float *v_scales,
                                           float alpha, float c, float eps, float *out,
                                           int32_t *n_surv, float *sel_scores, uint32_t *sel_hist,
                                           int32_t topk, int32_t recent, int32_t *idx,
                                           int32_t idx_stride, int32_t *count, void *workspace,
                                           size_t workspace_bytes, void *stream);

/*
 * Sparse-layer decode — "Three kinds of attention" (Sparse): for every query
 * head, softmax of tau * q_h . k_j over the selected keys of its KV head
 * (no normalisation, no position), then the weighted sum of their values.
 *   q          bf16 [B, Hq, D]   this sparse layer's own query
 *   k_cache, v_cache   the full layer's caches, as for embla_full_decode
 *   idx        int32 [B, Hkv, idx_stride]; the first count[b, g] entries are
 *              read and must lie in [0, n); an entry outside is skipped and
 *              recorded (see embla_device_check)
 *   count      int32 [B, Hkv], each in [0, idx_stride]; a unit with count 0
 *              gets a zero output
 *   tau        softmax scale, finite
 *   out        fp32 [B, Hq, D]
 */
size_t embla_sparse_decode_workspace_size(const embla_shape *shape, int32_t idx_stride);
embla_status embla_sparse_decode(const embla_shape *shape, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *idx, int32_t idx_stride,
                                 const int32_t *count, float tau, float *out, void *workspace,
                                 size_t workspace_bytes, void *stream);

/*
 * Sparse-layer decode over the full layer's 8-bit caches (the format of
 * embla_full_decode_e4m3): the same operation as embla_sparse_decode on the
 * decoded rows scale * decode(codes).
 *   k_codes, v_codes, k_scales, v_scales   as for embla_full_decode_e4m3
 *   every other argument, the workspace size and the result as for
 *   embla_sparse_decode.
 * The query enters the tensor cores in f16 after division by a power of two per
 * head (exact for every element at least 2^-24 times its head's largest); the
 * value sums run in fp32.
 */
embla_status embla_sparse_decode_e4m3(const embla_shape *shape, const void *q,
                                      const uint8_t *k_codes, const float *k_scales,
                                      const uint8_t *v_codes, const float *v_scales,
                                      const int32_t *idx, int32_t idx_stride,
                                      const int32_t *count, float tau, float *out,
                                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * Selection per query head — the other reading of which score the selection ranks
 * ("Three kinds of attention", Sparse: "the 1,024 keys that layer scored highest" under
 * grouped queries): every query head h ranks the keys by its own score s_hj and keeps its
 * own top-1024 plus the newest 128; the sparse layer's head h then attends over its own
 * set.  Three calls, used in this order:
 *
 * embla_full_decode_head_scores: the full-layer decode (out and n_surv exactly as
 *   embla_full_decode) that writes each head's scores instead of the group's:
 *   head_scores fp32 [B, Hq, cache_stride] (s_hj for j < n; rows >= n not written) and
 *   head_hist uint32 [B, Hq, 2048] (the order-key histogram of each head's scores).
 *   Workspace: embla_full_decode_workspace_size.
 * embla_select_topk_per_head: embla_select_topk over the B*Hq units of those scores:
 *   idx int32 [B, Hq, idx_stride], count int32 [B, Hq].
 * embla_sparse_decode_per_head: embla_sparse_decode where query head h reads its own
 *   idx[b, h] rows of KV head h / G (workspace: embla_sparse_decode_workspace_size).
 */
embla_status embla_full_decode_head_scores(const embla_shape *shape, const void *q,
                                           const void *k_cache, const void *v_cache, float alpha,
                                           float c, float eps, float *out, int32_t *n_surv,
                                           float *head_scores, uint32_t *head_hist,
                                           void *workspace, size_t workspace_bytes, void *stream);
size_t embla_select_topk_per_head_workspace_size(const embla_shape *shape, int32_t topk,
                                                  int32_t recent);
embla_status embla_select_topk_per_head(const embla_shape *shape, const float *head_scores,
                                        const uint32_t *head_hist, int32_t topk, int32_t recent,
                                        int32_t *idx, int32_t idx_stride, int32_t *count,
                                        void *workspace, size_t workspace_bytes, void *stream);
embla_status embla_sparse_decode_per_head(const embla_shape *shape, const void *q,
                                          const void *k_cache, const void *v_cache,
                                          const int32_t *idx, int32_t idx_stride,
                                          const int32_t *count, float tau, float *out,
                                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * Full-layer prefill — causal ReLU^2 attention over a prompt ("KV bridge, KV reuse, and
 * prefill": the early layers run on every prompt token; "Sevren Sparse Attention learns
 * to be sparse": the same weights as embla_full_decode).  The prompt's n_new tokens are
 * the last n_new of the ctx_len keys already in the caches: query t of head h sits at
 * position p = ctx_len - n_new + t and sees keys 0 .. p (a full layer has no position
 * encoding).  out = sum_{j<=p} w v_j / (c + sum_{j<=p} w), 0 where that is 0.
 *   n_new      0 <= n_new <= ctx_len
 *   q          bf16 [B, Hq, n_new, D]   raw queries (normalised inside), head-major
 *   k_cache, v_cache   bf16 [B, Hkv, cache_stride, D], rows 0 .. ctx_len-1 read
 *   alpha, c, eps      as for embla_full_decode
 *   out        fp32 [B, Hq, n_new, D]
 *   workspace  the keys' norms, fp32 [B, Hkv, ctx_len rounded up to 4]
 *              (embla_prefill_workspace_size)
 * The scores and the value sums run on the tensor cores with fp32 accumulation; the
 * weights enter the value product as two bf16 parts (hi + lo), about 16 bits.
 */
size_t embla_prefill_workspace_size(const embla_shape *shape);
embla_status embla_prefill(const embla_shape *shape, int64_t n_new, const void *q,
                           const void *k_cache, const void *v_cache, float alpha, float c,
                           float eps, float *out, void *workspace, size_t workspace_bytes,
                           void *stream);

/*
 * ReLU^2 MLP of one token at batch size 1 ("ReLU^2 activation": a neuron at or below zero
 * contributes nothing, so only the down-projection rows of the neurons that fired are
 * read).  h_i = max(w_up_i . x, 0)^2;  y = sum over i with h_i > 0 of h_i w_down_i.
 * The pages' MLP shapes are not given; this call takes plain (non-gated) up and down
 * projections.
 *   d        width: 512, 1024 or 2048 (else EMBLA_ERR_UNSUPPORTED)
 *   f        neurons, 1 <= f <= 2^30
 *   x        bf16 [d]
 *   w_up     bf16 [f, d]   row i = neuron i's input weights (read in full)
 *   w_down   bf16 [f, d]   row i = neuron i's output weights (read only where h_i > 0)
 *   y        fp32 [d]
 *   n_live   int32 [1]     neurons with h_i > 0
 *   workspace  fp32 partial sums (embla_relu2_mlp_workspace_size; 0 if d or f < 1)
 * Sums are fp32 in a fixed order: the result is the same bits on every call.
 */
size_t embla_relu2_mlp_workspace_size(int64_t d, int64_t f);
embla_status embla_relu2_mlp(int64_t d, int64_t f, const void *x, const void *w_up,
                             const void *w_down, float *y, int32_t *n_live, void *workspace,
                             size_t workspace_bytes, void *stream);

/*
 * Window-layer decode — "Three kinds of attention" (Sliding window).
 *   q          bf16 [B, Hq, D]   raw query; rotated here at position pos:
 *              pair (2i, 2i+1) turned by pos * rope_base^(-2i/D)
 *   k_win      bf16 [B, Hkv, window, D] ring: position p lives in slot
 *              p % window and was rotated at p when it was written
 *   v_win      bf16 [B, Hkv, window, D] ring, same slots
 *   window     ring size, 1..1024 (128 in Embla 1)
 *   pos        position of the current token (>= 0); the valid positions are
 *              max(0, pos-window+1) .. pos
 *   rope_base  > 0 (10000 in the workloads here)
 *   tau        softmax scale, finite
 *   out        fp32 [B, Hq, D]
 * shape->ctx_len and shape->cache_stride are not used by this call.
 */
size_t embla_window_decode_workspace_size(const embla_shape *shape, int32_t window);
embla_status embla_window_decode(const embla_shape *shape, const void *q, const void *k_win,
                                 const void *v_win, int32_t window, int64_t pos, float rope_base,
                                 float tau, float *out, void *workspace, size_t workspace_bytes,
                                 void *stream);

/*
 * Cache append — the decode step's token written into the caches the calls above
 * read ("Three kinds of attention": a full layer keeps every token's K and V).
 * Row `pos` of every (b, g) plane is copied from a packed array of one row per plane:
 *   k_rows, v_rows     bf16 [B, Hkv, D]   the token's K and V (device memory)
 *   k_cache, v_cache   bf16 [B, Hkv, cache_stride, D], as for embla_full_decode
 *   pos                0 <= pos < cache_stride (the token's position, ctx_len - 1 of
 *                      the decode call that follows); shape->ctx_len is not used
 * 8-bit caches: the codes and the per-token scales of K and V:
 *   k_code_rows, v_code_rows   uint8 [B, Hkv, D];   k_codes, v_codes   uint8 [B, Hkv, cache_stride, D]
 *   k_scale_rows, v_scale_rows fp32 [B, Hkv];       k_scales, v_scales fp32 [B, Hkv, cache_stride]
 * One kernel per call, launched like every kernel of this library: the call after it may
 * begin its launch while it runs, and reads nothing before it has finished.  Any
 * alignment works; 16-byte aligned rows are copied 16 bytes at a time.
 */
embla_status embla_append_kv(const embla_shape *shape, int64_t pos, const void *k_rows,
                             const void *v_rows, void *k_cache, void *v_cache, void *stream);
embla_status embla_append_kv_e4m3(const embla_shape *shape, int64_t pos, const uint8_t *k_code_rows,
                                  const float *k_scale_rows, const uint8_t *v_code_rows,
                                  const float *v_scale_rows, uint8_t *k_codes, float *k_scales,
                                  uint8_t *v_codes, float *v_scales, void *stream);

/*
 * V-read accounting — "The Architecture of Embla 1", "Skipping V": a value row
 * is read only when some query head of the group gives its key a weight above
 * zero, i.e. when sigma_j > 0; the page's own kernel decides this for groups of
 * keys (8 at a time).  From the selection scores of embla_full_decode:
 *   sel_scores     fp32 [B, Hkv, cache_stride], as embla_full_decode wrote them
 *   chunk          a power of two, 1..1024 (8 on the page)
 *   keys_needed    int32 [B, Hkv]: keys j < n with sigma_j > 0 (equals n_surv)
 *   chunks_needed  int32 [B, Hkv]: chunks [c*chunk, (c+1)*chunk) of [0, n)
 *                  holding at least one such key
 * Reading V chunk by chunk reads (chunks_needed * chunk) rows, the last chunk
 * cut at n; per-key compaction (embla_full_decode) reads keys_needed rows.
 */
embla_status embla_skip_stats(const embla_shape *shape, const float *sel_scores, int32_t chunk,
                              int32_t *keys_needed, int32_t *chunks_needed, void *stream);

/*
 * Device-side check word.  Kernels record failed checks (an index outside
 * [0, n) handed to embla_sparse_decode, a pipeline wait that exceeded its
 * time limit) by OR-ing flag bits into a word in device memory instead of
 * trapping.  This call synchronises `stream`, copies the word to *flags and,
 * if `clear` is non-zero, resets it.  Returns EMBLA_ERR_DEVICE_CHECK when any
 * flag was set, EMBLA_OK otherwise.
 *   bit 0  index out of range (sparse decode)
 *   bit 1  a wait for data in flight timed out (full decode, selection)
 */
embla_status embla_device_check(uint32_t *flags, int clear, void *stream);

/*
 * Exercises the timed-out-wait path on the device without touching any kernel's
 * data: one thread waits, through the same bounded wait the pipelined kernels
 * use, on a shared-memory barrier that nothing arrives at, gives up after
 * limit_us microseconds (1 .. 1,000,000, else EMBLA_ERR_INVALID_ARG) and sets
 * bit 1 of the check word, as a kernel's timed-out wait does; the context stays
 * usable.  With `arrive` non-zero the thread arrives first, the wait succeeds
 * at once and nothing is set.  Asynchronous on `stream`; read the result with
 * embla_device_check.
 */
embla_status embla_self_test_wait_limit(uint32_t limit_us, int arrive, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* EMBLA_ATTN_H */
