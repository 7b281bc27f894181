/*
 * nosa.h -- C ABI of the NOSA decode-step hot path on one GB300 (sm_103a).
 *
 * NOSA (Native and Offloadable Sparse Attention) keeps the full bf16 K/V cache
 * in pinned host memory.  The GPU keeps only compressed keys, pooled eviction
 * scores and a small per-sequence block cache.  One decode step per layer is
 *
 *   append  -> new K/V to the host store (and to its cache slot), eviction
 *              score s^e = softplus(v W1) W2, new compressed key when a
 *              16-token stride completes                        (a1)
 *   select  -> query-aware score over all compressed keys, mean->max pooling
 *              onto 64-token blocks, top-k_q query-aware blocks, then k_e
 *              blocks by pooled s^e among never-dropped candidates, plus the
 *              sink and sliding-window blocks; set difference against the
 *              cache; list of blocks to fetch                  (a2-a4)
 *   fetch   -> persistent UVA gather of the newly needed 16 KiB K and V
 *              chunks from pinned host memory into cache slots  (a5)
 *   attend  -> split-K flash-decode over the selected blocks    (a6)
 *
 * Sources: the NOSA wiki page (aiwiki.ai), sections "How NOSA works",
 * "Main-experiment configuration" and "NOSI: the inference system"; the
 * NOSA-1B blog (wmrh.cn), sections on the key compressor, the CIS pooling
 * kernel and the two-stage top-k; the NOSA explainer (l189.com), section 2.1
 * (eq. 4-8); the SparDA summary (developer.aliyun.com), section on the KV
 * prefetch runtime (persistent UVA kernel, CTA-count rule).
 *
 * Conventions for every entry point
 *   * Every call returns nosa_status; no exception or abort crosses the ABI.
 *   * Argument errors are reported synchronously and change no state.
 *   * Device work is asynchronous on the context's stream.  Errors detected on
 *     the device (bounds, timeouts, capacity) are latched in a device error
 *     word and reported by nosa_sync() (and by later calls, which then fail
 *     with NOSA_ERR_STATE until nosa_reset_state()).
 *   * Pointers marked "device" must be device (or managed) memory and must stay
 *     valid until the stream reaches the call; "host" pointers are read or
 *     written before the call returns unless stated otherwise.
 *   * A context is not thread-safe: its calls come from one host thread at a
 *     time (or are serialised by the caller).  Different contexts are
 *     independent, except the file-scope scratch of nosa_attend_noalloc.
 *   * bf16 tensors are passed as uint16_t bit patterns.
 *   * Units: a unit is one (sequence b, kv head g) of one layer; within a layer
 *     units are ordered u = b * num_kv_heads + g.  GQA: q head h uses kv head
 *     h / (num_q_heads / num_kv_heads).
 *   * All sequences of a context share one length T per layer.
 *   * The library allocates in nosa_create only; the step calls allocate
 *     nothing and can be captured in a CUDA graph (per-step values such as the
 *     context length live in device memory).
 */
#ifndef NOSA_H_
#define NOSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NOSA_OK = 0,
  NOSA_ERR_INVALID_ARG = 1, /* bad pointer, layer, size or config field */
  NOSA_ERR_OOM = 2,         /* device allocation failed */
  NOSA_ERR_HOST_ALLOC = 3,  /* pinned host allocation failed */
  NOSA_ERR_CUDA = 4,        /* a CUDA runtime call failed (e.g. no GPU) */
  NOSA_ERR_CAPACITY = 5,    /* append past max_context */
  NOSA_ERR_TIMEOUT = 6,     /* a bounded device-side wait gave up */
  NOSA_ERR_BOUNDS = 7,      /* a device-side index check failed */
  NOSA_ERR_STATE = 8        /* call out of order, or the context is in a failed state */
} nosa_status;

/* Flags for nosa_config.flags.  Both are test hooks that fault and hang nothing:
 * NOSA_F_TEST_ZERO_WAIT  the attention kernel's waits for blocks staged through its
 *                        copy ring give up without waiting, so the timeout path
 *                        runs (copies already in flight are still drained with the
 *                        normal bound) and NOSA_ERR_TIMEOUT is latched.  A step whose
 *                        blocks all come from host memory into dedicated stages (the
 *                        first step after a cold start, small batches) has no such
 *                        wait; the first step that reads a cached block latches it;
 * NOSA_F_TEST_BAD_SLOT   the selector publishes an out-of-range cache slot for the
 *                        first selected block of unit 0; the attention kernel clamps
 *                        it and NOSA_ERR_BOUNDS is latched. */
#define NOSA_F_TEST_ZERO_WAIT 1u
#define NOSA_F_TEST_BAD_SLOT 2u
/* NOSA_F_UNFUSED_STEP: nosa_step launches the selector (which appends the token
 * first), the attention (with the fetch inside) and the merge of its split-K
 * partials instead of the fused one-kernel decode step.  Same selections; the
 * attention's split-K partition differs, so outputs may differ in the last bits.
 * The fused kernel is also skipped when the device cannot schedule all units'
 * thread-block clusters at once or the cache has more slots than a CTA has
 * threads. */
#define NOSA_F_UNFUSED_STEP 4u
/* NOSA_F_DMA_BIAS: the attention adds each attended token's eviction score s^e_j
 * to its scaled logit, softmax_j(q.k_j / sqrt(d) + s^e_j): the additive attention
 * bias of DMA, from which the eviction head is adapted (NOSA wiki, "How NOSA
 * works"; the NOSA-1B blog names the score CIS).  Off: plain attention (NOSA
 * explainer eq. 8). */
#define NOSA_F_DMA_BIAS 8u
/* NOSA_F_TEST_RADIX_TOPK (test hook): the query-agnostic top-k_e always takes the warp radix
 * select, which otherwise runs only when more than 1024 blocks are eligible (the first
 * selection over a context of more than about 66K tokens).  Same selections either way. */
#define NOSA_F_TEST_RADIX_TOPK 16u
/* NOSA_F_TEST_PREFILL_WIDE (test hook): nosa_prefill takes the kernel forms it otherwise takes only
 * for prompts of more than 65,536 tokens (two positions per warp for the query-aware picks instead
 * of four, two bitmap words per lane in the walk instead of one).  Same selections either way. */
#define NOSA_F_TEST_PREFILL_WIDE 32u

typedef struct {
  uint32_t struct_size;   /* sizeof(nosa_config) */
  int32_t num_layers;     /* L >= 1 */
  int32_t batch;          /* B >= 1 sequences */
  int32_t num_q_heads;    /* Hq; Hq % Hkv == 0 and 1 <= Hq/Hkv <= 8 */
  int32_t num_kv_heads;   /* Hkv >= 1 */
  int32_t head_dim;       /* d; must be 128 */
  int32_t block_size;     /* n_b; must be 64 (wiki: block size 64 tokens) */
  int32_t cmp_kernel;     /* CompressK window; must be 32 */
  int32_t cmp_stride;     /* CompressK stride; must be 16 */
  int32_t k_q;            /* query-aware blocks per step (>= 0) */
  int32_t k_e;            /* query-agnostic blocks per step (>= 0); sink/window not counted */
  int32_t sink_blocks;    /* leading blocks always selected (>= 0) */
  int32_t window_tokens;  /* sliding window, a multiple of block_size (>= 0) */
  int32_t max_context;    /* capacity per sequence in tokens, 1 .. 262144 */
  int32_t evict_hidden;   /* eviction-head hidden size h: multiple of 32, 32..256 */
  int32_t gather_ctas;    /* CTAs of the persistent fetch kernel; 0 = rule 16 if B<32 else 32 */
  float softmax_scale;    /* 0 => 1/sqrt(head_dim) */
  uint32_t flags;         /* 0, or NOSA_F_* flags */
  /* Kernel sizing.  0 takes the library's rule for each (set from measurements on
   * GB300); a non-zero value overrides it, for sweeps and tests.  Selections, fetch
   * lists and state do not depend on them; outputs may differ in the last bits (the
   * order in which split-K partials are merged). */
  int32_t score_ctas;            /* selector CTAs (one thread-block cluster) per unit, 1..8;
                                    rule: about two CTAs per SM over a layer's units, more while
                                    one CTA's window logits would not fit its shared memory */
  int32_t attend_blocks_per_cta; /* selected blocks per attention CTA (split-K chunk), 1..64;
                                    rule: 8..16 for about four CTAs per SM */
  int32_t attend_merge;          /* how split-K partials are merged: NOSA_MERGE_* */
  int32_t decode_cluster;        /* fused step: CTAs per unit cluster, 1..8 (rule: the largest of 8
                                    and 4 whose clusters for all units are resident at once, else
                                    the three-kernel chain); a forced size must be schedulable */
  int32_t decode_teams;          /* fused step: attention workers of four warps per CTA, 1 or 2 */
  int32_t decode_stages;         /* fused step: 32 KiB staging buffers per worker, 2..6 (rule: 3) */
  int32_t forecast_streams;      /* forecast pipeline: 2 = selections and gathers on two streams
                                    (a layer's selection overlaps the previous layer's gather),
                                    1 = both in order on one stream */
  int32_t cache_slots;           /* GPU block cache slots per unit, from one selection's blocks
                                    (sink + window/64 + k_q + k_e) up to 256; 0 = rule: twice a
                                    selection, at most 256.
                                    Slots beyond a selection keep blocks that left it, so a block
                                    selected again later is not fetched again (the least recently
                                    selected are replaced first).  Selections and outputs do not
                                    depend on it; fetch lists, slots and transfers do. */
} nosa_config;

/* Values of nosa_config.attend_merge. */
#define NOSA_MERGE_AUTO 0    /* the rule: NOSA_MERGE_KERNEL */
#define NOSA_MERGE_KERNEL 1  /* CTAs store partials; a dependent merge kernel combines them */
#define NOSA_MERGE_TICKET 2  /* the unit's last CTA (atomic ticket) combines them */
#define NOSA_MERGE_CLUSTER 3 /* the unit's CTAs form one cluster and combine through DSMEM */

/* Derived sizes; filled by nosa_query_sizes (host only, no GPU needed). */
typedef struct {
  int32_t units_per_layer; /* B * Hkv */
  int32_t group;           /* Hq / Hkv */
  int32_t cache_slots;     /* slots per unit in the GPU block cache (nosa_config.cache_slots) */
  int32_t max_blocks;      /* ceil(max_context / 64) */
  int32_t max_windows;     /* complete CompressK windows at max_context */
  int32_t evict_words;     /* 32-bit words of the per-unit eviction bitmap */
  uint64_t host_store_bytes;   /* pinned K/V store: L*U*max_blocks*2*64*d*2 */
  uint64_t device_state_bytes; /* everything nosa_create allocates on the device */
  int32_t select_slots;    /* blocks of one selection at most: sink + window/64 + k_q + k_e */
  int32_t pad_;
} nosa_sizes;

typedef struct nosa_ctx nosa_ctx;

/* Per-context counters, accumulated on the device by nosa_select. */
typedef struct {
  uint64_t selections;      /* unit-selections made */
  uint64_t gamma_samples;   /* unit-selections that had a previous selection */
  double gamma_mean;        /* mean over those of |D_t & S_{t-1}| / |D_t| */
  double gamma_min;         /* minimum of the same (1.0 if no sample) */
  uint64_t blocks_fetched;  /* blocks copied host -> device (each 2 x 16 KiB) */
  uint64_t bytes_fetched;   /* blocks_fetched * 32 KiB */
  uint64_t short_selections;/* unit-selections whose query-agnostic part came up short */
} nosa_stats;

/* Host-side view for nosa_export_state: every pointer is host memory or NULL
 * (skipped).  Shapes are per layer; U = units_per_layer, cap = select_slots,
 * cs = cache_slots. */
typedef struct {
  int32_t* sel;       /* [U][cap] selected blocks S, ascending, -1 padded */
  int32_t* sel_kind;  /* [U][cap] 0 sink, 1 window, 2 query-aware, 3 query-agnostic, -1 pad */
  int32_t* sel_slot;  /* [U][cap] cache slot of each selected block, -1 pad */
  int32_t* n_sel;     /* [U] */
  int32_t* fetch;     /* [U][cap][2] (block, slot) fetched by the last selection, ascending */
  int32_t* n_fetch;   /* [U] */
  int32_t* slot_blk;  /* [U][cs] block held by each cache slot, -1 empty */
  uint32_t* evicted;  /* [U][evict_words] sticky eviction bitmap, bit b%32 of word b/32 */
  uint16_t* kt;       /* [U][max_windows][d] compressed keys (bf16 bits) */
  float* se_win;      /* [U][max_windows] window means of the eviction score */
  float* se_blk;      /* [U][max_blocks] pooled eviction score (-inf before any window) */
  int32_t* gamma;     /* [U][2] |D_t & S_{t-1}| and |D_t| of the last selection */
  int32_t* last_used; /* [U][cs] context length of the last selection holding each slot's
                         block, -1 for a slot no selection has used */
} nosa_state_view;

/* Validate a config without touching the GPU.  NOSA_OK or NOSA_ERR_INVALID_ARG. */
nosa_status nosa_validate_config(const nosa_config* cfg);

/* Sizes derived from a valid config (host only). */
nosa_status nosa_query_sizes(const nosa_config* cfg, nosa_sizes* out);

/* Create a context on the current CUDA device.  `stream` is a cudaStream_t
 * (NULL = legacy default stream) owned by the caller; every later call of the
 * context is queued on it.  Allocates the pinned, mapped host K/V store and
 * all device state; eviction heads start at zero.  On failure *out is NULL. */
nosa_status nosa_create(const nosa_config* cfg, void* stream, nosa_ctx** out);

/* Drain the stream and free everything.  NULL is accepted. */
nosa_status nosa_destroy(nosa_ctx* ctx);

/* Change the stream later calls are queued on (e.g. a capture stream). */
nosa_status nosa_set_stream(nosa_ctx* ctx, void* stream);

/* Eviction head of one layer: host float32 W1 [Hkv][d][h] and W2 [Hkv][h], copied before
 * return.  Defined by: NOSA explainer, section 2.1, eq. 4 (s^e = softplus(v W1) W2); NOSA wiki,
 * "How NOSA works" (the query-agnostic eviction head, one per kv head, ranked before any
 * exponential as in ED-DMA). */
nosa_status nosa_set_eviction_head(nosa_ctx* ctx, int layer, const float* W1, const float* W2);

/* Append n_tokens >= 1 tokens to every sequence of `layer` (row a1).
 * Defined by: NOSA explainer, section 2.1, eq. 4-6 (eviction score of each token, mean pooling
 * of keys and scores over compression windows); NOSA-1B blog, key compressor (kernel 32,
 * stride 16); NOSA wiki, "NOSI: the inference system" (the full K/V lives in host memory).
 * k, v: bf16 [B][Hkv][n_tokens][d]; device memory, or pinned/pageable host
 * memory when src_is_host != 0 (then copied before the kernels run).
 * n_tokens == 1 is the decode-step append; n_tokens > 1 is a bulk context load
 * (host store, eviction scores, compressed keys; cached blocks are kept in step).
 * Returns NOSA_ERR_CAPACITY (no state change) if T + n_tokens > max_context. */
nosa_status nosa_append_kv(nosa_ctx* ctx, int layer, const uint16_t* k, const uint16_t* v,
                           int n_tokens, int src_is_host);

/* Score and select the blocks of every unit of `layer` for query q
 * (device bf16 [B][Hq][d]), update the eviction bitmap and the slot map, and
 * build the fetch list (rows a2-a4).  Defined by: NOSA wiki, "How NOSA works" (query-aware
 * top-k_q scores set to +inf, the rest filled from the query-agnostic score, a block dropped
 * by that part never re-selected by it) and "Main-experiment configuration" (sink block,
 * sliding-window blocks, 64-token blocks); NOSA explainer, section 2.1, eq. 5-6 (pooled block
 * scores, the selection); SparDA summary, "lightweight design" (softmax aggregation over a GQA
 * group); NOSA wiki, "NOSI" (set difference against the cached blocks: a selected block is
 * fetched only when no cache slot holds it).  Optional device outputs: sel_out
 * [B][Hkv][select_slots] (S ascending, -1 padded) and nfetch_out [B][Hkv] (blocks to fetch). */
nosa_status nosa_select(nosa_ctx* ctx, int layer, const uint16_t* q, int32_t* sel_out,
                        int32_t* nfetch_out);

/* Copy the blocks listed by the last nosa_select of `layer` from the pinned
 * host store into their cache slots (persistent UVA gather kernel, row a5).  Defined by:
 * NOSA wiki, "NOSI: the inference system" (a host-to-device kernel reading host memory
 * through unified virtual addressing, block-wise 16 KiB transfers); SparDA summary, KV
 * prefetch runtime (a resident set of copy CTAs, their count chosen by batch size). */
nosa_status nosa_fetch(nosa_ctx* ctx, int layer);

/* Attention of q (device bf16 [B][Hq][d]) over the selected blocks; writes
 * out (device bf16 [B][Hq][d]) (row a6).  Defined by: NOSA explainer, section 2.1, eq. 8
 * (softmax attention over the keys and values of the selected blocks); NOSA-1B blog, decode
 * stage (attention over the top-k block indices only).  Needs a selection for the current T.  If
 * nosa_fetch has not run since that selection, the attention CTAs copy the
 * newly selected blocks from the pinned host store themselves (and write them
 * to their cache slots), so no separate gather pass is needed. */
nosa_status nosa_attend(nosa_ctx* ctx, int layer, const uint16_t* q, uint16_t* out);

/* One decode step of `layer`: append the token (k_new, v_new), score and select,
 * fetch the new blocks and attend with q, as one fused kernel or a short kernel
 * chain (nosa_step_plan says which): rows a1-a6 as defined at nosa_append_kv,
 * nosa_select, nosa_fetch and nosa_attend (NOSA wiki, "How NOSA works" and "NOSI";
 * NOSA explainer, section 2.1, eq. 4-8); the same selections and state as
 * nosa_append_kv + nosa_select + nosa_attend.  k_new, v_new: device bf16
 * [B][Hkv][d]; q, out: device bf16 [B][Hq][d].  NOSA_ERR_CAPACITY (nothing queued)
 * when the layer's context is full. */
nosa_status nosa_step(nosa_ctx* ctx, int layer, const uint16_t* q, const uint16_t* k_new,
                      const uint16_t* v_new, uint16_t* out);

/* nosa_step with host q, k_new, v_new and out (the same step and sources as nosa_step).  When all four are page-locked
 * (cudaHostAlloc / cudaHostRegister) the kernels read the inputs and write the
 * output in place over the host link; otherwise the inputs are copied to
 * context-owned device buffers and the output back, on the stream.  Either way
 * the buffers must stay untouched until the stream reaches the end of the step,
 * when out is written. */
nosa_status nosa_step_host(nosa_ctx* ctx, int layer, const uint16_t* q, const uint16_t* k_new,
                           const uint16_t* v_new, uint16_t* out);

/* One decode step of every layer from host buffers (nosa_step per layer, same sources): q and out [L][B][Hq][d], k_new and
 * v_new [L][B][Hkv][d], bf16, layer-major.  Copies q, k_new and v_new to
 * context-owned device buffers (one cudaMemcpyAsync each), runs nosa_step for layers
 * 0 .. L-1 in order on those, and copies every layer's output back (one
 * cudaMemcpyAsync), all on the context's stream, so that the layers' kernels stay
 * chained and no layer waits on the host link for its inputs.  Every layer is checked
 * before anything is queued: on an error nothing runs and no state changes
 * (NOSA_ERR_CAPACITY if any layer is full).  Page-locked buffers (cudaHostAlloc /
 * cudaHostRegister) let the copies run asynchronously and be captured in a CUDA
 * graph; pageable ones work outside a capture.  The buffers must stay untouched until
 * the stream reaches the end of the step, when out is written. */
nosa_status nosa_step_host_all(nosa_ctx* ctx, const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                               uint16_t* out);

/* SparDA-style forecast selection (SparDA summary: a forecast vector of layer l picks
 * layer l+1's blocks one layer ahead, so the copy of those blocks overlaps layer l's
 * work; one forecast head per kv head; sink and local blocks by position).  Selects
 * the blocks of `layer` for its context after the NEXT append (T+1): candidates, sink
 * and window of T+1, query-aware scores from the forecast f (device bf16 [B][Hkv][d])
 * over the windows complete at T, query-agnostic part, eviction, slots and fetch list
 * as in nosa_select.  Then nosa_fetch (optional), nosa_append_kv of the token and
 * nosa_attend use it.  NOSA_ERR_STATE if a forecast for T+1 was already made. */
nosa_status nosa_forecast_select(nosa_ctx* ctx, int layer, const uint16_t* f);

/* Pipelined forecast step of `layer` (needs a forecast selection for this token, from
 * nosa_forecast_select or an earlier nosa_step_forecast).  If f_next is not NULL it
 * first starts, on the context's own streams, the forecast selection of next_layer
 * (!= layer) with f_next and, after it, the copy of its new blocks (the selection on
 * a selection stream, the copy on a prefetch stream, so that one layer's selection
 * overlaps the previous layer's copy); then, on the context's stream, waits for this
 * layer's prefetch (if one was started by an earlier call), appends k_new/v_new and
 * attends with q.  Those streams fork from and join the context's stream through
 * events, so a CUDA graph capture of a sequence of calls stays one graph; call
 * nosa_forecast_join before ending a capture.  Pointers as in nosa_step; f_next:
 * device bf16 [B][Hkv][d].
 * When it pays (measured on GB300 against nosa_step per layer, block cache of twice a
 * selection): at small batch, where the step is a latency chain (1B shape, 16K, batch 8:
 * 12.1K against 8.6K tok/s, +40 %); not once the step is bound by HBM (8B shape, 32K, batch 32:
 * 4.66K against 5.02K, -7 %), where the next layer's selection reads its compressed keys from
 * HBM beside the attention and costs more than the overlap saves.  (With a cache of one
 * selection, when the host link set the pace, it also paid at the 8B shape: +2-5 %.) */
nosa_status nosa_step_forecast(nosa_ctx* ctx, int layer, const uint16_t* q, const uint16_t* k_new,
                               const uint16_t* v_new, uint16_t* out, const uint16_t* f_next, int next_layer);

/* Makes the context's stream wait for every prefetch started by nosa_step_forecast.
 * (Every entry point that works on a layer also waits for that layer's pending
 * prefetch first, and the calls that read or reset state wait for all of the
 * context's streams, so the forecast and plain entry points may be mixed.) */
nosa_status nosa_forecast_join(nosa_ctx* ctx);

/* Dense GQA decode attention over a device-resident KV store: the full-attention
 * comparator of the NOSA wiki's decode-throughput table (section "Decoding throughput") (every token attended; no
 * selection, no host memory).  Context-free; allocates nothing.
 *   q        device bf16 [units][group][d]
 *   kv       device bf16 [units][max_blocks][2][64][d]: block b of unit u holds keys
 *            then values of tokens 64b .. 64b+63 (the layout of the host store and
 *            of the block cache); 16-byte aligned
 *   context_len  tokens attended (<= max_blocks * 64 and <= 1,048,576)
 *   out      device bf16 [units][group][d]
 *   scratch  device memory of at least nosa_dense_scratch_bytes(units, context_len)
 *            bytes, 256-byte aligned; its first 4 bytes receive device-side error bits
 *            (zero them before the call to read them after it)
 * Asynchronous on `stream`.  NOSA_ERR_CAPACITY if the scratch is too small. */
nosa_status nosa_dense_attend(const uint16_t* q, const uint16_t* kv, int units, int group, int max_blocks,
                              int context_len, float softmax_scale, uint16_t* out, void* scratch,
                              size_t scratch_bytes, void* stream);

/* Scratch bytes nosa_dense_attend needs (0 on a bad argument or without a device). */
size_t nosa_dense_scratch_bytes(int units, int context_len);

/* NOSA_S sparse prefill of an empty `layer` (T = 0): appends a prompt of n_tokens tokens to
 * every sequence and attends every prompt position over its own block selection, in one call.
 * Defined by: NOSA wiki, "Results" (NOSA_S: sparse attention in prefill as well as in
 * decoding) and "How NOSA works" (a block the query-agnostic part drops at one step is never
 * re-selected by it, so a position's selection depends on the earlier positions').  The
 * selection for prompt position t is the one the decode step at T = t + 1 makes, with the
 * eviction state carried from position t - 1.  The query-aware picks of all positions are made
 * at once (they do not depend on that state); one warp per unit then walks the positions in
 * order for the query-agnostic picks and the eviction update; the attention of all positions
 * runs in one launch, reading the prompt's K/V from k and v.  Afterwards the layer's selection
 * state (host store, compressed keys, scores, eviction bitmap, last selection, the selection
 * and locality counters) is the state n_tokens calls of nosa_step with the same tokens would
 * leave; the block cache holds exactly the last selection, its i-th block (ascending) in slot i,
 * each marked as selected at T = n_tokens, with nothing left to fetch (the prompt's blocks never
 * cross the host link, so blocks_fetched does not grow).  Decoding continues with nosa_step.
 *   q, out   device bf16 [B][Hq][n_tokens][d] (out[b][h][t] is position t's attention output)
 *   k, v     device bf16 [B][Hkv][n_tokens][d]; q, k and v 16-byte aligned
 *   scratch  device memory of at least nosa_prefill_scratch_bytes(ctx, n_tokens) bytes, 16-byte
 *            aligned.  Afterwards it holds every position's selection as two bitmaps over the
 *            prompt's blocks: uint32 [2][B][Hkv][n_tokens][W], W = ceil(ceil(n_tokens / 64) / 32),
 *            block b at bit b % 32 of word b / 32; [0] the query-aware picks, [1] the
 *            query-agnostic ones.  Position t's selection is those blocks plus the sink blocks
 *            and the window blocks of a context of t + 1 tokens.
 * NOSA_ERR_INVALID_ARG on a misaligned pointer; NOSA_ERR_STATE if the layer is not empty;
 * NOSA_ERR_CAPACITY if n_tokens exceeds max_context or 131,072 (the longest prompt the kernels'
 * block bitmaps cover), or if the scratch is too small. */
nosa_status nosa_prefill(nosa_ctx* ctx, int layer, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         int n_tokens, uint16_t* out, void* scratch, size_t scratch_bytes);

/* Scratch bytes nosa_prefill needs for a prompt of n_tokens (0 on a bad argument). */
size_t nosa_prefill_scratch_bytes(nosa_ctx* ctx, int n_tokens);

/* How nosa_step runs on this context: *kernels_per_layer = the kernel launches of
 * one layer's step: 1 (the fused decode kernel, one thread-block cluster of
 * *cluster_size CTAs per unit), or 3 (the selector kernel, which also appends the
 * token, the attention kernel and the kernel merging its split-K partials;
 * *cluster_size = 0) — 2 when the attention merges its partials itself.  Either
 * pointer may be NULL. */
nosa_status nosa_step_plan(nosa_ctx* ctx, int32_t* kernels_per_layer, int32_t* cluster_size);

/* Wait for the stream; report and latch any device-side error. */
nosa_status nosa_sync(nosa_ctx* ctx);

/* Clear a latched error (the device state may be inconsistent afterwards). */
nosa_status nosa_reset_state(nosa_ctx* ctx);

/* Current context length of `layer` (synchronises the stream). */
nosa_status nosa_context_length(nosa_ctx* ctx, int layer, int32_t* T_out);

/* Counters (synchronises the stream); nosa_reset_stats zeroes them. */
nosa_status nosa_get_stats(nosa_ctx* ctx, nosa_stats* out);
nosa_status nosa_reset_stats(nosa_ctx* ctx);

/* Pooled block scores of the last selection of `layer` (plain or forecast), host float
 * [U][max_blocks] each (sq_blk: query-aware, se_blk: query-agnostic); either may
 * be NULL.  Each layer keeps its own.  Synchronises. */
nosa_status nosa_debug_scores(nosa_ctx* ctx, int layer, float* sq_blk, float* se_blk);

/* Copy selection / cache / compression state of `layer` to host memory. Synchronises. */
nosa_status nosa_export_state(nosa_ctx* ctx, int layer, const nosa_state_view* view);

const char* nosa_status_string(nosa_status s);

/* Sparse attention over a caller-owned block cache that allocates nothing.
 * The paper has no counterpart: this exists for callers that must not call
 * cudaMalloc (a memory pool they do not own, an allocator under capture or
 * audit, a path that may not grow the device footprint after start-up).
 * It runs the same split-K kernel as nosa_attend without a context; its
 * scratch (split-K partials, merge tickets, context length) is one fixed
 * file-scope device array of about 8.5 MB that every GPU loading this library
 * keeps until the process exits.
 *   q        device bf16 [units][group][128]
 *   cache    device bf16 [units][cache_slots][2][64][128] (K then V of each
 *            slot's block, 16-byte aligned), the layout of a context's cache
 *   sel      device int32 [units][cache_slots] selected block ids, ascending
 *   sel_slot device int32 [units][cache_slots] slot of each selected block
 *   n_sel    device int32 [units] number of selected blocks per unit, at most
 *            cache_slots
 *   context_len  tokens per sequence; block ceil(context_len/64)-1 is the
 *            partial tail and only its first tokens are attended
 *   softmax_scale 0 => 1/sqrt(128);  out device bf16 [units][group][128]
 *   err_out  optional device int32 (4-byte aligned): cleared on the stream, then
 *            receives the device-side error bits of this call: 1 = an n_sel above
 *            cache_slots or a slot outside [0, cache_slots) was met (clamped into
 *            range; that unit's output is meaningless), 2 = a bounded wait for a
 *            staged block gave up (that unit's outputs are NaN).  NULL: the bits
 *            go to the library's own scratch and are not reported.
 * Limits: units <= 1024 and units * ceil(cache_slots / chunk) <= 2048 split-K
 * partials, where chunk (blocks per CTA) is widened up to 64 to fit; larger
 * requests return NOSA_ERR_CAPACITY before anything is queued.  Calls never
 * allocate, so their scratch is shared: calls that overlap on the GPU (other
 * streams, other threads) race and must be serialised by the caller; each call
 * clears the tickets it uses.  The first call on a device does a one-time set-up
 * (looks up the scratch address and sets the kernel's shared-memory limit); make
 * that first call before any stream capture.  Asynchronous on `stream`. */
nosa_status nosa_attend_noalloc(const uint16_t* q, const uint16_t* cache, const int32_t* sel,
                                const int32_t* sel_slot, const int32_t* n_sel, int units, int group,
                                int cache_slots, int context_len, float softmax_scale, uint16_t* out,
                                int32_t* err_out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* NOSA_H_ */
