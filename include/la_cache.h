/*
 * la_cache.h -- C ABI of the bounded KV cache and its block-causal chunk
 * attention (single GPU, sm_103a).
 *
 * What the calls compute follows two pages on streaming video DiTs:
 *   [LA]  "LiveAnimate: 实时稳定长时流式人体动画" (ai-feeds.com), 方法 / 实验:
 *         PR-Sink bounded cache = static sink (first generated block, kept
 *         forever) + dynamic sink (history blocks retrieved by pose
 *         similarity) + rolling window of the 3 most recent blocks; each block
 *         attends only to the reference and earlier blocks; cache size and
 *         per-block latency stay constant as the stream grows.
 *   [LX]  "Soul App开源实时数字人生成框架SoulX-LiveAct详解" (youleyou.com),
 *         技术内核 / 上手实践指南: ConvKV memory (recent K/V exact, older K/V
 *         compressed about 5:1 by a 1D convolution into fixed-length memory
 *         with RoPE positions reset) and an FP8 KV cache.
 *
 * Conventions for every call
 *   - Pointers named "device" must be CUDA device memory of the current
 *     device; "host" pointers are ordinary host memory.  The library never
 *     allocates device memory: the caller hands it one pool
 *     (la_cache_required_bytes) and owns every input and output buffer.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued on it; device buffers passed in must stay
 *     valid until that work completes.
 *   - Q/K/V/O tensors of one block are row-major [T][H][D]: T tokens in
 *     raster order (frame, row, column), H heads, D head dim; element type
 *     `q_dtype` (LA_F32 or LA_BF16).  Their device pointers, and the ConvKV
 *     weights, must be 16-byte aligned (the kernels move rows in 16-byte
 *     vectors); a call given one that is not returns LA_ERR_INVALID_ARG.
 *   - Errors: arguments and call order are checked synchronously and the
 *     status is returned.  Faults seen inside kernels (an index out of range,
 *     a wait that ran out of time) are latched in a device error word that
 *     la_get_error reads; after any error every call but la_get_error and
 *     la_cache_destroy returns LA_ERR_STATE.
 */
#ifndef LA_CACHE_H
#define LA_CACHE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LA_OK = 0,
  LA_ERR_INVALID_ARG = 1,   /* bad pointer, size or configuration            */
  LA_ERR_OOM = 2,           /* pool smaller than la_cache_required_bytes     */
  LA_ERR_CUDA = 3,          /* a CUDA runtime call failed                    */
  LA_ERR_STATE = 4,         /* call out of order, or an earlier error latched*/
  LA_ERR_TIMEOUT = 5,       /* a device-side wait ran out of time            */
  LA_ERR_UNSUPPORTED = 6,   /* valid but not built (shape/dtype combination) */
  LA_ERR_DEVICE = 7         /* a kernel reported an out-of-range index       */
} la_status;

typedef enum { LA_POLICY_PR_SINK = 0, LA_POLICY_CONVKV = 1 } la_policy;
typedef enum { LA_F32 = 0, LA_BF16 = 1, LA_E4M3 = 2 } la_dtype;

/* Where history blocks that left the window live.
 * RESIDENT: every appended block keeps its K/V pages in the pool, so any of
 *   them can be retrieved into the dynamic sink without help.
 * EXTERNAL: the pool holds only the attended blocks; when the dynamic sink
 *   picks a history block, the caller supplies its K/V with la_fill_block
 *   (the pages bound only the attended cache, [LA] 实验; history storage is
 *   left to the caller). */
typedef enum { LA_HISTORY_RESIDENT = 0, LA_HISTORY_EXTERNAL = 1 } la_history_mode;

/* Attention kernel choice: AUTO = tensor cores where the shape is built
 * for them (bf16/e4m3, D = 128), otherwise the CUDA-core kernel. */
typedef enum { LA_ATTN_AUTO = 0, LA_ATTN_TENSOR = 1, LA_ATTN_SIMT = 2 } la_attn_impl;

typedef struct {
  int32_t num_layers, num_heads, head_dim;       /* L, H, D (D = 64 or 128)           */
  int32_t frames_per_block, grid_h, grid_w;      /* T = F * GH * GW <= 2^20 tokens    */
  int32_t rope_t, rope_h, rope_w;                /* RoPE dims per axis, sum = D       */
  float   rope_theta;                            /* 10000                              */
  int32_t policy;                                /* la_policy                          */
  int32_t static_sink;                           /* 1 = block 0 kept forever [LA]      */
  int32_t dyn_topk;                              /* k of the dynamic sink, <= 8        */
  int32_t window;                                /* rolling window, 3 in [LA]          */
  int32_t pose_dim;                              /* 34 = 17 keypoints x (x, y)         */
  int32_t max_history;                           /* blocks the pose table can hold     */
  int32_t conv_kernel, conv_stride, mem_slots;   /* ConvKV: 5, 5, 4096 [LX]            */
  int32_t q_dtype, kv_dtype;                     /* la_dtype                           */
  float   softmax_scale;                         /* 1/sqrt(D)                          */
  int32_t history_mode;                          /* la_history_mode                    */
  int32_t attn_impl;                             /* la_attn_impl                       */
} la_cache_config;

#define LA_MAX_SLOTS 16
#define LA_MAX_TOPK 8

/* The context of the block being generated, in slot order:
 * [static sink, dynamic sink (ascending id), window (oldest first), current]
 * for PR-Sink; [window (oldest first), current] after `mem_tokens`
 * compressed memory tokens for ConvKV. */
typedef struct {
  int32_t block;                       /* id of the block being generated      */
  int32_t n_slots;                     /* exact slots, current block included  */
  int32_t kv_len;                      /* keys attended: mem_tokens + n_slots*T */
  int32_t mem_tokens;                  /* ConvKV memory tokens (0 for PR-Sink)  */
  int32_t block_id[LA_MAX_SLOTS];      /* block held by each exact slot         */
  int32_t t0[LA_MAX_SLOTS];            /* temporal RoPE base of each slot       */
  int32_t n_dyn;                       /* dynamic-sink blocks chosen            */
  int32_t dyn_ids[LA_MAX_TOPK];        /* ascending                             */
  float   dyn_scores[LA_MAX_TOPK];     /* cosine score of each chosen block     */
  float   topk_gap;                    /* score_k - score_(k+1); +inf if none   */
  int32_t need_fill[LA_MAX_TOPK];      /* EXTERNAL: 1 = la_fill_block required   */
} la_context;

typedef struct la_cache la_cache_t;

/* Device bytes the pool must have for `cfg` (0 if `cfg` is invalid). */
size_t la_cache_required_bytes(const la_cache_config* cfg);

/* Creates a cache inside `dev_pool` (device, >= la_cache_required_bytes,
 * 256-byte aligned, owned by the caller and borrowed until destroy).
 * `conv_w` (device, ConvKV only, else NULL): bf16 depthwise weights laid out
 * [L][2 (K, V)][H][D][conv_kernel], borrowed until destroy.  Initialises the
 * pool on `stream`.  On success *out receives the handle. */
la_status la_cache_create(const la_cache_config* cfg, void* dev_pool, size_t pool_bytes,
                          const void* conv_w, void* stream, la_cache_t** out);

/* Releases the host state.  It does not synchronise: call it only after the
 * work enqueued for this cache has completed.  The pool stays the caller's. */
la_status la_cache_destroy(la_cache_t* cache);

/* Checkpoint and resume of a stream between blocks (the pages describe no
 * such facility; it serves callers that restart a long stream).  The device
 * state is the pool, which the caller owns and copies; the host state -- the
 * block counter, the frame table and free frames, the window, the dynamic
 * sink and any picks fetched ahead, the ConvKV ring position -- goes into a
 * host buffer of la_cache_state_bytes(cache) bytes:
 *   la_cache_save_state: only between blocks (after the append of a block's
 *     last layer, before the next select; LA_ERR_STATE otherwise);
 *     LA_ERR_INVALID_ARG when `cap` is too small.  The pool bytes must be
 *     copied after the cache's enqueued work has completed.
 *   la_cache_restore: builds a cache over a pool that holds the saved pool
 *     bytes (at any device address; same size rule as la_cache_create) and
 *     continues the stream at the saved block.  The blob carries the config:
 *     a different config or a malformed blob gives LA_ERR_INVALID_ARG.
 *     The pool is not initialised.  `conv_w` as for la_cache_create. */
size_t la_cache_state_bytes(la_cache_t* cache);
la_status la_cache_save_state(la_cache_t* cache, void* host_buf, size_t cap);
la_status la_cache_restore(const la_cache_config* cfg, void* dev_pool, size_t pool_bytes,
                           const void* conv_w, const void* state, size_t state_bytes,
                           void* stream, la_cache_t** out);

/* Starts block b (b = number of blocks appended so far).  Runs the pose
 * retrieval kernel on `stream` ([LA] 方法, Dynamic Sink): the centred 34-value
 * descriptor of `query_pose` (host, 17 (x, y) keypoints) is scored by cosine
 * similarity against every history block that is neither the static sink,
 * nor in the window, nor block b, and the top-k under (score desc, id asc)
 * are taken.  Builds the slot table the attention reads.  Synchronises
 * `stream` once to read the k chosen ids.  `out` (host, optional) receives
 * the context. */
la_status la_select_context(la_cache_t* cache, const float* query_pose, la_context* out,
                            void* stream);

/* EXTERNAL history only: writes the K/V of history block `block_id` for
 * `layer` into the dynamic-sink page the last la_select_context (or
 * la_prefetch_context) gave it (need_fill = 1).  k, v: [T][H][D] q_dtype,
 * the block's final K/V as la_cache_append_block received them, in device
 * memory or in page-locked host memory the device can address (the kernel
 * then reads it over the bus: a host-memory history tier). */
la_status la_fill_block(la_cache_t* cache, int layer, int block_id, const void* k,
                        const void* v, void* stream);

/* EXTERNAL history only, while block b is in progress (after its
 * la_select_context): runs the pose retrieval of block b + 1 for
 * `next_pose` (host, 17 (x, y) keypoints) -- its candidates are all
 * committed already -- and reserves a page for every picked block not in
 * the pool.  `out` (host, optional) gets block b + 1's context; need_fill
 * marks the picks whose K/V must be written with la_fill_block (on any
 * stream, e.g. a copy stream, so the writes overlap block b's attention;
 * the caller orders them before block b + 1's first attention).  A later
 * la_select_context for block b + 1 with the same pose finds those blocks
 * in place.  This is the "block offload" deployment the LiveAct page names
 * (上手实践指南: 显存块卸载), with the next block's pose known ahead.  One
 * call per block; LA_ERR_STATE outside a block. */
la_status la_prefetch_context(la_cache_t* cache, const float* next_pose, la_context* out,
                              void* stream);

/* Block-causal chunk attention of the current block for one layer
 * ([LA] 方法): every query token of the block attends, without mask, to all
 * tokens of the context (memory, cached slots and the current block itself).
 * 3D RoPE over (t, h, w) positions is applied to queries and keys; the slot
 * at temporal base t0 holds positions (t0 + frame, row, column).
 * q, k_cur, v_cur: device [T][H][D] q_dtype (the current block's values at
 * this denoising step); out: device [T][H][D] q_dtype.
 * out = softmax(softmax_scale * RoPE(q) RoPE(K_ctx)^T) V_ctx, per head.
 * With an e4m3 cache the tensor-core kernel also rounds the rotated queries
 * (one scale per head and token) and the probabilities to e4m3 ([LX]
 * 技术内核: FP8 attention). */
la_status la_chunk_attention(la_cache_t* cache, int layer, const void* q, const void* k_cur,
                             const void* v_cur, void* out, void* stream);

/* Appends the current block's final K/V for `layer` (device [T][H][D]
 * q_dtype).  When every layer has been appended the block is committed: its
 * pose joins the history, the window rolls ([LA] 方法, Rolling Window) and,
 * for ConvKV, the block leaving the window is compressed into the memory
 * ([LX] 技术内核) -- the compression of each layer runs in that layer's
 * append.  For an e4m3 cache the K/V are quantised with one fp32 scale per
 * (head, block). */
la_status la_cache_append_block(la_cache_t* cache, int layer, const void* k, const void* v,
                                void* stream);

/* Refreshes the static sink of `layer` (PR-Sink with static_sink = 1, once
 * block 0 has been committed, between blocks): its K/V pages are replaced by
 * `k`, `v` (device [T][H][D] q_dtype), stored exactly as an appended block
 * (keys turned by their within-block position, e4m3 with fresh per-head
 * scales).  The sink keeps its slot and RoPE base.  This is the cache side of
 * the Rolling Sink Frame Mechanism ("Live Avatar", chatpaper.ai, 摘要 /
 * abstract): appearance is recalibrated from a cached reference image, i.e.
 * the caller re-encodes the reference at the current time and hands its K/V
 * here, at an interval of its choosing.  Returns LA_ERR_UNSUPPORTED for
 * ConvKV or without a static sink, LA_ERR_STATE inside a block or before
 * block 0 is committed. */
la_status la_refresh_sink(la_cache_t* cache, int layer, const void* k, const void* v,
                          void* stream);

/* Called by la_stream_step for each (layer, block) needing a fill. */
typedef la_status (*la_fill_fn)(la_cache_t* cache, int layer, int block_id, void* user,
                                void* stream);

/* One streamed block: select, n_steps x L chunk attentions, then L appends
 * of the last step's K/V.  q, k, v, out: host arrays of n_steps*L device
 * pointers, entry [step * L + layer].  `fill` (required in EXTERNAL mode
 * when a fill is needed) is called between select and the attentions.  The
 * last step's attention writes the block's K/V pages straight into the
 * block's own cache frame, so the appends that follow copy nothing (for
 * ConvKV they still compress the block leaving the window). */
la_status la_stream_step(la_cache_t* cache, const float* pose, int n_steps,
                         const void* const* q, const void* const* k, const void* const* v,
                         void* const* out, la_fill_fn fill, void* user, void* stream);

/* EXTERNAL history only: loads the pose history of blocks 0..n-1 (host,
 * n x 17 x 2 keypoints) into an empty cache, as when a stream resumes with
 * its K/V held by the caller; the next block is n.  Blocks n-window..n-1
 * must then be supplied with la_fill_window before attention. */
la_status la_cache_load_history(la_cache_t* cache, const float* kps, int n, void* stream);

/* EXTERNAL history after la_cache_load_history: writes the K/V of a block
 * that is the static sink or in the window (device [T][H][D]). */
la_status la_fill_window(la_cache_t* cache, int layer, int block_id, const void* k,
                         const void* v, void* stream);

/* Synchronises the device, reads the device error word and writes a
 * message (host, `cap` bytes) -- LA_OK if no kernel reported a fault. */
la_status la_get_error(la_cache_t* cache, char* msg, size_t cap);

/* Host only, no device work: the context of block `block` given the chosen
 * dynamic ids (ascending, n_dyn of them).  Lets callers and tests check the
 * slot order and RoPE bases without a GPU. */
la_status la_context_plan(const la_cache_config* cfg, int block, const int32_t* dyn_ids,
                          int n_dyn, la_context* out);

/* Host only, no device work: how the tensor-core attention deals its work
 * to a device with `num_sms` SMs, for blocks of T tokens, H heads and
 * contexts of at most n_slots slots.  Items: full units (h, p), numbered
 * h * n_full + p, each query tiles 2p and 2p+1 of head h (128 rows each)
 * against the whole context; when a head has an odd number of query tiles,
 * its last tile goes in pieces, one per slot, numbered
 * H * n_full + h * n_slots + s (the tile against slot s alone; a separate
 * pass merges the pieces).  out (host, `cap` entries) receives G + 1
 * offsets, then the items of CTA 0, CTA 1, ...: CTA c runs entries
 * out[G + 1 + out[c]] .. out[G + 1 + out[c + 1] - 1] in order.  Returns the
 * grid G, or -1 for bad arguments or a short buffer. */
int la_attention_schedule(int T, int H, int n_slots, int num_sms, int32_t* out, int cap);

/* Test access to stored pages.  Returns the device address of the page
 * holding `which` (0 = RoPE'd key, 1 = value, 2 = raw key [ConvKV]) of
 * `block_id` for `layer`, laid out [H][T][D] in kv_dtype, and for e4m3 the
 * device address of its H fp32 scales (else NULL). */
la_status la_debug_page(la_cache_t* cache, int layer, int block_id, int which,
                        void** page, void** scales);

/* Test access to the ConvKV memory of `layer`: device addresses of the raw
 * key ring, the value ring and the rotated key ring ([H][mem_slots][D] bf16),
 * the number of valid tokens and the ring index of the oldest token. */
la_status la_debug_memory(la_cache_t* cache, int layer, void** k_raw, void** v, void** k_rot,
                          int* n_tokens, int* oldest);

/* Profiling: `starts`/`stops` (host arrays of n cudaEvent_t, created by the
 * caller) -- the i-th attention launched after this call records starts[i]
 * immediately before it and stops[i] immediately after it on the caller's
 * stream (the tensor-core attention: its kernel and, when the block has an
 * odd number of 128-row query tiles, the merge of that tile's per-slot
 * pieces), for i < n; later launches record nothing.  n = 0 turns recording
 * off.  The arrays are copied; the events stay the caller's. */
la_status la_set_profile_events(la_cache_t* cache, void* const* starts, void* const* stops, int n);

/* Failure injection for tests of the failure path (no GPU fault is made).
 * LA_INJECT_ATTN_STALL: the next `count` tensor-core attention launches of
 * this cache first wait on a barrier that nothing completes, with a 0.1 s
 * limit.  The wait runs out, the kernel latches LA_ERR_TIMEOUT in the error
 * word, drains its in-flight copies and MMAs, frees its tensor memory and
 * returns; la_get_error then reports LA_ERR_TIMEOUT and the CUDA context
 * stays usable.  LA_ERR_UNSUPPORTED when the cache runs the CUDA-core
 * kernel. */
#define LA_INJECT_ATTN_STALL 1
/* LA_INJECT_BAD_FRAME: the next `count` attention launches of this cache (either
 * kernel) read a slot table whose first slot names a frame past the end of the
 * pool.  The kernel's bounds check rejects the table before any load, latches
 * LA_ERR_DEVICE in the error word (the message names the kernel) and returns;
 * the CUDA context stays usable. */
#define LA_INJECT_BAD_FRAME 2
la_status la_debug_inject(la_cache_t* cache, int what, int count);

/* Number of kernels this library has enqueued since it was loaded. */
uint64_t la_launch_count(void);

const char* la_status_string(la_status s);

/* Pose top-k without any device allocation (the pages have no counterpart:
 * this call exists for callers, not for the method).
 *
 * Some callers cannot call cudaMalloc at the moment they need a retrieval:
 * a host that hands out only pre-sized buffers and forbids allocation once
 * serving has started, or code on a real-time path where an allocation's
 * implicit device synchronisation would stall the stream.  la_select_context
 * keeps its retrieval scratch in the cache pool, which needs a created
 * cache.  This call runs the same retrieval kernel with its scratch (the
 * per-candidate scores, the top-k state and an error word) in one fixed
 * array inside the library: `static __device__`, LA_NOALLOC_MAX_ROWS scores
 * (256 KB + 256 B), held by every GPU that loads the library until the
 * process exits.
 *
 * table    device, [max_rows][36] fp32, caller-owned, 16-byte aligned: row j
 *          is block j's centred descriptor (x0, y0, ..., x16, y16, 0, 0);
 * inv_norm device, [max_rows] fp32, caller-owned: 1/|descriptor| (0 if zero);
 *          rows are written by this call itself when pose_row >= 0, so a
 *          caller builds its history by calling once per block;
 * query_kp host, 17 (x, y) keypoints of the block being generated;
 * pose_row table row that receives the query's descriptor, or -1 for none;
 *          it may not lie in [c0, c1) (that row would be written while it is
 *          being scored);
 * [c0, c1) candidate block ids scored against the query (rows already
 *          written); 0 <= c0 <= c1 <= min(max_rows, LA_NOALLOC_MAX_ROWS);
 *          the ids returned are table rows (absolute, not relative to c0);
 * k        0 .. LA_MAX_TOPK picks; k + 1 entries are ranked so that the gap
 *          score_k - score_(k+1) can be read;
 * ids_out, scores_out  device, k + 1 entries each, in rank order (score
 *          descending, id ascending); ranks at or past *n_out (fewer than
 *          k + 1 candidates) hold id -1 and score 0;
 * n_out    device, 1 int32: entries ranked, min(k + 1, c1 - c0);
 * status_out device, 1 int32: the kernel's error word, LA_OK (0) or the
 *          la_status of a fault it detected (the host checks above reject
 *          every input the kernel would fault on, so it reads LA_OK unless
 *          the library itself is wrong).
 *
 * Sizes beyond the scratch (c1 > LA_NOALLOC_MAX_ROWS) are rejected with
 * LA_ERR_INVALID_ARG before any work is enqueued, as are bad pointers and
 * ranges.  The call enqueues two memsets of the scratch header, the kernel
 * and four device-to-device copies on `stream`, and does not synchronise.
 * It calls no cudaMalloc, cudaFree or other allocating routine.  Its first
 * call on a device (with that device current) looks up the scratch array's
 * device address, and that lookup, like the first launch of the retrieval
 * kernel, may load the library's device code, which the CUDA runtime can
 * allocate memory for: a caller that may not allocate once it is serving
 * makes one call (or one la_select_context) on each device before it
 * starts, and before any stream capture.  The address is kept for the life
 * of the process, so cudaDeviceReset after the first call is not supported.
 * Every call shares the one array and it keeps the last call's contents:
 * calls that overlap on the GPU (different streams, no ordering) race and
 * give wrong results. */
#define LA_NOALLOC_MAX_ROWS 65536
la_status la_pose_topk_noalloc(float* table, float* inv_norm, int max_rows,
                               const float* query_kp, int pose_row, int c0, int c1, int k,
                               int32_t* ids_out, float* scores_out, int32_t* n_out,
                               int32_t* status_out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* LA_CACHE_H */
