/*
 * fs.h — C ABI of the continuous-batched decode step (decode_step_batch).
 *
 * One handle holds one dense Llama-style model on one GPU, a paged KV arena
 * shared by up to max_lanes lanes, and the scratch panels of one step. One
 * call advances up to max_lanes lanes by one token each: every weight byte is
 * read once for the whole batch, while attention stays per lane over that
 * lane's own pages.
 *
 * Sources of the operations (page title, section):
 *   - "Fat-station continuous batching — the live-path integration",
 *     "The capture": decode_step_batch(kv caches, positions, tokens) advances
 *     K lanes by one token with one weight read for the wave; "Components",
 *     item 3: fill (reset a free lane, position 0), gather, fold (sample with
 *     the lane's temperature/seed, retire, free the lane).
 *   - "MODEL-BATCHING-RESULTS — multi-user batched decode, measured",
 *     "The lever": the seven projection matmuls and the LM head run as one
 *     GEMM over a [B, *] panel; attention is per user over its own KV cache;
 *     "API": StepBatch(ids) is the per-step primitive a continuous-batching
 *     scheduler calls after admitting/evicting users between steps.
 *   - mlx-bun "Parallel slots — configurable batched serving", "KV memory",
 *     rung 3: fixed-size KV blocks in a shared pool with a block manager.
 *
 * Conventions
 *   - Every call returns FS_OK (0) or a negative FS_ERR_* code; the message
 *     of the last failure is available from fs_last_error(handle) (or
 *     fs_last_error(NULL) for a failed fs_create). No C++ exception crosses
 *     this boundary.
 *   - A handle is used by one host thread at a time.
 *   - Calls that change lane state are atomic: on any error no lane length,
 *     position or page changes.
 *   - Unless stated otherwise, pointers are HOST pointers owned by the caller
 *     and only read during the call.
 *   - All kernels run on the handle's stream (fs_set_stream). Calls that
 *     return host results synchronise that stream; fs_decode_step_batch does
 *     not (its logits are ready once the stream reaches that point).
 */
#ifndef FS_H_
#define FS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define FS_OK 0
#define FS_ERR_ARG (-1)       /* bad argument, size or descriptor field      */
#define FS_ERR_LANE (-2)      /* lane index outside [0, max_lanes)            */
#define FS_ERR_DUP_LANE (-3)  /* a lane appears twice in one step            */
#define FS_ERR_POSITION (-4)  /* positions[i] differs from the lane length   */
#define FS_ERR_TOKEN (-5)     /* token outside [0, vocab)                     */
#define FS_ERR_KV_FULL (-6)   /* page pool exhausted, or lane at max_pos      */
#define FS_ERR_OOM (-7)       /* device allocation failed                     */
#define FS_ERR_CUDA (-8)      /* a CUDA call failed (message has the detail)  */
#define FS_ERR_STATE (-9)     /* call out of order (e.g. sample before step)  */
#define FS_ERR_DEVICE (-10)   /* a kernel reported a device-side error flag   */
#define FS_ERR_SCRATCH (-11)  /* request exceeds fs_gemm_bf16_noalloc's static
                                 scratch                                      */

/* ---- element types ----------------------------------------------------- */
#define FS_DTYPE_F32 0   /* IEEE binary32                                     */
#define FS_DTYPE_BF16 1  /* bfloat16 bit patterns (uint16)                    */
#define FS_DTYPE_Q8_0 2  /* blocks of 32 inputs: fp16 scale d (little endian)
                            then 32 int8 codes q; value = q * d; 34 bytes.
                            A [rows, cols] matrix is rows*cols/32 blocks in
                            row-major order (cols must be a multiple of 32).  */

/* Model and arena description. */
typedef struct fs_model_desc {
  int32_t n_layers;        /* L                                              */
  int32_t d_model;         /* d                                              */
  int32_t n_heads;         /* H query heads                                  */
  int32_t n_kv_heads;      /* Hkv; H must be a multiple of Hkv (GQA)         */
  int32_t head_dim;        /* hd, even; RoPE pairs (i, i + hd/2)             */
  int32_t d_ffn;           /* F (SwiGLU width)                               */
  int32_t vocab;           /* V                                              */
  float rms_eps;           /* RMSNorm epsilon                                */
  double rope_theta;       /* RoPE base                                      */
  int32_t tied_embeddings; /* 1: LM head is the embedding matrix             */
  int32_t weight_dtype;    /* FS_DTYPE_F32 / _BF16 / _Q8_0 for all matrices  */
  int32_t kv_dtype;        /* FS_DTYPE_F32 or FS_DTYPE_BF16                  */
  int32_t max_lanes;       /* lanes addressable by fs_decode_step_batch      */
  int32_t page_size;       /* tokens per KV page (e.g. 16)                   */
  int32_t n_pages;         /* pages in the shared arena                      */
  int32_t max_pos;         /* tokens a lane may hold                         */
  int32_t act_split;       /* 0: the bf16 activation panels (normed x,
                              attention output, SwiGLU product) feed the
                              tensor-core GEMMs as they are; 1: each panel
                              also carries its rounding remainder
                              lo = bf16(v - hi), and every tcgen05 GEMM
                              multiplies W by hi and by lo into one f32
                              accumulator (two MMAs per k-step), which keeps
                              the products near f32 accuracy at depth (bf16
                              and Q8_0 weights only)                         */
} fs_model_desc;

/* Per-layer weights in Hugging Face layout W[out, in], row-major, in
 * weight_dtype; norm gains are always f32. Pointers may be host or device
 * memory (the library copies them during fs_create; the caller keeps
 * ownership). */
typedef struct fs_layer_weights {
  const void* wq;        /* [H*hd, d]   */
  const void* wk;        /* [Hkv*hd, d] */
  const void* wv;        /* [Hkv*hd, d] */
  const void* wo;        /* [d, H*hd]   */
  const void* w_gate;    /* [F, d]      */
  const void* w_up;      /* [F, d]      */
  const void* w_down;    /* [d, F]      */
  const float* attn_norm; /* [d]        */
  const float* ffn_norm;  /* [d]        */
} fs_layer_weights;

typedef struct fs_weights {
  const void* embed;              /* [V, d]                               */
  const void* lm_head;            /* [V, d]; NULL when tied_embeddings    */
  const float* final_norm;        /* [d]                                  */
  const fs_layer_weights* layers; /* n_layers entries                     */
} fs_weights;

typedef struct fs_handle fs_handle;

/* Creates a handle on the current CUDA device: validates the descriptor,
 * uploads and re-lays out the weights, allocates the KV arena and scratch.
 * Errors: FS_ERR_ARG (descriptor), FS_ERR_OOM, FS_ERR_CUDA. */
int fs_create(const fs_model_desc* desc, const fs_weights* weights,
              fs_handle** out);

/* Frees every device buffer of the handle. NULL is accepted. */
int fs_destroy(fs_handle* h);

/* Message of the last failed call on h (or of the last failed fs_create
 * when h is NULL). Valid until the next call on the same handle. */
const char* fs_last_error(const fs_handle* h);

/* Kernels of h run on `stream` (a cudaStream_t) from now on. NULL selects
 * the handle's own stream. */
int fs_set_stream(fs_handle* h, void* stream);

/* Fill step of the scheduler ("Components", item 3): lane k lets go of its
 * pages (a page returns to the pool once no lane holds it) and its length
 * becomes 0. Errors: FS_ERR_LANE. */
int fs_lane_reset(fs_handle* h, int32_t lane);

/* Clone, per-user prefix reuse kept under batching ("MODEL-BATCHING-RESULTS",
 * "Why in-kernel batching, not vLLM"): empty lane dst takes lane src's
 * history. dst shares src's full pages (a page holds a count of the lanes
 * that hold it; a full page is never written again), and src's partial last
 * page, which both lanes go on writing, is copied to a new page (lowest free
 * index) in every layer. Both lanes then have src's length, and a token fed
 * to either gives the logits the other gives for the same token. Enqueued
 * on the handle's stream; no synchronisation.
 * Errors: FS_ERR_LANE, FS_ERR_ARG (src == dst), FS_ERR_STATE (dst not
 * empty), FS_ERR_KV_FULL (a partial page and no free page); nothing changes
 * on error. */
int fs_lane_clone(fs_handle* h, int32_t src, int32_t dst);

/* Evict, quarantine of a span of one user's history (same passage as
 * fs_lane_clone): positions [start, end) leave the lane's cache. Entries at
 * positions p >= end move down to p - (end - start) and their keys are
 * rotated back by end - start positions, so the lane holds length - (end -
 * start) consecutive positions and the next token goes at that length.
 * K/V of the kept entries are not recomputed (they were computed while the
 * span was present). end == length drops a suffix and moves nothing. Pages
 * the lane writes (from the one holding `start` on) that another lane still
 * holds are first replaced by private copies (lowest free index); pages
 * past the new end are let go. Enqueued on the handle's stream.
 * Errors: FS_ERR_LANE, FS_ERR_ARG (not 0 <= start <= end <= length),
 * FS_ERR_KV_FULL (too few free pages for the copies); nothing changes on
 * error. */
int fs_lane_evict(fs_handle* h, int32_t lane, int32_t start, int32_t end);

/* decode_step_batch. For each i < n, lane lanes[i], whose length must equal
 * positions[i], consumes tokens[i]: its K/V at that position are appended to
 * its pages (a new page, lowest free index first, when the length is a
 * multiple of page_size) and its next-token logits are produced. On success
 * positions[i] is incremented. lanes, positions and tokens are host arrays.
 * logits_out: DEVICE pointer to f32 [n, vocab] in input order, or NULL to
 * keep the logits inside the handle for fs_sample. n == 0 is a no-op.
 * With logits_out == NULL the step's kernels run as one CUDA graph, captured
 * on the first call with that n and replayed afterwards; the first call
 * for an n therefore must not happen inside another stream capture.
 * Errors (nothing changes): FS_ERR_ARG (n outside [0, max_lanes]),
 * FS_ERR_LANE, FS_ERR_DUP_LANE, FS_ERR_POSITION, FS_ERR_TOKEN,
 * FS_ERR_KV_FULL; FS_ERR_CUDA if a launch fails (lane state is then
 * undefined). */
int fs_decode_step_batch(fs_handle* h, const int32_t* lanes,
                         int32_t* positions, const int32_t* tokens, int32_t n,
                         float* logits_out);

/* decode_step_batch followed by greedy sampling, without materialising the
 * logits: the LM head's GEMM epilogue keeps, per lane and 128-row vocab
 * tile, the largest logit and its lowest index, and a small kernel takes each
 * lane's argmax over its tiles (lowest index on ties), the token fs_sample
 * returns with temperature 0 for the same step. Lanes, positions, tokens and
 * errors as fs_decode_step_batch. tokens_out: int32 [n] in DEVICE memory
 * (ready once the stream reaches this point; the call does not synchronise)
 * or host memory (written before the call returns). When the handle's LM head
 * is split across blocks the logits are written and argmaxed by the sampler
 * kernel instead (same tokens). After this call fs_sample refuses
 * (FS_ERR_STATE): the step left no logits. The pages have this as "fused
 * sampling" in their cost notes (the LM head's [B, V] output dominates the
 * small model at large B). */
int fs_decode_step_greedy(fs_handle* h, const int32_t* lanes,
                          int32_t* positions, const int32_t* tokens, int32_t n,
                          int32_t* tokens_out);

/* decode_step_batch with chunked prefill: the prompt of a lane is consumed in
 * chunks ("Fat-station continuous batching", "What /generate does today":
 * the prompt is prefilled in chunks) within one batched step, next to the
 * decoding lanes ("DGR-012", "Prefill does not starve decode": prefill per
 * tick is capped in tokens). Rows i < n: lane lanes[i] consumes tokens[i] at
 * positions[i]; a lane may appear on several rows, and its rows' positions
 * must be exactly its length, length + 1, ..., length + rows - 1, in any
 * order. Every row's K/V are appended before attention, so a row attends to
 * its lane's keys 0..positions[i], including the other rows of this step
 * at earlier positions; a row's logits equal, bit for bit, those of feeding
 * the same tokens one per call through fs_decode_step_batch. Pages are taken
 * per lane in position order, lanes in order of first appearance. n counts
 * rows (at most max_lanes). On success every positions[i] is incremented
 * and each lane's length grows by its row count. logits_out, graphs and
 * errors as fs_decode_step_batch, except that FS_ERR_POSITION also reports
 * positions that are not the lane's next consecutive ones (repeated lanes
 * are not FS_ERR_DUP_LANE here). */
int fs_step_batch_chunked(fs_handle* h, const int32_t* lanes,
                          int32_t* positions, const int32_t* tokens, int32_t n,
                          float* logits_out);

/* Samples one token per row of the last step's logits ("Components", item 3,
 * fold: the lane's temperature and seed). Row i: temps[i] == 0 selects the
 * argmax (lowest index on ties); otherwise z = logit / temps[i] in double,
 * u = (Philox4x32-10(key = seeds[i], counter = counters[i]) >> 11) * 2^-53,
 * and the first index whose running sum of exp(z - max z) reaches u times
 * the total. temps/seeds/counters are host arrays of n entries, n must equal
 * the last step's n; tokens_out is a host array. Synchronises the stream.
 * Errors: FS_ERR_STATE (no step yet, or n differs), FS_ERR_ARG. */
int fs_sample(fs_handle* h, int32_t n, const float* temps,
              const uint64_t* seeds, const uint64_t* counters,
              int32_t* tokens_out);

/* fs_sample on device buffers, without synchronising: temps (f32), seeds and
 * counters (uint64) and tokens_out (int32) are DEVICE arrays of n entries.
 * The tokens are ready once the stream reaches this point. Same rule and
 * errors as fs_sample. */
int fs_sample_device(fs_handle* h, int32_t n, const float* temps,
                     const uint64_t* seeds, const uint64_t* counters,
                     int32_t* tokens_out);

/* ---- inspection and test hooks ---------------------------------------- */

/* Copies the last step's logits (f32 [n, vocab], input order) to `dst`
 * (host or device memory). Synchronises the stream. Errors: FS_ERR_STATE
 * (no step yet). */
int fs_copy_logits(fs_handle* h, float* dst);

/* Kernel classes of the profiler. */
#define FS_PROF_GEMM 0      /* weight-streaming GEMM (all matrices)          */
#define FS_PROF_ATTN 1      /* attention partial + combine                  */
#define FS_PROF_OTHER 2     /* embed, norms, RoPE/append, sampler           */
#define FS_PROF_CLASSES 3

/* Enables (1) or disables (0) CUDA-event timing of every kernel launch of
 * the handle, on the handle's stream. */
int fs_profile_enable(fs_handle* h, int32_t enable);

/* Synchronises the stream and returns, for kernel class `cls`, the summed
 * device time in ms, the number of launches and the algorithmic bytes those
 * launches move (weights, activations, KV and outputs, each counted once)
 * since the last read; then clears that class. */
int fs_profile_read(fs_handle* h, int32_t cls, double* ms_out,
                    int64_t* launches_out, double* bytes_out);

/* Tokens one lane can hold (the descriptor's max_pos). */
int fs_lane_capacity(const fs_handle* h, int32_t* tokens_out);

/* Kernel timeline tracing (a diagnostic; no counterpart on the pages).
 * With capacity > 0, thread 0 of every block of the library's step kernels
 * appends one record of four uint64 to a device buffer of `capacity`
 * records: word 0 = tag << 40 | waited << 39 | SM id << 24 | linear block
 * index (waited: the block passed its wait for the preceding kernel; tag: 1
 * embed, 2 RMSNorm, 3 sampler, 4 tile argmax, 5 attention (cp.async), 6
 * attention (TMA), 7 attention (tiled), 8 attention (fused), 9 RoPE +
 * KV append, 10 GEMV, 11 / 12 split attention partials / combine (the
 * three-kernel path), 13 GEMV with the SwiGLU epilogue, 16 + epilogue
 * kind for the tensor-core GEMM: 16
 * store, 17 residual, 18 SwiGLU, 19 argmax); words 1-3 = %globaltimer ns
 * at the block's entry, after its wait for the preceding kernel, and at its
 * end. Records past the capacity are counted, not stored. The buffer is
 * process-wide: one handle at a time may trace (FS_ERR_STATE otherwise);
 * capacity 0 turns tracing off and frees the buffer (also done by
 * fs_destroy). Synchronises the stream. */
int fs_trace_enable(fs_handle* h, int64_t capacity);

/* Copies min(appended, capacity, cap) records (4 uint64 each, in the order
 * they were appended) to host memory and the count appended so far to
 * *appended_out; reset != 0 then empties the buffer. Synchronises the
 * stream. Errors: FS_ERR_STATE (h is not tracing), FS_ERR_ARG. */
int fs_trace_read(fs_handle* h, uint64_t* records_out, int64_t cap, int64_t* appended_out,
                  int reset);

/* Current length (tokens held) of a lane. */
int fs_lane_length(const fs_handle* h, int32_t lane, int32_t* length_out);

/* Page table of a lane: writes min(cap, n_pages_of_lane) page indices and
 * the lane's page count to *n_out. */
int fs_lane_pages(const fs_handle* h, int32_t lane, int32_t* pages_out,
                  int32_t cap, int32_t* n_out);

/* Copies a lane's K (after RoPE) and V of one layer to host f32 arrays of
 * [length, Hkv, hd]. Synchronises the stream. */
int fs_lane_export_kv(fs_handle* h, int32_t lane, int32_t layer, float* k_out,
                      float* v_out);

/* Seeds lane `lane` (which must be empty) with n tokens of given K (already
 * rotated) and V for every layer: k and v are host f32 arrays
 * [n_layers, n, Hkv, hd]. Pages are allocated as by n decode steps.
 * Errors: FS_ERR_STATE (lane not empty), FS_ERR_KV_FULL, FS_ERR_ARG. */
int fs_lane_import_kv(fs_handle* h, int32_t lane, const float* k,
                      const float* v, int32_t n);

/* Seeds an empty lane with n tokens of pseudo-random K/V (values of unit
 * scale drawn on the device from `seed`) for timing long contexts, where
 * the content does not matter. Errors as fs_lane_import_kv. */
int fs_lane_fill_random_kv(fs_handle* h, int32_t lane, int32_t n,
                           uint64_t seed);

/* Q8_0 quantiser on the device: src is n f32 values (DEVICE pointer, n a
 * multiple of 32), blocks_out receives n/32 blocks of 34 bytes (DEVICE
 * pointer). Per block: d = max|x| / 127, q = round-half-away(x * (1/d))
 * clamped to [-127, 127], d stored as fp16 (round to nearest even); an
 * all-zero block stores d = 0 and q = 0. Runs on `stream` (a cudaStream_t,
 * NULL = default stream) and synchronises it. */
int fs_quantize_q8_0(const float* src, int64_t n, uint8_t* blocks_out,
                     void* stream);

/* Number of kernels the library launched on the handle since creation. */
int fs_kernel_launches(const fs_handle* h, int64_t* count_out);

/* Name of the GEMM path serving the handle's weight matrices: "tcgen05"
 * (bf16 weights on the tensor cores), "tcgen05-q8_0" (Q8_0 weights,
 * dequantised to bf16 in shared memory inside the GEMM), "tcgen05-q8_0+bf16"
 * or "warp-gemv" (f32 weights, d_ffn not a multiple of 64, or a device
 * without tcgen05). A Q8_0 handle whose lane capacity cuts a matrix's GEMM
 * into two or more lane groups (each of which would dequantise every weight
 * tile) also keeps that matrix as bf16(q * d), converted once by fs_create
 * (2 bytes per weight on top of the Q8_0 tiles); calls of that many groups
 * multiply the copy, the same operand bits ("tcgen05-q8_0+bf16"). The
 * environment variable FS_Q8_BF16_GROUPS, read by fs_create, sets that group
 * count (default 2; 0 keeps no copies). */
const char* fs_gemm_path(const fs_handle* h);

/* Work split of the tcgen05 GEMM for one weight matrix, as fs_create and the
 * decode step choose it (host arithmetic only: no device, handle or CUDA call;
 * a test and tuning hook). n_rows x k_inputs is the matrix (k_inputs a
 * multiple of 32), max_lanes the handle's lane capacity, n the call's lanes
 * (1 <= n <= max_lanes), sms the device's SM count, weight_dtype
 * FS_DTYPE_BF16 or FS_DTYPE_Q8_0. Writes out[8] (host):
 *   out[0] P, the stream-K width: blocks per lane group, a whole number of
 *          K splits of every 128-row tile; fixed per handle, never dependent
 *          on n (a lane's bits do not depend on its batch)
 *   out[1] lanes per group (the MMA's N), out[2] lane groups,
 *   out[3] TMEM columns a block allocates,
 *   out[4] 1 when a Q8_0 handle keeps a bf16 copy of the matrix,
 *   out[5] 1 when this call multiplies that copy,
 *   out[6] 128-row tiles, out[7] 64-wide k-blocks.
 * Reads the environment knobs fs_create reads for these choices.
 * Errors: FS_ERR_ARG (sizes, dtype, or a matrix too large for the GEMM). */
int fs_gemm_plan(int64_t n_rows, int64_t k_inputs, int max_lanes, int n, int sms,
                 int weight_dtype, int32_t* out);

/* Name of the decode-attention kernel serving the handle: "tma-mma" (KV
 * tiles by TMA, warp MMAs; bf16 KV, page_size a multiple of 8 that divides
 * or is a multiple of 64), "cp.async-mma" (KV tiles by cp.async, warp MMAs;
 * bf16 KV), "tiled", "fused" or "three-kernel" (the f32-KV and odd-shape
 * paths). The environment variable FS_ATTN=mma|tiled|fused, read by
 * fs_create, selects a slower kernel (a comparison point). */
const char* fs_attention_path(const fs_handle* h);

/* Synchronises the stream, returns the handle's device error code (0: none;
 * non-zero: a kernel gave up on a bounded wait) and clears it. fs_sample
 * reports a set code as FS_ERR_DEVICE. */
int fs_device_error(fs_handle* h, int32_t* code_out);

/* Failure-detection check (no counterpart on the pages): launches on the
 * handle's stream a kernel that waits, bounded by timeout_us microseconds
 * (1 .. 1e6), on a barrier nothing arrives on, the way every wait of the
 * step kernels is bounded; on giving up it sets the handle's device error
 * code to 99 and returns. Then as fs_device_error: synchronises, writes the
 * code (99 when the check worked) and clears it. The handle stays usable.
 * Errors: FS_ERR_ARG, FS_ERR_CUDA. */
int fs_selftest_bounded_wait(fs_handle* h, int32_t timeout_us, int32_t* code_out);

/* Test hook: Y[b, n] = sum_k X[b, k] * W[n, k] for bf16 W [N, K] and
 * X [B, K] (K a multiple of 64), f32 Y [B, N]; all DEVICE pointers owned by
 * the caller. path 1 = tcgen05 kernel with `splits` equal K splits per
 * 128-row tile (1 <= splits <= min(8, K/64)); the splits of a tile sum
 * through a thread-block cluster where the partial tile fits in shared
 * memory, else through the workspace; path 2 = the same with the workspace
 * reduction always; path 0 = warp-GEMV kernel. Paths 1 and 2 give the same
 * bits. Allocates its own workspace; runs on
 * `stream` (NULL = default) and synchronises it. Errors: FS_ERR_ARG,
 * FS_ERR_OOM, FS_ERR_CUDA, FS_ERR_DEVICE (a bounded wait timed out). */
int fs_gemm_bf16(const uint16_t* W, int32_t N, int32_t K, const uint16_t* X,
                 int32_t B, float* Y, int32_t splits, int32_t path,
                 void* stream);

/* Test hook: the tcgen05 path of fs_gemm_bf16 with the stream-K width given
 * directly: the ceil(N/128) * K/64 k-blocks (row tile after row tile) are
 * cut into `width` equal ranges, one block per range and lane group, so a
 * range may end inside a row tile and cover parts of several
 * (1 <= width <= ceil(N/128) * K/64). Same operands, ownership, stream and
 * errors as fs_gemm_bf16. The pages have no counterpart; it exists to test
 * the work split that the decode step uses. */
int fs_gemm_bf16_width(const uint16_t* W, int32_t N, int32_t K, const uint16_t* X,
                       int32_t B, float* Y, int32_t width, void* stream);

/* Tuning hook: fs_gemm_bf16_width launched once and then `reps` times, each
 * launch between two CUDA events and after a 256 MiB memset that evicts the
 * operands from L2; *ms_out receives the mean device time of one launch in
 * ms. Same operands, ownership and errors as fs_gemm_bf16. The pages have
 * no counterpart. */
int fs_gemm_bf16_time(const uint16_t* W, int32_t N, int32_t K, const uint16_t* X,
                      int32_t B, float* Y, int32_t width, int32_t reps,
                      double* ms_out, void* stream);

/* fs_gemm_bf16 without any device allocation. The pages have no counterpart
 * of this entry point; it exists for callers that cannot call cudaMalloc or
 * cudaFree: for example a process whose device memory belongs to another
 * framework's caching allocator, a latency-critical loop in which cudaFree's
 * device-wide synchronisation or an unbounded allocation time is not
 * acceptable, or an embedder with a fixed device-memory budget.
 *
 * Computes Y[b, n] = sum_k X[b, k] * W[n, k] on the tcgen05 path with
 * `splits` K splits (1 <= splits <= min(8, K/64)), exactly as
 * fs_gemm_bf16(..., splits, path = 1, ...): bf16 W [N, K], bf16 X [B, K],
 * f32 Y [B, N], K a multiple of 64, all DEVICE pointers owned by the caller.
 * Runs on `stream` (NULL = default) and synchronises it.
 *
 * Scratch: a static device array of 8 MiB in this library (every GPU that
 * loads the library holds it until exit). It holds up to 16384 arrival
 * counters (ceil(N/128) * lane groups + 1 <= 16384) and, when splits > 1,
 * splits * B * ceil(N/128) * 128 f32 partials within 8 MiB - 64 KiB (for
 * example N = 4096, splits = 4, B <= 127). Larger requests return
 * FS_ERR_SCRATCH and run nothing. Every call looks up the array's device
 * address on the current device (cudaGetSymbolAddress), synchronises
 * `stream` after the launch and copies the kernel's error flag to the host
 * before returning. Every call shares the array and clears its counters and
 * error flag first; calls that overlap on the GPU race and must be
 * serialised by the caller.
 * Errors: FS_ERR_ARG, FS_ERR_SCRATCH, FS_ERR_CUDA, FS_ERR_DEVICE. */
int fs_gemm_bf16_noalloc(const uint16_t* W, int32_t N, int32_t K,
                         const uint16_t* X, int32_t B, float* Y,
                         int32_t splits, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* FS_H_ */
