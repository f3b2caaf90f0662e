/*
 * g4.h -- C ABI of libg4, the GB300 (sm_103a) greedy decode step of a Gemma-4-E2B-shaped
 * decoder with bf16 or W4A16 weights.
 *
 * The problem statement this library follows:
 *   - "Gemma 4 E2B in JAX on One TPU v5e", Step 2: a jitted prefill, a static per-sequence KV
 *     cache, and one decode step per token; Step 3: W4A16 weights (int4, bf16 scale per 32)
 *     unpacked inside every matmul.
 *   - "Porting Gemma 4 E2B to SGLang-JAX on One Cloud TPU v5e", Step 1 (config fields),
 *     Step 3 (per-layer embeddings), Step 4 (KV-shared layers read their source layer's
 *     post-norm, post-RoPE K/V), Step 5 (double-wide MLP on the sharing layers).
 *   - "One TPU chip, eight agents", The engine (kv_share_map; RoPE follows the logical
 *     position; cached decode equals a full re-forward) and Feasibility part 1 (only the
 *     K/V-owning layers hold a cache: 18 KiB per token).
 *
 * Conventions shared by every entry point:
 *   - Pointers named d_* are DEVICE pointers on the handle's device; others are host pointers.
 *   - Calls are asynchronous on the given stream (a cudaStream_t; NULL = legacy default
 *     stream).  Outputs are valid once the stream has synchronised.
 *   - No entry point aborts, exits or traps.  Errors the host can see (bad arguments, sizes
 *     over the configured maxima, context overflow known from host metadata, allocation
 *     failure) return a negative g4_status before any device work.  Errors only the device
 *     can see (a token id >= vocab, a position >= max_context, a bounded wait that ran out)
 *     set a sticky device error word and the offending work is skipped or clamped; read it
 *     with g4_get_device_error.
 *   - All functions are thread-compatible, not thread-safe: one handle, one host thread at
 *     a time.
 *   - Entry points that take a handle or a device index make that device current for the
 *     call and restore the caller's current device before returning.
 */
#ifndef G4_H
#define G4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* g4_stream; /* == cudaStream_t */

typedef enum g4_status {
  G4_OK = 0,
  G4_ERR_INVALID_ARG = -1,      /* NULL where a pointer is required, inconsistent sizes */
  G4_ERR_UNSUPPORTED = -2,      /* a config this build does not implement */
  G4_ERR_OOM = -3,              /* device allocation failed (nothing leaked) */
  G4_ERR_CUDA = -4,             /* a CUDA runtime call failed; see g4_last_cuda_error */
  G4_ERR_CONTEXT_OVERFLOW = -5, /* a position would reach max_context */
  G4_ERR_TIMEOUT = -6,          /* a device-side bounded wait ran out */
  G4_ERR_DEVICE_CHECK = -7      /* a device-side argument check failed (bad token/position) */
} g4_status;

enum { G4_BF16 = 0, G4_W4A16 = 1 };
/* KV cache row formats: bf16 values, or int8 codes with one fp32 scale per row ("One TPU
 * chip, eight agents", Measured: the raw JAX decode kernel, int8 KV cache). */
enum { G4_KV_BF16 = 0, G4_KV_INT8 = 1 };

/* Device error word bits (g4_get_device_error). */
enum { G4_DEV_BAD_TOKEN = 1, G4_DEV_BAD_POSITION = 2, G4_DEV_TIMEOUT = 4, G4_DEV_BAD_SLOT = 8 };

/* Model shape and the numeric constants the pages leave open (every one is a field).
 * Layer l is "full" iff l % full_every == full_every - 1, else "sliding" ("4 sliding, 1 full,
 * repeating").  The last num_kv_shared_layers layers take their K/V from the last earlier
 * layer of the same type; a sharing layer with no earlier layer of its type keeps its own.
 * Width of the MLP is mlp for layers below the first sharing layer and mlp_shared from it on.
 * Constraints: num_kv_heads == 1; group_size == 32; hidden, mlp, mlp_shared, ple_dim and
 * num_q_heads * head_dim_{sliding,full} multiples of 32; head dims in {64, 128, 256, 512}. */
typedef struct g4_config {
  int32_t num_layers, num_kv_shared_layers, hidden, num_q_heads, num_kv_heads;
  int32_t head_dim_sliding, head_dim_full, sliding_window, full_every;
  int32_t mlp, mlp_shared, ple_dim, vocab;
  int32_t max_batch;   /* cache slots: sequences held at once */
  int32_t max_context; /* positions per slot */
  int32_t weight_format; /* G4_BF16 or G4_W4A16 */
  int32_t group_size;    /* 32 */
  float rms_eps, rope_theta_sliding, rope_theta_full;
  float attn_scale_sliding, attn_scale_full; /* 0 => 1/sqrt(head_dim) */
  /* KV cache.  kv_format: G4_KV_BF16 or G4_KV_INT8 (row r of d values -> a = max|r|,
   * s = a / 127, c = round-half-even(r / s) clipped to +-127, stored value c * s).
   * kv_page_size: 0 = static rows (slot, position); else paged ("Six serving engines on one
   * Cloud TPU v5e chip", Step 3: page size 128), a power of two >= 16: a slot's positions
   * [k * page, (k+1) * page) live in the pool page its page table names (g4_kv_reserve).
   * kv_pages: pool pages (0 = max_batch * ceil(max_context / kv_page_size)). */
  int32_t kv_format, kv_page_size, kv_pages;
  /* Vocabulary tables (embed / lm_head and ple_table): G4_BF16, or G4_W4A16 with the
   * linears' int4 layout and bf16 scales per 32 columns ("Six serving engines on one Cloud
   * TPU v5e chip", What Changes and What Stays: int4 embedding tables). */
  int32_t table_format;
} g4_config;

/* One projection y = W x, W [N, K].
 *   G4_BF16 : w = bf16 [N, K] row-major; scales unused.
 *   G4_W4A16: w = int32 [N, K/8], element k of a row in word k/8, bits 4*(k%8).., signed
 *             two's-complement nibble, low nibble first ("eight int4 values per int32");
 *             scales = bf16 [N, K/32].  The dequantised weight is bf16(q * scale). */
typedef struct g4_linear {
  const void* w;
  const void* scales;
} g4_linear;

/* Per-layer tensors (device pointers).  Norm gains are bf16 vectors (input, post-attention,
 * pre-FFW, post-FFW, post-per-layer-input of length hidden; q_norm/k_norm of length
 * head_dim).  k, v and k_norm are read only for layers that keep their own K/V.
 * gate/up are [mlp_l, hidden], down [hidden, mlp_l], ple_gate [ple_dim, hidden],
 * ple_proj [hidden, ple_dim]. */
typedef struct g4_layer_weights {
  g4_linear q, k, v, o, gate, up, down, ple_gate, ple_proj;
  const void *in_norm, *post_attn_norm, *pre_ffw_norm, *post_ffw_norm, *post_ple_norm;
  const void *q_norm, *k_norm;
  float layer_scale;
} g4_layer_weights;

/* Whole-model tensors.  embed: bf16 [vocab, hidden], also the tied lm_head.
 * ple_table: bf16 [vocab, num_layers * ple_dim].  ple_model_proj: [num_layers*ple_dim, hidden].
 * layers: HOST array of num_layers entries.  With table_format G4_W4A16, embed and ple_table
 * are int32 [rows, cols/8] in the linears' int4 layout and embed_scales / ple_table_scales
 * bf16 [rows, cols/32]; the dequantised value is bf16(q * scale). */
typedef struct g4_weights {
  const void* embed;
  const void* ple_table;
  g4_linear ple_model_proj;
  const void* ple_proj_norm; /* bf16 [ple_dim] */
  const void* final_norm;    /* bf16 [hidden] */
  const g4_layer_weights* layers;
  const void* embed_scales;     /* table_format G4_W4A16 only */
  const void* ple_table_scales; /* table_format G4_W4A16 only */
} g4_weights;

typedef struct g4_handle g4_handle;

/* Build a decoder on `device` (made current).  Ownership: every linear is copied into a
 * library-owned, GEMV-tiled device layout (int4 re-nibbled for 128-bit loads), so the
 * caller may free its linear tensors after this returns.  embed, ple_table and every norm
 * gain are BORROWED: they must outlive the handle.  The KV cache (max_batch x max_context
 * positions of the K/V-owning layers only; shared layers alias their source's cache) and
 * all workspaces are owned by the handle.  Synchronises the device before returning.
 * Errors: G4_ERR_INVALID_ARG, G4_ERR_UNSUPPORTED, G4_ERR_OOM, G4_ERR_CUDA (nothing leaks). */
g4_status g4_create(const g4_config* cfg, const g4_weights* weights, int device,
                    g4_handle** out);
/* Testing hook: with the environment variable G4_FAIL_ALLOC_AT=n (n >= 1), the n-th device
 * allocation of a g4_create call reports out-of-memory without allocating; g4_create then
 * frees everything it took and returns G4_ERR_OOM. */

/* Prefill (teacher-forced): for each sequence i, feed tokens d_tokens[offsets[i] ..
 * offsets[i+1]) at positions start_pos[i] + 0, 1, ... of cache slot slots[i], writing the
 * K/V of every position ("Gemma 4 E2B in JAX on One TPU v5e", Step 2: jitted prefill into a
 * static cache).  The problem statement passes slots, offsets and start positions as device
 * arrays; here they are HOST arrays (a reading): the prompt rows are planned into blocks of up
 * to 64 and, with a paged cache, pages are reserved on the host before any launch, both from
 * the lengths, so device metadata would cost a device-to-host copy and a synchronisation per
 * call.  The token ids stay on the device.  Appending to an existing context is start_pos >
 * 0.  d_next_ids[i] = greedy argmax after the sequence's last token; d_logits (nullable)
 * receives those logits [n_seq, vocab] fp32.  slots, offsets, start_pos are HOST arrays
 * (n_seq, n_seq + 1, n_seq entries); d_tokens is a DEVICE array of offsets[n_seq] ids.
 * The prompt rows run in blocks of up to 64 (sequence by sequence, positions ascending): one
 * step per block, with every row's K/V written before the block's attention, so a block's
 * rows see each other's keys causally.  While a per-layer trace is set, one step per prompt
 * position instead (trace rows are sequences).
 * Errors: G4_ERR_INVALID_ARG (n_seq outside 1..max_batch, empty or decreasing offsets, slot
 * out of range or repeated), G4_ERR_CONTEXT_OVERFLOW (start_pos + length > max_context). */
g4_status g4_prefill(g4_handle* h, g4_stream stream, int32_t n_seq, const int32_t* slots,
                     const int32_t* offsets, const int32_t* start_pos, const int32_t* d_tokens,
                     int32_t* d_next_ids, float* d_logits);

/* One greedy decode step for n_seq sequences: d_tokens[i] at logical position
 * d_positions[i] (== its cache slot index) of cache slot d_slots[i].  Writes the owning
 * layers' K/V at that position, returns d_next_ids[i] = argmax of the logits (lowest index
 * among equal maxima) and, if d_logits != NULL, the logits [n_seq, vocab] fp32.  All
 * arguments are device pointers, so the step never synchronises with the host; it runs as
 * one CUDA-graph launch, re-captured when the pointer set or n_seq changes.  A position >=
 * max_context or a token >= vocab sets the device error word (the sequence's work is
 * clamped).  Errors: G4_ERR_INVALID_ARG (n_seq outside 1..max_batch, NULL pointers). */
g4_status g4_decode_step(g4_handle* h, g4_stream stream, int32_t n_seq, const int32_t* d_slots,
                         const int32_t* d_tokens, const int32_t* d_positions,
                         int32_t* d_next_ids, float* d_logits);

/* Paged KV cache (kv_page_size > 0): make cache slot `slot` hold positions [0,
 * n_positions), taking pool pages as needed and writing the slot's page-table entries on
 * `stream` (host arrays are not touched after return).  Pages already held stay; none is
 * taken when the pool is short.  A decode step whose position has no page sets
 * G4_DEV_BAD_POSITION and leaves that row's K/V unwritten.  g4_prefill reserves its own
 * positions.  With static rows (kv_page_size == 0) this only checks n_positions.
 * Errors: G4_ERR_INVALID_ARG (slot out of range, n_positions < 0), G4_ERR_CONTEXT_OVERFLOW
 * (n_positions > max_context), G4_ERR_OOM (not enough free pages). */
g4_status g4_kv_reserve(g4_handle* h, g4_stream stream, int32_t slot, int32_t n_positions);

/* Paged KV cache: return every page of `slot` to the pool (its positions become unheld).
 * No-op with static rows.  Errors: G4_ERR_INVALID_ARG. */
g4_status g4_kv_release(g4_handle* h, g4_stream stream, int32_t slot);

/* Free pool pages (paged KV cache), or -1 with static rows or a NULL handle. */
int32_t g4_kv_pages_free(const g4_handle* h);

/* Failure-detection probe (tests): launch one warp on `stream` that waits, bounded by
 * wait_ns of %globaltimer, for a device flag that nothing sets; when the wait runs out it sets
 * G4_DEV_TIMEOUT in the device error word and returns, as every bounded wait of the step's
 * kernels does.  The next g4_get_device_error then returns G4_ERR_TIMEOUT and the handle stays
 * usable.  Errors: G4_ERR_INVALID_ARG (wait_ns outside 0..2e9). */
g4_status g4_timeout_probe(g4_handle* h, g4_stream stream, int64_t wait_ns);

/* Synchronise `stream`, read and clear the device error word.  *word_out (nullable) gets
 * the G4_DEV_* bits.  Returns G4_ERR_TIMEOUT if the timeout bit is set, else
 * G4_ERR_DEVICE_CHECK if any other bit is set, else G4_OK. */
g4_status g4_get_device_error(g4_handle* h, g4_stream stream, int32_t* word_out);

/* Optional per-layer trace for tests: while d_trace != NULL, every step (decode and each
 * prefill position) writes, for sequence i and layer l, the attention output (n_q_heads *
 * head_dim floats, zero-padded to n_q_heads * head_dim_full) and the residual stream after
 * the layer (hidden floats), as
 *   d_trace[((l * 2 + 0) * max_batch + i) * stride ...]  attention output
 *   d_trace[((l * 2 + 1) * max_batch + i) * stride ...]  residual after layer l
 * with stride = max(hidden, n_q_heads * head_dim_full).  The buffer must hold
 * num_layers * 2 * max_batch * stride floats; pass NULL to stop.  Errors: INVALID_ARG. */
g4_status g4_set_trace(g4_handle* h, float* d_trace, int64_t capacity_floats);

/* Per-phase timing of the decode step (profiling).  Runs `repeats` decode steps with the
 * same arguments as g4_decode_step, launched directly (not from a graph) with a CUDA event
 * pair on `stream` around every phase launch, synchronises, and fills one entry per phase
 * name in first-launch order: launches, total milliseconds between its events, and the
 * bytes of weights its launches stream (the KV bytes of attention phases are not counted:
 * the host does not know the positions).  Each repeat rewrites the same K/V rows, so the
 * cache state is that of one step.  Errors: INVALID_ARG. */
typedef struct g4_phase_stat {
  char name[32];
  int32_t launches;
  double ms_total;
  double bytes_total;
} g4_phase_stat;
g4_status g4_profile_step(g4_handle* h, g4_stream stream, int32_t n_seq, const int32_t* d_slots,
                          const int32_t* d_tokens, const int32_t* d_positions, int32_t* d_next_ids,
                          float* d_logits, int32_t repeats, g4_phase_stat* stats, int32_t max_stats,
                          int32_t* n_stats);

/* Bytes of device memory the handle owns (weights copies, KV cache, workspaces). */
int64_t g4_device_bytes(const g4_handle* h);

/* Which implementation a step of n_seq sequences runs: 1 = the persistent single-launch step
 * (selected with g4_set_step_mode and n_seq <= 2), 0 = one launch per phase (replayed as a
 * CUDA graph), -1 = NULL handle. */
int32_t g4_step_mode(const g4_handle* h, int32_t n_seq);

/* Select the implementation of steps with n_seq <= 2: mode 0 (the default) launches one kernel
 * per phase; mode 1 runs the whole step as one persistent cooperative kernel (phases separated
 * by a bounded grid barrier).  Both compute the same step; their fp32 sums are ordered
 * differently.  Not thread-safe against concurrent steps on the same handle.  Errors:
 * G4_ERR_INVALID_ARG (NULL handle, mode not 0/1), G4_ERR_UNSUPPORTED (mode 1 on a model the
 * persistent step was not planned for, e.g. an lm_head input wider than 2048). */
g4_status g4_set_step_mode(g4_handle* h, int32_t mode);

/* Release everything the handle owns (after synchronising its device).  NULL is a no-op. */
void g4_free(g4_handle* h);

const char* g4_status_string(g4_status s);
/* Text of the last CUDA error seen by any g4_* call on this thread ("" if none). */
const char* g4_last_cuda_error(void);

/* ----------------------------------------------------------------------------------------
 * Standalone kernels (the same device code the decode step runs), for per-kernel checks.
 * --------------------------------------------------------------------------------------*/

typedef struct g4_linear_op g4_linear_op;

/* Copy one projection (format and layout as g4_linear) into the library's tiled layout on
 * `device`.  Errors: INVALID_ARG (n_in not a multiple of 32, n_out < 1), OOM, CUDA. */
g4_status g4_linear_create(int device, int32_t weight_format, int32_t n_out, int32_t n_in,
                           const void* d_w, const void* d_scales, g4_linear_op** out);
/* y[b, n] = sum_k W[n, k] x[b, k] for b < n_rows; d_x fp32 [n_rows, n_in], d_y fp32
 * [n_rows, n_out], fp32 accumulation of the bf16 (or bf16(q*s)) weights.
 * Errors: INVALID_ARG (n_rows outside 1..64, NULL). */
g4_status g4_linear_forward(g4_linear_op* op, g4_stream stream, int32_t n_rows,
                            const float* d_x, float* d_y);
void g4_linear_free(g4_linear_op* op);

/* Row-wise greedy argmax of fp32 logits [n_rows, n_cols]: d_ids[r] = lowest index of the
 * maximum (NaNs never win).  Uses the same block-partial + last-block reduction as the
 * lm_head.  Errors: INVALID_ARG (n_rows outside 1..64, n_cols < 1). */
g4_status g4_argmax_rows(int device, g4_stream stream, int32_t n_rows, int32_t n_cols,
                         const float* d_logits, int32_t* d_ids);

/* Row-wise greedy argmax like g4_argmax_rows, for callers that must not allocate device
 * memory: it calls no cudaMalloc, cudaFree or allocating library routine.  Such callers
 * include a serving loop that has handed all device memory to its own pool (an allocation
 * here would fail, or would synchronise the whole device in the middle of a step) and code
 * running between a stream capture's begin and end, where cudaMalloc may not be called.
 * (The pages have no counterpart: this is an interface convenience, not part of the method.)
 *
 * Its scratch is one fixed array in the library (about 129 KB), held by every GPU that
 * loads the library until the process exits.  Limits: n_rows <= 64 and n_cols <= 1,048,576;
 * larger sizes return G4_ERR_INVALID_ARG (g4_last_cuda_error names the limits) with no
 * device work.  The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  Every call clears the
 * array's counters with a memset on `stream` and then reuses the array, which keeps the
 * last call's partial results: calls that overlap on the GPU (other streams, other
 * threads) race on it and must be serialised by the caller. */
g4_status g4_argmax_rows_static(int device, g4_stream stream, int32_t n_rows, int32_t n_cols,
                                const float* d_logits, int32_t* d_ids);

#ifdef __cplusplus
}
#endif

#endif /* G4_H */
