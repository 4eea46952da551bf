/*
 * zerogr.h - C ABI of the GB300 (sm_103a) filtering-first constrained beam
 * decoder over semantic IDs (SIDs).
 *
 * Method: "ZeroGR: Filtering-First Constrained Decoding for Generative
 * Recommendation" (paper-daily.com digest).  Section names used below:
 *   [Problem]  "What problem does it solve"  (SID beam search, validity filter)
 *   [Order]    "Does filtering first change the result"  (legal-only softmax)
 *   [Pipeline] "Overall flow"  (three parts; four stages per decoding step)
 *   [Index]    "Why slice the index by decoding step"  (step tables, dense vs
 *              sparse, implicit successor rows)
 *   [Speed]    "Why computing fewer scores is not automatically faster"
 *              (padded candidate slots, in-place weight rows, per-step
 *              full-vs-selective choice made on warm-up requests)
 *   [Results]  "Is the scheme really better"  (unconstrained decode as the
 *              speed reference; chunked CPU rebuild streamed through two
 *              buffers)
 *
 * Conventions (every call):
 *   - Every call returns a zg_status; nothing exits, throws or traps.  After
 *     a non-OK status, zg_last_error() gives a message (thread-local).
 *   - "host" pointers are CPU memory; "device" pointers are CUDA device
 *     memory of the current device (for example torch.Tensor.data_ptr()).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).
 *   - Inputs are read-only and stay owned by the caller.  Handles
 *     (zg_index, zg_plan) are owned by the library and released with their
 *     *_free call.  Indexes and plans are read-only after creation and may be
 *     shared by concurrent decodes; a workspace may not.
 *   - Limits: 1 <= L <= 8, 1 <= V <= 65536, L * ceil(log2 V) <= 64,
 *     d % 8 == 0 with d * sizeof(weight) <= 2048 bytes,
 *     1 <= K <= beam <= 512, B >= 1.  Anything outside returns
 *     ZG_ERR_INVALID_ARG (or ZG_ERR_UNSUPPORTED for the key-width limit).
 */
#ifndef ZEROGR_H
#define ZEROGR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define ZG_API __attribute__((visibility("default")))
#else
#define ZG_API
#endif

#define ZG_MAX_STEPS 8
#define ZG_MAX_BEAM 512

typedef enum {
  ZG_OK = 0,
  ZG_ERR_INVALID_ARG = 1,
  ZG_ERR_OUT_OF_MEMORY = 2,
  ZG_ERR_CUDA = 3,
  ZG_ERR_UNSUPPORTED = 4,
  ZG_ERR_TIMEOUT = 5,
  ZG_ERR_DEVICE_STATUS = 6,
  ZG_ERR_IO = 7
} zg_status;

typedef enum { ZG_F32 = 0, ZG_BF16 = 1, ZG_F16 = 2 } zg_dtype;
typedef enum { ZG_FMT_SPARSE = 0, ZG_FMT_DENSE = 1 } zg_format;
typedef enum { ZG_SELECTIVE = 0, ZG_FULL = 1, ZG_NAIVE = 2 } zg_variant;
typedef enum { ZG_RESIDENT_DEVICE = 0, ZG_RESIDENT_HOST = 1 } zg_residency;
typedef enum { ZG_FORMAT_AUTO = 0, ZG_FORMAT_ALL_SPARSE = 1, ZG_FORMAT_ALL_DENSE = 2 } zg_format_mode;
typedef enum { ZG_ORDER_FILTER_FIRST = 0, ZG_ORDER_SCORE_FIRST = 1 } zg_order;
typedef enum { ZG_HIDDEN_SPLIT = 0, ZG_HIDDEN_SINGLE = 1 } zg_hidden_rounding;
typedef enum { ZG_SCORES_AUTO = 0, ZG_SCORES_WRITTEN = 1, ZG_SCORES_CHUNK_TOPS = 2 } zg_full_scores;

typedef struct zg_index zg_index; /* opaque: step tables + host header */
typedef struct zg_plan zg_plan;   /* opaque: per-step variant choice   */

#define ZG_MAX_DECO_LAYERS 4

/* A light causal decoder producing each step's hidden vector ("Separating
 * Thinking from Spelling", AI Papers Daily digest: the backbone emits a fixed
 * next-item concept once; a light 2-layer, 256-wide causal decoder
 * conditioned on the concept and the generated prefix runs the
 * trie-constrained beam search).  The hidden vector of a beam with prefix
 * t_1..t_{s-1} at step s is the output of the last position of the sequence
 * [c_1 .. c_M, E_1[t_1] .. E_{s-1}[t_{s-1}]], each row plus its position
 * embedding, after `layers` pre-norm layers
 *   x += attn(norm(x)) Wo^T,  attn = causal multi-head attention of
 *        (norm(x) Wq^T, norm(x) Wk^T, norm(x) Wv^T), scores / sqrt(d/heads);
 *   x += relu(norm(x) W1^T) W2^T;
 * and a final norm; norm(x) = x / sqrt(mean(x^2) + 1e-6) per row.
 * All device float32, row-major [out][in], 16-byte aligned, caller-owned:
 *   E[s]: [V][d], s = 0..L-2;  P: [M + L - 1][d];
 *   Wq, Wk, Wv, Wo[l]: [d][d];  W1[l]: [ffn][d];  W2[l]: [d][ffn].
 * Limits: 1 <= M <= 8, 1 <= layers <= ZG_MAX_DECO_LAYERS, heads divides d
 * with d / heads <= 256, ffn a multiple of 4. */
typedef struct {
  int32_t M, heads, ffn, layers;
  const float* E[ZG_MAX_STEPS];
  const float* P;
  const float* Wq[ZG_MAX_DECO_LAYERS];
  const float* Wk[ZG_MAX_DECO_LAYERS];
  const float* Wv[ZG_MAX_DECO_LAYERS];
  const float* Wo[ZG_MAX_DECO_LAYERS];
  const float* W1[ZG_MAX_DECO_LAYERS];
  const float* W2[ZG_MAX_DECO_LAYERS];
} zg_deco;

/* The model the decoder scores with ([Pipeline] stage 1 is the model's
 * hidden vector).  Without a light decoder (deco NULL) it is the synthetic
 * model h = u + sum_{j<s} C_j[t_j]:
 *   C[s]: device float32 [V][d], row-major, s = 0..L-2 (the table added after
 *         choosing the token of step s+1); C[L-1] is unused and may be NULL.
 *   W[s]: device w_dtype [V][d], row-major, s = 0..L-1 (output head of step
 *         s+1); rows must be 16-byte aligned (d % 8 == 0 ensures it).
 *   deco: NULL, or a light decoder (zg_deco) producing the hidden vectors;
 *         then C is unused and the decode's input u holds each request's M
 *         concept vectors, device float32 [B][M][d], and zg_decode runs the
 *         decoder before every step's projection (steps are not fused).
 * The struct and its pointer arrays are caller-owned. */
typedef struct {
  int32_t L, V, d, w_dtype;
  const float* C[ZG_MAX_STEPS];
  const void* W[ZG_MAX_STEPS];
  const zg_deco* deco;
} zg_model;

/* Index build options.  Zero-initialised = defaults. */
typedef struct {
  int32_t n_threads;           /* host threads; <= 0: all hardware threads          */
  int32_t format_mode;         /* ZG_FORMAT_AUTO (per-step rule), ZG_FORMAT_ALL_SPARSE
                                  or ZG_FORMAT_ALL_DENSE                             */
  int32_t reserved;
  int32_t residency;           /* ZG_RESIDENT_DEVICE (decodable) or ZG_RESIDENT_HOST
                                  (no CUDA use at all: stats/export/save only)       */
  uint64_t pinned_chunk_bytes; /* size of each of the two pinned staging buffers;
                                  0: 64 MiB.  Grown if one first-token subtree's
                                  slice of a step is larger.                         */
} zg_build_opts;

typedef struct {
  int32_t format;          /* ZG_FMT_SPARSE or ZG_FMT_DENSE                  */
  uint32_t rows;           /* distinct length-(s-1) prefixes                 */
  uint32_t nnz;            /* legal (row, token) entries = rows of step s+1  */
  uint32_t words_per_row;  /* 32-bit words of a dense bitmap row            */
  uint32_t max_fanout;     /* slots per beam of this step (largest row)     */
  uint32_t reserved;
  double mean_fanout;      /* nnz / rows                                     */
  double legal_fraction;   /* nnz / (rows * V)                               */
  uint64_t bytes;          /* bytes of this step's table                     */
} zg_step_stats;

typedef struct {
  int32_t L, V, residency, reserved;
  int64_t n_input;           /* SIDs given                                     */
  int64_t n_unique;          /* distinct SIDs (duplicates merged)              */
  uint64_t bytes;            /* all step tables                                */
  uint64_t dense_trie_bytes; /* the same catalogue as a dense prefix-trie
                                tensor, one int32 child per (row, token):
                                sum_s rows_s * V * 4 (computed, not allocated)  */
  double ms_sort, ms_count, ms_fill, ms_total; /* build phases, host wall time */
} zg_index_info;

/* ---------------------------------------------------------------- index ---
 * zg_index_build - [Index], [Results] (rebuild pipeline).
 * Builds the step-sliced index from n catalogue SIDs on host threads: pack
 * and sort, merge duplicates, count each first-token subtree's rows and
 * entries (pass 1), lay the subtrees out by prefix sums, then fill them in
 * parallel into two pinned buffers in turn while the other buffer's
 * cudaMemcpyAsync to HBM runs on `stream` (pass 2).  No kernels run.
 *   sids: host int32 [n][L], tokens in [0, V).  Caller-owned, read only.
 * Table layout of step s (1-based): rows are the distinct length-(s-1)
 * prefixes in lexicographic order; uint32 rowptr[rows+1]; a row's legal
 * tokens ascending; entry e (in (row, token) order) is row e of step s+1.
 * Sparse steps store uint16 col[nnz]; dense steps a uint32 bitmap
 * [rows][ceil(V/32)] (bit t%32 of word t/32).  Automatic format: dense iff
 * 4*rows*ceil(V/32) < 2*nnz.
 * Returns ZG_ERR_INVALID_ARG for n < 1, bad L/V or a token out of range,
 * ZG_ERR_UNSUPPORTED if L*ceil(log2 V) > 64, ZG_ERR_OUT_OF_MEMORY /
 * ZG_ERR_CUDA on allocation or copy failure.  Returns after the copies end. */
ZG_API zg_status zg_index_build(const int32_t* sids, int64_t n, int32_t L, int32_t V,
                         const zg_build_opts* opts, void* stream, zg_index** out);

/* Per-step table statistics (step is 1-based). */
ZG_API zg_status zg_index_stats(const zg_index* idx, int32_t step, zg_step_stats* out);
ZG_API zg_status zg_index_info_get(const zg_index* idx, zg_index_info* out);

/* Canonical bytes of one step's table, for bit-exact comparison: uint32
 * {format, rows, nnz, words_per_row}, uint32 rowptr[rows+1], then uint16
 * col[nnz] zero-padded to 4 bytes (sparse) or uint32 bitmap[rows][words]
 * (dense), little-endian.  If buf is NULL or *bytes is too small, *bytes is
 * set to the size needed and ZG_ERR_INVALID_ARG is returned (buf NULL:
 * ZG_OK). */
ZG_API zg_status zg_index_export(const zg_index* idx, int32_t step, void* buf, size_t* bytes);

/* Save to / load from a file: header, step metadata, table bytes and a
 * 64-bit FNV-1a checksum.  Load fails with ZG_ERR_IO on a short, corrupt or
 * foreign file. */
ZG_API zg_status zg_index_save(const zg_index* idx, const char* path);
ZG_API zg_status zg_index_load(const char* path, int32_t residency, void* stream, zg_index** out);
ZG_API void zg_index_free(zg_index* idx);

/* ---------------------------------------------------------------- plan ----
 * [Speed]: before serving, warm-up requests time each scoring variant at
 * every step; the fastest is kept until the next model update.
 *   ZG_SELECTIVE: score only legal tokens, reading their weight rows in place
 *                 into padded slots (one slot per legal token; every beam of
 *                 the step gets max_fanout slots, or V on dense steps).
 *   ZG_FULL:      project every token (a dense contraction), then pick the
 *                 legal ones.
 *   ZG_NAIVE:     measurement contrast only (never chosen by zg_tune): legal
 *                 tokens scored the straightforward way of [Speed]'s figure -
 *                 compact every beam's candidates into one list (count, scan,
 *                 list), copy their weight rows into a temporary matrix, dot
 *                 each row with its beam's hidden vector.  Its workspace holds
 *                 B * min(beams * max_fanout, nnz) listed rows of the step;
 *                 ZG_ERR_UNSUPPORTED above 16 GiB.
 * zg_tune runs the decode step by step on warm_u (device float32 [B][d]):
 * each variant of step s runs 2 warm-up times and `reps` timed times on the
 * same entering state (CUDA events on `stream`); the faster is kept and
 * advances the state.  Allocates and frees its own workspace.  Synchronous. */
ZG_API zg_status zg_tune(const zg_index* idx, const zg_model* model, const float* warm_u, int32_t B,
                  int32_t beam, int32_t K, int32_t reps, void* stream, zg_plan** out);
/* A plan with a fixed variant per step (variant: host uint8 [L], each
 * ZG_SELECTIVE, ZG_FULL or ZG_NAIVE). */
ZG_API zg_status zg_plan_force(const zg_index* idx, int32_t B, int32_t beam, const uint8_t* variant,
                        zg_plan** out);
/* How zg_decode runs the plan's trailing run of ZG_SELECTIVE steps: as one
 * fused kernel with a thread-block cluster of cluster_ctas CTAs (1, 2, 4, 8
 * or 16) per request and cluster barriers between scoring and selection, or
 * (0) as stand-alone step kernels.  Default 8; zg_tune times every size and
 * keeps the fastest.  Results are identical either way. */
ZG_API zg_status zg_plan_set_fusion(zg_plan* plan, int32_t cluster_ctas);
/* variant: host uint8 [L]; step_ms: host float [L][2] timings of {SELECTIVE,
 * FULL} from zg_tune (-1 when not timed); cluster_ctas: the fused kernel's
 * cluster size (0: not fused); fused_ms: host float [5] timings of the fused
 * kernel with 1, 2, 4, 8, 16 CTAs a cluster (-1 when not timed or not
 * schedulable).  Any output may be NULL. */
ZG_API zg_status zg_plan_describe(const zg_plan* plan, uint8_t* variant, float* step_ms,
                                  int32_t* cluster_ctas, float* fused_ms);
/* Order of filtering and normalisation (the comparison of [Order]).
 *   ZG_ORDER_FILTER_FIRST (default): log-softmax over the legal tokens only.
 *   ZG_ORDER_SCORE_FIRST: the conventional baseline of [Problem] - project
 *     every token (one dense contraction), normalise the log-softmax over the
 *     whole codebook, then mask the illegal tokens and select among the legal
 *     ones.  Every step runs ZG_FULL whatever the plan's variants, unfused;
 *     sparse-format steps first expand each beam's legal list into a token
 *     bitmap (workspace), dense-format steps read the index bitmap.  Scores
 *     are the score-first cumulative log-probabilities (at most the
 *     filter-first ones: the mass of illegal tokens is not redistributed).
 * Changes the workspace size: size the workspace after setting the order.
 * ZG_ERR_INVALID_ARG for another value. */
ZG_API zg_status zg_plan_set_order(zg_plan* plan, int32_t order);
/* How ZG_FULL steps run ([Speed]: a dense step scores every token in one
 * large product, then picks the legal ones).
 *   hidden_rounding (bf16/fp16 weights; the tensor cores take both operands
 *   in the weights' type):
 *     ZG_HIDDEN_SPLIT (default): the fp32 hidden vector enters as two half
 *       operands (hi + lo, two products into one fp32 accumulator), so full
 *       and selective scores agree to ~1e-6;
 *     ZG_HIDDEN_SINGLE: one rounding of the hidden vector (half the tensor
 *       work; scores off by ~1e-3 for bf16, ~1e-4 for fp16, inside the 2e-2
 *       tolerance of half weights).
 *   scores:
 *     ZG_SCORES_WRITTEN: every score goes to the workspace, the select reads
 *       them back;
 *     ZG_SCORES_CHUNK_TOPS: no score is written: per 32-token chunk of a beam
 *       the projection keeps the legal (max, sum exp), the second-largest
 *       legal score and the position of the largest; the select cuts on the
 *       chunk maxima and re-scores the rare chunk whose second-largest also
 *       clears the cut (exact; same results as written scores);
 *     ZG_SCORES_AUTO (default): written (chunk tops measured slower: their
 *       re-scores cost more than the stores they save).
 * Results agree with the other settings within the rounding stated above.
 * Changes the workspace size: size the workspace after setting it.
 * ZG_ERR_INVALID_ARG for other values. */
ZG_API zg_status zg_plan_set_full_projection(zg_plan* plan, int32_t hidden_rounding, int32_t scores);
/* Save / load a plan ([Speed]: the variant chosen per step on warm-up
 * requests is kept until the next model update, so a serving process can
 * reuse a tuned plan across restarts).  The file holds the steps, batch,
 * beam, order, fusion, the per-step variants and the tuner's timings, and a
 * 64-bit FNV-1a checksum.  zg_plan_load returns ZG_ERR_IO for a missing,
 * short, corrupt or foreign file, or one whose fields are out of range; the
 * new plan is owned by the caller (zg_plan_free). */
ZG_API zg_status zg_plan_save(const zg_plan* plan, const char* path);
ZG_API zg_status zg_plan_load(const char* path, zg_plan** out);
ZG_API void zg_plan_free(zg_plan* plan);

/* --------------------------------------------------------------- decode ---
 * Workspace bytes zg_decode needs for (idx, plan, model, B, beam, K); idx
 * NULL = unconstrained decode. */
ZG_API zg_status zg_decode_workspace_size(const zg_index* idx, const zg_plan* plan,
                                   const zg_model* model, int32_t B, int32_t beam, int32_t K,
                                   size_t* bytes);

/* zg_decode - [Pipeline] online part, all L steps.  Per step and beam:
 * look up the legal tokens of the beam's row, form the hidden vector
 * (gather-add), score legal tokens (plan's variant), log-softmax over the
 * legal tokens only ([Order]), add to the cumulative score, keep the best
 * `beam` candidates per request (best K at the last step).  Ties order by
 * lower parent-beam rank, then lower slot (ascending token).  One root beam
 * per request.
 *   idx:  device-resident index, or NULL for the unconstrained decode of
 *         [Results] (every token legal, every step full, SIDs need not
 *         exist; of the plan only its full-projection settings apply).
 *   plan: per-step variants; NULL = ZG_SELECTIVE at every step.
 *   u:    device float32 [B][d] request vectors.
 *   out_sids:   device int32 [B][K][L]; out_scores: device float32 [B][K],
 *               best first; rows beyond a request's candidates are -1/-inf.
 *   workspace:  device, >= zg_decode_workspace_size bytes, 256-byte aligned;
 *               caller-owned scratch, contents undefined on return.
 * Asynchronous on `stream`: only kernel launches, so it can be captured in
 * a CUDA graph.  Launch errors are returned; device-side invariant breaches
 * are recorded for zg_check_device_status. */
ZG_API zg_status zg_decode(const zg_index* idx, const zg_plan* plan, const zg_model* model,
                    const float* u, int32_t B, int32_t beam, int32_t K, int32_t* out_sids,
                    float* out_scores, void* workspace, size_t ws_bytes, void* stream);

/* zg_decode with host buffers: copies u (host float32 [B][d], pinned memory
 * recommended) to the device, decodes, copies out_sids (host int32
 * [B][K][L]) and out_scores (host float32 [B][K]) back, and synchronises
 * `stream`.  The workspace must be sized with zg_decode_host_workspace_size. */
ZG_API zg_status zg_decode_host_workspace_size(const zg_index* idx, const zg_plan* plan,
                                        const zg_model* model, int32_t B, int32_t beam,
                                        int32_t K, size_t* bytes);
ZG_API zg_status zg_decode_host(const zg_index* idx, const zg_plan* plan, const zg_model* model,
                         const float* u_host, int32_t B, int32_t beam, int32_t K,
                         int32_t* out_sids_host, float* out_scores_host, void* workspace,
                         size_t ws_bytes, void* stream);

/* Per-step record of zg_decode_trace. */
typedef struct {
  int32_t variant;        /* ZG_SELECTIVE or ZG_FULL (always ZG_FULL unconstrained) */
  int32_t live_beams;     /* beams entering the step with a finite score           */
  int64_t legal_slots;    /* sum of legal fan-outs F_b over live beams (V each when
                             unconstrained)                                        */
  int64_t chunks;         /* 32-slot chunks the selective kernel scores            */
  int64_t unique_tokens;  /* distinct legal tokens = distinct W_s rows touched     */
  int64_t index_bytes;    /* table bytes the filter reads: rowptr pairs plus column
                             entries (sparse) or bitmap rows (dense)               */
  float ms_gather;        /* gather-add kernel (full steps at s >= 2) or the       */
                          /* selective step's chunk-counting kernel, else 0        */
  float ms_project;       /* selective or full projection kernel                   */
  float ms_select;        /* masked log-softmax + cumulative add + top-K kernel     */
  float ms_model;         /* the light decoder's kernels of this step (0 without)   */
} zg_step_trace;

typedef struct {
  int32_t L;
  int32_t fused_from;     /* first step zg_decode runs in its fused cluster kernel
                             (0: none)                                              */
  zg_step_trace step[ZG_MAX_STEPS]; /* stand-alone step kernels, step by step       */
  float ms_fused;         /* zg_decode's fused cluster kernel                        */
  float ms_total;         /* all kernels of zg_decode's own launch sequence          */
} zg_trace;

/* zg_decode_trace - two timed passes of the zg_decode computation on
 * `stream` (CUDA events around every kernel launch): first zg_decode's own
 * launch sequence (ms_fused, ms_total), then the stand-alone step kernels
 * step by step (ms_gather/ms_project/ms_select) with an untimed counting
 * kernel after each step that fills the work counts (the observability the
 * per-step variant choice of [Speed] rests on).  Each step of the second
 * pass is queued behind a 50 us device-side delay so that its launches are
 * all enqueued before it starts: the events time the kernels, not the
 * host's launch gaps.  Both passes give the same
 * results; the outputs hold the second pass's.  Synchronous; not for CUDA
 * graph capture.  The workspace is the one sized by zg_decode_workspace_size. */
ZG_API zg_status zg_decode_trace(const zg_index* idx, const zg_plan* plan, const zg_model* model,
                                 const float* u, int32_t B, int32_t beam, int32_t K,
                                 int32_t* out_sids, float* out_scores, void* workspace,
                                 size_t ws_bytes, void* stream, zg_trace* trace);

/* Bytes of the static device scratch zg_decode_static decodes in. */
#define ZG_STATIC_SCRATCH_BYTES (16u << 20)

/* zg_decode_static - the paper has no counterpart; this is a deployment
 * convenience.  zg_decode with no caller workspace and no allocation at all:
 * the scratch is a fixed ZG_STATIC_SCRATCH_BYTES (16 MiB) array in the
 * library's device memory, held by every GPU that loads the library until
 * the process exits.  It serves callers that cannot allocate device memory
 * when they decode: processes whose device memory is pre-reserved by another
 * framework's allocator, request threads on which allocation (and the
 * synchronisation that freeing implies) is not allowed, runtimes that plan
 * memory statically.
 * Arguments and results are those of zg_decode without workspace/ws_bytes.
 * A decode whose zg_decode_workspace_size exceeds ZG_STATIC_SCRATCH_BYTES is
 * rejected with ZG_ERR_INVALID_ARG before anything runs.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.  The
 * address is cached per device and CUDA context: after cudaDeviceReset the
 * next call (again outside any capture) looks it up in the new context.
 * Every call on a device shares the one array and it keeps the previous
 * call's contents (the decode writes every scratch word before reading it,
 * so nothing needs clearing): calls whose executions can overlap on the GPU
 * (concurrent streams, other host threads) race and must not be issued. */
ZG_API zg_status zg_decode_static(const zg_index* idx, const zg_plan* plan, const zg_model* model,
                                  const float* u, int32_t B, int32_t beam, int32_t K,
                                  int32_t* out_sids, float* out_scores, void* stream);

/* ZG_STATIC_SCRATCH_BYTES as compiled into the library (for bindings that
 * cannot read the header). */
ZG_API size_t zg_static_scratch_bytes(void);

/* Test and diagnosis hook, no counterpart in the paper: the number of polls
 * after which a pipeline wait (an mbarrier) of the tensor-core full
 * projection gives up, records bit 2 in the device status word and ends the
 * kernel early (its copies and tensor-core operations drained, tensor memory
 * freed).  0 restores the default (2^26 polls, about a second).  Applies to
 * launches issued after the call, process-wide.  A limit too small for the
 * work makes decodes fail with ZG_ERR_DEVICE_STATUS. */
ZG_API void zg_debug_set_wait_limit(uint32_t polls);

/* Test hook, no counterpart in the paper: makes the index builder's next
 * pinned staging allocation (ZG_INJECT_PINNED_ALLOC) or host-to-device copy
 * (ZG_INJECT_COPY) report a failure after `after` successful ones, once, so
 * the error paths of zg_index_build (status, cleanup of the device image and
 * staging buffers) can be exercised without a real failure.  point 0 disarms.
 * Process-wide; only builds with ZG_RESIDENT_DEVICE stage or copy. */
#define ZG_INJECT_PINNED_ALLOC 1
#define ZG_INJECT_COPY 2
ZG_API void zg_debug_inject_build_failure(int32_t point, int32_t after);

/* Synchronises `stream`, then reports and clears the device status word that
 * kernels set instead of trapping (bit 0: row out of range, bit 1: token out
 * of range, bit 2: a bounded wait in the tensor-core kernel expired, bit 3:
 * tensor-memory allocation failed, bit 4: a select found fewer candidates
 * than its own cut guarantees).  Non-zero -> ZG_ERR_DEVICE_STATUS. */
ZG_API zg_status zg_check_device_status(void* stream);

ZG_API const char* zg_last_error(void);
ZG_API const char* zg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ZEROGR_H */
