/*
 * tria.h - TriAttention KV-cache eviction pass (score -> select -> compact) on
 * one NVIDIA GB300 (sm_103a).
 *
 * Sources, cited by page title and section:
 *   [Worklog] "TriAttention Native C++ Worklog" (TensorRT-Model-Connect).
 *   [Doc]     "TriAttention KV-Cache Eviction (--triattention)" (llama.cpp fork
 *             documentation).
 *
 * What one pass computes, for every segment = (sequence s, KV head g) of one
 * layer with n live rows (rows ascend in token position):
 *   1. score  - for each query head h of g's GQA group and each live row r
 *        raw_h(r) = (1/|D|) sum_{d in D} sum_f Re( qbar_{h,f} e^{i w_f (p_s + d)} conj(k_{r,f}) )
 *                   + sum_f (q_abs_{h,f} - |qbar_{h,f}|) |k_{r,f}|
 *      on the stored RoPE-rotated key k_r (NEOX pairs k_{r,f} = K[r][f] + i K[r][f+hd/2]),
 *      with p_s the absolute decode position ([Worklog] Phase 9: scored on the
 *      stored rotated keys, rotation on the query side only, a norm term on
 *      the keys' magnitudes added; 2026-04-18 section: phases from the
 *      absolute position). Then per query head
 *      z = (raw - mean) / (std + 1e-6) over the n live rows, and the row's
 *      score s(r) = max over the group ([Doc] §5 Phase C).
 *   2. select - with B = budget rows, keep rows [0, sink) and [n - window, n)
 *      and the B - sink - window best of the rest by (s descending, row
 *      ascending) ([Doc] §1 CLI flags, §5 Phase B steps 1-3).
 *   3. compact - move kept row i (ascending) to row i of K, V, the q8_0 scale
 *      planes and pos, in place; set n_live = B ([Doc] §5 Phase B step 4;
 *      [Worklog] exact-gather checks of K and V after compaction).
 *
 * Conventions for every call:
 *   - Pointers marked "device" are CUDA device pointers owned by the caller;
 *     pointers marked "host" are read during the call only.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = legacy default stream) unless stated otherwise. They return the
 *     errors detected on the host. Errors found on the device (bad n_live, bad
 *     keep list, a bounded wait that gave up) are recorded in the workspace
 *     and read with tria_device_status().
 *   - The library keeps no global mutable state; all per-call state lives in
 *     the caller's workspace, which calls must not share while they overlap
 *     on the GPU.
 *   - Nothing here falls back to the CPU: without a usable GPU the calls fail.
 */
#ifndef TRIA_H
#define TRIA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TRIA_VERSION 2
#define TRIA_MAX_SEQS 128      /* sequences per call */
#define TRIA_MAX_HEAD_DIM 256  /* [Doc] §4/§6: head_dim <= 256, freq_count <= 128 */
#define TRIA_MAX_GROUP 8       /* query heads per KV head supported */

typedef enum tria_status {
  TRIA_OK = 0,
  TRIA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, layout overlap */
  TRIA_ERR_UNSUPPORTED = 2,   /* gate: head_dim > 256 or % 32, n_q % n_kv, group > 8, dtype */
  TRIA_ERR_BUDGET = 3,        /* budget rows < sink + window */
  TRIA_ERR_CUDA = 4,          /* a CUDA runtime call failed */
  TRIA_ERR_WORKSPACE = 5,     /* workspace too small or not 256-byte aligned */
  TRIA_ERR_TIMEOUT = 6,       /* device: a bounded wait gave up */
  TRIA_ERR_DEVICE_ARG = 7,    /* device: n_live < 0 or > capacity (sequence skipped) */
  TRIA_ERR_KEEP_LIST = 8,     /* device: keep list not strictly ascending / out of range */
  TRIA_ERR_CAPACITY = 9       /* rows to append do not fit the physical capacity */
} tria_status;

typedef enum tria_dtype {
  TRIA_F32 = 0,
  TRIA_F16 = 1,
  /* q8_0 (ggml Q8_0 values, stored planar): int8 codes [row][head_dim] in the
   * data plane plus fp16 block scales [row][head_dim/32] in the scale plane;
   * value = scale of its 32-wide block x code ([Doc] §4 "--cache-type-k q8_0"). */
  TRIA_Q8_0 = 2
} tria_dtype;

/* Calibration statistics of one model ([Doc] §2 "Calibration file (.tria)":
 * per-layer, per-head RoPE-direction statistics; §5 Phase C: omega and
 * per-head q_mean / q_abs laid out [n_layers x n_heads x freq_count]).
 * All arrays are host memory, copied by tria_load_stats. */
typedef struct tria_stats_desc {
  int32_t n_layers;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;           /* every layer's head_dim unless layer_head_dim is given */
  double rope_theta;          /* w_f = theta^(-2f/rot) when omega is NULL (rot = head_dim - nonrot_dim) */
  const double* omega;        /* [rot/2] optional RoPE angular frequencies */
  const float* q_mean;        /* [n_layers][n_q_heads][rot/2][2] pre-RoPE mean query (re, im) */
  const float* q_abs;         /* [n_layers][n_q_heads][rot/2] mean |q_f|; NULL: no norm term */
  const int32_t* kv_of_q;     /* [n_q_heads] optional query->KV head map ([Worklog] "sampled-head
                                 mapping"); NULL: h / (n_q_heads / n_kv_heads). Each KV head must
                                 get the same number of query heads. */
  const int64_t* offsets;     /* [n_offsets] future query offsets D; NULL: {1, 2, 4, ..., 65536} */
  int32_t n_offsets;
  /* Hybrid models ([Doc] §6 "Hybrid head_dim models": head_dim varies across
   * layers, e.g. 256 / 512; the follow-on it names is a per-layer stats
   * offset table so that the eligible layers score on the GPU):
   * layer_head_dim [n_layers] optional; NULL: every layer has head_dim. When
   * given, head_dim is ignored and q_mean / q_abs (and omega, if given) are
   * packed layer after layer: layer l holds n_q_heads * (layer_head_dim[l] -
   * nonrot_dim) / 2 pairs (omega: (layer_head_dim[l] - nonrot_dim) / 2
   * frequencies). Every entry must be even and > nonrot_dim. Layers whose
   * head_dim fails the gate (> 256, not a multiple of 32, rotary dims not a
   * multiple of 16) are not loaded; passes on them return
   * TRIA_ERR_UNSUPPORTED. */
  const int32_t* layer_head_dim;
  const double* layer_rope_theta;  /* [n_layers] optional per-layer theta; NULL: rope_theta */
  /* Non-rotary (content) dims ([Doc] §4 gate line field nonrot=, §6 "Non-
   * rotary models"; the pages give no formula, the reading here): the last
   * nonrot_dim dims of every head are never rotated and the first
   * rot = head_dim - nonrot_dim are NEOX-rotary, paired (f, f + rot/2), with
   * w_f = theta^(-2f/rot). q_mean / q_abs / omega then hold rot/2 pairs per
   * head (per layer: layer_head_dim[l] - nonrot_dim), and a row's score gains
   *   sum_e q_nonrot[h][e] * K[r][rot + e]
   * (the mean non-rotary query dotted with the key's non-rotary dims: no
   * phase, no offset average, no norm term). 0: every dim is rotary. */
  int32_t nonrot_dim;
  const float* q_nonrot;      /* [n_layers][n_q_heads][nonrot_dim] mean non-rotary query;
                                 NULL: no content term */
} tria_stats_desc;

typedef struct tria_stats tria_stats;  /* opaque, device resident, immutable after load */

/* One layer's cache for all sequences of the call.
 * Rows: sequence s owns n_kv_heads * capacity[s] consecutive rows from row
 * seq_row0[s]; KV head g of it (one segment) starts at row
 * seq_row0[s] + g * capacity[s]. Row r of every plane is at byte offset
 * r * (row bytes of that plane). Row bytes: f32 4*hd, f16 2*hd, q8_0 data hd,
 * q8_0 scales hd/16; pos 4. Segments must not overlap. */
typedef struct tria_layer_cache {
  int32_t n_seqs;             /* 1 .. TRIA_MAX_SEQS */
  int32_t n_kv_heads;
  int32_t head_dim;
  tria_dtype k_type;          /* F32, F16 or Q8_0 */
  tria_dtype v_type;          /* F32, F16 or Q8_0 */
  void* k;                    /* device, 16-byte aligned, rotated keys */
  void* k_scale;              /* device, q8_0 keys only (else NULL) */
  void* v;                    /* device, 16-byte aligned */
  void* v_scale;              /* device, q8_0 values only (else NULL) */
  int32_t* pos;               /* device [rows] absolute token positions (moved with the rows) */
  int32_t* n_live;            /* device [n_seqs] live rows per sequence (all its KV heads);
                                 read at the start, set to the budget by compaction */
  const int64_t* seq_row0;    /* host [n_seqs] */
  const int32_t* capacity;    /* host [n_seqs] physical rows per segment */
} tria_layer_cache;

/* Eviction policy ([Doc] §1 CLI flags: --tri-budget N % of n_ctx, --tri-window
 * (default 512), --tri-interval (default 128), --tri-sink (default 0);
 * [Worklog] absolute decode position). Host arrays, read during the call. */
typedef struct tria_policy {
  double budget_frac;         /* (0, 1]: budget rows B_s = floor(budget_frac * n_ctx[s]) */
  const int32_t* n_ctx;       /* [n_seqs] context length the fraction refers to */
  const int32_t* budget_rows; /* [n_seqs] optional absolute budget; overrides the fraction */
  int32_t window;             /* most recent rows always kept */
  int32_t sink;               /* first rows always kept */
  int32_t interval;           /* decode steps between passes (used by tria_should_evict) */
  const int64_t* cur_pos;     /* [n_seqs] absolute decode position p_s (not the row count) */
  const int32_t* sink_rows;   /* [n_seqs] optional per-sequence sink (e.g. the prompt rows
                                 that a schedule protects); overrides `sink` when not NULL */
} tria_policy;

/* Host-only gate of [Doc] §4 "GPU scoring requirements" (n_q % n_kv == 0,
 * head_dim <= 256 and % 32 == 0) plus this library's limit of group <= 8. The page's gate
 * also wants no non-rotary dims ([Doc] §6 "Non-rotary models" are scored on the
 * CPU there); here heads with nonrot_dim non-rotary dims are eligible when the
 * rotary dims head_dim - nonrot_dim are a multiple of 16 (UNSUPPORTED
 * otherwise). nonrot_dim < 0 or >= head_dim: INVALID_ARG. No GPU use. */
tria_status tria_gate_check(int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t nonrot_dim);

/* The gate as one log line, in the form of the [Doc] §4 startup log
 * ("tria: gpu gate - is_q8_0=1 nh=32 nkv=8 hd=128 nonrot=0 -> eligible"), with
 * the reason appended when ineligible; written to buf (NUL-terminated,
 * truncated to buf_size). Returns tria_gate_check's status. No GPU use. */
tria_status tria_gate_describe(int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t nonrot_dim,
                               tria_dtype k_type, char* buf, size_t buf_size);

/* Budget rows floor(budget_frac * n_ctx) computed in double ([Doc] §1). */
int64_t tria_budget_rows(double budget_frac, int64_t n_ctx);

/* Decode-loop trigger: 1 when n_live >= budget + interval ([Worklog] "Final
 * apples-to-apples check": compaction starts at kv_budget + divide_length). */
int32_t tria_should_evict(int64_t n_live, int64_t budget, int64_t interval);

/* Copies the statistics to the device (allocates with cudaMalloc), folds the
 * offset average and the norm weights (q_abs - |q_mean|) in a kernel, and
 * synchronises `stream`. *out is NULL on error. */
tria_status tria_load_stats(const tria_stats_desc* desc, tria_stats** out, void* stream);
void tria_free_stats(tria_stats* stats);

/* Workspace bytes for calls on `cache` with `group` query heads per KV head
 * (0 when only tria_select / tria_compact are used). 0 on invalid input. */
size_t tria_workspace_size(const tria_layer_cache* cache, int32_t group);

/* Zeroes a workspace (required once after allocation and after any device
 * error). Asynchronous. */
tria_status tria_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Step 1 only: writes s(r) to score_out[row] (device float, global row index)
 * and, if raw_out is not NULL, raw_h(r) to raw_out[row * G + j] for the j-th
 * query head of the segment's group (ascending head index). Rows at or past
 * n_live are not written. The cache is not modified. */
tria_status tria_score(const tria_stats* stats, int32_t layer, const tria_layer_cache* cache,
                       const tria_policy* policy, float* score_out, float* raw_out,
                       void* ws, size_t ws_bytes, void* stream);

/* Step 2 only, on a caller-given score array (device float, global row
 * index). Writes each segment's kept rows (segment-local indices, ascending)
 * to keep_out[seg_row0 + i] (device int32): B entries when n_live > B, else
 * the n_live identity entries. The cache is not modified. */
tria_status tria_select(const float* score, const tria_layer_cache* cache, const tria_policy* policy,
                        int32_t* keep_out, void* ws, size_t ws_bytes, void* stream);

/* tria_select without a workspace argument. The paper has no counterpart to
 * this entry point: it exists for callers that cannot allocate device memory
 * where they select (an allocator-free decode step, a runtime that owns every
 * allocation and forbids cudaMalloc after start-up). It allocates nothing and
 * calls no allocating routine; its scratch is a fixed 4 MiB array compiled
 * into the library, which every GPU that loads the library holds until the
 * process exits. Same inputs, outputs and results as tria_select.
 *  - Limit: control words + per-segment state and 8 KiB histogram + 20 bytes
 *    per 32-row chunk of the largest capacity, for all n_seqs * n_kv_heads
 *    segments, must fit in 4 MiB (e.g. 32 segments of 131072 rows do);
 *    larger calls return TRIA_ERR_WORKSPACE.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture. The address belongs to the CUDA context it
 *    was looked up in: a call made in another context of the device (for
 *    instance after cudaDeviceReset, which replaces the primary context)
 *    looks it up again, so after a reset the next call must also be made
 *    outside stream capture.
 *  - Host checks are those of tria_select (the cache layout, including
 *    sequences whose rows overlap, pointer alignment, budget / sink / window
 *    and n_ctx of every sequence).
 *  - All calls share the one array, which keeps the previous call's contents;
 *    each call clears what must start at zero. Calls that overlap on the GPU
 *    (different streams, no ordering) race and give undefined results.
 *  - Device-detected errors are not reported (only host-side checks return
 *    an error). Asynchronous on `stream`. */
tria_status tria_select_noalloc(const float* score, const tria_layer_cache* cache, const tria_policy* policy,
                                int32_t* keep_out, void* stream);

/* Step 3 only: compacts every segment with n_live > B using the caller's
 * keep list (as tria_select writes it: B strictly ascending entries in
 * [0, n_live) per segment), then sets n_live = B. Rows at or past B keep their
 * old contents. A keep list that breaks the rules is reported as
 * TRIA_ERR_KEEP_LIST and nothing is moved. */
tria_status tria_compact(const tria_layer_cache* cache, const tria_policy* policy,
                         const int32_t* keep, void* ws, size_t ws_bytes, void* stream);

/* The whole pass (steps 1-3) for one layer and all sequences of the call.
 * Calls with fp16 or q8_0 keys, head_dim 64 or 128 (any group) or 256
 * (group <= 4) and every dim rotary (statistics with nonrot_dim 0) run as one
 * fused persistent kernel (see tria_evict_model) when they have at least 128
 * segments (n_seqs x n_kv_heads), or at least 32 with no capacity above 65536
 * rows; the others run the three staged kernels of tria_evict_staged. Same
 * results either way. */
tria_status tria_evict(const tria_stats* stats, int32_t layer, const tria_layer_cache* cache,
                       const tria_policy* policy, void* ws, size_t ws_bytes, void* stream);

/* tria_evict as three kernels in sequence (score; select with the z-max
 * score; compaction), whatever the shape. */
tria_status tria_evict_staged(const tria_stats* stats, int32_t layer, const tria_layer_cache* cache,
                              const tria_policy* policy, void* ws, size_t ws_bytes, void* stream);

/* Byte offset, in a workspace laid out for `cache` (tria_workspace_size), of
 * the float array [rows] where the staged evict path keeps the z-max score it
 * selected with ([Doc] §5 Phase C): after tria_evict_staged, element r holds
 * s(r) for every live row r (before compaction) of each segment above its
 * budget; other rows are not written. The fused kernel keeps its scores
 * elsewhere (tria_evict_model's score_out). 0 on invalid input. No GPU use. */
size_t tria_workspace_score_offset(const tria_layer_cache* cache);

/* Workspace bytes for tria_evict_model over n_layers layers of caches shaped
 * like `cache` (also enough for every single-layer call on one of them). 0 on
 * invalid input (n_layers outside 1 .. 128). */
size_t tria_model_workspace_size(const tria_layer_cache* cache, int32_t n_layers, int32_t group);

/* The pass over several layers of a model in one call ([Doc] §5 Phase B: the
 * pass runs per layer and KV head; layers only change the statistics and the
 * cache planes). caches[i] (host array of n_layers structs) is the cache of
 * layer layers[i] (host int32 [n_layers]): the same sequences (n_seqs,
 * seq_row0, capacity), n_kv_heads, head_dim and dtypes in every layer, each
 * with its own planes and its own n_live array (device, updated in place).
 * Every layer must be loaded with the first layer's RoPE frequencies
 * (TRIA_ERR_UNSUPPORTED otherwise) and appear once. One policy for all
 * layers. Shapes of the fused kernel (see tria_evict) with up to 2048
 * segments (n_layers x n_seqs x n_kv_heads; at least 128, or 32 with no
 * capacity above 65536 rows, or any count from 1 when score_out is given)
 * run as ONE persistent kernel for all layers: every warp streams a
 * run of the keys, each scored segment is selected by one CTA as soon as its
 * warps finish, and the rows move once segments are selected; other calls run
 * tria_evict_staged per layer.
 * score_out (device float, optional): the z-max score s(r) of every live row
 * of every compacted segment, at score_out[i * layer_rows + row] for layer
 * i of the call (layer_rows = max over s of seq_row0[s] + n_kv_heads *
 * capacity[s]); rows of segments at or below budget are not written. Only
 * with the fused kernel (else TRIA_ERR_UNSUPPORTED). ws: at least
 * tria_model_workspace_size(caches, n_layers, group) bytes. */
tria_status tria_evict_model(const tria_stats* stats, const int32_t* layers, int32_t n_layers,
                             const tria_layer_cache* caches, const tria_policy* policy, float* score_out,
                             void* ws, size_t ws_bytes, void* stream);

/* Which kernels tria_evict_model runs for these arguments without score_out:
 * 1 = the fused kernel (one launch for all layers), 0 = tria_evict_staged per
 * layer (three launches each), -1 = arguments that tria_evict_model rejects.
 * Same arguments and meaning as there. Host only: reads the stats handle's
 * host metadata and the caches' host arrays, launches nothing, needs no GPU
 * work (a stats handle still comes from tria_load_stats). */
int32_t tria_evict_model_fused(const tria_stats* stats, const int32_t* layers, int32_t n_layers,
                               const tria_layer_cache* caches);

/* tria_evict over sequences of different layers in one call (the pass is
 * per segment, so layers only change which statistics a segment uses): the
 * caller lays several layers' caches out as the sequences of one
 * tria_layer_cache (for instance one allocation per plane, a layer's rows
 * after the previous layer's) and sequence s is scored with the statistics of
 * layer layer_of_seq[s] (host int32 [n_seqs]). All those layers must be loaded,
 * have the cache's head_dim and the same RoPE frequencies (else
 * TRIA_ERR_UNSUPPORTED). The fixed costs of a pass (launches, ramps) are paid
 * once for all of them. */
tria_status tria_evict_layers(const tria_stats* stats, const int32_t* layer_of_seq, const tria_layer_cache* cache,
                              const tria_policy* policy, void* ws, size_t ws_bytes, void* stream);

/* tria_evict with CUDA events recorded on `stream` between its stages;
 * synchronises `stream` and writes the stage times in milliseconds to
 * stage_ms[5] = {raw scores, z-max scores (0: computed inside select), select,
 * compact, whole pass} and the
 * number of kernels launched to *launches. For benchmarks and tracing. */
tria_status tria_evict_profiled(const tria_stats* stats, int32_t layer, const tria_layer_cache* cache,
                                const tria_policy* policy, void* ws, size_t ws_bytes, void* stream,
                                float* stage_ms, int32_t* launches);

/* tria_evict with the caller's CUDA events (events[4], cudaEvent_t passed as
 * void*) recorded on `stream` before the scoring kernel, between the kernels
 * and after the compaction kernel: {start, scored, selected, compacted}.
 * Does not synchronise, so it can be captured in a CUDA graph; read the
 * stage times with cudaEventElapsedTime once the stream has reached
 * events[3]. For benchmarks and tracing. */
tria_status tria_evict_marked(const tria_stats* stats, int32_t layer, const tria_layer_cache* cache,
                              const tria_policy* policy, void* ws, size_t ws_bytes, void* stream,
                              void* const* events);

/* Synchronises `stream`, returns the first device-detected error of the
 * calls since the last check (TRIA_OK if none) and clears it. After
 * TRIA_ERR_TIMEOUT a call may have stopped with its counters mid-way and its
 * cache rows part moved (their contents are then unspecified): re-initialise
 * the workspace (tria_workspace_init) before the next call. */
tria_status tria_device_status(void* ws, void* stream);

/* Runs the bounded wait used by the compaction kernel on a flag that nothing
 * sets, with `spin_limit` polls, and returns what the kernel reported
 * (TRIA_ERR_TIMEOUT expected). Synchronises `stream`. For failure tests. */
tria_status tria_selftest_bounded_wait(int32_t spin_limit, void* ws, size_t ws_bytes, void* stream);

/* ---- Shared-slot variant -----------------------------------------------
 * For caches whose token cells are shared by every layer (llama.cpp cells):
 * one keep-set per token for all layers and KV heads ([Doc] §5 Phase B/C:
 * per-query-head z-normalisation and max across the GQA group; the Vulkan
 * port's global z-normalisation shader; [Worklog] cross-layer aggregation).
 * The pages do not state the combine rule. Reading taken: a token's score is
 * the maximum of its z-max scores (tria_score, one per layer and KV head)
 * over all layers and KV heads; NaN scores are ignored unless all are NaN.
 * A pass over L layers whose caches share one layout:
 *   tria_score(stats, l, cache_l, ..., scores + l * layer_stride, NULL, ...)  for every l
 *   tria_shared_combine(scores, layer_stride, L, cache_0, combined, ...)
 *   tria_shared_select(combined, cache_0, policy, keep, ...)
 *   tria_compact(cache_l, policy, keep, ...)                                  for every l
 * Each layer's tria_layer_cache keeps its own n_live array (equal values):
 * tria_compact sets it for that layer only.
 *
 * tria_shared_combine: scores device float [n_layers][layer_stride] (row
 * index of the cache layout, layer_stride >= the layout's rows); writes
 * combined[seq_row0[s] + t] for t < n_live[s] (the KV-head-0 slot of every
 * sequence); other entries are not written. ws: a workspace of this cache
 * (its control words report a bad n_live, TRIA_ERR_DEVICE_ARG). */
tria_status tria_shared_combine(const float* scores, int64_t layer_stride, int32_t n_layers,
                                const tria_layer_cache* cache, float* combined, void* ws, size_t ws_bytes,
                                void* stream);

/* tria_shared_select: selects on the combined scores of every sequence (the
 * rules of tria_select, one segment per sequence) and writes the keep list to
 * keep_out[seq_row0[s] + g * capacity[s] + i] for every KV head g, i.e. the
 * same list in every segment of the sequence, as tria_compact reads it. */
tria_status tria_shared_select(const float* combined, const tria_layer_cache* cache, const tria_policy* policy,
                               int32_t* keep_out, void* ws, size_t ws_bytes, void* stream);

/* ---- Decode-loop lifecycle ---------------------------------------------
 * A decode loop appends rows to each sequence and runs a pass when its
 * schedule says so. Sources, [Worklog] sections: "Why this is still fair even
 * though the TriAttention bundle is tri12288" (compaction starts once the
 * cache length reaches kv_budget + divide_length), "Sample9 compaction was
 * then proven live" (passes at positions 3200, 3328, 3456, ... each taking
 * 3200 rows to 3072), "Same-prompt boundary runs localized the divergence to
 * the first compaction" (158-token prompt, first pass at absolute position
 * 7168 keeping 6144), "Sample9 boundary replay exposed a prompt-token
 * accounting mismatch" and "Aligned sample9 replay" (prompt rows need not
 * count toward the cache length), "Phase 6: overflow bug during prompt
 * prefill" and "4. Separate physical cache limit from logical TriAttention
 * budget" (no compaction during prefill; physical capacity apart from the
 * logical budget); [Doc] §1 CLI flags (--tri-interval, --tri-budget,
 * --tri-sink, --tri-window) and §5 Phase B (the evictor fires only on
 * single-token decode steps).
 *
 * tria_append writes n_tokens new rows after the live rows of every segment
 * and adds n_tokens to n_live, on the device, so that a loop never has to read
 * n_live back.
 *   k_new        device, rows of k_type laid out [n_seqs][n_kv_heads][n_tokens]
 *                (row bytes as in the cache), 16-byte aligned
 *   k_scale_new  device, q8_0 keys only (else NULL): scale rows, same layout,
 *                2-byte aligned
 *   v_new, v_scale_new  likewise for the values
 *   pos_new      device int32 [n_seqs][n_tokens]: absolute positions, written
 *                to the new row of every KV head
 *   ws           a workspace of this cache (only its control words are used)
 * Host errors: TRIA_ERR_INVALID_ARG (null or misaligned pointer, n_tokens < 0,
 * a scale plane given for a non-q8_0 type or missing for q8_0),
 * TRIA_ERR_WORKSPACE. Device errors (tria_device_status): TRIA_ERR_DEVICE_ARG
 * when n_live is outside [0, capacity], TRIA_ERR_CAPACITY when n_live +
 * n_tokens > capacity; that sequence is left unchanged. n_tokens = 0 does
 * nothing. */
tria_status tria_append(const tria_layer_cache* cache, const void* k_new, const void* k_scale_new,
                        const void* v_new, const void* v_scale_new, const int32_t* pos_new,
                        int32_t n_tokens, void* ws, size_t ws_bytes, void* stream);

/* When a pass runs and what it keeps. Host only; no GPU use. */
typedef enum tria_trigger {
  /* [Worklog]: a pass once the counted rows reach kv_budget + divide_length;
   * it keeps kv_budget counted rows */
  TRIA_TRIGGER_LENGTH = 0,
  /* [Doc] §1: a pass every divide_length decode steps (--tri-interval); it
   * keeps floor(budget_frac * n_ctx) counted rows (--tri-budget) */
  TRIA_TRIGGER_INTERVAL = 1
} tria_trigger;

typedef struct tria_schedule {
  int32_t trigger;             /* tria_trigger */
  int32_t count_prompt_tokens; /* 1: prompt rows count toward the trigger and the budget;
                                  0: only rows appended by decode steps count */
  int32_t protect_prefill;     /* 1: prompt rows are never evicted (they join the sink) */
  int32_t sink;                /* first rows always kept */
  int32_t window;              /* most recent rows always kept */
  int32_t pad;
  int64_t kv_budget;           /* LENGTH: counted rows a pass keeps (>= 1) */
  int64_t divide_length;       /* LENGTH: counted rows between passes; INTERVAL: decode
                                  steps between passes (>= 1) */
  double budget_frac;          /* INTERVAL: (0, 1] */
  int64_t n_ctx;               /* INTERVAL: context length the fraction refers to */
} tria_schedule;

/* One sequence's place in the loop. Owned by the caller; changed only by the
 * calls below. */
typedef struct tria_seq_state {
  int64_t capacity;      /* physical rows per segment */
  int64_t rows;          /* live rows: the host's copy of n_live */
  int64_t counted;       /* live rows that count toward the budget */
  int64_t prompt_rows;   /* rows appended by the prompt (prefill) */
  int64_t next_pos;      /* absolute position of the next token = tokens appended so far */
  int64_t decode_steps;  /* single-token steps since the prompt */
  int64_t passes;        /* passes run */
  int32_t due;           /* 1: a pass must run before the next append */
  int32_t pad;
} tria_seq_state;

#define TRIA_NO_PASS INT32_MAX  /* budget of a sequence whose pass is not due */

/* Checks a schedule: TRIA_ERR_INVALID_ARG for a bad trigger, a flag other
 * than 0 / 1, a negative sink or window, divide_length < 1, kv_budget < 1
 * (LENGTH) or budget_frac outside (0, 1] or n_ctx < 0 (INTERVAL). */
tria_status tria_schedule_check(const tria_schedule* sch);

/* Empty sequence with `capacity` physical rows per segment. */
tria_status tria_seq_init(tria_seq_state* st, int64_t capacity);

/* The prompt: n_tokens rows appended before the first decode step (never
 * makes a pass due). TRIA_ERR_CAPACITY when they do not fit (the state is
 * unchanged: the prompt is not compacted while it is being built);
 * TRIA_ERR_INVALID_ARG after the first decode step or for n_tokens < 0. */
tria_status tria_seq_prefill(const tria_schedule* sch, tria_seq_state* st, int64_t n_tokens);

/* One decode step: one row appended; sets st->due by the trigger.
 * TRIA_ERR_INVALID_ARG while a pass is still due; TRIA_ERR_CAPACITY when the
 * row does not fit (state unchanged). */
tria_status tria_seq_decode(const tria_schedule* sch, tria_seq_state* st);

/* The policy values of the next pass over n_seqs sequences: budget_rows[s]
 * (TRIA_NO_PASS when s is not due), sink_rows[s] and cur_pos[s] = next_pos
 * (the absolute position, [Worklog] "2026-04-18: later-compaction
 * absolute-position bug isolated and fixed"), ready for tria_policy's
 * budget_rows / sink_rows / cur_pos; *n_due = sequences due. A due sequence
 * keeps B = (counted budget) + (prompt rows outside the count, when
 * protected) rows, with sink = max(sink, prompt rows) when protected.
 * TRIA_ERR_BUDGET when B < sink + window for a due sequence. */
tria_status tria_schedule_plan(const tria_schedule* sch, const tria_seq_state* st, int32_t n_seqs,
                               int32_t* budget_rows, int32_t* sink_rows, int64_t* cur_pos, int32_t* n_due);

/* Records that the planned pass ran: rows = min(rows, B) and the counts of
 * every due sequence, clears due. */
tria_status tria_schedule_passed(const tria_schedule* sch, tria_seq_state* st, int32_t n_seqs);

/* ---- Calibration statistics --------------------------------------------
 * The scoring statistics of one layer from a stream of its pre-RoPE queries
 * ([Doc] §2 Calibration file: statistics per layer and head, gathered over
 * calibration text from the pre-RoPE Q of every layer;
 * §5 Phase C: q_mean / q_abs arrays laid out [layers][heads][frequency
 * pairs]). With rot = head_dim - nonrot_dim rotary dims and NEOX pairs
 * z = q[f] + i q[f + rot/2] (f < rot/2):
 *   q_mean[h][f]   = mean over tokens of z   (stored as re, im)
 *   q_abs[h][f]    = mean over tokens of |z|
 *   q_nonrot[h][e] = mean over tokens of q[rot + e]   (e < nonrot_dim; the
 *                    content term of tria_stats_desc)
 * Feed batches with tria_calib_accumulate, then tria_calib_finish; both take
 * the same nonrot_dim (even, in [0, head_dim); else TRIA_ERR_INVALID_ARG).
 *
 * tria_calib_accumulate:
 *   q      device, [n_tokens][n_q_heads][head_dim] values of q_type (TRIA_F32
 *          or TRIA_F16), row-major, 4-byte aligned; read only.
 *   acc    device, double [n_q_heads][head_dim/2][3] running sums (re, im,
 *          modulus) of the rot/2 rotary pairs, then of nonrot_dim/2 content
 *          pairs (q[rot + e], q[rot + nonrot_dim/2 + e]), owned by the
 *          caller and zeroed before the first batch;
 *          the batch's sums are added to it (fp32 within a block of tokens,
 *          fp64 across blocks; the order of the fp64 additions is not fixed,
 *          so repeated runs may differ in the last bits of acc).
 *   Errors: TRIA_ERR_INVALID_ARG (null acc, null q with n_tokens > 0,
 *   n_tokens < 0, n_q_heads < 1, misalignment), TRIA_ERR_UNSUPPORTED (q_type
 *   other than f32 / f16, head_dim odd, below 2 or above 512). n_tokens = 0
 *   adds nothing (q may then be null).
 * tria_calib_finish:
 *   acc       as above; n_tokens = tokens accumulated (> 0).
 *   q_mean    device float [n_q_heads][rot/2][2]; q_abs device float
 *             [n_q_heads][rot/2]; q_nonrot device float
 *             [n_q_heads][nonrot_dim] (may be NULL when nonrot_dim is 0): one
 *             layer's rows of the tria_stats_desc arrays. Errors as above. */
tria_status tria_calib_accumulate(const void* q, tria_dtype q_type, int32_t n_tokens, int32_t n_q_heads,
                                  int32_t head_dim, int32_t nonrot_dim, double* acc, void* stream);
tria_status tria_calib_finish(const double* acc, int64_t n_tokens, int32_t n_q_heads, int32_t head_dim,
                              int32_t nonrot_dim, float* q_mean, float* q_abs, float* q_nonrot, void* stream);

const char* tria_status_string(tria_status status);
int32_t tria_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TRIA_H */
