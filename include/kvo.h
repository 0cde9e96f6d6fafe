/*
 * kvo.h -- C ABI of the GB300-native sparse-decode KV offload hot path.
 *
 * The operation follows two web pages:
 *  [LS] "Layerwise and Sparse KV Cache Offloading Design", section 4 "Sparse
 *       Decode Offload": "Memory layout" (full main KV in a pinned host pool;
 *       indexer cache and per-layer hot K/V buffers in device memory) and
 *       "Decode step" (steps 1-6: new-token rows to their logical host slots,
 *       indexer top-k, LRU residency table, miss-row copy host -> device,
 *       logical -> physical remap).  Section 2 "Transfer granularity": token
 *       rows device -> host, top-k miss rows host -> device.
 *  [FO] "FlashOffloading offloads all KV cache ... What does it mean?", the
 *       decode paragraphs: fixed-size hot shelf, MTP3 per-position miss lists
 *       merged and deduplicated, the cache_slots reverse index (-1 when
 *       absent), token index and slot packed into one int32 before selection.
 *
 * Units.  A unit is one (request r, layer l) pair, u = r * n_layers + l.
 * Every unit owns: a host row pool [max_tokens][row_elems] bf16 (pinned,
 * mapped), an indexer cache [max_tokens][128] bf16 and a hot buffer
 * [hot_capacity][row_elems] bf16 in device memory, cache_slots[max_tokens]
 * (token -> hot slot, -1 absent), slot_token[hot_capacity] (slot -> token,
 * -1 free), last_use[hot_capacity] (stamp of the last step that used the
 * slot) and a step stamp.  Units never interact.
 *
 * Semantics fixed by this library where the pages are silent (the CPU oracle
 * shipped with the tests states the same rules):
 *  - score: single-head fp32 dot product of bf16 query and key, summed as 16
 *    FMA chains over d = 8j..8j+7 followed by the tree c_j += c_{j+w},
 *    w = 8, 4, 2, 1; zero returned as +0.
 *  - selection order: score descending, then token ascending; outputs keep
 *    that order.  Position p (of P) sees tokens t < len - (P - 1 - p).
 *  - payload: cache_slots[t] when >= 0 (hit: the slot), else -(t + 1)
 *    (miss: the token); read before the step's update.  Padding entries (a
 *    position sees fewer than k tokens): token -1, score -inf, payload
 *    KVO_PAD_PAYLOAD, slot -1.
 *  - merge: the step's wanted set W is the distinct tokens of all P lists;
 *    misses are filled in token order.
 *  - LRU: the unit's stamp grows by one per successful step; victims are the
 *    slots not holding a token of W, in (last_use asc, slot asc) order
 *    (free slots have last_use 0); every slot of W gets last_use = stamp.
 *  - capacity: |W| > hot_capacity -> unit status KVO_ECAPACITY, the unit's
 *    state and hot rows stay unchanged, its slots are -1.
 *
 * Conventions.  Every call returns 0 (KVO_OK) or a negative KVO_E* code;
 * kvo_last_error() gives a thread-local message.  kvo_append and kvo_step
 * are asynchronous on the caller's CUDA stream (a cudaStream_t passed as
 * void*, NULL = legacy default stream) and never synchronise the device;
 * they return only argument and launch errors.  Per-unit results go to the
 * device array unit_status.  The caller owns queries, inputs, outputs and
 * the stream; the library owns the host pool, the indexer cache, the hot
 * buffers and the residency metadata.  A handle is not thread-safe, and calls
 * on one handle must be ordered (same stream, or synchronised by the caller).
 * Device pointers are plain CUDA device addresses (any allocator).
 */
#ifndef KVO_H
#define KVO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVO_OK 0
#define KVO_EINVAL (-1)    /* bad argument or configuration */
#define KVO_ENOMEM (-2)    /* host or device allocation failed */
#define KVO_ERANGE (-3)    /* append past max_tokens, unit index out of range */
#define KVO_ECUDA (-4)     /* CUDA runtime error (no device, launch failure) */
#define KVO_ETIMEOUT (-5)  /* a bounded device-side wait expired (unit status) */
#define KVO_ECAPACITY (-6) /* |W| > hot_capacity (unit status only) */

#define KVO_PAD_PAYLOAD INT32_MIN

typedef struct kvo_handle kvo_handle;

typedef struct kvo_config {
  int32_t n_requests;   /* >= 1 */
  int32_t n_layers;     /* >= 1; units = n_requests * n_layers */
  int64_t max_tokens;   /* cached tokens per unit, upper bound, >= 1, < 2^31 */
  int32_t idx_dim;      /* indexer dimension: must be 128 */
  int32_t row_elems;    /* bf16 elements of one main-KV row (576 for MLA), multiple of 8 */
  int32_t topk;         /* k, 1..4096, <= hot_capacity */
  int32_t hot_capacity; /* hot slots per unit, 1..2^24 */
  int32_t n_positions;  /* P query positions per step, 1..8 (4 = MTP3) */
  int32_t device;       /* CUDA device ordinal */
  int32_t idx_dtype;    /* KVO_IDX_BF16 (0) or KVO_IDX_INT8 (1): indexer cache format */
  int32_t host_block_tokens; /* 0: each unit owns rows 0..max_tokens-1 of the host pool.  > 0
                                (a multiple of 8): the pool is host_blocks blocks of this many
                                rows, shared by all units through per-unit block tables
                                (kvo_set_blocks; "SFA Remote D2H Connector Design",
                                "Data Ownership": main-KV block IDs) */
  int64_t host_blocks;       /* blocks of a paged pool (0: enough for every unit's max_tokens) */
} kvo_config;

/* Indexer cache formats ("FlashOffloading ... What does it mean?", LIM C8
 * paragraph).  BF16: keys stored as given, canonical fp32 score.  INT8: each
 * key (at prefill/append) and each query (at kvo_step) is rotated by the
 * 128-point Walsh-Hadamard transform and quantized to int8 codes with one
 * fp16 scale per vector; the score is the exact int32 dot product of the
 * codes times both scales / 128 (half the key bytes of BF16).  Inputs are
 * bf16 in both formats. */
#define KVO_IDX_BF16 0
#define KVO_IDX_INT8 1

typedef struct kvo_stats {
  uint64_t steps;           /* kvo_step calls */
  uint64_t unit_steps;      /* unit steps that ended KVO_OK */
  uint64_t capacity_errors; /* unit steps that ended KVO_ECAPACITY */
  uint64_t hits;            /* distinct selected tokens already resident */
  uint64_t misses;          /* distinct selected tokens filled from host */
  uint64_t rows_h2d;        /* rows copied host pool -> hot buffer (counted by the copy kernel) */
  uint64_t bytes_h2d;
  uint64_t rows_d2h;        /* rows appended device -> host pool (counted by the copy kernel) */
  uint64_t bytes_d2h;
  uint64_t timeouts;        /* bounded device waits that expired */
  uint64_t rescored;        /* units rescored because a speculative threshold was too high */
  uint64_t fused_steps;     /* kvo_step calls that ran as one fused launch (KVO_OPT_FUSED) */
  uint64_t block_errors;    /* paged pool: rows of unmapped blocks skipped by append or gather */
  uint64_t fetch_dup_bytes; /* deferred fill: host-pool bytes the attention kernel read for a row
                               part another CTA of the same call was still writing (read twice) */
  uint64_t split_steps;     /* staged kvo_step calls in unit groups whose row copies ran inside
                               the next group's score launch (KVO_OPT_GROUP_GATHER_SMS) */
  uint64_t launches;        /* kernels launched by kvo_append, kvo_step, kvo_reset and kvo_attend */
  uint64_t rows_h2d_in_score; /* of rows_h2d: rows copied by the first CTAs of a score launch
                                 (KVO_OPT_GROUP_GATHER_SMS) */
} kvo_stats;

/* Options for kvo_set_option. */
#define KVO_OPT_GATHER_MODE 1 /* value: KVO_GATHER_LDG (default) | KVO_GATHER_BULK */
#define KVO_OPT_WAIT_LIMIT_NS 2 /* bound of every device-side wait, ns (default 2e9) */
#define KVO_OPT_PROFILE 3       /* 1: bracket every launch with CUDA events (kvo_profile_read) */
#define KVO_OPT_GROUPS 4        /* 1..16 unit groups per kvo_step: the miss-row copy of group g runs
                                   on a library stream while group g+1 is scored (default 1) */
#define KVO_OPT_SCORE_CTAS 5    /* upper bound on scoring CTAs per launch, 0 = one per SM */
#define KVO_OPT_SPECULATE 6     /* 0: off; v in 1..1000: each (unit, position) starts its scan
                                   with threshold (previous step's k-th score) x (query norm
                                   ratio) x v/1000, and a unit whose candidates fall short is
                                   rescored exactly in the same call (default 900) */
#define KVO_OPT_FUSED 7         /* 1: kvo_step is one cooperative launch that overlaps the scoring of
                                   some units with the select, residency and miss-row fill of
                                   others; 0: one launch per stage; 2 (default): per call, the
                                   fused launch when the configuration fits its layout,
                                   hot_capacity <= 65536, the pinned pool is at most 16 GiB
                                   (the staged gather's fixed unit-to-CTA order reads a larger
                                   pool faster) and the miss rows of the previous step
                                   amount to at least 1.5% of the indexer key bytes (the staged
                                   step wins when few rows move or the LRU lists are long), else
                                   the staged one; that staged step runs in two unit groups, the
                                   first group's rows copied by some CTAs of the second group's
                                   score launch (KVO_OPT_GROUP_GATHER_SMS, default 4/25 of the
                                   SMs), when those rows amount to at least 1.5% of the key
                                   bytes, the call lists at least 64 units and KVO_OPT_GROUPS has
                                   not been set.  All give identical results.  When the
                                   configuration does not fit the fused layout the default is 0
                                   and setting 1 or 2 returns KVO_EINVAL.  The fused step moves
                                   miss rows with bulk async copies and ignores
                                   KVO_OPT_GATHER_MODE, GROUPS and SCORE_CTAS. */
#define KVO_OPT_GATHER_CTAS 8   /* fused step: CTAs that only fill miss rows, 0 .. SMs-1 (default 8);
                                   the others score and join the fill when no piece is left */
#define KVO_OPT_PIECE_TOKENS 9  /* fused step: tokens per scoring piece, a multiple of 128 in
                                   [128, 2^20] (default 4096); resizes scratch, synchronous */
#define KVO_OPT_HOST_HUGE_PAGE 10 /* read only (kvo_get_option): page size of transparent huge
                                     pages backing the pinned host pool; always 0 (the pool is
                                     driver-allocated pinned memory, cudaHostAlloc) */
#define KVO_OPT_DEFER_FILL 11   /* 1: kvo_step assigns the miss rows' hot slots but leaves the rows
                                   to the next kvo_attend on the same unit list, which reads them
                                   from the pinned pool inside the attention kernel and writes them
                                   to their slots (the Copy-SFA operator of "Layerwise and Sparse KV
                                   Cache Offloading Design", Chinese edition: misses fetched inside
                                   sparse attention).  Any other call that needs the hot rows first
                                   (kvo_step, kvo_reset, kvo_export_state, kvo_attend on another unit
                                   list) completes the fill with a copy kernel on its stream.
                                   Requires row_elems == 576; the first 1 allocates 12 bytes per
                                   hot slot of claim words (synchronous).  Default 0 */
#define KVO_OPT_GROUP_GATHER_SMS 12 /* staged step in unit groups: 0 copies each group's miss rows
                                   on a library stream beside the next group's scoring; s in
                                   1 .. SMs/2 makes the first s CTAs of group g+1's score launch
                                   (one per SM) copy group g's rows while the others score and
                                   then take the copy batches not yet claimed, all on the
                                   caller's stream (the last group's rows use every SM after its
                                   residency update).  Default 0 with KVO_OPT_GROUPS set by the
                                   caller; the two-group step that KVO_OPT_FUSED = 2 chooses uses
                                   4/25 of the SMs unless this option was set (kvo_get_option
                                   returns the value set, 0 if none) */
#define KVO_OPT_PROFILE_KINDS 13 /* with KVO_OPT_PROFILE 1: bit (1 << KVO_PROF_x) set brackets the
                                   launches of kind x with events (default every kind); each
                                   pair of events adds a few microseconds between launches */
#define KVO_GATHER_LDG 0  /* miss rows read by 16-byte loads from the mapped host pool */
#define KVO_GATHER_BULK 1 /* miss rows moved by bulk async copies through shared memory */

/*
 * kvo_create: allocate one handle ([LS] "Memory layout").  cfg is read, not
 * kept.  Allocates the pinned mapped host pool (units * max_tokens *
 * row_elems * 2 bytes), the device indexer cache, hot buffers, metadata and
 * step scratch; initialises cache_slots and slot_token to -1, last_use, stamps
 * and lengths to 0.  Synchronous.  Errors: KVO_EINVAL (cfg out of range),
 * KVO_ECUDA (no such device), KVO_ENOMEM.  On error *out is NULL.
 */
int kvo_create(const kvo_config* cfg, kvo_handle** out);

/* kvo_destroy: synchronise the device and free everything kvo_create made
 * (the pages define no teardown; this is the library's own).  NULL is a no-op. */
int kvo_destroy(kvo_handle* h);

/*
 * kvo_host_rows ([LS] "Memory layout": the full main-KV history of every
 * unit lives in the pinned host pool): host address of row 0 of unit's pool;
 * rows are contiguous, row_elems bf16 each, max_tokens rows.  The caller may write rows [0, n)
 * before kvo_prefill(unit, n) (bulk load of a prefilled context; untimed
 * set-up, outside the decode step).  NULL if unit is out of range.
 */
void* kvo_host_rows(kvo_handle* h, int32_t unit);

/*
 * Paged host pool (config host_block_tokens > 0; "SFA Remote D2H Connector
 * Design", "Data Ownership": the main KV is addressed by block IDs).  A unit's
 * token t lives in
 * row t mod B of physical block blocks[t / B] of its block table (B =
 * host_block_tokens); the indexer cache and the hot buffers stay per unit on
 * the device.  kvo_host_rows returns NULL for a paged pool.
 * kvo_set_blocks: entries first_block .. first_block+n_blocks-1 of unit's
 * table = blocks[0..n_blocks-1] (host array; -1 = unmapped), copied on
 * `stream`: from pageable memory the call returns once the array has been
 * staged (the caller may reuse it); from pinned memory it is asynchronous
 * (keep the array unchanged until the stream has passed the copy).  Rows of
 * unmapped blocks are never read or written: an append skips them and a
 * gather leaves the hot row as it was, and kvo_stats.block_errors counts
 * them.  Errors: KVO_EINVAL (not paged, a block id >= host_blocks),
 * KVO_ERANGE (unit or block range).
 * kvo_host_block: host address of physical block `block` ([B][row_elems]
 * bf16), for filling the cached rows; NULL on a bad argument.
 */
int kvo_set_blocks(kvo_handle* h, int32_t unit, int32_t first_block, int32_t n_blocks,
                   const int32_t* blocks, void* stream);
void* kvo_host_block(kvo_handle* h, int64_t block);

/*
 * kvo_prefill ([LS] section 5, "Request flow", steps 1 and 5: the decode
 * side takes a prefilled request into its main host destination and its
 * indexer destination): set an empty unit's context to n_tokens tokens whose
 * rows are
 * already in the host pool; copies idx_keys (bf16 [n_tokens][128], host or
 * device memory) into the indexer cache on the given stream.  Errors:
 * KVO_EINVAL (unit not empty), KVO_ERANGE (unit or n_tokens out of range).
 */
int kvo_prefill(kvo_handle* h, int32_t unit, int64_t n_tokens, const void* idx_keys,
                void* stream);

/*
 * kvo_append ([LS] Decode step 1-2; "Transfer granularity": token rows
 * device -> host): for each listed unit, copy its n_tokens new rows to host
 * pool rows len..len+n_tokens-1 and their indexer keys to the indexer cache,
 * then len += n_tokens.  New tokens are not resident (cache_slots -1).
 *   units     : host array [n_units] of distinct unit ids, or NULL = all units
 *               in order (then n_units must equal the unit count).
 *   main_rows : device bf16 [n_units][n_tokens][row_elems]
 *   idx_keys  : device bf16 [n_units][n_tokens][128]
 * Errors (nothing launched): KVO_EINVAL (bad pointer, duplicate unit),
 * KVO_ERANGE (unit id out of range or len + n_tokens > max_tokens).
 */
int kvo_append(kvo_handle* h, const int32_t* units, int32_t n_units, int32_t n_tokens,
               const void* main_rows, const void* idx_keys, void* stream);

/*
 * kvo_step ([LS] Decode step 3-6, [FO] decode paragraphs): one decode step
 * of every listed unit: indexer scoring of every cached token, fused top-k
 * carrying the packed payload, MTP merge and dedup, LRU residency update,
 * miss-row copy from the host pool into the hot buffer, remap to slots.
 *   units        : host array [n_units] of distinct unit ids, or NULL = all.
 *   queries      : device bf16 [n_units][P][128]
 *   topk_tokens  : device int32 [n_units][P][k] (out)
 *   topk_slots   : device int32 [n_units][P][k] (out) hot slot of each token
 *   topk_scores  : device float [n_units][P][k] (out, nullable)
 *   topk_payload : device int32 [n_units][P][k] (out, nullable) packed payload
 *   unit_status  : device int32 [n_units] (out) KVO_OK | KVO_ECAPACITY |
 *                  KVO_ETIMEOUT
 * Outputs are unspecified until the stream reaches the end of the step.
 */
int kvo_step(kvo_handle* h, const int32_t* units, int32_t n_units, const void* queries,
             int32_t* topk_tokens, int32_t* topk_slots, float* topk_scores,
             int32_t* topk_payload, int32_t* unit_status, void* stream);

/*
 * kvo_select ([LS] Decode step 3, [FO] packed-payload top-k): the scoring
 * and fused top-k of kvo_step alone, on caller buffers, stateless.
 *   keys        : device bf16; key of token t of unit i at
 *                 keys + (i * unit_stride + t) * 128 elements
 *   cache_slots : device int32, entry of token t of unit i at
 *                 cache_slots[i * unit_stride + t]; NULL = nothing resident
 *   lengths     : host int64 [n_units] cached tokens per unit (<= unit_stride)
 *   queries     : device bf16 [n_units][n_pos][128]
 *   tokens, scores, payload: device [n_units][n_pos][k] (scores, payload
 *                 nullable), same order and padding rules as kvo_step
 *   workspace   : device scratch of at least kvo_select_workspace_size()
 *                 bytes, 256-byte aligned, owned by the caller; its contents
 *                 need no initialisation and are not preserved
 *   status      : device uint32, nullable, 4-byte aligned: set to 0 at the
 *                 start of the call on the stream; the kernels OR in
 *                 KVO_SELECT_ERR_TIMEOUT (a bounded wait expired) or
 *                 KVO_SELECT_ERR_PLAN (an internal consistency check failed);
 *                 nonzero means the outputs are not valid
 * Errors: KVO_EINVAL, KVO_ECUDA.  Asynchronous on stream.
 */
#define KVO_SELECT_ERR_TIMEOUT 1u
#define KVO_SELECT_ERR_PLAN 2u
size_t kvo_select_workspace_size(int32_t n_units, int32_t n_pos, int32_t k, int32_t device);
int kvo_select(const void* keys, int64_t unit_stride, const int32_t* cache_slots,
               const int64_t* lengths, int32_t n_units, int32_t n_pos, int32_t k,
               const void* queries, int32_t* tokens, float* scores, int32_t* payload,
               void* workspace, size_t workspace_bytes, uint32_t* status, void* stream);

/*
 * kvo_reset (the pages define no reset; the library's own, for reusing a
 * unit): return every listed unit to its first keep_tokens cached tokens
 * with an empty hot shelf (cache_slots and slot_token -1, last_use and stamp
 * 0), as when a finished request's unit is reused for a new request whose
 * prefilled context is already in place.  keep_tokens must not exceed any
 * listed unit's length.  Asynchronous on stream.  Errors: KVO_EINVAL,
 * KVO_ERANGE.
 */
int kvo_reset(kvo_handle* h, const int32_t* units, int32_t n_units, int64_t keep_tokens,
              void* stream);

/*
 * Per-kernel device time (measurement support; no passage of the pages),
 * recorded when KVO_OPT_PROFILE is 1: CUDA events on
 * the launching stream bracket every kernel the library launches.
 * kvo_profile_read synchronises those events, adds their durations into
 * ms[kind] and the launch counts into launches[kind] for kind <
 * min(n_kinds, KVO_PROF_KINDS), and forgets them.
 */
#define KVO_PROF_APPEND 0
#define KVO_PROF_PLAN 1
#define KVO_PROF_SCORE 2
#define KVO_PROF_SELECT 3
#define KVO_PROF_RESIDENCY 4
#define KVO_PROF_GATHER 5
#define KVO_PROF_RESET 6
#define KVO_PROF_RESCORE 7   /* rescoring pass of units whose speculative threshold was too high */
#define KVO_PROF_RESELECT 8
#define KVO_PROF_FUSED 9     /* the fused step launch (KVO_OPT_FUSED) */
#define KVO_PROF_ATTEND 10   /* kvo_attend */
#define KVO_PROF_KINDS 11
int kvo_profile_read(kvo_handle* h, double* ms, uint64_t* launches, int32_t n_kinds);

/* kvo_set_option: KVO_OPT_* above (library tuning; no passage of the pages).
 * KVO_EINVAL on unknown key or value. */
int kvo_set_option(kvo_handle* h, int32_t key, int64_t value);

/* kvo_get_option: the current value of KVO_OPT_* key into *value (host
 * memory).  KVO_EINVAL on unknown key or NULL arguments. */
int kvo_get_option(kvo_handle* h, int32_t key, int64_t* value);

/* kvo_get_stats (library counters; no passage of the pages): synchronises the
 * device, then copies the counters. */
int kvo_get_stats(kvo_handle* h, kvo_stats* out);

/*
 * kvo_export_state (test accessor of the state [LS] "Memory layout" and
 * Decode step 4 describe): synchronises the device and copies one unit's state to
 * host buffers (any may be NULL): cache_slots [max_tokens] int32,
 * slot_token [hot_capacity] int32, last_use [hot_capacity] uint32, length
 * and stamp scalars, hot_rows [hot_capacity][row_elems] bf16.
 */
int kvo_export_state(kvo_handle* h, int32_t unit, int32_t* cache_slots, int32_t* slot_token,
                     uint32_t* last_use, int64_t* length, uint32_t* stamp, void* hot_rows);

/*
 * kvo_select_noalloc: kvo_select for callers that cannot allocate memory.
 * The pages have no counterpart of this call; it exists for callers such as
 * an operator hosted by a framework that owns all device memory and forbids
 * its extensions to call cudaMalloc, or a latency-critical loop that cannot
 * afford an allocation.  Same arguments and results as kvo_select, without
 * the workspace: the scratch is a fixed 16 MiB device array inside the
 * library, held until exit by every GPU that loads the library (under lazy
 * module loading, from the first call on that device), and an accepted call
 * allocates nothing on the host or the device.  Limits: n_units <= 64
 * and a scratch need (the kvo_select_workspace_size formula) of at most
 * 16 MiB, else KVO_ERANGE with a message.  All calls share the array: the
 * call clears what must start at zero, but calls that overlap on the GPU race
 * (order them on one stream).  The first call on a device looks up the
 * array's address for that device; make it before any stream capture.  That
 * address is kept until exit, so calls after a cudaDeviceReset of that device
 * are not supported.  status (device uint32, nullable) reports the kernels'
 * completion as for kvo_select; without it an expired wait goes unreported.
 */
int kvo_select_noalloc(const void* keys, int64_t unit_stride, const int32_t* cache_slots,
                       const int64_t* lengths, int32_t n_units, int32_t n_pos, int32_t k,
                       const void* queries, int32_t* tokens, float* scores, int32_t* payload,
                       uint32_t* status, void* stream);

/*
 * kvo_attend ([LS] Decode step 7: the sparse-attention operator reads the
 * K/V rows now resident on the device; the pages name an SFA/MLA model without its formula, so this is the
 * absorbed latent attention of the DeepSeek family, reading R13 of the
 * oracle): for each listed unit u, position p and head h, over the hot rows
 * named by that position's top-k slots (slot < 0 or >= hot_capacity: pad,
 * skipped), with a row = [latent 512 | rope key 64] and the query of the same
 * split,
 *   s_i = scale * q[u][p][h] . row_i,
 *   out[u][p][h][d] = sum_i softmax(s)_i * row_i[d]  (d < 512),
 *   lse[u][p][h] = log sum_i exp(s_i)  (-inf when the list has no row).
 * Run it after kvo_step on the same stream with that step's topk_slots: the
 * hot rows it reads are the ones the step made resident.  When that step ran
 * with KVO_OPT_DEFER_FILL = 1 and this call lists the same units in the same
 * order, the step's miss rows are not in the hot buffer yet: this kernel reads
 * each from the pinned pool (the token its packed payload names), uses it, and
 * writes it to its slot, one CTA per row part (claim words in device memory;
 * a CTA that finds a part claimed but not yet written reads the pool again),
 * so that on return the hot buffer is as a filling kvo_step would have left it
 * (the pages' Copy-SFA operator, Chinese edition of "Layerwise and Sparse KV
 * Cache Offloading Design": misses copied inside sparse attention).  Those
 * rows count in kvo_stats.rows_h2d / bytes_h2d, re-reads in fetch_dup_bytes.
 *   units      : host array [n_units] (as kvo_step), or NULL = all units.
 *   queries    : device bf16 [n_units][P][n_heads][576], 16-byte aligned.
 *   n_heads    : a multiple of 128 (one CTA pair per 128 heads).
 *   scale      : softmax scale (e.g. 1/sqrt(192)), finite.
 *   topk_slots : device int32 [n_units][P][k], as written by kvo_step.
 *   out        : device bf16 [n_units][P][n_heads][512] (written), 16-byte aligned.
 *   lse        : device float [n_units][P][n_heads] (written), nullable.
 * Precision: scores accumulate in fp32 on the tensor cores; softmax weights
 * are rounded to bf16 before the value product and normalised by the sum of
 * the rounded weights; out is rounded to bf16.  Requires row_elems == 576.
 * Errors (nothing launched): KVO_EINVAL (NULL or misaligned pointer, n_heads,
 * scale, row size), KVO_ERANGE (unit id).  A bounded device wait that expires
 * sets the error word read by kvo_get_stats (the output is then unspecified).
 */
int kvo_attend(kvo_handle* h, const int32_t* units, int32_t n_units, const void* queries,
               int32_t n_heads, float scale, const int32_t* topk_slots, void* out, float* lse,
               void* stream);

/* ------------------------------------------------------------------------
 * Layerwise prefill offload ([LS] section 3 "Layerwise Prefill Offload":
 * "Buffer planning", "Execution pipeline", "Reuse invariant"; [FO] prefill
 * paragraph: four trays, tray B0 bound to the first layer, onload_layer_map).
 * The main KV of every layer lives in a pinned host pool; N layers share
 * I + min(B, N - I) device buffers.  A prefill pass walks the layers in order:
 * the layer's cached prefix is loaded into its buffer (unless the buffer
 * still holds it), the caller's compute for the layer reads it and writes the
 * chunk's new rows after it, and those rows are saved back to the host pool.
 * Loads and saves run on the copy engines on two library streams; a buffer is
 * reloaded only after the save of its previous layer has finished.
 * ------------------------------------------------------------------------ */
typedef struct kvo_lw kvo_lw; /* opaque, library-owned */
typedef struct {
  int32_t n_layers;      /* N cache-bearing layers, >= 1 */
  int32_t n_independent; /* I: layers 0..I-1 keep a dedicated buffer (tray B0 = layer 0); 0..N */
  int32_t n_shared;      /* B shared buffers, round robin over layers I..N-1; >= 1 if I < N */
  int32_t lookahead;     /* onload_layer_map: a layer's load is issued when the compute of the
                            layer `lookahead` before it starts (>= 1) */
  int64_t max_tokens;    /* rows per layer in the host pool and in every buffer */
  int32_t row_elems;     /* bf16 elements per row (576); row bytes a multiple of 16 */
  int32_t device;
} kvo_lw_config;

/* kvo_lw_create: the plan (reading R14 of the oracle: independent layers take
 * buffers 0..I-1, the k-th reusable layer buffer I + k mod min(B, N - I)), the
 * device buffers [n_phys][max_tokens][row_elems] bf16 and the pinned host pool
 * [N][max_tokens][row_elems] bf16 (zeroed).  Cached length starts at 0.
 * Errors: KVO_EINVAL (config), KVO_ENOMEM, KVO_ECUDA. */
int kvo_lw_create(const kvo_lw_config* cfg, kvo_lw** out);
int kvo_lw_destroy(kvo_lw* lw);

/* kvo_lw_plan: *n_phys = the number of device buffers; phys_of_layer [N]
 * (nullable) = the buffer of each layer. */
int kvo_lw_plan(kvo_lw* lw, int32_t* n_phys, int32_t* phys_of_layer);

/* kvo_lw_host_rows: host address of layer `layer`'s rows [max_tokens][row_elems]
 * in the pinned pool (NULL on a bad argument).  Write the cached prefix there
 * before kvo_lw_set_length; the library reads and writes it during passes. */
void* kvo_lw_host_rows(kvo_lw* lw, int32_t layer);

/* kvo_lw_set_length: the cached prefix now has `tokens` rows in every layer
 * (host pool rows 0..tokens-1); forgets what the buffers hold.  Synchronises
 * the library streams.  Errors: KVO_EINVAL (inside a pass), KVO_ERANGE. */
int kvo_lw_set_length(kvo_lw* lw, int64_t tokens);

/* kvo_lw_begin: start a pass over `chunk_tokens` new tokens on the caller's
 * stream (loads wait for the work already on it).  Errors: KVO_EINVAL (pass
 * already open), KVO_ERANGE (length + chunk_tokens > max_tokens). */
int kvo_lw_begin(kvo_lw* lw, int64_t chunk_tokens, void* stream);

/* kvo_lw_layer: the next layer of the pass (layers in order 0..N-1).  Issues
 * the loads up to `lookahead` layers ahead, makes `stream` wait until this
 * layer's buffer holds its cached rows 0..L-1, and returns the buffer
 * (device, [max_tokens][row_elems] bf16) in *buffer.  The caller's compute on
 * `stream` reads rows 0..L-1 and writes the chunk's rows L..L+c-1.
 * Errors: KVO_EINVAL (no open pass, layer out of order). */
int kvo_lw_layer(kvo_lw* lw, int32_t layer, void** buffer, void* stream);

/* kvo_lw_layer_done: the compute of `layer` has been enqueued on `stream`;
 * its rows L..L+c-1 are saved to the host pool once it finishes. */
int kvo_lw_layer_done(kvo_lw* lw, int32_t layer, void* stream);

/* kvo_lw_end: after the last layer: `stream` waits for every save of the pass;
 * the cached length grows by the chunk.  Errors: KVO_EINVAL (layers missing). */
int kvo_lw_end(kvo_lw* lw, void* stream);

/* kvo_lw_stats: bytes copied host -> device and device -> host so far. */
int kvo_lw_stats(kvo_lw* lw, uint64_t* bytes_h2d, uint64_t* bytes_d2h);

/*
 * kvo_wait_selftest (failure detection of the library's own bounded waits;
 * no passage of the pages): runs, on `device`, one thread through the two bounded
 * waits every kernel of the library relies on (a spin on a global flag and an
 * mbarrier phase wait), each on a condition nothing satisfies and limited to
 * limit_ns (1 us .. 10 s).  Both must give up; the call returns KVO_ETIMEOUT
 * when they did, with the time waited in *waited_ns (nullable), and leaves
 * the device usable.  Synchronous.  Errors: KVO_EINVAL (limit), KVO_ECUDA.
 */
int kvo_wait_selftest(int32_t device, int64_t limit_ns, int64_t* waited_ns);

/* kvo_last_error (library error reporting; no passage of the pages): message
 * of the last failing call on this thread ("" if none). */
const char* kvo_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVO_H */
