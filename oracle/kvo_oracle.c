/*
 * CPU ORACLE for the sparse-decode KV offload step.  TEST INFRASTRUCTURE ONLY:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load it.  It shares no code, header or constant table with the CUDA path.
 *
 * Plain, slow, obviously correct: every unit (request, layer) is processed on
 * its own, every selection is a full qsort, every LRU choice a full sort.
 *
 * Sources (web pages; section names as printed there):
 *  [LS]  "Layerwise and Sparse KV Cache Offloading Design", section 4
 *        "Sparse Decode Offload" -> "Memory layout" and "Decode step" (the
 *        seven numbered steps), and section 2 "Transfer granularity".
 *  [FO]  "FlashOffloading offloads all KV cache ... What does it mean?",
 *        the decode paragraphs: hot shelf of fixed size, MTP3 per-position
 *        miss lists merged and deduplicated, the cache_slots reverse index
 *        (-1 when absent), the index/slot pair packed into one int32 before
 *        selection.
 *
 * Readings where the pages are silent (all of them are choices of this
 * project, applied identically by the CUDA path):
 *  R1 score   : s = single-head dot product of the bf16 indexer query and key,
 *               fp32, canonical order: 16 chunk sums c_j, each an FMA chain
 *               over d = 8j..8j+7 starting from +0, then the tree
 *               c_j += c_{j+w} for w = 8, 4, 2, 1 (j < w); s = c_0; a zero
 *               result is returned as +0.
 *  R2 ties    : ordering (score desc, token asc); output in that order.
 *  R3 MTP     : position p of P sees tokens t < len - (P - 1 - p).
 *  R4 payload : pay = cache_slots[t] if >= 0 (hit: the slot) else -(t + 1)
 *               (miss: the token), read before this step's update; padding
 *               entries (fewer visible tokens than k) carry token -1, score
 *               -inf, payload INT32_MIN, slot -1.
 *  R5 merge   : W = distinct tokens over the P lists; misses sorted by token
 *               ascending.
 *  R6 LRU     : per-unit stamp, +1 per successful step; candidate slots are
 *               those not holding a token of W, taken in (last_use asc,
 *               slot asc) order (free slots have last_use 0); i-th miss takes
 *               i-th candidate; every slot of W gets last_use = stamp.
 *  R7 capacity: |W| > capacity -> unit status ORACLE_ECAPACITY, nothing
 *               changes, slots -1.
 *  R8 append  : new rows go to the host rows only; their cache_slots are -1.
 *  R9-R11     : an empty shelf at the start, the benchmark workloads' shared
 *               queries across MTP positions and one contiguous 576-element
 *               row per token need no arithmetic of their own here.
 *  R12 int8 indexer ("FlashOffloading ... What does it mean?", the LIM C8
 *               paragraph: Hadamard rotation and int8 quantization of the
 *               indexer query and key, fp16 dequantization scales that follow
 *               the indexer layout):
 *               rotation y = H x with the 128-point Walsh-Hadamard matrix
 *               (entries +-1, unnormalised), computed in fp32 by the fast
 *               transform: stages h = 1, 2, ..., 64, each pair (i, i + h)
 *               with i & h == 0 becomes (a + b, a - b);
 *               scale s = fp16(max|y| / 127) (fp32 division, then
 *               round-to-nearest-even to fp16), one per vector (per key, per
 *               query position); codes c = clamp(rint(y / s), -127, 127) with
 *               s read back as fp32 (all 0 when s = 0);
 *               score = (((float)(sum c_q c_k) * s_q) * s_k) / 128, in that
 *               order (the integer sum is exact; / 128 undoes the unnormalised
 *               rotation, H H = 128 I, so the score estimates q . k); a zero
 *               score is +0.  Keys are quantized when they are appended,
 *               queries at each step; the bf16 keys are kept only for tests.
 *  R13 sparse attention ([LS] Decode step 7: attention runs on the rows
 *               made resident by the step; the pages name an SFA/MLA model but give no
 *               formula, so the absorbed multi-head latent attention of the
 *               DeepSeek family is taken): per unit, position p and head h,
 *               over the tokens t of that position's top-k list (pads
 *               skipped), with the 576-element row r_t = [latent (512) |
 *               rope key (64)] of the main-KV history and the query
 *               q_h (576, same split):
 *                 s_t = scale * sum_{d<576} q_h[d] r_t[d],
 *                 w_t = exp(s_t - max s) / sum_t' exp(s_t' - max s),
 *                 out_h[d] = sum_t w_t r_t[d] for d < 512 (the latent part
 *                 is the value), lse_h = max s + log(sum exp(s - max s)),
 *               all in fp64; a list with no token gives out 0, lse -inf.
 *               scale is the caller's softmax scale.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)
#define ORACLE_ERANGE (-3)
#define ORACLE_ECAPACITY (-6)
#define ORACLE_DIM 128
#define ORACLE_PAD_PAYLOAD INT32_MIN

typedef struct oracle_unit {
  int64_t tmax;
  int32_t row_elems, topk, capacity, n_pos, keep_rows;
  int32_t idx_int8;      /* R12: 1 = scores from the int8 indexer */
  int8_t* kcode;         /* [tmax][128] int8 key codes (R12), or NULL */
  uint16_t* kscale;      /* [tmax] fp16 key scales (R12), or NULL */
  int64_t len;
  uint32_t stamp;
  uint16_t* keys;        /* [tmax][128] indexer keys (device copy in the real system) */
  uint16_t* rows;        /* [tmax][row_elems] full main-KV history ("host pool"), or NULL */
  int32_t* cache_slots;  /* [tmax] token -> hot slot, -1 when absent */
  int32_t* slot_token;   /* [capacity] hot slot -> token, -1 when free */
  uint32_t* last_use;    /* [capacity] stamp of the last step that used the slot */
  uint16_t* hot;         /* [capacity][row_elems] hot buffer rows, or NULL */
} oracle_unit;

static float bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* R1: canonical fp32 score of one key against one query (both 128 bf16). */
float oracle_score(const uint16_t* q, const uint16_t* k) {
  float c[16];
  for (int j = 0; j < 16; ++j) {
    float acc = 0.0f;
    for (int e = 0; e < 8; ++e) acc = fmaf(bf16_value(q[8 * j + e]), bf16_value(k[8 * j + e]), acc);
    c[j] = acc;
  }
  for (int w = 8; w >= 1; w >>= 1)
    for (int j = 0; j < w; ++j) c[j] = c[j] + c[j + w];
  float s = c[0];
  if (s == 0.0f) s = 0.0f;
  return s;
}

/* ---- R12: int8 indexer ------------------------------------------------ */

/* fp32 -> fp16 bits, round to nearest even (IEEE 754 binary16). */
uint16_t oracle_f32_to_f16(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  const uint32_t sign = (x >> 16) & 0x8000u;
  const int32_t exp = (int32_t)((x >> 23) & 0xffu);
  uint32_t man = x & 0x7fffffu;
  if (exp == 0xff) return (uint16_t)(sign | 0x7c00u | (man ? 0x200u : 0u));
  const int32_t e = exp - 127 + 15;
  if (e >= 31) return (uint16_t)(sign | 0x7c00u);
  if (e <= 0) {
    /* half subnormal: units of 2^-24; value = (1.man) 2^(exp-127) */
    if (exp == 0) return (uint16_t)sign; /* fp32 subnormals are far below 2^-25 */
    const uint32_t full = man | 0x800000u;
    const int32_t shift = 14 - e;
    if (shift > 24) return (uint16_t)sign;
    uint32_t hm = full >> shift;
    const uint32_t rem = full & ((1u << shift) - 1u), half = 1u << (shift - 1);
    if (rem > half || (rem == half && (hm & 1u))) ++hm;
    return (uint16_t)(sign | hm); /* hm == 0x400 is the smallest normal */
  }
  uint32_t hm = man >> 13;
  const uint32_t rem = man & 0x1fffu;
  int32_t he = e;
  if (rem > 0x1000u || (rem == 0x1000u && (hm & 1u))) ++hm;
  if (hm == 0x400u) {
    hm = 0;
    if (++he >= 31) return (uint16_t)(sign | 0x7c00u);
  }
  return (uint16_t)(sign | ((uint32_t)he << 10) | hm);
}

/* fp16 bits -> fp32 (exact). */
float oracle_f16_to_f32(uint16_t h) {
  const uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
  const uint32_t e = (h >> 10) & 0x1fu, m = h & 0x3ffu;
  uint32_t x;
  if (e == 0) {
    float v = (float)m * 5.9604644775390625e-8f; /* m * 2^-24, exact */
    memcpy(&x, &v, 4);
    x |= sign;
  } else if (e == 31) {
    x = sign | 0x7f800000u | (m << 13);
  } else {
    x = sign | ((e - 15 + 127) << 23) | (m << 13);
  }
  float f;
  memcpy(&f, &x, 4);
  return f;
}

/* R12 rotation: unnormalised fast Walsh-Hadamard transform, fixed stage order. */
void oracle_fwht128(const float* in, float* out) {
  float y[ORACLE_DIM];
  memcpy(y, in, sizeof(y));
  for (int h = 1; h < ORACLE_DIM; h <<= 1)
    for (int i = 0; i < ORACLE_DIM; ++i)
      if ((i & h) == 0) {
        const float a = y[i], b = y[i + h];
        y[i] = a + b;
        y[i + h] = a - b;
      }
  memcpy(out, y, sizeof(y));
}

/* R12 quantization of an already rotated vector: fp16 scale, int8 codes. */
void oracle_quant_rotated(const float* y, int8_t* code, uint16_t* scale) {
  float m = 0.0f;
  for (int d = 0; d < ORACLE_DIM; ++d) {
    const float a = fabsf(y[d]);
    if (a > m) m = a;
  }
  const uint16_t s16 = oracle_f32_to_f16(m / 127.0f);
  const float s = oracle_f16_to_f32(s16);
  for (int d = 0; d < ORACLE_DIM; ++d) {
    float c = s > 0.0f ? rintf(y[d] / s) : 0.0f;
    if (c > 127.0f) c = 127.0f;
    if (c < -127.0f) c = -127.0f;
    code[d] = (int8_t)c;
  }
  *scale = s16;
}

/* R12: rotate and quantize one bf16 vector of 128. */
void oracle_quant128(const uint16_t* x, int8_t* code, uint16_t* scale) {
  float v[ORACLE_DIM], y[ORACLE_DIM];
  for (int d = 0; d < ORACLE_DIM; ++d) v[d] = bf16_value(x[d]);
  oracle_fwht128(v, y);
  oracle_quant_rotated(y, code, scale);
}

/* R12 score of int8 codes with their fp16 scales. */
float oracle_score_i8(const int8_t* q, uint16_t sq, const int8_t* k, uint16_t sk) {
  int32_t dot = 0;
  for (int d = 0; d < ORACLE_DIM; ++d) dot += (int32_t)q[d] * (int32_t)k[d];
  float s = (((float)dot * oracle_f16_to_f32(sq)) * oracle_f16_to_f32(sk)) / 128.0f;
  if (s == 0.0f) s = 0.0f;
  return s;
}

oracle_unit* oracle_unit_new(int64_t tmax, int32_t dim, int32_t row_elems, int32_t topk,
                             int32_t capacity, int32_t n_pos, int32_t keep_rows) {
  if (dim != ORACLE_DIM || tmax < 0 || row_elems <= 0 || topk <= 0 || capacity <= 0 ||
      n_pos <= 0)
    return NULL;
  oracle_unit* u = (oracle_unit*)calloc(1, sizeof(oracle_unit));
  if (!u) return NULL;
  u->tmax = tmax;
  u->row_elems = row_elems;
  u->topk = topk;
  u->capacity = capacity;
  u->n_pos = n_pos;
  u->keep_rows = keep_rows;
  u->keys = (uint16_t*)malloc((size_t)(tmax > 0 ? tmax : 1) * ORACLE_DIM * 2);
  u->cache_slots = (int32_t*)malloc((size_t)(tmax > 0 ? tmax : 1) * 4);
  u->slot_token = (int32_t*)malloc((size_t)capacity * 4);
  u->last_use = (uint32_t*)calloc((size_t)capacity, 4);
  if (keep_rows) {
    u->rows = (uint16_t*)malloc((size_t)(tmax > 0 ? tmax : 1) * row_elems * 2);
    u->hot = (uint16_t*)calloc((size_t)capacity * row_elems, 2);
  }
  if (!u->keys || !u->cache_slots || !u->slot_token || !u->last_use ||
      (keep_rows && (!u->rows || !u->hot))) {
    free(u->keys); free(u->cache_slots); free(u->slot_token); free(u->last_use);
    free(u->rows); free(u->hot); free(u);
    return NULL;
  }
  for (int64_t t = 0; t < tmax; ++t) u->cache_slots[t] = -1;
  for (int32_t s = 0; s < capacity; ++s) u->slot_token[s] = -1;
  return u;
}

void oracle_unit_free(oracle_unit* u);

/* As oracle_unit_new; idx_int8 = 1 selects the int8 indexer (R12). */
oracle_unit* oracle_unit_new2(int64_t tmax, int32_t dim, int32_t row_elems, int32_t topk,
                              int32_t capacity, int32_t n_pos, int32_t keep_rows, int32_t idx_int8) {
  oracle_unit* u = oracle_unit_new(tmax, dim, row_elems, topk, capacity, n_pos, keep_rows);
  if (!u || !idx_int8) return u;
  u->idx_int8 = 1;
  u->kcode = (int8_t*)malloc((size_t)(tmax > 0 ? tmax : 1) * ORACLE_DIM);
  u->kscale = (uint16_t*)malloc((size_t)(tmax > 0 ? tmax : 1) * 2);
  if (!u->kcode || !u->kscale) {
    free(u->kcode); free(u->kscale);
    u->kcode = NULL; u->kscale = NULL;
    oracle_unit_free(u);
    return NULL;
  }
  return u;
}

void oracle_unit_free(oracle_unit* u) {
  if (!u) return;
  free(u->keys); free(u->cache_slots); free(u->slot_token); free(u->last_use);
  free(u->rows); free(u->hot); free(u->kcode); free(u->kscale); free(u);
}

/* R8 / [LS] Decode step 1-2: new rows land at their logical slots len..len+n-1. */
int32_t oracle_append(oracle_unit* u, int32_t n_tok, const uint16_t* rows, const uint16_t* keys) {
  if (n_tok < 0) return ORACLE_EINVAL;
  if (u->len + n_tok > u->tmax) return ORACLE_ERANGE;
  memcpy(u->keys + (size_t)u->len * ORACLE_DIM, keys, (size_t)n_tok * ORACLE_DIM * 2);
  if (u->idx_int8) /* R12: keys are quantized once, when they arrive */
    for (int32_t j = 0; j < n_tok; ++j)
      oracle_quant128(keys + (size_t)j * ORACLE_DIM, u->kcode + (size_t)(u->len + j) * ORACLE_DIM,
                      u->kscale + u->len + j);
  if (u->keep_rows && rows)
    memcpy(u->rows + (size_t)u->len * u->row_elems, rows, (size_t)n_tok * u->row_elems * 2);
  for (int32_t j = 0; j < n_tok; ++j) u->cache_slots[u->len + j] = -1;
  u->len += n_tok;
  return ORACLE_OK;
}

typedef struct { float score; int32_t token; } scored_t;

/* R2: score descending, then token ascending. */
static int cmp_scored(const void* a, const void* b) {
  const scored_t* x = (const scored_t*)a;
  const scored_t* y = (const scored_t*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->token > y->token) - (x->token < y->token);
}

static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

typedef struct { uint32_t last_use; int32_t slot; } lru_t;

/* R6: least recently used first, lower slot index first among equals. */
static int cmp_lru(const void* a, const void* b) {
  const lru_t* x = (const lru_t*)a;
  const lru_t* y = (const lru_t*)b;
  if (x->last_use != y->last_use) return x->last_use < y->last_use ? -1 : 1;
  return (x->slot > y->slot) - (x->slot < y->slot);
}

/* Score of token t for query q under the unit's indexer (R1 or R12). */
static float unit_score(const oracle_unit* u, const uint16_t* q, const int8_t* qcode, uint16_t qscale,
                        int64_t t) {
  if (u->idx_int8)
    return oracle_score_i8(qcode, qscale, u->kcode + (size_t)t * ORACLE_DIM, u->kscale[t]);
  return oracle_score(q, u->keys + (size_t)t * ORACLE_DIM);
}

/* Scores of every visible token for one query (used by tests). */
void oracle_scores(const oracle_unit* u, const uint16_t* q, int64_t n, float* out) {
  int8_t qc[ORACLE_DIM];
  uint16_t qs = 0;
  if (u->idx_int8) oracle_quant128(q, qc, &qs);
  for (int64_t t = 0; t < n && t < u->len; ++t) out[t] = unit_score(u, q, qc, qs, t);
}

/*
 * One decode step of one unit ([LS] Decode step 3-6, [FO] decode paragraphs).
 * queries: [P][128] bf16.  Outputs (all [P][k]): tok, score, pay (payload
 * before the update), slot (after the update).  status: OK or ECAPACITY.
 * miss_tok/miss_slot: [<= P*k] the (token -> slot) pairs filled, token order;
 * n_miss: their count (rows copied host -> hot).
 */
int32_t oracle_step(oracle_unit* u, const uint16_t* queries, int32_t* tok, float* score,
                    int32_t* pay, int32_t* slot, int32_t* status, int32_t* miss_tok,
                    int32_t* miss_slot, int32_t* n_miss) {
  const int32_t P = u->n_pos, K = u->topk, C = u->capacity;
  *n_miss = 0;
  scored_t* buf = (scored_t*)malloc((size_t)(u->len > 0 ? u->len : 1) * sizeof(scored_t));
  int32_t* wl = (int32_t*)malloc((size_t)P * K * sizeof(int32_t));
  char* hit_slot = (char*)calloc((size_t)C, 1);
  lru_t* cand = (lru_t*)malloc((size_t)C * sizeof(lru_t));
  if (!buf || !wl || !hit_slot || !cand) {
    free(buf); free(wl); free(hit_slot); free(cand);
    return ORACLE_ENOMEM;
  }

  /* [LS] step 3 + [FO] packed payload: top-k per position, payload read now. */
  for (int32_t p = 0; p < P; ++p) {
    int64_t vis = u->len - (P - 1 - p); /* R3 */
    if (vis < 0) vis = 0;
    const uint16_t* q = queries + (size_t)p * ORACLE_DIM;
    int8_t qc[ORACLE_DIM];
    uint16_t qs = 0;
    if (u->idx_int8) oracle_quant128(q, qc, &qs); /* R12: the query, each step */
    for (int64_t t = 0; t < vis; ++t) {
      buf[t].score = unit_score(u, q, qc, qs, t);
      buf[t].token = (int32_t)t;
    }
    qsort(buf, (size_t)vis, sizeof(scored_t), cmp_scored);
    for (int32_t i = 0; i < K; ++i) {
      size_t o = (size_t)p * K + i;
      if (i < vis) {
        int32_t t = buf[i].token;
        tok[o] = t;
        score[o] = buf[i].score;
        int32_t cs = u->cache_slots[t];
        pay[o] = cs >= 0 ? cs : -(t + 1); /* R4 */
      } else {
        tok[o] = -1;
        score[o] = -INFINITY;
        pay[o] = ORACLE_PAD_PAYLOAD;
      }
    }
  }

  /* [FO] MTP merge + dedup (R5): distinct tokens; misses sorted ascending. */
  int32_t n_w = 0;
  for (int32_t o = 0; o < P * K; ++o)
    if (tok[o] >= 0) wl[n_w++] = tok[o];
  qsort(wl, (size_t)n_w, sizeof(int32_t), cmp_i32);
  int32_t n_distinct = 0;
  for (int32_t i = 0; i < n_w; ++i)
    if (i == 0 || wl[i] != wl[i - 1]) wl[n_distinct++] = wl[i];
  int32_t n_m = 0;
  for (int32_t i = 0; i < n_distinct; ++i) {
    int32_t t = wl[i];
    int32_t cs = u->cache_slots[t];
    if (cs >= 0) hit_slot[cs] = 1;
  }
  /* misses, in token order, moved to the front of wl */
  for (int32_t i = 0; i < n_distinct; ++i)
    if (u->cache_slots[wl[i]] < 0) wl[n_m++] = wl[i];

  if (n_distinct > C) { /* R7 */
    *status = ORACLE_ECAPACITY;
    for (int32_t o = 0; o < P * K; ++o) slot[o] = -1;
    free(buf); free(wl); free(hit_slot); free(cand);
    return ORACLE_OK;
  }

  /* [LS] step 4: LRU residency table (R6). */
  u->stamp += 1;
  int32_t n_c = 0;
  for (int32_t s = 0; s < C; ++s)
    if (!hit_slot[s]) { cand[n_c].last_use = u->last_use[s]; cand[n_c].slot = s; ++n_c; }
  qsort(cand, (size_t)n_c, sizeof(lru_t), cmp_lru);
  for (int32_t i = 0; i < n_m; ++i) {
    int32_t t = wl[i], s = cand[i].slot;
    int32_t old = u->slot_token[s];
    if (old >= 0) u->cache_slots[old] = -1; /* eviction */
    u->slot_token[s] = t;
    u->cache_slots[t] = s;
    /* [LS] step 5: only miss rows are copied host -> hot buffer. */
    if (u->keep_rows)
      memcpy(u->hot + (size_t)s * u->row_elems, u->rows + (size_t)t * u->row_elems,
             (size_t)u->row_elems * 2);
    miss_tok[i] = t;
    miss_slot[i] = s;
  }
  *n_miss = n_m;
  for (int32_t s = 0; s < C; ++s)
    if (hit_slot[s]) u->last_use[s] = u->stamp;
  for (int32_t i = 0; i < n_m; ++i) u->last_use[miss_slot[i]] = u->stamp;

  /* [LS] step 6: logical top-k positions -> physical hot slots. */
  for (int32_t o = 0; o < P * K; ++o) slot[o] = tok[o] >= 0 ? u->cache_slots[tok[o]] : -1;
  *status = ORACLE_OK;
  free(buf); free(wl); free(hit_slot); free(cand);
  return ORACLE_OK;
}

/*
 * Many units, one step each, OpenMP over units (used only to time the CPU
 * baseline).  queries: [n][P][128]; outputs [n][P][k]; miss arrays [n][P*k].
 */
int32_t oracle_step_many(oracle_unit** units, int32_t n, const uint16_t* queries, int32_t* tok,
                         float* score, int32_t* pay, int32_t* slot, int32_t* status,
                         int32_t* miss_tok, int32_t* miss_slot, int32_t* n_miss) {
  int32_t rc = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t i = 0; i < n; ++i) {
    oracle_unit* u = units[i];
    size_t pk = (size_t)u->n_pos * u->topk;
    int32_t r = oracle_step(u, queries + (size_t)i * u->n_pos * ORACLE_DIM, tok + i * pk,
                            score + i * pk, pay + i * pk, slot + i * pk, status + i,
                            miss_tok + i * pk, miss_slot + i * pk, n_miss + i);
    if (r != ORACLE_OK) {
#pragma omp atomic write
      rc = r;
    }
  }
  return rc;
}

/*
 * R13: sparse attention of one position over rows of the main-KV history.
 * rows: [tmax][row_elems] bf16 (row_elems >= 576); tok: [k] tokens of the
 * position's top-k list (< 0: pad, skipped); q: [n_heads][576] bf16.
 * out: [n_heads][512] fp64; lse: [n_heads] fp64.  Plain two-pass softmax.
 */
void oracle_attend_rows(const uint16_t* rows, int32_t row_elems, int64_t n_rows, const int32_t* tok,
                        int32_t k, const uint16_t* q, int32_t n_heads, double scale, double* out,
                        double* lse) {
  double* s = (double*)malloc((size_t)(k > 0 ? k : 1) * sizeof(double));
  for (int32_t h = 0; h < n_heads; ++h) {
    const uint16_t* qh = q + (size_t)h * 576;
    double mx = -INFINITY;
    for (int32_t i = 0; i < k; ++i) {
      s[i] = -INFINITY;
      if (tok[i] < 0 || tok[i] >= n_rows) continue;
      const uint16_t* r = rows + (size_t)tok[i] * row_elems;
      double dot = 0.0;
      for (int d = 0; d < 576; ++d) dot += (double)bf16_value(qh[d]) * (double)bf16_value(r[d]);
      s[i] = scale * dot;
      if (s[i] > mx) mx = s[i];
    }
    double* o = out + (size_t)h * 512;
    for (int d = 0; d < 512; ++d) o[d] = 0.0;
    if (mx == -INFINITY) {
      lse[h] = -INFINITY;
      continue;
    }
    double sum = 0.0;
    for (int32_t i = 0; i < k; ++i)
      if (s[i] != -INFINITY) sum += exp(s[i] - mx);
    for (int32_t i = 0; i < k; ++i) {
      if (s[i] == -INFINITY) continue;
      const double w = exp(s[i] - mx) / sum;
      const uint16_t* r = rows + (size_t)tok[i] * row_elems;
      for (int d = 0; d < 512; ++d) o[d] += w * (double)bf16_value(r[d]);
    }
    lse[h] = mx + log(sum);
  }
  free(s);
}

/* R13 over the unit's own history (kept when the unit was made with rows). */
int32_t oracle_attend(const oracle_unit* u, const int32_t* tok, int32_t k, const uint16_t* q,
                      int32_t n_heads, double scale, double* out, double* lse) {
  if (!u->rows || u->row_elems < 576) return ORACLE_EINVAL;
  oracle_attend_rows(u->rows, u->row_elems, u->len, tok, k, q, n_heads, scale, out, lse);
  return ORACLE_OK;
}

int32_t oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* accessors */
int64_t oracle_len(const oracle_unit* u) { return u->len; }
uint32_t oracle_stamp(const oracle_unit* u) { return u->stamp; }
int32_t* oracle_cache_slots(oracle_unit* u) { return u->cache_slots; }
int32_t* oracle_slot_token(oracle_unit* u) { return u->slot_token; }
uint32_t* oracle_last_use(oracle_unit* u) { return u->last_use; }
uint16_t* oracle_hot(oracle_unit* u) { return u->hot; }
uint16_t* oracle_rows(oracle_unit* u) { return u->rows; }
uint16_t* oracle_keys(oracle_unit* u) { return u->keys; }
int8_t* oracle_kcode(oracle_unit* u) { return u->kcode; }
uint16_t* oracle_kscale(oracle_unit* u) { return u->kscale; }
