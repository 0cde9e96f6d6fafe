// C ABI of libkvo: argument checks, allocation, launch order.
//
// Memory layout ("Layerwise and Sparse KV Cache Offloading Design", section 4
// "Memory layout"): the full main-KV history lives in one pinned, mapped host
// allocation [units][stride][row_elems] bf16 that kernels read and write in
// place over the host link; the indexer cache [units][stride][128] bf16, the
// hot buffers [units][C][row_elems] bf16 and the residency metadata live in
// device memory.  A decode step is either one fused cooperative launch or
// five launches on the caller's stream: plan -> score -> select -> residency
// -> gather.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
#include <stdlib.h>
#include <sys/mman.h>
#include <unistd.h>

#include <string>
#include <vector>

#include "kvo_internal.cuh"

using kvo::DevStats;

struct kvo_handle {
  kvo_config cfg{};
  int device = 0, n_sm = 0;
  int U = 0, C = 0, P = 0, k = 0, R = 0, cap = 0;
  int64_t stride = 0;
  int G_max = 0;
  uint16_t* host_pool = nullptr;      // host address
  uint16_t* host_pool_dev = nullptr;  // device-visible address of the same memory
  int32_t block_tokens = 0;           // > 0: paged pool of n_blocks blocks of this many rows
  int64_t n_blocks = 0;
  int32_t max_blocks = 0;             // block-table entries per unit
  int32_t* blocks = nullptr;          // [U][max_blocks] block tables (device), -1 = unmapped
  size_t pool_map_bytes = 0;          // always 0: cudaHostAlloc memory
  size_t pool_bytes = 0;              // size of the pinned pool
  size_t pool_huge_page = 0;
  uint16_t* idx = nullptr;           // bf16 indexer [U][stride][128]
  int8_t* idx8 = nullptr;            // int8 indexer codes [U][stride][128]
  uint16_t* idxs = nullptr;          // their fp16 scales [U][stride]
  int8_t* q8 = nullptr;              // per-step query codes [U][P][128]
  uint16_t* qscale = nullptr;        // their fp16 scales [U][P]
  uint32_t* qdone = nullptr;         // fused launch: CTAs done quantizing queries
  bool int8 = false;
  uint16_t* hot = nullptr;
  int32_t* cache_slots = nullptr;
  int32_t* slot_token = nullptr;
  uint32_t* last_use = nullptr;
  uint32_t* stamp = nullptr;
  int32_t* len = nullptr;
  std::vector<int64_t> len_host;
  int32_t* all_units = nullptr;  // identity list
  int32_t* units_dev = nullptr;  // last uploaded explicit list
  std::vector<int32_t> units_cached;
  int64_t* off = nullptr;
  uint64_t* gthr = nullptr;
  uint32_t* tok_bits = nullptr; // [U][tok_words] scratch, kept all zero
  int64_t tok_words = 0;
  int32_t* order = nullptr;     // [2][U][C] LRU lists
  int32_t* order_par = nullptr; // [U]
  uint64_t* spec = nullptr;     // [U][P] persistent: k-th best key of each unit's last step
  float* qn_prev = nullptr;     // [U][P] persistent: that step's squared query norms
  float* qn_cur = nullptr;      // [U][P] scratch
  uint64_t* tspec = nullptr;    // [U][P] scratch
  int32_t* fb = nullptr;        // [U] scratch
  uint32_t* fb_any = nullptr;   // scratch
  int speculate = 900;          // permille, 0 = off
  uint64_t* seg_keys = nullptr;
  int32_t* seg_cnt = nullptr;
  int32_t* sel_pay = nullptr;
  int32_t* miss_tok = nullptr;
  int32_t* miss_slot = nullptr;
  int32_t* miss_cnt = nullptr;
  int32_t* claim_batches = nullptr;  // [U] copy batches claimed per unit (staged step in unit groups)
  int64_t* miss_off = nullptr;
  uint32_t* done_ctr = nullptr;
  uint32_t* err = nullptr;
  DevStats* stats = nullptr;
  uint64_t host_steps = 0;
  int gather_mode = KVO_GATHER_LDG;
  uint64_t wait_ns = 2000000000ull;
  // fused step (one cooperative launch per kvo_step)
  bool fused_ok = false;        // the configuration fits the fused kernel's layout
  int fused = 2;                // KVO_OPT_FUSED mode: 0 staged, 1 fused, 2 per call
  int gather_ctas = 8;
  uint64_t fused_steps = 0;
  uint64_t split_steps = 0;
  unsigned long long* bytes_prev_host = nullptr;  // pinned, mapped: previous step's miss bytes
  unsigned long long* bytes_prev_dev = nullptr;   // its device address
  unsigned long long* bytes_seen = nullptr;       // device
  uint64_t planned_steps = 0;
  int piece_tokens = 4096;
  int64_t fseg_pieces = 0;      // pieces the segment buffers hold
  int64_t* pbeg = nullptr;      // [U+1]
  int32_t* pdone = nullptr;     // [U]
  unsigned long long* ctr = nullptr;  // [4]
  uint32_t* plan_flag = nullptr;      // [1]
  uint64_t* fseg_keys = nullptr;      // [pieces][P][k]
  int32_t* fseg_cnt = nullptr;        // [pieces][P]
  int32_t* chunk_unit = nullptr;
  int32_t* chunk_start = nullptr;
  int32_t* chunk_cnt = nullptr;
  uint32_t* chunk_flag = nullptr;
  int64_t chunk_cap = 0;
  uint32_t epoch = 0;
  // deferred fill (KVO_OPT_DEFER_FILL): kvo_step assigns the miss rows' slots and
  // leaves the rows to the next kvo_attend on the same units, which reads them
  // from the host pool inside the attention kernel and writes them to the hot buffer
  int defer_fill = 0;
  bool fill_pending = false;           // a deferred step's rows are not yet in the hot buffer
  std::vector<int32_t> pending_units;  // its unit list (materialised)
  const int32_t* pending_du = nullptr; // its device unit list
  uint32_t* claim = nullptr;           // [U][C][3] claim words of the fetching attention
  uint32_t fetch_epoch = 0;
  // unit groups: miss-row copies overlap the next group's scoring
  int groups = 1;
  int group_gather_sms = 0;     // KVO_OPT_GROUP_GATHER_SMS
  bool groups_set = false, group_gather_sms_set = false;  // set by the caller (else chosen per call)
  int score_ctas = 0;
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  cudaEvent_t ev_group[16] = {};
  // opt-in launch profiling
  bool profile = false;
  uint32_t profile_kinds = (1u << KVO_PROF_KINDS) - 1;  // KVO_OPT_PROFILE_KINDS
  uint64_t launches = 0;  // kernels launched through timed()
  struct Rec {
    int kind;
    cudaEvent_t e0, e1;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> free_events;
};

namespace {

thread_local std::string g_err;

int fail(int code, const std::string& msg) {
  g_err = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  g_err = std::string(what) + ": " + cudaGetErrorString(e);
  return KVO_ECUDA;
}

// Makes the handle's device current for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

template <class T>
cudaError_t dalloc(T** p, size_t count) {
  return cudaMalloc(reinterpret_cast<void**>(p), count * sizeof(T) > 0 ? count * sizeof(T) : 16);
}

void free_all(kvo_handle* h) {
  for (auto& r : h->recs) {
    cudaEventDestroy(r.e0);
    cudaEventDestroy(r.e1);
  }
  for (auto e : h->free_events) cudaEventDestroy(e);
  h->recs.clear();
  h->free_events.clear();
  if (h->side) cudaStreamDestroy(h->side);
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  if (h->ev_join) cudaEventDestroy(h->ev_join);
  for (auto& ev : h->ev_group)
    if (ev) cudaEventDestroy(ev);
  void* dev[] = {h->idx, h->idx8, h->idxs, h->q8, h->qscale, h->qdone, h->blocks, h->hot, h->cache_slots, h->slot_token, h->last_use, h->stamp, h->len,
                 h->all_units, h->units_dev, h->off, h->gthr, h->spec, h->qn_prev, h->qn_cur,
                 h->tspec, h->fb, h->fb_any, h->tok_bits, h->order, h->order_par, h->seg_keys, h->seg_cnt, h->sel_pay,
                 h->miss_tok, h->miss_slot, h->miss_cnt, h->miss_off, h->done_ctr, h->err,
                 h->stats, h->pbeg, h->pdone, h->ctr, h->plan_flag, h->fseg_keys, h->fseg_cnt, h->chunk_unit,
                 h->chunk_start, h->chunk_cnt, h->chunk_flag, h->claim, h->claim_batches};
  for (void* p : dev)
    if (p) cudaFree(p);
  if (h->bytes_seen) cudaFree(h->bytes_seen);
  if (h->bytes_prev_host) cudaFreeHost(h->bytes_prev_host);
  kvo::free_pinned(h->host_pool, h->pool_map_bytes);
}

size_t residency_smem_bytes(int C, int P, int k) {
  const int nwords = (C + 31) / 32;
  return (size_t)((nwords + 3) & ~3) * 4 + (size_t)P * k * 8;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The pinned host pool: driver-allocated pinned memory (cudaHostAlloc), mapped
// into the GPU's address space.  An anonymous mapping backed by transparent huge
// pages and registered with cudaHostRegister gathered faster while its huge pages
// stayed whole, but the host kernel split some of them while the GPU read the pool
// (vmstat thp_split_pmd), and each split cost the following steps tens to hundreds
// of milliseconds of GPU address translation; driver-allocated memory is never
// split, compacted or migrated.
cudaError_t alloc_host_pool(kvo_handle* h, size_t bytes) {
  void* p = nullptr;
  cudaError_t e = kvo::alloc_pinned(bytes, &p, &h->pool_map_bytes, &h->pool_huge_page);
  h->host_pool = static_cast<uint16_t*>(p);
  return e;
}

// Largest hot capacity for which kvo_step takes the fused path by default.
constexpr int kFusedDefaultMaxCapacity = 65536;
// Largest pinned pool for which kvo_step takes the fused path by default.  The fused
// fill hands out rows in chunks from a counter, so its CTAs read rows of many units at
// once and in a different order every step; from a large pool such reads wait for address
// translations (measured on a 38.7 GB pool: 89-107 GB/s), while the staged gather, whose
// CTAs keep the same units from step to step, moves the same rows at 203-208 GB/s.
constexpr size_t kFusedDefaultMaxPoolBytes = (size_t)16 << 30;

// Whether the fused step's shared-memory layout holds this configuration:
// the finisher's select and residency reuse the candidate buffers.
bool fused_fits(int P, int k, int cap, int C, bool int8) {
  const size_t region = (size_t)P * cap * 8 + (size_t)k * 8;
  int kpad = 1;
  while (kpad < k) kpad <<= 1;
  return kvo::fused_smem_bytes(P, k, cap, int8) <= 227 * 1024 && residency_smem_bytes(C, P, k) <= region &&
         (size_t)kpad * 8 + 8 * 256 <= region;
}

// (Re)allocates the per-piece candidate segments for the current piece size.
cudaError_t alloc_fused_segments(kvo_handle* h) {
  if (h->fseg_keys) cudaFree(h->fseg_keys);
  if (h->fseg_cnt) cudaFree(h->fseg_cnt);
  h->fseg_keys = nullptr;
  h->fseg_cnt = nullptr;
  // every unit at the full piece size, plus the finer pieces of the first units
  const int64_t small = kvo::kSmallPieceUnits < h->U ? kvo::kSmallPieceUnits : h->U;
  const int64_t lmax = h->cfg.max_tokens, lsmall = lmax < kvo::kSmallPieceMaxLen ? lmax : kvo::kSmallPieceMaxLen;
  h->fseg_pieces = (int64_t)h->U * kvo::pieces_of(h->U, lmax, h->piece_tokens) +
                   small * kvo::pieces_of(0, lsmall, h->piece_tokens);  // unit 0 has the finest pieces
  cudaError_t e = dalloc(&h->fseg_keys, (size_t)h->fseg_pieces * h->P * h->k);
  if (e == cudaSuccess) e = dalloc(&h->fseg_cnt, (size_t)h->fseg_pieces * h->P);
  if (e != cudaSuccess) h->fseg_pieces = 0;
  return e;
}

cudaError_t alloc_fused(kvo_handle* h) {
  const size_t U = (size_t)h->U;
  const int rows = kvo::fused_chunk_rows();
  h->chunk_cap = (int64_t)U * ((h->P * h->k + rows - 1) / rows);
  cudaError_t e = dalloc(&h->pbeg, U + 1);
  if (e == cudaSuccess) e = dalloc(&h->pdone, U);
  if (e == cudaSuccess) e = dalloc(&h->ctr, 4);
  if (e == cudaSuccess) e = dalloc(&h->plan_flag, 1);
  if (e == cudaSuccess) e = cudaMemset(h->plan_flag, 0, 4);
  if (e == cudaSuccess) e = dalloc(&h->chunk_unit, (size_t)h->chunk_cap);
  if (e == cudaSuccess) e = dalloc(&h->chunk_start, (size_t)h->chunk_cap);
  if (e == cudaSuccess) e = dalloc(&h->chunk_cnt, (size_t)h->chunk_cap);
  if (e == cudaSuccess) e = dalloc(&h->chunk_flag, (size_t)h->chunk_cap);
  if (e == cudaSuccess) e = cudaMemset(h->chunk_flag, 0, (size_t)h->chunk_cap * 4);
  if (e == cudaSuccess) e = cudaMemset(h->ctr, 0, 4 * 8);
  if (e == cudaSuccess) e = alloc_fused_segments(h);
  return e;
}

// Token -> host-pool row translation of the handle (contiguous or paged).
kvo::HostRows host_rows_of(const kvo_handle* h) {
  kvo::HostRows r{};
  r.blocks = h->blocks;
  r.block_tokens = h->block_tokens;
  r.max_blocks = h->max_blocks;
  r.n_blocks = h->n_blocks;
  r.stride = h->stride;
  return r;
}

// Resolve the unit list of a call: NULL = all; else validate and upload.
int resolve_units(kvo_handle* h, const int32_t* units, int32_t n_units, cudaStream_t s,
                  const int32_t** dev_units) {
  if (units == nullptr) {
    if (n_units != h->U) return fail(KVO_EINVAL, "units == NULL requires n_units == unit count");
    *dev_units = h->all_units;
    return KVO_OK;
  }
  if (n_units < 1 || n_units > h->U) return fail(KVO_EINVAL, "n_units out of range");
  std::vector<uint8_t> seen((size_t)h->U, 0);
  for (int32_t i = 0; i < n_units; ++i) {
    const int32_t u = units[i];
    if (u < 0 || u >= h->U) return fail(KVO_ERANGE, "unit id out of range");
    if (seen[(size_t)u]) return fail(KVO_EINVAL, "duplicate unit id in list");
    seen[(size_t)u] = 1;
  }
  bool same = (int32_t)h->units_cached.size() == n_units &&
              memcmp(h->units_cached.data(), units, (size_t)n_units * 4) == 0;
  if (!same) {
    h->units_cached.assign(units, units + n_units);
    cudaError_t e = cudaMemcpyAsync(h->units_dev, h->units_cached.data(), (size_t)n_units * 4,
                                    cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "unit list upload");
  }
  *dev_units = h->units_dev;
  return KVO_OK;
}


cudaEvent_t take_event(kvo_handle* h) {
  if (!h->free_events.empty()) {
    cudaEvent_t e = h->free_events.back();
    h->free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Runs one launch, bracketed by events when profiling is on.
template <class F>
cudaError_t timed(kvo_handle* h, int kind, cudaStream_t s, F launch) {
  ++h->launches;
  if (!h->profile || !((h->profile_kinds >> kind) & 1u)) return launch();
  cudaEvent_t e0 = take_event(h), e1 = take_event(h);
  if (e0) cudaEventRecord(e0, s);
  cudaError_t e = launch();
  if (e1) cudaEventRecord(e1, s);
  if (e0 && e1) h->recs.push_back({kind, e0, e1});
  return e;
}

// The unit list of a call, materialised (NULL = all units in order).
std::vector<int32_t> unit_list(const kvo_handle* h, const int32_t* units, int32_t n_units) {
  std::vector<int32_t> v;
  if (units) {
    v.assign(units, units + (n_units > 0 ? n_units : 0));
  } else {
    v.resize((size_t)h->U);
    for (int32_t u = 0; u < h->U; ++u) v[(size_t)u] = u;
  }
  return v;
}

// Completes a deferred fill on stream s: the pending step's miss rows are copied
// into the hot buffer (used when no fetching kvo_attend on the same units follows).
int flush_pending(kvo_handle* h, cudaStream_t s) {
  if (!h->fill_pending) return KVO_OK;
  kvo::GatherArgs ga{};
  ga.units = h->pending_du;
  ga.n = (int32_t)h->pending_units.size();
  ga.row_elems = h->R;
  ga.C = h->C;
  ga.stride = h->stride;
  ga.rows = host_rows_of(h);
  ga.host_pool = h->host_pool_dev;
  ga.hot = h->hot;
  ga.miss_tok = h->miss_tok;
  ga.miss_slot = h->miss_slot;
  ga.miss_cnt = h->miss_cnt;
  ga.pk = h->P * h->k;
  ga.stats = h->stats;
  ga.err = h->err;
  ga.wait_ns = h->wait_ns;
  cudaError_t e = timed(h, KVO_PROF_GATHER, s, [&] { return kvo::launch_flush_fill(ga, s); });
  if (e != cudaSuccess) return cuda_fail(e, "deferred fill");
  h->fill_pending = false;
  return KVO_OK;
}

// Records a step whose fill was deferred.
void set_pending(kvo_handle* h, const int32_t* units, int32_t n_units, const int32_t* du) {
  h->pending_units = unit_list(h, units, n_units);
  h->pending_du = du;
  h->fill_pending = true;
}

int grid_for(int64_t T, int G_max) {
  const int64_t per = 4096;  // fewest tokens worth a CTA
  int64_t g = (T + per - 1) / per;
  if (g < 1) g = 1;
  if (g > G_max) g = G_max;
  return (int)g;
}

// Step path of this call.  Mode 2 measures: the fused launch pays when miss
// rows keep the host link busy for a good part of the step (it overlaps them
// with scoring); with few rows, or long LRU lists that make its one-SM
// finishers slow, the staged launches are faster.  The previous step's row
// bytes come from plan through mapped host memory (one or two steps old).
bool use_fused(kvo_handle* h, const int32_t* units, int32_t n_units) {
  if (h->fused == 0 || !h->fused_ok) return false;
  if (h->fused == 1) return true;
  if (h->C > kFusedDefaultMaxCapacity) return false;
  if (h->pool_bytes > kFusedDefaultMaxPoolBytes) return false;
  if (h->planned_steps < 2 || !h->bytes_prev_host) return true;
  int64_t T = 0;
  for (int32_t i = 0; i < n_units; ++i) T += h->len_host[(size_t)(units ? units[i] : i)];
  const unsigned long long rows = *reinterpret_cast<volatile unsigned long long*>(h->bytes_prev_host);
  return (double)rows >= 0.015 * (double)T * kvo::kKeyBytes;
}

// Staged step of the per-call choice (mode 2): two unit groups, the first group's miss
// rows copied by the first 4/25 of the CTAs of the second group's score launch (24 of 152,
// one per SM) while its other CTAs score, when the previous step's rows were at least 1.5%
// of the key bytes and the call lists enough units for two groups.  The copying CTAs keep
// a fixed unit assignment and start with the launch, on the caller's stream.
constexpr int kSplitMinUnits = 64;
bool use_split(kvo_handle* h, const int32_t* units, int32_t n_units) {
  if (h->fused != 2 || h->groups_set || h->defer_fill || n_units < kSplitMinUnits) return false;
  if (h->planned_steps < 2 || !h->bytes_prev_host) return true;
  int64_t T = 0;
  for (int32_t i = 0; i < n_units; ++i) T += h->len_host[(size_t)(units ? units[i] : i)];
  const unsigned long long rows = *reinterpret_cast<volatile unsigned long long*>(h->bytes_prev_host);
  return (double)rows >= 0.015 * (double)T * kvo::kKeyBytes;
}

// kvo_step as one fused launch (its CTA 0 plans the step).
int fused_step(kvo_handle* h, const int32_t* du, const int32_t* units, int32_t n_units, const void* queries,
               int32_t* topk_tokens, int32_t* topk_slots, float* topk_scores, int32_t* topk_payload,
               int32_t* unit_status, cudaStream_t s) {
  const int PK = h->P * h->k;
  int64_t T = 0, NP = 0;
  for (int32_t i = 0; i < n_units; ++i) {
    const int64_t L = h->len_host[(size_t)(units ? units[i] : i)];
    T += L;
    NP += kvo::pieces_of(i, L, h->piece_tokens);
  }
  if (NP > h->fseg_pieces) return fail(KVO_EINVAL, "more pieces than the segment buffers hold");
  kvo::FusedArgs f{};
  kvo::SelectArgs& sa = f.s;
  sa.keys = h->idx;
  sa.keys8 = h->idx8;
  sa.kscale = h->idxs;
  sa.q8 = h->q8;
  sa.qscale = h->qscale;
  sa.stride = h->stride;
  sa.units = du;
  sa.len = h->len;
  sa.queries = static_cast<const uint16_t*>(queries);
  sa.cache_slots = h->cache_slots;
  sa.n = n_units;
  sa.P = h->P;
  sa.k = h->k;
  sa.cap = h->cap;
  sa.T = T;
  sa.G = 1;
  sa.off = h->off;
  sa.gthr = h->gthr;
  sa.seg_keys = h->fseg_keys;
  sa.seg_cnt = h->fseg_cnt;
  sa.out_tok = topk_tokens;
  sa.out_score = topk_scores;
  sa.out_pay = h->sel_pay;
  sa.out_pay_user = topk_payload;
  sa.err = h->err;
  sa.stats = h->stats;
  sa.wait_ns = h->wait_ns;
  sa.spec = h->spec;
  sa.qn_prev = h->qn_prev;
  sa.qn_cur = h->qn_cur;
  sa.tspec = h->tspec;
  sa.spec_scale = h->speculate > 0 ? (float)h->speculate / 1000.f : 0.f;
  sa.fallback = 0;
  sa.pbeg = h->pbeg;
  sa.pdone = h->pdone;
  sa.ctr = h->ctr;
  sa.status_init = unit_status;
  sa.piece_tokens = h->piece_tokens;
  sa.n_pieces = NP;
  sa.bytes_prev = h->bytes_prev_dev;
  sa.bytes_seen = h->bytes_seen;

  kvo::ResidencyArgs& ra = f.r;
  ra.units = du;
  ra.n = n_units;
  ra.P = h->P;
  ra.k = h->k;
  ra.C = h->C;
  ra.stride = h->stride;
  ra.tok = topk_tokens;
  ra.pay = h->sel_pay;
  ra.cache_slots = h->cache_slots;
  ra.slot_token = h->slot_token;
  ra.last_use = h->last_use;
  ra.stamp = h->stamp;
  ra.out_slot = topk_slots;
  ra.status = unit_status;
  ra.miss_tok = h->miss_tok;
  ra.miss_slot = h->miss_slot;
  ra.miss_cnt = h->miss_cnt;
  ra.err = h->err;
  ra.stats = h->stats;
  ra.len = h->len;
  ra.tok_bits = h->tok_bits;
  ra.tok_words = h->tok_words;
  ra.order = h->order;
  ra.order_par = h->order_par;
  ra.U = h->U;

  kvo::GatherArgs& ga = f.g;
  ga.units = du;
  ga.n = n_units;
  ga.row_elems = h->R;
  ga.C = h->C;
  ga.mode = KVO_GATHER_BULK;
  ga.stride = h->stride;
  ga.rows = host_rows_of(h);
  ga.host_pool = h->host_pool_dev;
  ga.hot = h->hot;
  ga.miss_tok = h->miss_tok;
  ga.miss_slot = h->miss_slot;
  ga.pk = PK;
  ga.stats = h->stats;
  ga.err = h->err;
  ga.wait_ns = h->wait_ns;

  f.chunk_unit = h->chunk_unit;
  f.chunk_start = h->chunk_start;
  f.chunk_cnt = h->chunk_cnt;
  f.chunk_flag = h->chunk_flag;
  f.chunk_cap = h->chunk_cap;
  if (++h->epoch == 0) ++h->epoch;  // 0 marks a never-written chunk
  f.epoch = h->epoch;
  f.n_gather = h->gather_ctas < h->n_sm ? h->gather_ctas : h->n_sm - 1;
  f.smem_bytes = (int)kvo::fused_smem_bytes(h->P, h->k, h->cap, h->int8);
  f.plan_flag = h->plan_flag;
  f.qdone = h->qdone;
  f.defer = h->defer_fill;
  if (f.defer) f.n_gather = 0;  // nothing to fill: every CTA scores

  // the plan runs inside the fused launch (its CTA 0)
  cudaError_t e = timed(h, KVO_PROF_FUSED, s, [&] { return kvo::launch_fused(f, h->n_sm, s); });
  if (e != cudaSuccess) return cuda_fail(e, "fused step launch");
  ++h->host_steps;
  ++h->fused_steps;
  ++h->planned_steps;
  return KVO_OK;
}

}  // namespace

namespace kvo {
void set_last_error(const char* msg) { g_err = msg; }
}  // namespace kvo

namespace kvo {

int set_error(int code, const char* msg) { return fail(code, msg); }
int set_cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }

// Pinned, device-mapped host memory from the driver (cudaHostAlloc); map_bytes
// and huge_page are always 0 (no anonymous mapping of this library's own).
cudaError_t alloc_pinned(size_t bytes, void** out, size_t* map_bytes, size_t* huge_page) {
  *map_bytes = 0;
  *huge_page = 0;
  cudaError_t e = cudaHostAlloc(out, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
  if (e != cudaSuccess) *out = nullptr;
  return e;
}

void free_pinned(void* p, size_t /*map_bytes*/) {
  if (p) cudaFreeHost(p);
}

}  // namespace kvo

extern "C" {

const char* kvo_last_error(void) { return g_err.c_str(); }

int kvo_create(const kvo_config* cfg, kvo_handle** out) {
  if (!out) return fail(KVO_EINVAL, "out is NULL");
  *out = nullptr;
  if (!cfg) return fail(KVO_EINVAL, "cfg is NULL");
  const kvo_config c = *cfg;
  if (c.n_requests < 1 || c.n_layers < 1 || (int64_t)c.n_requests * c.n_layers > (1 << 20))
    return fail(KVO_EINVAL, "n_requests * n_layers must be in [1, 2^20]");
  if (c.max_tokens < 1 || c.max_tokens >= (int64_t)1 << 31) return fail(KVO_EINVAL, "max_tokens out of range");
  if (c.idx_dim != kvo::kDim) return fail(KVO_EINVAL, "idx_dim must be 128");
  if (c.idx_dtype != KVO_IDX_BF16 && c.idx_dtype != KVO_IDX_INT8) return fail(KVO_EINVAL, "bad idx_dtype");
  if (c.row_elems < 8 || c.row_elems > 4096 || c.row_elems % 8)
    return fail(KVO_EINVAL, "row_elems must be a multiple of 8 in [8, 4096]");
  if (c.topk < 1 || c.topk > 4096) return fail(KVO_EINVAL, "topk must be in [1, 4096]");
  if (c.hot_capacity < c.topk || c.hot_capacity > (1 << 24))
    return fail(KVO_EINVAL, "hot_capacity must be in [topk, 2^24]");
  if (c.n_positions < 1 || c.n_positions > 8) return fail(KVO_EINVAL, "n_positions must be in [1, 8]");
  if (c.host_block_tokens < 0 || c.host_block_tokens % 8 || (c.host_block_tokens == 0 && c.host_blocks != 0) ||
      c.host_blocks < 0)
    return fail(KVO_EINVAL, "host_block_tokens must be 0 or a positive multiple of 8 (host_blocks only with it)");
  const int cap = kvo::score_cap_for(c.n_positions, c.topk, c.idx_dtype == KVO_IDX_INT8);
  if (cap == 0) return fail(KVO_EINVAL, "topk too large for n_positions (shared-memory candidate buffer)");
  if (residency_smem_bytes(c.hot_capacity, c.n_positions, c.topk) > 224 * 1024)
    return fail(KVO_EINVAL, "hot_capacity / n_positions * topk too large for the residency kernel");

  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) return fail(KVO_ECUDA, "no CUDA device");
  if (c.device < 0 || c.device >= ndev) return fail(KVO_ECUDA, "device ordinal out of range");
  DeviceGuard guard(c.device);
  if (!guard.ok) return fail(KVO_ECUDA, "cudaSetDevice failed");

  kvo_handle* h = new (std::nothrow) kvo_handle();
  if (!h) return fail(KVO_ENOMEM, "handle");
  h->cfg = c;
  h->device = c.device;
  cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, c.device);
  h->U = c.n_requests * c.n_layers;
  h->C = c.hot_capacity;
  h->P = c.n_positions;
  h->k = c.topk;
  h->R = c.row_elems;
  h->cap = cap;
  h->stride = (c.max_tokens + 7) & ~(int64_t)7;
  h->G_max = h->n_sm;
  h->len_host.assign((size_t)h->U, 0);

  const size_t U = (size_t)h->U, S = (size_t)h->stride, C = (size_t)h->C, PK = (size_t)h->P * h->k;
  size_t pool_rows = U * S;
  if (c.host_block_tokens > 0) {
    h->block_tokens = c.host_block_tokens;
    h->max_blocks = (int32_t)((c.max_tokens + c.host_block_tokens - 1) / c.host_block_tokens);
    h->n_blocks = c.host_blocks > 0 ? c.host_blocks : (int64_t)U * h->max_blocks;
    pool_rows = (size_t)h->n_blocks * (size_t)h->block_tokens;
  }
  h->pool_bytes = pool_rows * h->R * 2;
  cudaError_t e = alloc_host_pool(h, h->pool_bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();  // the failed allocation is not left as this thread's last CUDA error
    delete h;
    return fail(KVO_ENOMEM, std::string("pinned host pool: ") + cudaGetErrorString(e));
  }
  e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->host_pool_dev), h->host_pool, 0);
  const size_t segs = (size_t)h->G_max + U;
  h->int8 = c.idx_dtype == KVO_IDX_INT8;
  if (h->int8) {
    if (e == cudaSuccess) e = dalloc(&h->idx8, U * S * kvo::kDim);
    if (e == cudaSuccess) e = dalloc(&h->idxs, U * S);
    if (e == cudaSuccess) e = dalloc(&h->q8, U * h->P * kvo::kDim);
    if (e == cudaSuccess) e = dalloc(&h->qscale, U * h->P);
    if (e == cudaSuccess) e = dalloc(&h->qdone, 1);
    if (e == cudaSuccess) e = cudaMemset(h->qdone, 0, 4);
  } else if (e == cudaSuccess) {
    e = dalloc(&h->idx, U * S * kvo::kDim);
  }
  if (e == cudaSuccess) e = dalloc(&h->hot, U * C * h->R);
  if (e == cudaSuccess && h->block_tokens > 0) {
    e = dalloc(&h->blocks, U * (size_t)h->max_blocks);
    if (e == cudaSuccess) e = cudaMemset(h->blocks, 0xff, U * (size_t)h->max_blocks * 4);  // all unmapped
  }
  if (e == cudaSuccess) e = dalloc(&h->cache_slots, U * S);
  if (e == cudaSuccess) e = dalloc(&h->slot_token, U * C);
  if (e == cudaSuccess) e = dalloc(&h->last_use, U * C);
  if (e == cudaSuccess) e = dalloc(&h->stamp, U);
  if (e == cudaSuccess) e = dalloc(&h->len, U);
  if (e == cudaSuccess) e = dalloc(&h->all_units, U);
  if (e == cudaSuccess) e = dalloc(&h->units_dev, U);
  if (e == cudaSuccess) e = dalloc(&h->off, U + 1);
  if (e == cudaSuccess) e = dalloc(&h->gthr, U * h->P);
  h->tok_words = (h->stride + 31) / 32;
  if (e == cudaSuccess) e = dalloc(&h->tok_bits, U * (size_t)h->tok_words);
  if (e == cudaSuccess) e = dalloc(&h->order, 2 * U * C);
  if (e == cudaSuccess) e = dalloc(&h->order_par, U);
  if (e == cudaSuccess) e = dalloc(&h->spec, U * h->P);
  if (e == cudaSuccess) e = dalloc(&h->qn_prev, U * h->P);
  if (e == cudaSuccess) e = dalloc(&h->qn_cur, U * h->P);
  if (e == cudaSuccess) e = dalloc(&h->tspec, U * h->P);
  if (e == cudaSuccess) e = dalloc(&h->fb, U);
  if (e == cudaSuccess) e = dalloc(&h->fb_any, 1);
  if (e == cudaSuccess) e = dalloc(&h->seg_keys, segs * PK);
  if (e == cudaSuccess) e = dalloc(&h->seg_cnt, segs * h->P);
  if (e == cudaSuccess) e = dalloc(&h->sel_pay, U * PK);
  if (e == cudaSuccess) e = dalloc(&h->miss_tok, U * PK);
  if (e == cudaSuccess) e = dalloc(&h->miss_slot, U * PK);
  if (e == cudaSuccess) e = dalloc(&h->miss_cnt, U);
  if (e == cudaSuccess) e = dalloc(&h->claim_batches, U);
  if (e == cudaSuccess) e = dalloc(&h->miss_off, U + 16);
  if (e == cudaSuccess) e = dalloc(&h->done_ctr, 16);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming);
  for (int g = 0; g < 16 && e == cudaSuccess; ++g) e = cudaEventCreateWithFlags(&h->ev_group[g], cudaEventDisableTiming);
  if (e == cudaSuccess) e = dalloc(&h->err, 1);
  if (e == cudaSuccess) e = dalloc(&h->stats, 1);
  h->fused_ok = fused_fits(h->P, h->k, h->cap, h->C, h->int8);
  if (e == cudaSuccess && h->fused_ok) e = alloc_fused(h);
  h->fused = h->fused_ok ? 2 : 0;
  if (e == cudaSuccess) e = dalloc(&h->bytes_seen, 1);
  if (e == cudaSuccess) e = cudaMemset(h->bytes_seen, 0, 8);
  if (e == cudaSuccess) {
    e = cudaHostAlloc(reinterpret_cast<void**>(&h->bytes_prev_host), 8, cudaHostAllocMapped);
    if (e == cudaSuccess) {
      *h->bytes_prev_host = 0;
      e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->bytes_prev_dev), h->bytes_prev_host, 0);
    } else {
      h->bytes_prev_host = nullptr;
    }
  }
  if (h->gather_ctas > h->n_sm - 1) h->gather_ctas = h->n_sm - 1;
  if (e != cudaSuccess) {
    free_all(h);
    delete h;
    // A failed cudaMalloc is also recorded as the thread's last CUDA error; left there,
    // the caller's next kernel launch check (this library's or PyTorch's) would report it.
    cudaGetLastError();
    return fail(KVO_ENOMEM, std::string("device allocation: ") + cudaGetErrorString(e));
  }
  // initial state: nothing resident, every slot free, stamps and lengths 0
  e = kvo::launch_fill_i32(h->cache_slots, -1, U * S, 0);
  if (e == cudaSuccess) e = kvo::launch_fill_i32(h->slot_token, -1, U * C, 0);
  if (e == cudaSuccess) e = cudaMemset(h->last_use, 0, U * C * 4);
  if (e == cudaSuccess) e = cudaMemset(h->stamp, 0, U * 4);
  if (e == cudaSuccess) e = cudaMemset(h->tok_bits, 0, U * (size_t)h->tok_words * 4);
  if (e == cudaSuccess) e = kvo::launch_order_init(h->order, h->order_par, h->U, h->C, 0);
  if (e == cudaSuccess) e = cudaMemset(h->spec, 0, U * h->P * 8);
  if (e == cudaSuccess) e = cudaMemset(h->qn_prev, 0, U * h->P * 4);
  if (e == cudaSuccess) e = cudaMemset(h->fb, 0, U * 4);
  if (e == cudaSuccess) e = cudaMemset(h->fb_any, 0, 4);
  if (e == cudaSuccess) e = cudaMemset(h->len, 0, U * 4);
  if (e == cudaSuccess) e = cudaMemset(h->miss_cnt, 0, U * 4);
  if (e == cudaSuccess) e = cudaMemset(h->miss_off, 0, (U + 16) * 8);
  if (e == cudaSuccess) e = cudaMemset(h->done_ctr, 0, 16 * 4);
  if (e == cudaSuccess) e = cudaMemset(h->err, 0, 4);
  if (e == cudaSuccess) e = cudaMemset(h->stats, 0, sizeof(DevStats));
  if (e == cudaSuccess) {
    std::vector<int32_t> ident(U);
    for (size_t u = 0; u < U; ++u) ident[u] = (int32_t)u;
    e = cudaMemcpy(h->all_units, ident.data(), U * 4, cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    free_all(h);
    delete h;
    return cuda_fail(e, "initialisation");
  }
  *out = h;
  g_err.clear();
  return KVO_OK;
}

int kvo_destroy(kvo_handle* h) {
  if (!h) return KVO_OK;
  DeviceGuard guard(h->device);
  cudaDeviceSynchronize();
  free_all(h);
  delete h;
  return KVO_OK;
}

void* kvo_host_rows(kvo_handle* h, int32_t unit) {
  if (!h || unit < 0 || unit >= h->U) return nullptr;
  if (h->block_tokens > 0) {
    fail(KVO_EINVAL, "paged pool: use kvo_host_block");
    return nullptr;
  }
  return h->host_pool + (size_t)unit * h->stride * h->R;
}

void* kvo_host_block(kvo_handle* h, int64_t block) {
  if (!h || h->block_tokens <= 0 || block < 0 || block >= h->n_blocks) {
    fail(KVO_EINVAL, "not a block of a paged pool");
    return nullptr;
  }
  return h->host_pool + (size_t)block * h->block_tokens * h->R;
}

int kvo_set_blocks(kvo_handle* h, int32_t unit, int32_t first_block, int32_t n_blocks, const int32_t* blocks,
                   void* stream) {
  if (!h) return fail(KVO_EINVAL, "handle is NULL");
  if (h->block_tokens <= 0) return fail(KVO_EINVAL, "the host pool is not paged");
  if (unit < 0 || unit >= h->U) return fail(KVO_ERANGE, "unit out of range");
  if (n_blocks < 0 || first_block < 0 || (int64_t)first_block + n_blocks > h->max_blocks)
    return fail(KVO_ERANGE, "block range past the table");
  if (n_blocks == 0) return KVO_OK;
  if (!blocks) return fail(KVO_EINVAL, "blocks is NULL");
  for (int32_t j = 0; j < n_blocks; ++j)
    if (blocks[j] < -1 || (int64_t)blocks[j] >= h->n_blocks) return fail(KVO_EINVAL, "block id out of range");
  DeviceGuard guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // pageable source: the copy is staged before the call returns, so the caller may reuse the array
  cudaError_t e = cudaMemcpyAsync(h->blocks + (size_t)unit * h->max_blocks + first_block, blocks,
                                  (size_t)n_blocks * 4, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "block table upload");
  return KVO_OK;
}

int kvo_prefill(kvo_handle* h, int32_t unit, int64_t n_tokens, const void* idx_keys, void* stream) {
  if (!h) return fail(KVO_EINVAL, "handle is NULL");
  if (unit < 0 || unit >= h->U) return fail(KVO_ERANGE, "unit out of range");
  if (n_tokens < 0 || n_tokens > h->cfg.max_tokens) return fail(KVO_ERANGE, "n_tokens out of range");
  if (h->len_host[(size_t)unit] != 0) return fail(KVO_EINVAL, "prefill needs an empty unit");
  if (n_tokens > 0 && !idx_keys) return fail(KVO_EINVAL, "idx_keys is NULL");
  DeviceGuard guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  const size_t row0 = (size_t)unit * h->stride;
  if (n_tokens > 0 && !h->int8) {
    e = cudaMemcpyAsync(h->idx + row0 * kvo::kDim, idx_keys, (size_t)n_tokens * kvo::kKeyBytes, cudaMemcpyDefault,
                        s);
  } else if (n_tokens > 0) {
    // int8 indexer: the bf16 keys are rotated and quantized on the device
    // (staged through a stream-ordered buffer when they are host memory)
    cudaPointerAttributes at{};
    const bool on_dev = cudaPointerGetAttributes(&at, idx_keys) == cudaSuccess &&
                        (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged);
    cudaGetLastError();
    const uint16_t* src = static_cast<const uint16_t*>(idx_keys);
    void* staging = nullptr;
    if (!on_dev) {
      e = cudaMallocAsync(&staging, (size_t)n_tokens * kvo::kKeyBytes, s);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(staging, idx_keys, (size_t)n_tokens * kvo::kKeyBytes, cudaMemcpyDefault, s);
      src = static_cast<const uint16_t*>(staging);
    }
    if (e == cudaSuccess) e = kvo::launch_quant_keys(src, n_tokens, h->idx8 + row0 * kvo::kDim, h->idxs + row0, s);
    if (staging) {
      const cudaError_t f = cudaFreeAsync(staging, s);
      if (e == cudaSuccess) e = f;
    }
  }
  if (e == cudaSuccess) e = kvo::launch_set_len(h->len, unit, (int32_t)n_tokens, s);
  if (e != cudaSuccess) return cuda_fail(e, "prefill");
  h->len_host[(size_t)unit] = n_tokens;
  return KVO_OK;
}

int kvo_append(kvo_handle* h, const int32_t* units, int32_t n_units, int32_t n_tokens,
               const void* main_rows, const void* idx_keys, void* stream) {
  if (!h) return fail(KVO_EINVAL, "handle is NULL");
  if (n_tokens < 0) return fail(KVO_EINVAL, "n_tokens < 0");
  if (n_tokens > 0 && (!main_rows || !idx_keys)) return fail(KVO_EINVAL, "NULL rows or keys");
  if (!aligned16(main_rows) || !aligned16(idx_keys)) return fail(KVO_EINVAL, "rows/keys not 16-byte aligned");
  DeviceGuard guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // range check before anything is launched
  for (int32_t i = 0; i < n_units; ++i) {
    const int32_t u = units ? units[i] : i;
    if (u < 0 || u >= h->U) return fail(KVO_ERANGE, "unit id out of range");
    if (h->len_host[(size_t)u] + n_tokens > h->cfg.max_tokens)
      return fail(KVO_ERANGE, "append past max_tokens");
  }
  const int32_t* du = nullptr;
  int rc = resolve_units(h, units, n_units, s, &du);
  if (rc != KVO_OK) return rc;
  if (n_tokens == 0) return KVO_OK;
  kvo::AppendArgs a{};
  a.units = du;
  a.n = n_units;
  a.n_tok = n_tokens;
  a.row_elems = h->R;
  a.stride = h->stride;
  a.rows = static_cast<const uint16_t*>(main_rows);
  a.keys = static_cast<const uint16_t*>(idx_keys);
  a.hrows = host_rows_of(h);
  a.host_pool = h->host_pool_dev;
  a.idx = h->idx;
  a.idx8 = h->idx8;
  a.idxs = h->idxs;
  a.len = h->len;
  a.stats = h->stats;
  cudaError_t e = timed(h, KVO_PROF_APPEND, s, [&] { return kvo::launch_append(a, s); });
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  for (int32_t i = 0; i < n_units; ++i) h->len_host[(size_t)(units ? units[i] : i)] += n_tokens;
  return KVO_OK;
}

int kvo_step(kvo_handle* h, const int32_t* units, int32_t n_units, const void* queries,
             int32_t* topk_tokens, int32_t* topk_slots, float* topk_scores, int32_t* topk_payload,
             int32_t* unit_status, void* stream) {
  if (!h) return fail(KVO_EINVAL, "handle is NULL");
  if (!queries || !topk_tokens || !topk_slots || !unit_status) return fail(KVO_EINVAL, "NULL argument");
  if (!aligned16(queries)) return fail(KVO_EINVAL, "queries not 16-byte aligned");
  DeviceGuard guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int rc = flush_pending(h, s);  // a deferred fill no attention call took up
  if (rc != KVO_OK) return rc;
  const int32_t* du = nullptr;
  rc = resolve_units(h, units, n_units, s, &du);
  if (rc != KVO_OK) return rc;
  if (use_fused(h, units, n_units)) {
    rc = fused_step(h, du, units, n_units, queries, topk_tokens, topk_slots, topk_scores, topk_payload,
                    unit_status, s);
    if (rc == KVO_OK && h->defer_fill) set_pending(h, units, n_units, du);
    return rc;
  }
  const int PK = h->P * h->k;
  int NG = h->groups < n_units ? h->groups : n_units;
  int gsm = h->group_gather_sms;
  if (use_split(h, units, n_units)) {
    NG = 2;
    if (!h->group_gather_sms_set) gsm = h->n_sm * 4 / 25 > 0 ? h->n_sm * 4 / 25 : 1;
  }
  if (NG < 1) NG = 1;
  const int g_max = h->score_ctas > 0 && h->score_ctas < h->G_max ? h->score_ctas : h->G_max;
  // split: the score launch of group g > 0 carries the copy of group g-1's rows in its
  // first gsm CTAs (one stream); else each group's copy runs on the side stream
  const bool split = NG > 1 && gsm > 0 && !h->defer_fill;
  const bool side = NG > 1 && !split;
  kvo::GatherArgs ga_prev{};
  bool have_prev = false;
  cudaError_t e = cudaSuccess;
  if (side) {
    e = cudaEventRecord(h->ev_fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->side, h->ev_fork, 0);
  }
  for (int g = 0; g < NG && e == cudaSuccess; ++g) {
    const int b = (int)((int64_t)n_units * g / NG), en = (int)((int64_t)n_units * (g + 1) / NG);
    const int ng = en - b;
    if (ng <= 0) continue;
    int64_t T = 0;
    for (int32_t i = b; i < en; ++i) T += h->len_host[(size_t)(units ? units[i] : i)];
    const size_t ob = (size_t)b * PK;

    kvo::SelectArgs sa{};
    sa.keys = h->idx;
    sa.keys8 = h->idx8;
    sa.kscale = h->idxs;
    sa.q8 = h->q8 ? h->q8 + (size_t)b * h->P * kvo::kDim : nullptr;
    sa.qscale = h->qscale ? h->qscale + (size_t)b * h->P : nullptr;
    sa.stride = h->stride;
    sa.units = du + b;
    sa.len = h->len;
    sa.queries = static_cast<const uint16_t*>(queries) + (size_t)b * h->P * kvo::kDim;
    sa.cache_slots = h->cache_slots;
    sa.n = ng;
    sa.P = h->P;
    sa.k = h->k;
    sa.cap = h->cap;
    sa.T = T;
    const bool carry = split && have_prev;  // this launch also copies the previous group's rows
    sa.G = grid_for(T, carry && g_max > h->n_sm - gsm ? h->n_sm - gsm : g_max);
    if (carry) {
      sa.gather_ctas = gsm;
      sa.prev = ga_prev;
      have_prev = false;
      // the batch counters the copying and helping CTAs claim from start at zero
      e = cudaMemsetAsync(ga_prev.claim, 0, (size_t)ga_prev.n * sizeof(int32_t), s);
    }
    sa.off = h->off;
    sa.gthr = h->gthr;
    sa.seg_keys = h->seg_keys;
    sa.seg_cnt = h->seg_cnt;
    sa.out_tok = topk_tokens + ob;
    sa.out_score = topk_scores ? topk_scores + ob : nullptr;
    sa.out_pay = h->sel_pay + ob;
    sa.out_pay_user = topk_payload ? topk_payload + ob : nullptr;
    sa.err = h->err;
    sa.stats = h->stats;
    sa.wait_ns = h->wait_ns;
    const bool spec_on = h->speculate > 0;
    sa.spec = h->spec;
    sa.qn_prev = h->qn_prev;
    sa.qn_cur = h->qn_cur + (size_t)b * h->P;
    sa.tspec = h->tspec + (size_t)b * h->P;
    sa.fb = h->fb + b;
    sa.fb_any = h->fb_any;
    sa.spec_scale = spec_on ? (float)h->speculate / 1000.f : 0.f;
    sa.fallback = 0;
    if (g == 0) {
      sa.bytes_prev = h->bytes_prev_dev;
      sa.bytes_seen = h->bytes_seen;
    }
    if (sa.q8 && e == cudaSuccess)  // int8 indexer: this group's queries, one warp each
      e = timed(h, KVO_PROF_PLAN, s, [&] {
        return kvo::launch_quant_keys(sa.queries, (int64_t)ng * h->P, sa.q8, sa.qscale, s);
      });
    if (e == cudaSuccess) e = timed(h, KVO_PROF_PLAN, s, [&] { return kvo::launch_plan(sa, s); });
    if (e == cudaSuccess) e = timed(h, KVO_PROF_SCORE, s, [&] { return kvo::launch_score(sa, s); });
    if (e == cudaSuccess) e = timed(h, KVO_PROF_SELECT, s, [&] { return kvo::launch_select(sa, s); });
    if (spec_on) {
      // units whose speculative threshold was too high are rescored exactly
      kvo::SelectArgs fa = sa;
      fa.fallback = 1;
      fa.gather_ctas = 0;
      if (e == cudaSuccess) e = timed(h, KVO_PROF_RESCORE, s, [&] { return kvo::launch_score(fa, s); });
      if (e == cudaSuccess) e = timed(h, KVO_PROF_RESELECT, s, [&] { return kvo::launch_select(fa, s); });
    }

    kvo::ResidencyArgs ra{};
    ra.units = du + b;
    ra.n = ng;
    ra.P = h->P;
    ra.k = h->k;
    ra.C = h->C;
    ra.stride = h->stride;
    ra.tok = topk_tokens + ob;
    ra.pay = h->sel_pay + ob;
    ra.cache_slots = h->cache_slots;
    ra.slot_token = h->slot_token;
    ra.last_use = h->last_use;
    ra.stamp = h->stamp;
    ra.out_slot = topk_slots + ob;
    ra.status = unit_status + b;
    ra.miss_tok = h->miss_tok + ob;
    ra.miss_slot = h->miss_slot + ob;
    ra.miss_cnt = h->miss_cnt + b;
    ra.miss_off = h->miss_off + b + g;
    ra.done_ctr = h->done_ctr + g;
    ra.err = h->err;
    ra.stats = h->stats;
    ra.len = h->len;
    ra.tok_bits = h->tok_bits;
    ra.tok_words = h->tok_words;
    ra.order = h->order;
    ra.order_par = h->order_par;
    ra.U = h->U;
    if (e == cudaSuccess) e = timed(h, KVO_PROF_RESIDENCY, s, [&] { return kvo::launch_residency(ra, s); });

    kvo::GatherArgs ga{};
    ga.units = du + b;
    ga.n = ng;
    ga.row_elems = h->R;
    ga.C = h->C;
    ga.mode = h->gather_mode;
    ga.stride = h->stride;
    ga.rows = host_rows_of(h);
    ga.host_pool = h->host_pool_dev;
    ga.hot = h->hot;
    ga.miss_tok = h->miss_tok + ob;
    ga.miss_slot = h->miss_slot + ob;
    ga.miss_off = h->miss_off + b + g;
    ga.pk = PK;
    ga.stats = h->stats;
    ga.err = h->err;
    ga.wait_ns = h->wait_ns;
    if (h->defer_fill) {
      // the rows are left for the attention call (or the next call's flush)
    } else if (split && en < n_units) {
      ga_prev = ga;  // copied by the next group's score launch
      ga_prev.claim = h->claim_batches + b;
      have_prev = true;
    } else if (side) {
      if (e == cudaSuccess) e = cudaEventRecord(h->ev_group[g], s);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(h->side, h->ev_group[g], 0);
      if (e == cudaSuccess)
        e = timed(h, KVO_PROF_GATHER, h->side, [&] { return kvo::launch_gather(ga, h->n_sm, h->side); });
    } else if (e == cudaSuccess) {
      e = timed(h, KVO_PROF_GATHER, s, [&] { return kvo::launch_gather(ga, h->n_sm, s); });
    }
  }
  if (side && e == cudaSuccess) {
    e = cudaEventRecord(h->ev_join, h->side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h->ev_join, 0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "step launch");
  ++h->host_steps;
  ++h->planned_steps;
  if (split) ++h->split_steps;
  if (h->defer_fill) set_pending(h, units, n_units, du);
  return KVO_OK;
}

size_t kvo_select_workspace_size(int32_t n_units, int32_t n_pos, int32_t k, int32_t device) {
  int n_sm = 0;
  if (n_units < 1 || n_pos < 1 || k < 1) return 0;
  if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t n = (size_t)n_units, PK = (size_t)n_pos * k, segs = (size_t)n_sm + n;
  return up(n * 4) * 2 + up((n + 1) * 8) + up(n * n_pos * 8) + up(segs * PK * 8) + up(segs * n_pos * 4) +
         up(n * PK * 4) + up(4);
}

int kvo_select(const void* keys, int64_t unit_stride, const int32_t* cache_slots,
               const int64_t* lengths, int32_t n_units, int32_t n_pos, int32_t k,
               const void* queries, int32_t* tokens, float* scores, int32_t* payload,
               void* workspace, size_t workspace_bytes, uint32_t* status, void* stream) {
  if (!keys || !lengths || !queries || !tokens || !workspace) return fail(KVO_EINVAL, "NULL argument");
  if (reinterpret_cast<uintptr_t>(status) & 3u) return fail(KVO_EINVAL, "status not 4-byte aligned");
  if (n_units < 1 || n_pos < 1 || n_pos > 8 || k < 1 || k > 4096) return fail(KVO_EINVAL, "size out of range");
  if (unit_stride < 1 || unit_stride >= (int64_t)1 << 31) return fail(KVO_EINVAL, "unit_stride out of range");
  if (!aligned16(keys) || !aligned16(queries)) return fail(KVO_EINVAL, "keys/queries not 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return fail(KVO_EINVAL, "workspace not 256-byte aligned");
  const int cap = kvo::score_cap_for(n_pos, k, false);
  if (cap == 0) return fail(KVO_EINVAL, "k too large for n_pos");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(KVO_ECUDA, "no current device");
  const size_t need = kvo_select_workspace_size(n_units, n_pos, k, dev);
  if (need == 0 || workspace_bytes < need) return fail(KVO_EINVAL, "workspace too small");
  std::vector<int32_t> host(2 * (size_t)n_units);
  int64_t T = 0;
  for (int32_t i = 0; i < n_units; ++i) {
    if (lengths[i] < 0 || lengths[i] > unit_stride) return fail(KVO_EINVAL, "length out of range");
    host[i] = i;
    host[n_units + i] = (int32_t)lengths[i];
    T += lengths[i];
  }
  int n_sm = 0;
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t n = (size_t)n_units, PK = (size_t)n_pos * k, segs = (size_t)n_sm + n;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  int32_t* d_units = reinterpret_cast<int32_t*>(w); w += up(n * 4);
  int32_t* d_len = reinterpret_cast<int32_t*>(w); w += up(n * 4);
  int64_t* d_off = reinterpret_cast<int64_t*>(w); w += up((n + 1) * 8);
  uint64_t* d_gthr = reinterpret_cast<uint64_t*>(w); w += up(n * n_pos * 8);
  uint64_t* d_seg_keys = reinterpret_cast<uint64_t*>(w); w += up(segs * PK * 8);
  int32_t* d_seg_cnt = reinterpret_cast<int32_t*>(w); w += up(segs * n_pos * 4);
  int32_t* d_pay = reinterpret_cast<int32_t*>(w); w += up(n * PK * 4);
  uint32_t* d_err = status ? status : reinterpret_cast<uint32_t*>(w);  // the caller's word when given
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(d_units, host.data(), n * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(d_len, host.data() + n, n * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(d_err, 0, 4, s);
  if (e != cudaSuccess) return cuda_fail(e, "select set-up");
  kvo::SelectArgs sa{};
  sa.keys = static_cast<const uint16_t*>(keys);
  sa.stride = unit_stride;
  sa.units = d_units;
  sa.len = d_len;
  sa.queries = static_cast<const uint16_t*>(queries);
  sa.cache_slots = cache_slots;
  sa.n = n_units;
  sa.P = n_pos;
  sa.k = k;
  sa.cap = cap;
  sa.T = T;
  sa.G = grid_for(T, n_sm);
  sa.off = d_off;
  sa.gthr = d_gthr;
  sa.seg_keys = d_seg_keys;
  sa.seg_cnt = d_seg_cnt;
  sa.out_tok = tokens;
  sa.out_score = scores;
  sa.out_pay = payload ? payload : d_pay;
  sa.out_pay_user = nullptr;
  sa.err = d_err;
  sa.stats = nullptr;
  sa.wait_ns = 2000000000ull;
  e = kvo::launch_plan(sa, s);
  if (e == cudaSuccess) e = kvo::launch_score(sa, s);
  if (e == cudaSuccess) e = kvo::launch_select(sa, s);
  if (e != cudaSuccess) return cuda_fail(e, "select launch");
  return KVO_OK;
}

int kvo_set_option(kvo_handle* h, int32_t key, int64_t value) {
  if (!h) return fail(KVO_EINVAL, "handle is NULL");
  switch (key) {
    case KVO_OPT_GATHER_MODE:
      if (value != KVO_GATHER_LDG && value != KVO_GATHER_BULK) return fail(KVO_EINVAL, "bad gather mode");
      h->gather_mode = (int)value;
      return KVO_OK;
    case KVO_OPT_PROFILE:
      if (value != 0 && value != 1) return fail(KVO_EINVAL, "profile is 0 or 1");
      h->profile = value == 1;
      return KVO_OK;
    case KVO_OPT_PROFILE_KINDS:
      if (value < 1 || value >= (1 << KVO_PROF_KINDS)) return fail(KVO_EINVAL, "profile kinds: a non-empty mask of KVO_PROF_*");
      h->profile_kinds = (uint32_t)value;
      return KVO_OK;
    case KVO_OPT_GROUPS:
      if (value < 1 || value > 16) return fail(KVO_EINVAL, "groups must be in [1, 16]");
      h->groups = (int)value;
      h->groups_set = true;
      return KVO_OK;
    case KVO_OPT_GROUP_GATHER_SMS:
      if (value < 0 || value > h->n_sm / 2) return fail(KVO_EINVAL, "group_gather_sms must be in [0, SMs/2]");
      h->group_gather_sms = (int)value;
      h->group_gather_sms_set = true;
      return KVO_OK;
    case KVO_OPT_SCORE_CTAS:
      if (value < 0 || value > 1 << 20) return fail(KVO_EINVAL, "score_ctas out of range");
      h->score_ctas = (int)value;
      return KVO_OK;
    case KVO_OPT_SPECULATE:
      if (value < 0 || value > 1000) return fail(KVO_EINVAL, "speculate must be in [0, 1000]");
      h->speculate = (int)value;
      return KVO_OK;
    case KVO_OPT_FUSED:
      if (value < 0 || value > 2) return fail(KVO_EINVAL, "fused is 0, 1 or 2");
      if (value != 0 && !h->fused_ok) return fail(KVO_EINVAL, "configuration does not fit the fused step");
      h->fused = (int)value;
      return KVO_OK;
    case KVO_OPT_GATHER_CTAS:
      if (value < 0 || value > h->n_sm - 1) return fail(KVO_EINVAL, "gather_ctas must be in [0, SMs-1]");
      h->gather_ctas = (int)value;
      return KVO_OK;
    case KVO_OPT_PIECE_TOKENS: {
      if (value < kvo::kDim || value > (1 << 20) || value % 128) return fail(KVO_EINVAL, "bad piece_tokens");
      if (!h->fused_ok) return fail(KVO_EINVAL, "configuration does not fit the fused step");
      DeviceGuard guard(h->device);
      cudaError_t e = cudaDeviceSynchronize();
      if (e != cudaSuccess) return cuda_fail(e, "piece_tokens");
      h->piece_tokens = (int)value;
      e = alloc_fused_segments(h);
      if (e != cudaSuccess) {
        cudaGetLastError();  // as in kvo_create: not left as the thread's last CUDA error
        return fail(KVO_ENOMEM, std::string("piece segments: ") + cudaGetErrorString(e));
      }
      return KVO_OK;
    }
    case KVO_OPT_HOST_HUGE_PAGE:
      return fail(KVO_EINVAL, "read-only option");
    case KVO_OPT_DEFER_FILL: {
      if (value != 0 && value != 1) return fail(KVO_EINVAL, "defer_fill is 0 or 1");
      if (value == 1 && h->R != 576) return fail(KVO_EINVAL, "defer_fill needs the attention row (576 elements)");
      if (value == 1 && !h->claim) {
        DeviceGuard guard(h->device);
        const size_t n = (size_t)h->U * (size_t)h->C * 3;
        cudaError_t e = dalloc(&h->claim, n);
        if (e == cudaSuccess) e = cudaMemset(h->claim, 0, n * 4);
        if (e != cudaSuccess) {
          if (h->claim) cudaFree(h->claim);
          h->claim = nullptr;
          cudaGetLastError();  // as in kvo_create: not left as the thread's last CUDA error
          return fail(KVO_ENOMEM, std::string("claim words: ") + cudaGetErrorString(e));
        }
        h->fetch_epoch = 0;
      }
      h->defer_fill = (int)value;
      return KVO_OK;
    }
    case KVO_OPT_WAIT_LIMIT_NS:
      if (value < 1000) return fail(KVO_EINVAL, "wait limit below 1 us");
      h->wait_ns = (uint64_t)value;
      return KVO_OK;
    default:
      return fail(KVO_EINVAL, "unknown option");
  }
}

int kvo_get_option(kvo_handle* h, int32_t key, int64_t* value) {
  if (!h || !value) return fail(KVO_EINVAL, "NULL argument");
  switch (key) {
    case KVO_OPT_GATHER_MODE: *value = h->gather_mode; return KVO_OK;
    case KVO_OPT_WAIT_LIMIT_NS: *value = (int64_t)h->wait_ns; return KVO_OK;
    case KVO_OPT_PROFILE: *value = h->profile ? 1 : 0; return KVO_OK;
    case KVO_OPT_PROFILE_KINDS: *value = h->profile_kinds; return KVO_OK;
    case KVO_OPT_GROUPS: *value = h->groups; return KVO_OK;
    case KVO_OPT_GROUP_GATHER_SMS: *value = h->group_gather_sms; return KVO_OK;
    case KVO_OPT_SCORE_CTAS: *value = h->score_ctas; return KVO_OK;
    case KVO_OPT_SPECULATE: *value = h->speculate; return KVO_OK;
    case KVO_OPT_FUSED: *value = h->fused; return KVO_OK;
    case KVO_OPT_GATHER_CTAS: *value = h->gather_ctas; return KVO_OK;
    case KVO_OPT_PIECE_TOKENS: *value = h->piece_tokens; return KVO_OK;
    case KVO_OPT_HOST_HUGE_PAGE: *value = (int64_t)h->pool_huge_page; return KVO_OK;
    case KVO_OPT_DEFER_FILL: *value = h->defer_fill; return KVO_OK;
    default: return fail(KVO_EINVAL, "unknown option");
  }
}

int kvo_reset(kvo_handle* h, const int32_t* units, int32_t n_units, int64_t keep_tokens, void* stream) {
  if (!h) return fail(KVO_EINVAL, "handle is NULL");
  if (keep_tokens < 0) return fail(KVO_EINVAL, "keep_tokens < 0");
  DeviceGuard guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int32_t i = 0; i < n_units; ++i) {
    const int32_t u = units ? units[i] : i;
    if (u < 0 || u >= h->U) return fail(KVO_ERANGE, "unit id out of range");
    if (h->len_host[(size_t)u] < keep_tokens) return fail(KVO_ERANGE, "keep_tokens beyond a unit's length");
  }
  int rc = flush_pending(h, s);
  if (rc != KVO_OK) return rc;
  const int32_t* du = nullptr;
  rc = resolve_units(h, units, n_units, s, &du);
  if (rc != KVO_OK) return rc;
  kvo::ResetArgs a{};
  a.units = du;
  a.n = n_units;
  a.keep = (int32_t)keep_tokens;
  a.stride = h->stride;
  a.C = h->C;
  a.cache_slots = h->cache_slots;
  a.slot_token = h->slot_token;
  a.last_use = h->last_use;
  a.stamp = h->stamp;
  a.len = h->len;
  a.P = h->P;
  a.spec = h->spec;
  a.qn_prev = h->qn_prev;
  a.order = h->order;
  a.order_par = h->order_par;
  cudaError_t e = timed(h, KVO_PROF_RESET, s, [&] { return kvo::launch_reset(a, s); });
  if (e != cudaSuccess) return cuda_fail(e, "reset launch");
  for (int32_t i = 0; i < n_units; ++i) h->len_host[(size_t)(units ? units[i] : i)] = keep_tokens;
  return KVO_OK;
}

int kvo_attend(kvo_handle* h, const int32_t* units, int32_t n_units, const void* queries, int32_t n_heads,
               float scale, const int32_t* topk_slots, void* out, float* lse, void* stream) {
  if (!h) return fail(KVO_EINVAL, "handle is NULL");
  if (!queries || !topk_slots || !out) return fail(KVO_EINVAL, "NULL argument");
  if (!aligned16(queries) || !aligned16(out)) return fail(KVO_EINVAL, "queries or out not 16-byte aligned");
  if (h->R != 576) return fail(KVO_EINVAL, "attention needs 576-element rows");
  if (n_heads < 128 || n_heads % 128 != 0 || n_heads > 8192)
    return fail(KVO_EINVAL, "n_heads must be a positive multiple of 128 (at most 8192)");
  if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return fail(KVO_EINVAL, "scale is not finite");
  DeviceGuard guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // After a deferred step on the same units, the attention kernel fills the
  // step's miss rows itself; any other unit list completes the fill first.
  bool fetch = false;
  if (h->fill_pending) {
    fetch = unit_list(h, units, n_units) == h->pending_units;
    if (!fetch) {
      const int rf = flush_pending(h, s);
      if (rf != KVO_OK) return rf;
    }
  }
  const int32_t* du = nullptr;
  int rc = resolve_units(h, units, n_units, s, &du);
  if (rc != KVO_OK) return rc;
  kvo::AttendArgs a{};
  if (fetch) {
    if (h->fetch_epoch >= 0x7ffffff0u) {  // 2e + 1 must stay below 2^32: start the claim words again
      cudaError_t ez = cudaMemsetAsync(h->claim, 0, (size_t)h->U * h->C * 3 * 4, s);
      if (ez != cudaSuccess) return cuda_fail(ez, "claim words");
      h->fetch_epoch = 0;
    }
    a.pay = h->sel_pay;
    a.host_pool = h->host_pool_dev;
    a.hrows = host_rows_of(h);
    a.hot_w = h->hot;
    a.claim = h->claim;
    a.epoch = ++h->fetch_epoch;
    const int pairs = h->n_sm / 2, per_unit = h->P * (n_heads / 128);
    a.group = pairs / per_unit > 0 ? pairs / per_unit : 1;
    a.stats = h->stats;
  }
  a.units = du;
  a.slots = topk_slots;
  a.q = static_cast<const uint16_t*>(queries);
  a.hot = h->hot;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.n = n_units;
  a.P = h->P;
  a.k = h->k;
  a.H = n_heads;
  a.C = h->C;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.err = h->err;
  a.wait_ns = h->wait_ns;
  cudaError_t e = timed(h, KVO_PROF_ATTEND, s, [&] { return kvo::launch_attend(a, s); });
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  if (fetch) h->fill_pending = false;
  return KVO_OK;
}

int kvo_wait_selftest(int32_t device, int64_t limit_ns, int64_t* waited_ns) {
  if (limit_ns < 1000 || limit_ns > 10000000000ll) return fail(KVO_EINVAL, "limit_ns must be in [1 us, 10 s]");
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return fail(KVO_ECUDA, "no such device");
  DeviceGuard guard(device);
  unsigned long long out[3] = {0, 0, 0};
  cudaError_t e = kvo::run_wait_selftest((uint64_t)limit_ns, out);
  if (e != cudaSuccess) return cuda_fail(e, "wait self-test");
  if (waited_ns) *waited_ns = (int64_t)out[2];
  if (out[0] == 1 && out[1] == 1) return fail(KVO_ETIMEOUT, "both bounded waits expired, as designed");
  return fail(KVO_ECUDA, "a wait on a condition nothing satisfies reported success");
}

int kvo_profile_read(kvo_handle* h, double* ms, uint64_t* launches, int32_t n_kinds) {
  if (!h || !ms || !launches || n_kinds < 0) return fail(KVO_EINVAL, "NULL argument");
  DeviceGuard guard(h->device);
  for (auto& r : h->recs) {
    float t = 0.f;
    cudaError_t e = cudaEventSynchronize(r.e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.e0, r.e1);
    if (e != cudaSuccess) return cuda_fail(e, "profile events");
    if (r.kind < n_kinds && r.kind < KVO_PROF_KINDS) {
      ms[r.kind] += t;
      launches[r.kind] += 1;
    }
    h->free_events.push_back(r.e0);
    h->free_events.push_back(r.e1);
  }
  h->recs.clear();
  return KVO_OK;
}

int kvo_get_stats(kvo_handle* h, kvo_stats* out) {
  if (!h || !out) return fail(KVO_EINVAL, "NULL argument");
  DeviceGuard guard(h->device);
  cudaError_t e = cudaDeviceSynchronize();
  DevStats d{};
  uint32_t err = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&d, h->stats, sizeof(d), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&err, h->err, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "stats");
  out->steps = h->host_steps;
  out->unit_steps = d.unit_steps;
  out->capacity_errors = d.capacity_errors;
  out->hits = d.hits;
  out->misses = d.misses;
  out->rows_h2d = d.rows_h2d;
  out->bytes_h2d = d.bytes_h2d;
  out->rows_d2h = d.rows_d2h;
  out->bytes_d2h = d.bytes_d2h;
  out->timeouts = (err & kvo::kErrTimeout) ? 1 : 0;
  out->rescored = d.rescored;
  out->fused_steps = h->fused_steps;
  out->block_errors = d.block_errors;
  out->fetch_dup_bytes = d.fetch_dup_bytes;
  out->split_steps = h->split_steps;
  out->launches = h->launches;
  out->rows_h2d_in_score = d.rows_h2d_in_score;
  return KVO_OK;
}

int kvo_export_state(kvo_handle* h, int32_t unit, int32_t* cache_slots, int32_t* slot_token,
                     uint32_t* last_use, int64_t* length, uint32_t* stamp, void* hot_rows) {
  if (!h) return fail(KVO_EINVAL, "handle is NULL");
  if (unit < 0 || unit >= h->U) return fail(KVO_ERANGE, "unit out of range");
  DeviceGuard guard(h->device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess && h->fill_pending) {  // the state is exported complete
    const int rf = flush_pending(h, 0);
    if (rf != KVO_OK) return rf;
    e = cudaDeviceSynchronize();
  }
  const size_t S = (size_t)h->stride, C = (size_t)h->C;
  if (e == cudaSuccess && cache_slots)
    e = cudaMemcpy(cache_slots, h->cache_slots + unit * S, (size_t)h->cfg.max_tokens * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && slot_token)
    e = cudaMemcpy(slot_token, h->slot_token + unit * C, C * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && last_use)
    e = cudaMemcpy(last_use, h->last_use + unit * C, C * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && stamp) e = cudaMemcpy(stamp, h->stamp + unit, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && hot_rows)
    e = cudaMemcpy(hot_rows, h->hot + unit * C * h->R, C * h->R * 2, cudaMemcpyDeviceToHost);
  int32_t dlen = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&dlen, h->len + unit, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "export");
  if (length) *length = dlen;
  return KVO_OK;
}

}  // extern "C"
