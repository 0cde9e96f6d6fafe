// Internal declarations shared by the kernels of libkvo (sm_103a only).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvo.h"

namespace kvo {

constexpr int kDim = 128;            // indexer dimension
constexpr int kKeyBytes = kDim * 2;  // one indexer key row
constexpr uint32_t kFull = 0xffffffffu;

// Error bits of the sticky device error word.
constexpr uint32_t kErrTimeout = 1u;
constexpr uint32_t kErrPlan = 2u;

// Device-side counters (mirrors kvo_stats).
struct DevStats {
  unsigned long long steps, unit_steps, capacity_errors, hits, misses, rows_h2d, bytes_h2d,
      rows_d2h, bytes_d2h, timeouts, rescored, block_errors, fetch_dup_bytes,
      rows_h2d_in_score;  // of rows_h2d: copied by the first CTAs of a score launch
};

// Host-pool row of token t of unit u: contiguous per unit (blocks == nullptr),
// or row t mod B of physical block blocks[u][t / B] of a paged pool.  Returns
// -1 for a row of an unmapped block (or a block id out of range).
struct HostRows {
  const int32_t* blocks;  // [U][max_blocks] block tables, or nullptr
  int32_t block_tokens, max_blocks;
  int64_t n_blocks;
  int64_t stride;         // rows per unit when contiguous
};
__device__ __forceinline__ int64_t host_row(const HostRows& h, int64_t u, int64_t t) {
  if (!h.blocks) return u * h.stride + t;
  const int32_t b = __ldg(h.blocks + u * h.max_blocks + t / h.block_tokens);
  if (b < 0 || (int64_t)b >= h.n_blocks) return -1;
  return (int64_t)b * h.block_tokens + t % h.block_tokens;
}

// ---------------------------------------------------------------------------
// Ordering keys.  A selection key is larger for a better candidate: the fp32
// score mapped to an order-preserving unsigned word in the high half, the
// bitwise complement of the token in the low half (lower token wins a tie).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_bits(float f) {
  uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float unorder_bits(uint32_t k) {
  uint32_t b = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(b);
}
__device__ __forceinline__ uint64_t sel_key(float s, uint32_t t) {
  return ((uint64_t)order_bits(s) << 32) | (uint64_t)(~t);
}
__device__ __forceinline__ uint32_t key_token(uint64_t key) { return ~(uint32_t)key; }
__device__ __forceinline__ float key_score(uint64_t key) { return unorder_bits((uint32_t)(key >> 32)); }

// bf16 pair (packed in a 32-bit word) -> two exact fp32 values.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ---------------------------------------------------------------------------
// mbarrier + bulk async copy (inline PTX)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on a phase parity.  Returns false when limit_ns elapsed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0 && global_ns() - t0 > limit_ns) return false;
  }
}
// 1-D bulk copy global -> shared; completion counted in bytes on bar.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// L2 policy for data read or written once per step (the indexer key stream,
// miss rows): evicted first, so that per-unit state stays in L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
// 1-D bulk copy shared -> global with an L2 cache policy.
__device__ __forceinline__ void bulk_s2g_hint(void* dst, const void* src, uint32_t bytes, uint64_t pol) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
               "r"(smem_u32(src)), "r"(bytes), "l"(pol)
               : "memory");
}
// 1-D bulk copy shared -> global, tracked by the issuing thread's bulk group.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Named barrier among the first n_threads threads of the block (id 1..15).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t n_threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n_threads) : "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Upper bound search: largest i in [0, n) with off[i] <= x (off non-decreasing).
__device__ __forceinline__ int find_segment(const int64_t* off, int n, int64_t x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// CTA of the flat partition [floor(c*T/G), floor((c+1)*T/G)) holding token x.
__device__ __forceinline__ int cta_of(int64_t x, int64_t T, int G) {
  return (int)(((x + 1) * (int64_t)G - 1) / T);
}
__device__ __forceinline__ int64_t cta_start(int c, int64_t T, int G) {
  return ((int64_t)c * T) / G;
}

// ---------------------------------------------------------------------------
// Launch-side structures
// ---------------------------------------------------------------------------
struct GatherArgs {
  const int32_t* units;
  int32_t n, row_elems, C, mode;
  int64_t stride;              // host pool rows per unit
  HostRows rows;               // token -> host-pool row
  const uint16_t* host_pool;   // device-visible address of the pinned pool
  uint16_t* hot;               // [U][C][row_elems]
  const int32_t* miss_tok;
  const int32_t* miss_slot;
  const int64_t* miss_off;     // [n+1]
  const int32_t* miss_cnt;     // [n] (the deferred fill's flush)
  int32_t pk;                  // stride of the miss lists
  int32_t* claim;              // [n] batches claimed per unit (zero before the launch), or nullptr
  DevStats* stats;
  uint32_t* err;
  uint64_t wait_ns;
};

struct SelectArgs {
  const uint16_t* keys;        // bf16 [.][stride][128], unit id major (bf16 indexer)
  const int8_t* keys8;         // int8 [.][stride][128] codes (int8 indexer), else nullptr
  const uint16_t* kscale;      // fp16 [.][stride] key scales (int8 indexer)
  int8_t* q8;                  // [n][P][128] query codes of this step (int8 indexer)
  uint16_t* qscale;            // [n][P] their fp16 scales
  int64_t stride;              // token stride between units
  const int32_t* units;        // [n] unit ids (device)
  const int32_t* len;          // device lengths indexed by unit id
  const uint16_t* queries;     // [n][P][128]
  const int32_t* cache_slots;  // [.][stride] or nullptr
  int32_t n, P, k, cap;        // cap: candidate buffer entries per position
  int64_t T;                   // total cached tokens of the listed units
  int32_t G;                   // score CTAs
  // Separate score launch of a staged step in unit groups (0: none): the first
  // gather_ctas CTAs of the launch copy the miss rows of the previous group
  // (prev) instead of scoring; the G scoring CTAs follow them.
  int32_t gather_ctas;
  GatherArgs prev;
  int64_t* off;                // [n+1] flat offsets (scratch, written by plan)
  uint64_t* gthr;              // [n][P] shared lower bounds of each k-th best key (zeroed by plan)
  uint64_t* seg_keys;          // [(G+n)][P][k] candidates per segment
  int32_t* seg_cnt;            // [(G+n)][P]
  int32_t* out_tok;            // [n][P][k]
  float* out_score;            // nullable
  int32_t* out_pay;            // [n][P][k] (internal copy, may equal user payload)
  int32_t* out_pay_user;       // nullable, second destination
  uint32_t* err;               // sticky error word
  DevStats* stats;             // nullable
  uint64_t wait_ns;
  // Speculative thresholds (all nullable: off).  spec[u][p] is the k-th best
  // key of unit u's last step and qn_prev[u][p] that step's squared query
  // norm; plan turns them into tspec[i][p] for this step, select verifies the
  // result is exact and flags units to rescore (fb, fb_any) otherwise.
  uint64_t* spec;
  float* qn_prev;
  float* qn_cur;
  uint64_t* tspec;
  int32_t* fb;
  uint32_t* fb_any;
  float spec_scale;            // threshold = previous k-th score * norm ratio * spec_scale
  int32_t fallback;            // 1: rescoring pass over the flagged units, no speculation
  // Fused step only (all nullable: off).  Unit i's tokens are cut into
  // max(1, ceil(len / piece_tokens)) pieces numbered unit-major from pbeg[i];
  // plan writes pbeg, zeroes pdone and the work counters, and marks every
  // status KVO_ETIMEOUT until the unit's finisher overwrites it.
  int64_t* pbeg;               // [n+1]
  int32_t* pdone;              // [n] pieces of the unit completed
  unsigned long long* ctr;     // [4] work counters of the fused step
  int32_t* status_init;        // [n]
  int32_t piece_tokens;        // multiple of the 128-token tile
  int64_t n_pieces;            // pbeg[n], checked by plan
  // Miss-row bytes of the previous step for the host's choice of step path
  // (nullable): plan writes stats->bytes_h2d - *bytes_seen to *bytes_prev
  // (mapped host memory) and stores the total in *bytes_seen.
  unsigned long long* bytes_prev;
  unsigned long long* bytes_seen;
};

struct ResidencyArgs {
  const int32_t* units;
  int32_t n, P, k, C;
  int64_t stride;              // cache_slots stride per unit
  const int32_t* tok;          // [n][P][k]
  const int32_t* pay;          // [n][P][k]
  int32_t* cache_slots;        // [U][stride]
  int32_t* slot_token;         // [U][C]
  uint32_t* last_use;          // [U][C]
  uint32_t* stamp;             // [U]
  int32_t* out_slot;           // [n][P][k]
  int32_t* status;             // [n]
  int32_t* miss_tok;           // [n][P*k]
  int32_t* miss_slot;          // [n][P*k]
  int32_t* miss_cnt;           // [n]
  int64_t* miss_off;           // [n+1]
  uint32_t* done_ctr;          // last-block counter (self-resetting)
  uint32_t* err;
  DevStats* stats;
  const int32_t* len;          // [U] cached tokens
  uint32_t* tok_bits;          // [U][tok_words] token bitmap scratch (all zero between calls)
  int64_t tok_words;
  int32_t* order;              // [2][U][C] LRU lists (double buffered)
  int32_t* order_par;          // [U] which buffer is current
  int32_t U;
};


// Sparse attention over the hot buffer (kvo_attend.cu).
struct AttendArgs {
  const int32_t* units;   // [n] unit ids
  const int32_t* slots;   // [n][P][k] hot slots of each position's top-k list (< 0: pad)
  const uint16_t* q;      // [n][P][H][576] bf16 queries
  const uint16_t* hot;    // [U][C][576] bf16 hot rows
  uint16_t* out;          // [n][P][H][512] bf16
  float* lse;             // [n][P][H] or null
  int n, P, k, H, C;
  float scale_log2;       // softmax scale * log2(e)
  uint32_t* err;
  uint64_t wait_ns;
  // In-kernel fill of the step's miss rows (used by the fetching variant only):
  // an entry whose payload is a miss (pay < 0, not the pad value) names token
  // -pay-1 of the host pool, read inside the kernel and written to its slot.
  const int32_t* pay;         // [n][P][k] the step's packed payloads
  const uint16_t* host_pool;  // device-visible address of the pinned pool
  HostRows hrows;             // token -> host-pool row
  uint16_t* hot_w;            // == hot, for the writes of filled rows
  uint32_t* claim;            // [U][C][3] claim words of (slot, part): 2e claimed, 2e + 1 written
  uint32_t epoch;             // this call's e (>= 1)
  int group;                  // units per round of the pair order
  DevStats* stats;
};

struct AppendArgs {
  const int32_t* units;
  int32_t n, n_tok, row_elems;
  int64_t stride;
  const uint16_t* rows;        // [n][n_tok][row_elems]
  const uint16_t* keys;        // [n][n_tok][128]
  HostRows hrows;              // token -> host-pool row
  uint16_t* host_pool;         // device-visible address
  uint16_t* idx;               // [U][stride][128] bf16 indexer, or nullptr
  int8_t* idx8;                // [U][stride][128] int8 codes, or nullptr
  uint16_t* idxs;              // [U][stride] fp16 scales of idx8
  int32_t* len;                // [U]
  DevStats* stats;
};

struct ResetArgs {
  const int32_t* units;
  int32_t n, keep, C, P;
  uint64_t* spec;              // [U][P] cleared
  float* qn_prev;              // [U][P] cleared
  int32_t* order;              // [U][C] first LRU buffer set to 0..C-1
  int32_t* order_par;          // [U] set to 0
  int64_t stride;
  int32_t* cache_slots;
  int32_t* slot_token;
  uint32_t* last_use;
  uint32_t* stamp;
  int32_t* len;
};

// Tokens per scoring piece of listed unit i (length len) in the fused step.
// The first units are cut finer (when they are not long): the first
// kTinyPieceUnits eight times, the next ones up to kSmallPieceUnits four
// times, so that they complete, and their miss rows start moving, early in
// the step.
constexpr int kTinyPieceUnits = 4;
constexpr int kSmallPieceUnits = 16;
constexpr int64_t kSmallPieceMaxLen = 65536;
__host__ __device__ inline int64_t piece_tokens_of(int i, int64_t len, int piece_tokens) {
  if (i < kSmallPieceUnits && len <= kSmallPieceMaxLen) {
    const int div = i < kTinyPieceUnits ? 8 : 4;
    const int64_t ps = (piece_tokens / div) & ~127;
    if (ps >= 128) return ps;
  }
  return piece_tokens;
}
__host__ __device__ inline int64_t pieces_of(int i, int64_t len, int piece_tokens) {
  const int64_t ps = piece_tokens_of(i, len, piece_tokens);
  return len > 0 ? (len + ps - 1) / ps : 1;
}

// One fused launch of the decode step: scoring, select, residency and the
// miss-row fill of every listed unit, overlapped across units.
struct FusedArgs {
  SelectArgs s;                // pbeg, pdone, ctr, status_init set
  ResidencyArgs r;             // miss_off / done_ctr unused
  GatherArgs g;                // miss_off unused
  int32_t* chunk_unit;         // [chunk_cap] published gather work: listed unit index,
  int32_t* chunk_start;        //   first row in the unit's miss list,
  int32_t* chunk_cnt;          //   row count,
  uint32_t* chunk_flag;        //   == epoch once the entry is valid
  int64_t chunk_cap;
  uint32_t epoch;              // differs between consecutive launches
  int32_t n_gather;            // CTAs 0 .. n_gather-1 only fill miss rows
  int32_t smem_bytes;          // dynamic shared memory of one CTA
  uint32_t* plan_flag;         // == epoch once CTA 0 has run the plan
  uint32_t* qdone;             // CTAs done quantizing queries (int8 indexer); zero between launches
  int32_t defer;               // 1: the miss rows are left for the attention call (nothing is published)
};

// Sets the thread-local message returned by kvo_last_error().
void set_last_error(const char* msg);

// Host-side launchers (return cudaError_t of the launch).
int score_cap_for(int P, int k, bool int8);
cudaError_t launch_plan(const SelectArgs& a, cudaStream_t s);
cudaError_t launch_score(const SelectArgs& a, cudaStream_t s);
cudaError_t launch_select(const SelectArgs& a, cudaStream_t s);
cudaError_t launch_residency(const ResidencyArgs& a, cudaStream_t s);
cudaError_t launch_gather(const GatherArgs& a, int n_sm, cudaStream_t s);
cudaError_t launch_flush_fill(const GatherArgs& a, cudaStream_t s);  // one CTA per listed unit, miss_cnt rows each
cudaError_t launch_append(const AppendArgs& a, cudaStream_t s);
cudaError_t launch_attend(const AttendArgs& a, cudaStream_t s);  // a.pay != nullptr: fetching variant
cudaError_t run_wait_selftest(uint64_t limit_ns, unsigned long long* host_out);  // out[3]
// host helpers shared by the entry points (kvo_api.cu)
int set_error(int code, const char* msg);
int set_cuda_error(cudaError_t e, const char* what);
cudaError_t alloc_pinned(size_t bytes, void** out, size_t* map_bytes, size_t* huge_page);
void free_pinned(void* p, size_t map_bytes);
size_t attend_smem_bytes();
cudaError_t launch_reset(const ResetArgs& a, cudaStream_t s);
cudaError_t launch_order_init(int32_t* order, int32_t* par, int U, int C, cudaStream_t s);
cudaError_t launch_set_len(int32_t* len, int32_t unit, int32_t value, cudaStream_t s);
cudaError_t launch_fill_i32(int32_t* p, int32_t v, size_t n, cudaStream_t s);
size_t fused_smem_bytes(int P, int k, int cap, bool int8);
cudaError_t launch_quant_keys(const uint16_t* src, int64_t n, int8_t* codes, uint16_t* scales, cudaStream_t s);
int fused_chunk_rows();
cudaError_t launch_fused(const FusedArgs& a, int grid, cudaStream_t s);

}  // namespace kvo
