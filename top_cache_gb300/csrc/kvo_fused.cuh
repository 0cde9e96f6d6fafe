// The decode step as one persistent launch ("Layerwise and Sparse KV Cache
// Offloading Design", section 4 "Sparse Decode Offload", Decode steps 3-6:
// indexer scoring and top-k, residency update, miss-row transfer, remap).
//
// The separate-launch path runs scoring, select, residency and the miss-row
// fill one after the other, so the host link idles while the SMs score and
// the SMs idle while the link fills rows.  Here each unit moves on as soon as
// its own scores are complete:
//
//  scorer CTAs   a producer warp claims pieces (up to piece_tokens tokens of
//                one unit, a quarter of that for the first units; numbered
//                unit-major) from a global counter and
//                streams their keys through the bulk-copy ring; the 16
//                consumer warps score and filter them exactly as the score
//                kernel does and write each piece's candidates.  The CTA that
//                holds a unit's last-claimed piece finishes the unit (its
//                producer claims nothing more meanwhile): exact top-k
//                of every position (after checking the speculative threshold,
//                rescanning the unit from global memory when it was too high),
//                the residency update, then it publishes the unit's miss rows
//                as gather chunks.
//  gather CTAs   (the first n_gather) copy published miss rows host -> shared
//                -> hot buffer with bulk async copies, several rows in flight
//                per warp; scorer CTAs join them once no piece is left.
//
// Every wait that depends on another CTA or on the copy engine is bounded
// (wait_ns) and sets the sticky error bit when it expires; the launch is
// cooperative so that all CTAs are resident together.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kvo_device.cuh"
#include "kvo_internal.cuh"

namespace kvo {

using namespace dev;

namespace {

constexpr int kFusedThreads = kScoreThreads;  // 16 consumer warps + 1 producer warp
constexpr int kFusedWarps = kFusedThreads / 32;
constexpr int kPieceRing = 16;                // claimed pieces passed to the consumers
constexpr int kFusedSegs = 1024;              // segment offsets the finisher holds (both groups)
constexpr int kFusedExtra = kPieceRing * 8 + 64 + kFusedSegs * 4 + 256 * 4 + 12 * 4;
constexpr int kChunkRows = 32;                // miss rows per gather work item
constexpr int kGatherLag = 2;                 // hot-buffer stores left in flight per warp
constexpr int kGatherMinSlots = 4;
constexpr int kGatherMaxSlots = 32;
constexpr uint32_t kPieceEnd = 0xffffffffu;

__device__ __forceinline__ uint64_t ld_volatile_u64(const void* p) {
  return *reinterpret_cast<const volatile unsigned long long*>(p);
}
__device__ __forceinline__ uint32_t ld_volatile_u32(const void* p) {
  return *reinterpret_cast<const volatile uint32_t*>(p);
}

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Polls cond() until it holds or limit_ns elapses.
template <class Cond>
__device__ __forceinline__ bool spin_until(Cond cond, uint64_t limit_ns) {
  if (cond()) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (cond()) return true;
    if ((it & 15u) == 0 && global_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------------------
// Miss-row fill: one warp, lane 0 drives a ring of D shared-memory row slots.
// Row j lands in slot j % D (bulk copy from the mapped host pool, completion
// on bar[j % D]); once it has landed a bulk store moves it to its hot slot.
// A slot is refilled only when the store of its previous row has finished
// reading it, which wait_group.read guarantees: at least kGatherLag younger
// stores separate the two.
// ---------------------------------------------------------------------------
struct RowPipe {
  uint64_t* bar;
  uint64_t* dstq;
  uint8_t* slots;
  int D;
  uint32_t bytes, slot_bytes;
  uint32_t issued, stored;
  uint64_t wait_ns;
  uint64_t pol;  // L2 policy of the rows (read and written once)
  bool timed_out;

  __device__ __forceinline__ bool retire(bool block) {
    if (stored == issued) return false;
    const int d = (int)(stored % (uint32_t)D);
    const uint32_t parity = (stored / (uint32_t)D) & 1u;
    if (block) {
      if (!timed_out && !mbar_wait(&bar[d], parity, wait_ns)) timed_out = true;
    } else if (!mbar_try_wait(&bar[d], parity)) {
      return false;
    }
    bulk_s2g_hint(reinterpret_cast<void*>(dstq[d]), slots + (size_t)d * slot_bytes, bytes, pol);
    bulk_commit();
    ++stored;
    return true;
  }
  __device__ __forceinline__ void push(uint64_t src, uint64_t dst) {
    if (issued - stored >= (uint32_t)(D - kGatherLag)) retire(true);
    bulk_wait_read<kGatherLag>();
    const int d = (int)(issued % (uint32_t)D);
    dstq[d] = dst;
    mbar_arrive_expect_tx(&bar[d], bytes);
    bulk_g2s_hint(slots + (size_t)d * slot_bytes, reinterpret_cast<const void*>(src), bytes, &bar[d], pol);
    ++issued;
  }
  __device__ __forceinline__ void drain() {
    while (stored < issued) retire(true);
    bulk_wait_all();
  }
};

// Waits until gather chunk c is published.  1: ready; 0: every unit has
// published and c is past the last chunk; -1: timed out.  idle() runs
// between polls.
template <class Idle>
__device__ __forceinline__ int wait_chunk(const FusedArgs& f, unsigned long long c, Idle idle) {
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (c < (unsigned long long)f.chunk_cap && ld_volatile_u32(&f.chunk_flag[c]) == f.epoch) {
      __threadfence();
      return 1;
    }
    if (ld_volatile_u64(&f.s.ctr[3]) == (unsigned long long)f.s.n) {
      // every unit has published: chunk c exists (and its flag is visible on
      // the next poll) or never will
      __threadfence();
      if (c >= ld_volatile_u64(&f.s.ctr[1])) return 0;
    }
    idle();
    if ((it & 7u) == 7u && global_ns() - t0 > f.s.wait_ns) return -1;
    __nanosleep(256);
  }
}

// One warp moves chunks of miss rows until none is left.  slice: this warp's
// shared memory (128-byte aligned).
__device__ __forceinline__ void gather_warp(const FusedArgs& f, uint8_t* slice, int D, int lane) {
  const GatherArgs& g = f.g;
  RowPipe pipe;
  pipe.bar = reinterpret_cast<uint64_t*>(slice);
  pipe.dstq = pipe.bar + D;
  ulonglong2* abuf = reinterpret_cast<ulonglong2*>(pipe.dstq + D);  // [32] (src, dst)
  const uint32_t row_bytes = (uint32_t)g.row_elems * 2u;
  pipe.bytes = row_bytes;
  pipe.slot_bytes = (row_bytes + 127u) & ~127u;
  pipe.slots = slice + ((16 * D + 32 * 16 + 127) & ~127);
  pipe.D = D;
  pipe.issued = pipe.stored = 0;
  pipe.wait_ns = g.wait_ns;
  pipe.pol = l2_evict_first();
  pipe.timed_out = false;
  if (lane == 0) {
    for (int d = 0; d < D; ++d) mbar_init(&pipe.bar[d], 1);
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  __syncwarp();
  unsigned long long rows = 0, bad_rows = 0;
  bool failed = false;
  for (;;) {
    unsigned long long c = 0;
    int st = 0;
    if (lane == 0) {
      c = atomicAdd(&f.s.ctr[2], 1ull);
      st = wait_chunk(f, c, [&] { pipe.retire(false); });
    }
    st = __shfl_sync(kFull, st, 0);
    if (st <= 0) {
      failed = st < 0;
      break;
    }
    c = __shfl_sync(kFull, c, 0);
    const int i = __ldcg(&f.chunk_unit[c]);
    const int r0 = __ldcg(&f.chunk_start[c]);
    const int cnt = __ldcg(&f.chunk_cnt[c]);
    bool bad = false;
    if (lane < cnt) {
      const int64_t e = (int64_t)i * g.pk + r0 + lane;
      const int32_t t = __ldcg(&g.miss_tok[e]);
      const int32_t s = __ldcg(&g.miss_slot[e]);
      const int64_t u = g.units[i];
      const int64_t hr = host_row(g.rows, u, t);
      uint16_t* dst = g.hot + (u * g.C + s) * g.row_elems;
      // a row of an unmapped block (paged pool) is copied onto itself, which
      // leaves the hot row as it was
      const uint16_t* src = hr < 0 ? dst : g.host_pool + hr * g.row_elems;
      bad = hr < 0;
      abuf[lane] = make_ulonglong2(reinterpret_cast<uint64_t>(src), reinterpret_cast<uint64_t>(dst));
    }
    __syncwarp();
    if (lane == 0)
      for (int r = 0; r < cnt; ++r) pipe.push(abuf[r].x, abuf[r].y);
    __syncwarp();
    const unsigned long long nb = __popc(__ballot_sync(kFull, bad));
    rows += (unsigned long long)cnt - nb;
    bad_rows += nb;
  }
  if (lane == 0) {
    pipe.drain();
    if (failed || pipe.timed_out) atomicOr(g.err, kErrTimeout);
    if (rows && g.stats) {
      atomicAdd(&g.stats->rows_h2d, rows);
      atomicAdd(&g.stats->bytes_h2d, rows * row_bytes);
    }
    if (bad_rows && g.stats) atomicAdd(&g.stats->block_errors, bad_rows);
  }
  __syncwarp();
}

// The CTA's warps split its shared memory and fill miss rows.
__device__ __forceinline__ void gather_cta(const FusedArgs& f, uint8_t* smem, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t slot_bytes = ((uint32_t)f.g.row_elems * 2u + 127u) & ~127u;
  const int per_min = kGatherMinSlots * ((int)slot_bytes + 16) + 640;
  int nw = f.smem_bytes / per_min;
  if (nw > kFusedWarps) nw = kFusedWarps;
  if (warp >= nw) return;
  const int slice = (f.smem_bytes / nw) & ~127;
  int D = (slice - 640) / ((int)slot_bytes + 16);
  if (D > kGatherMaxSlots) D = kGatherMaxSlots;
  gather_warp(f, smem + (size_t)warp * slice, D, lane);
}

// Warp 0 of a finisher: the unit's miss rows become gather chunks.
__device__ __forceinline__ void publish_chunks(const FusedArgs& f, int i, uint32_t m, int lane) {
  const int nch = (int)((m + kChunkRows - 1) / kChunkRows);
  unsigned long long base = 0;
  if (lane == 0 && nch) base = atomicAdd(&f.s.ctr[1], (unsigned long long)nch);
  base = __shfl_sync(kFull, base, 0);
  for (int c = lane; c < nch; c += 32) {
    const unsigned long long e = base + c;
    if (e >= (unsigned long long)f.chunk_cap) continue;  // cannot happen: capacity covers every unit's rows
    f.chunk_unit[e] = i;
    f.chunk_start[e] = c * kChunkRows;
    f.chunk_cnt[e] = (int32_t)min((uint32_t)kChunkRows, m - (uint32_t)c * kChunkRows);
  }
  __threadfence();
  for (int c = lane; c < nch; c += 32) {
    const unsigned long long e = base + c;
    if (e < (unsigned long long)f.chunk_cap) *reinterpret_cast<volatile uint32_t*>(&f.chunk_flag[e]) = f.epoch;
  }
  __threadfence();
  __syncwarp();
  if (lane == 0) atomicAdd(&f.s.ctr[3], 1ull);
}

// ---------------------------------------------------------------------------
// Scorer CTA
// ---------------------------------------------------------------------------
struct FusedSmem {
  ScoreSmem sm;
  uint8_t* region;        // candidate buffers + scratch, reused by the finisher
  size_t region_bytes;
  uint64_t* pring;        // [kPieceRing] (sequence << 32 | piece)
  volatile int64_t* s_piece;
  volatile int32_t* pcons;  // pieces the consumers have taken from the ring
  volatile int32_t* s_flag;
  volatile int32_t* s_ready;  // pieces the consumers have completed, finishing included
  uint32_t* s_tot;          // [8] candidates per position of the unit being finished
  uint32_t* seg_off;        // [kFusedSegs]
  uint32_t* hist1;          // [256] histogram / scan words of the second select group
  uint32_t* rx1;            // [12] (8-byte aligned)
  template <class KF>
  __device__ void carve(uint8_t* smem, int P, int cap, int k) {
    sm.carve<KF>(smem, P, cap);
    region = reinterpret_cast<uint8_t*>(sm.cand);
    region_bytes = (size_t)P * cap * 8 + (size_t)k * 8;
    pring = reinterpret_cast<uint64_t*>(region + region_bytes);
    s_piece = reinterpret_cast<volatile int64_t*>(pring + kPieceRing);
    pcons = reinterpret_cast<volatile int32_t*>(s_piece + 1);
    s_flag = pcons + 1;
    s_ready = s_flag + 1;
    s_tot = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(pring + kPieceRing) + 32);
    seg_off = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(pring + kPieceRing) + 64);
    hist1 = seg_off + kFusedSegs;
    rx1 = hist1 + 256;
  }
};

// Producer (one lane): claim pieces, post them to the consumers, stream
// their keys.  Consumers see the same sequence of pieces and tiles.
template <class KF>
__device__ __forceinline__ void fused_producer(const FusedArgs& f, const FusedSmem& fs) {
  const SelectArgs& a = f.s;
  uint32_t seq = 0;
  bool finishes = false;  // the last piece claimed is its unit's last: the consumers finish that unit
  const uint64_t pol = l2_evict_first();  // keys are read once per step
  for (uint32_t q = 0;; ++q) {
    // nothing is claimed behind a finisher (that piece would wait for it);
    // the ring stays idle meanwhile and the finisher uses it
    if (finishes) {
      if (!spin_until([&] { return *fs.s_ready >= (int)q; }, a.wait_ns)) {
        atomicOr(a.err, kErrTimeout);
        return;
      }
      // the finisher wrote the ring with ordinary stores; bulk copies follow
      __threadfence_block();
      fence_proxy_async_smem();
    }
    if (q >= (uint32_t)kPieceRing) {
      // the ring entry about to be replaced must have been taken
      const int need = (int)(q - kPieceRing + 1);
      if (!spin_until([&] { return *fs.pcons >= need; }, a.wait_ns)) {
        atomicOr(a.err, kErrTimeout);
        return;
      }
    }
    const unsigned long long piece = atomicAdd(&a.ctr[0], 1ull);
    const bool end = piece >= (unsigned long long)a.n_pieces;
    *reinterpret_cast<volatile unsigned long long*>(&fs.pring[q % kPieceRing]) =
        ((unsigned long long)q << 32) | (end ? kPieceEnd : (uint32_t)piece);
    if (end) return;
    const int i = find_segment(a.pbeg, a.n, (int64_t)piece);
    finishes = (int64_t)piece == a.pbeg[i + 1] - 1;
    const int64_t len = a.off[i + 1] - a.off[i];
    const int64_t ps = piece_tokens_of(i, len, a.piece_tokens);
    const int64_t t0 = ((int64_t)piece - a.pbeg[i]) * ps;
    const int64_t t1 = min(t0 + ps, len);
    const int u = a.units[i];
    for (int64_t t = t0; t < t1; t += kTile, ++seq) {
      const int stage = seq % KF::kStages;
      const uint32_t round = seq / KF::kStages;
      if (round > 0 && !mbar_wait(&fs.sm.empty[stage], (round - 1) & 1u, a.wait_ns)) {
        atomicOr(a.err, kErrTimeout);  // consumers stopped: issue nothing more
        return;
      }
      const int nt = (int)((t1 - t) < kTile ? (t1 - t) : kTile);
      issue_tile<KF>(a, fs.sm.ring + stage * KF::kStageBytes, &fs.sm.full[stage], u, t, nt, pol);
    }
  }
}

// Rescores unit i from global memory without a speculative threshold and
// leaves its exact candidates in its first segment (the others emptied).
template <int PP, class SC>
__device__ __forceinline__ void rescan_unit(const SelectArgs& a, const FusedSmem& fs, SC& sc, int i,
                                            int64_t pb, int64_t pe, int ctid) {
  const int P = a.P, k = a.k, cap = a.cap;
  const int64_t L = a.off[i + 1] - a.off[i];
  const int u = a.units[i];
  uint64_t* gth = a.gthr + (int64_t)i * P;
  sc.load_queries(a, i, P);
  piece_begin(fs.sm, P, nullptr, ctid);
  int ti = 0;
  for (int64_t t = 0; t < L; t += kTile, ++ti) {
    const int nt = (int)((L - t) < kTile ? (L - t) : kTile);
    float acc[SC::V];
    sc.score_global(a, u, t, nt, acc);
    sc.filter(acc, t, nt, L, P, fs.sm.thr, fs.sm.cnt, fs.sm.cand, cap);
    if (t + kTile < L && (ti + 1) % kCheckTiles == 0) piece_check(fs.sm, P, k, cap, gth, ctid);
  }
  piece_end(fs.sm, P, k, cap, gth, pb, a.seg_keys, a.seg_cnt, ctid);
  for (int64_t e = (pb + 1) * P + ctid; e < pe * P; e += kCT) a.seg_cnt[e] = 0;
  consumer_sync();
}

// Exact top-k of positions p0, p0 + step, ... of unit i by one group of NTG
// consumer threads (barrier `sync`) in its own part of the finisher's
// shared memory: bucket sort when the candidates fit and spread, radix
// select and bitonic sort otherwise.
template <int NTG, class Sync>
__device__ __forceinline__ void select_positions(const SelectArgs& a, int i, int p0, int step, int64_t pb, int nseg,
                                                 uint8_t* region, size_t bytes, uint32_t* seg_off, int seg_cap,
                                                 uint32_t* hist, uint32_t* rx, int gtid, Sync sync) {
  const int k = a.k;
  int kpad = 1;
  while (kpad < k) kpad <<= 1;
  uint64_t* keys = reinterpret_cast<uint64_t*>(region);
  const uint32_t words = (uint32_t)(bytes / 8);
  int log2B = 12;
  while ((1 << log2B) > 8 * NTG || (log2B > 9 && (8u << log2B) > bytes / 4)) --log2B;
  for (int p = p0; p < a.P; p += step) {
    bool done = false;
    if (nseg + 1 <= seg_cap) {
      segment_offsets<NTG>(a, p, 1, pb, nseg, seg_off, gtid, sync);
      done = bucket_select<NTG>(a, i, p, pb, nseg, seg_off, region, bytes, log2B, hist, gtid, sync);
    }
    if (!done)
      select_body<NTG>(a, i, p, pb, nseg, false, keys, words - (uint32_t)kpad, keys + (words - kpad), hist, rx, gtid,
                       sync);
  }
}

// Select, residency and publication of unit i (the consumer threads).
template <int PP, class KF, class SC>
__device__ __forceinline__ void finish_unit(const FusedArgs& f, const FusedSmem& fs, SC& sc, int i, int ctid) {
  const SelectArgs& a = f.s;
  const int P = a.P, k = a.k;
  const int64_t pb = a.pbeg[i], pe = a.pbeg[i + 1];
  const int nseg = (int)(pe - pb);
  const int warp = ctid >> 5, lane = ctid & 31;
  // candidates per position (warp p sums position p's segment counts)
  auto totals = [&] {
    if (warp < P) {
      uint32_t t = 0;
      for (int c = lane; c < nseg; c += 32) t += (uint32_t)__ldcg(&a.seg_cnt[(pb + c) * P + warp]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(kFull, t, o);
      if (lane == 0) fs.s_tot[warp] = t;
    }
    consumer_sync();
  };
  totals();
  bool exact = true;
  for (int p = 0; p < P; ++p) exact = exact && !spec_short(a, i, p, fs.s_tot[p]);
  if (!exact) {
    rescan_unit<PP>(a, fs, sc, i, pb, pe, ctid);
    if (ctid == 0 && a.stats) atomicAdd(&a.stats->rescored, 1ull);
  }
  // positions in two concurrent groups of 256 threads (their barriers and
  // memory waits overlap), one in the idle key ring and one in the candidate
  // buffers; or all 512 threads on one position at a time
  int kpad = 1;
  while (kpad < k) kpad <<= 1;
  const size_t ring_bytes = (size_t)KF::kStages * KF::kStageBytes;
  if (P >= 2 && kpad <= 8 * (kCT / 2)) {
    const int g = ctid / (kCT / 2), gtid = ctid % (kCT / 2);
    auto gsync = [g] { named_sync(2 + g, kCT / 2); };
    select_positions<kCT / 2>(a, i, g, 2, pb, nseg, g ? fs.region : fs.sm.ring, g ? fs.region_bytes : ring_bytes,
                              fs.seg_off + g * (kFusedSegs / 2), kFusedSegs / 2, g ? fs.hist1 : fs.sm.hist,
                              g ? fs.rx1 : fs.sm.rx, gtid, gsync);
  } else {
    const bool in_ring = ring_bytes > fs.region_bytes;
    select_positions<kCT>(a, i, 0, 1, pb, nseg, in_ring ? fs.sm.ring : fs.region,
                          in_ring ? ring_bytes : fs.region_bytes, fs.seg_off, kFusedSegs, fs.sm.hist, fs.sm.rx, ctid,
                          [] { consumer_sync(); });
  }
  consumer_sync();
  const int nwords_pad = (((f.r.C + 31) >> 5) + 3) & ~3;
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(fs.region);
  int32_t* M = reinterpret_cast<int32_t*>(bitmap + nwords_pad);
  int32_t* V = M + P * k;
  // the unit's miss rows are published as soon as their slots are assigned
  residency_body<kCT>(f.r, i, bitmap, M, V, fs.sm.hist, ctid, [] { consumer_sync(); }, nullptr, [&](uint32_t m) {
    __threadfence();
    consumer_sync();
    if (ctid < 32) publish_chunks(f, i, f.defer ? 0u : m, ctid);  // deferred: the rows stay for the attention call
  });
}

template <int PP, class KF>
__device__ __forceinline__ void fused_consumers(const FusedArgs& f, const FusedSmem& fs, int tid) {
  const SelectArgs& a = f.s;
  const int ctid = tid, warp = tid >> 5, lane = tid & 31;
  const int P = a.P, k = a.k, cap = a.cap;
  typename ScorerFor<PP, KF>::type sc;
  sc.init(warp, lane);
  constexpr int V = ScorerFor<PP, KF>::type::V;
  uint32_t seq = 0;
  bool stalled = false;  // a wait of this thread expired: later tiles are not waited for
  for (uint32_t q = 0;; ++q) {
    if (ctid == 0) {
      uint64_t e = 0;
      const bool ok = spin_until(
          [&] {
            e = ld_volatile_u64(&fs.pring[q % kPieceRing]);
            return (uint32_t)(e >> 32) == q;
          },
          a.wait_ns);
      int64_t piece = -1;
      if (!ok) atomicOr(a.err, kErrTimeout);
      else if ((uint32_t)e != kPieceEnd) piece = (int64_t)(uint32_t)e;
      *fs.s_piece = piece;
      *fs.pcons = (int32_t)(q + 1);
    }
    consumer_sync();
    const int64_t piece = *fs.s_piece;
    if (piece < 0) break;
    const int i = find_segment(a.pbeg, a.n, piece);
    const int64_t len = a.off[i + 1] - a.off[i];
    const int64_t ps = piece_tokens_of(i, len, a.piece_tokens);
    const int64_t t0 = (piece - a.pbeg[i]) * ps;
    const int64_t t1 = min(t0 + ps, len);
    uint64_t* gth = a.gthr + (int64_t)i * P;
    sc.load_queries(a, i, P);
    piece_begin(fs.sm, P, a.tspec ? a.tspec + (int64_t)i * P : nullptr, ctid);
    int ti = 0;
    for (int64_t t = t0; t < t1; t += kTile, ++seq, ++ti) {
      const int stage = seq % KF::kStages;
      const uint32_t round = seq / KF::kStages;
      if (!stalled && !mbar_wait(&fs.sm.full[stage], round & 1u, a.wait_ns)) {
        stalled = true;
        atomicOr(a.err, kErrTimeout);
      }
      const int nt = (int)((t1 - t) < kTile ? (t1 - t) : kTile);
      float acc[V];
      sc.score(fs.sm.ring + stage * KF::kStageBytes, t, acc, [&] {
        __syncwarp();
        if (lane == 0) mbar_arrive(&fs.sm.empty[stage]);
      });
      sc.filter(acc, t, nt, len, P, fs.sm.thr, fs.sm.cnt, fs.sm.cand, cap);
      if (t + kTile < t1 && (ti + 1) % kCheckTiles == 0) piece_check(fs.sm, P, k, cap, gth, ctid);
    }
    piece_end(fs.sm, P, k, cap, gth, piece, a.seg_keys, a.seg_cnt, ctid);
    // The CTA holding a unit's last-claimed piece finishes the unit, once the
    // unit's other pieces (claimed earlier, by CTAs that claim nothing
    // behind a finisher) are complete.
    __threadfence();
    consumer_sync();
    const int np = (int)(a.pbeg[i + 1] - a.pbeg[i]);
    const bool finisher = piece == a.pbeg[i + 1] - 1;
    if (ctid == 0) {
      atomicAdd(&a.pdone[i], 1);
      if (finisher) {
        if (!spin_until([&] { return ld_volatile_u32(&a.pdone[i]) >= (uint32_t)np; }, a.wait_ns))
          atomicOr(a.err, kErrTimeout);
        __threadfence();
      }
    }
    consumer_sync();
    if (finisher) {
      finish_unit<PP, KF>(f, fs, sc, i, ctid);
      consumer_sync();
    }
    if (ctid == 0) {
      __threadfence_block();
      *fs.s_ready = (int32_t)(q + 1);
    }
  }
}

template <int PP, class KF>
__global__ void __launch_bounds__(kFusedThreads, 1) fused_step_kernel(FusedArgs f) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // int8 indexer: every warp of the grid quantizes some of the step's queries
  if (f.s.q8) {
    const int nq = f.s.n * f.s.P;
    for (int e = blockIdx.x * (kFusedThreads / 32) + warp; e < nq; e += gridDim.x * (kFusedThreads / 32))
      warp_quant128(f.s.queries + (int64_t)e * kDim, f.s.q8 + (int64_t)e * kDim, f.s.qscale + e, lane);
    __threadfence();
    __syncthreads();
    if (tid == 0) atomicAdd(f.qdone, 1u);
  }
  // CTA 0 plans the step (offsets, piece table, thresholds, counters); every
  // CTA starts once the plan (and the queries' codes) are published
  if (blockIdx.x == 0) {
    plan_body<kFusedThreads>(f.s, tid, reinterpret_cast<int64_t*>(smem), reinterpret_cast<int64_t*>(smem) + 32);
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      if (f.s.q8) {
        if (!spin_until([&] { return ld_volatile_u32(f.qdone) >= gridDim.x; }, f.s.wait_ns))
          atomicOr(f.s.err, kErrTimeout);
        // every CTA adds one in each launch, so the counter is back at zero
        // once this launch ends, even if the wait above gave up early
        atomicSub(f.qdone, gridDim.x);
        __threadfence();  // the codes seen through the counter reach readers of the flag
      }
      *reinterpret_cast<volatile uint32_t*>(f.plan_flag) = f.epoch;
    }
  }
  if (tid == 0) {
    if (!spin_until([&] { return ld_volatile_u32(f.plan_flag) == f.epoch; }, f.s.wait_ns))
      atomicOr(f.s.err, kErrTimeout);
    __threadfence();
  }
  __syncthreads();
  if ((int)blockIdx.x >= f.n_gather) {
    FusedSmem fs;
    fs.carve<KF>(smem, f.s.P, f.s.cap, f.s.k);
    if (tid == 0) {
      for (int s = 0; s < KF::kStages; ++s) {
        mbar_init(&fs.sm.full[s], 1);
        mbar_init(&fs.sm.empty[s], kCW);
      }
      for (int q = 0; q < kPieceRing; ++q) fs.pring[q] = ~0ull;
      *fs.pcons = 0;
      *fs.s_ready = 0;
      fence_mbar_init();
    }
    __syncthreads();
    if (warp == kCW) {
      if (lane == 0) fused_producer<KF>(f, fs);
      __syncwarp();
    } else {
      fused_consumers<PP, KF>(f, fs, tid);
    }
    // no piece left: the ring and the candidate buffers become row slots
    __syncthreads();
    if (tid == 0) {
      for (int s = 0; s < KF::kStages; ++s) {
        mbar_inval(&fs.sm.full[s]);
        mbar_inval(&fs.sm.empty[s]);
      }
    }
    __syncthreads();
  }
  gather_cta(f, smem, tid);
}

template <int PP, class KF>
cudaError_t launch_fused_pp(const FusedArgs& a, int grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(fused_step_kernel<PP, KF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       a.smem_bytes);
  if (e != cudaSuccess) return e;
  FusedArgs copy = a;
  void* args[] = {&copy};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(fused_step_kernel<PP, KF>), dim3(grid),
                                     dim3(kFusedThreads), args, (size_t)a.smem_bytes, s);
}


template <class KF>
cudaError_t launch_fused_kf(const FusedArgs& a, int grid, cudaStream_t s) {
  if (a.s.P <= 1) return launch_fused_pp<1, KF>(a, grid, s);
  if (a.s.P <= 2) return launch_fused_pp<2, KF>(a, grid, s);
  if (a.s.P <= 4) return launch_fused_pp<4, KF>(a, grid, s);
  return launch_fused_pp<8, KF>(a, grid, s);
}

}  // namespace
}  // namespace kvo
