// Device building blocks shared by the step kernels (separate launches) and the
// fused persistent step kernel: indexer scoring of a tile, candidate filter and
// compaction, exact top-k select of one (unit, position), residency update of
// one unit.  Every block-level routine takes its thread count NT and a barrier
// functor, so it runs both as a whole CTA (__syncthreads) and as the consumer
// warps of a warp-specialised CTA (named barrier).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <cuda_fp16.h>

#include <type_traits>

#include "kvo_internal.cuh"

namespace kvo {
namespace dev {

constexpr int kTile = 128;                  // keys per ring stage
constexpr int kTileBytes = kTile * kKeyBytes;
constexpr int kStages = 3;
constexpr int kCW = 16;                     // consumer warps
constexpr int kCT = kCW * 32;               // consumer threads
constexpr int kScoreThreads = kCT + 32;     // + one producer warp
constexpr int kCheckTiles = 8;              // tiles between candidate-buffer checks
constexpr int kSmemMax = 222 * 1024;        // leaves room for a co-resident copy CTA
constexpr int kSelThreads = 512;
constexpr int kSelSmemKeys = 8192;          // candidates held in shared memory by select (fallback)
constexpr int kSelLog2B = 11;               // buckets of the select kernel's bucket sort
constexpr int kSelMaxSegs = 512;            // segments whose offsets the select kernel holds
constexpr int kSelSmemBytes = 104 * 1024;   // two CTAs per SM
constexpr int kMaxK = 4096;
constexpr int kScoreGatherRows = 90;        // rows per batch of a score launch's copying CTAs (x 72 chunks <= 12 x 544)

__device__ __forceinline__ void consumer_sync() { named_sync(1, kCT); }

// Indexer key formats.  A ring stage holds one tile of kTile keys; int8
// stages hold the keys' 128-byte code rows followed by their fp16 scales.
struct KeysBf16 {
  static constexpr bool kInt8 = false;
  static constexpr int kRowBytes = kKeyBytes;
  static constexpr int kStages = 3;
  static constexpr int kStageBytes = kTile * kKeyBytes;  // 32 KB
};
struct KeysInt8 {
  static constexpr bool kInt8 = true;
  static constexpr int kRowBytes = kDim;
  static constexpr int kStages = 6;
  static constexpr int kScaleOff = kTile * kDim;         // codes, then scales
  // the scales are copied from the 8-token boundary at or below the tile's
  // first token (16-byte aligned source): up to 7 + kTile of them
  static constexpr int kScaleBytes = ((kTile + 7) * 2 + 15) & ~15;
  static constexpr int kStageBytes = kScaleOff + kScaleBytes;
};
// Shared memory of a scoring CTA besides the candidate buffers.
template <class KF>
constexpr int smem_fixed() {
  return KF::kStages * KF::kStageBytes + 2 * KF::kStages * 8 + 8 * 4 + 8 * 8 + 256 * 4 + 10 * 4 + 8;
}

// Rotation and int8 quantization of one 128-element bf16 vector by a warp
// (reading R12 of the oracle; "FlashOffloading ... What does it mean?", the
// LIM C8 paragraph): y = H x by the unnormalised fast Walsh-Hadamard
// transform in fp32, stages h = 1 .. 64, pair (i, i + h) -> (a + b, a - b);
// scale = fp16(max|y| / 127) (round to nearest even); codes =
// clamp(rint(y / scale), -127, 127).  Lane l holds elements 4l .. 4l+3.
// Returns the scale as fp32; lane 0 writes its fp16 bits to *scale.
__device__ __forceinline__ float warp_quant128(const uint16_t* x, int8_t* code, uint16_t* scale, int lane) {
  // scale: nullable
  const uint2 raw = *reinterpret_cast<const uint2*>(x + 4 * lane);
  float v[4] = {bf_lo(raw.x), bf_hi(raw.x), bf_lo(raw.y), bf_hi(raw.y)};
  // h = 1, 2 inside the lane
  float a = v[0], b = v[1];
  v[0] = a + b; v[1] = a - b;
  a = v[2]; b = v[3];
  v[2] = a + b; v[3] = a - b;
  a = v[0]; b = v[2];
  v[0] = a + b; v[2] = a - b;
  a = v[1]; b = v[3];
  v[1] = a + b; v[3] = a - b;
  // h = 4 .. 64 across lanes (partner lane l ^ (h / 4))
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float o = __shfl_xor_sync(kFull, v[e], m);
      v[e] = upper ? o - v[e] : v[e] + o;  // lower: a + b; upper: a - b
    }
  }
  float mx = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
  const __half h = __float2half_rn(__fdiv_rn(mx, 127.0f));
  const float sc = __half2float(h);
  uint32_t packed = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float c = sc > 0.f ? rintf(__fdiv_rn(v[e], sc)) : 0.f;
    c = fminf(fmaxf(c, -127.f), 127.f);
    packed |= (uint32_t)(uint8_t)(int8_t)c << (8 * e);
  }
  *reinterpret_cast<uint32_t*>(code + 4 * lane) = packed;
  if (lane == 0 && scale) *scale = __half_as_ushort(h);
  return sc;
}

// ---------------------------------------------------------------------------
// 16-lane tree reduction of chunk sums.  Lane j (of a half warp) holds chunk
// j's partial sums for V (token, position) pairs.  Levels pair lanes j and
// j^8, then j^4, j^2, j^1: exactly the tree c_j += c_{j+w}, w = 8, 4, 2, 1
// (fp32 addition is commutative, so either lane of a pair may add).  While
// more than one value is left per lane a level also transposes: each lane
// keeps the lower half of its slots and receives the partner's upper half, so
// V values cost V-1 shuffles and no selects.  That works because slot i of
// lane l holds pair (i ^ X_l), X_l = tree_perm<V>(l): partners differ in
// exactly the bit of X that the level splits on.
// ---------------------------------------------------------------------------
template <int CUR, int V, class T>
__device__ __forceinline__ void tree_level(T (&a)[V], int m) {
  if constexpr (CUR > 1) {
#pragma unroll
    for (int i = 0; i < CUR / 2; ++i) a[i] = a[i] + __shfl_xor_sync(kFull, a[i + CUR / 2], m);
  } else {
    a[0] = a[0] + __shfl_xor_sync(kFull, a[0], m);
  }
}

template <int V, class T>
__device__ __forceinline__ void tree16(T (&a)[V]) {
  tree_level<V, V>(a, 8);
  tree_level<(V >= 2 ? V / 2 : 1), V>(a, 4);
  tree_level<(V >= 4 ? V / 4 : 1), V>(a, 2);
  tree_level<(V >= 8 ? V / 8 : 1), V>(a, 1);
}

// The same tree over groups of 8 lanes (levels j^4, j^2, j^1), for sums whose
// order is free (exact integer sums of the int8 indexer).
template <int V, class T>
__device__ __forceinline__ void tree8(T (&a)[V]) {
  tree_level<V, V>(a, 4);
  tree_level<(V >= 2 ? V / 2 : 1), V>(a, 2);
  tree_level<(V >= 4 ? V / 4 : 1), V>(a, 1);
}

// X_l: the lane's slot permutation (slot i holds pair i ^ X_l), which is also
// the pair held in slot 0 after tree16.
template <int V, int G = 16>
__device__ __forceinline__ int tree_perm(int lane) {
  int x = 0, cur = V;
#pragma unroll
  for (int m = G / 2; m >= 1; m >>= 1) {
    if (cur > 1) {
      if (lane & m) x += cur / 2;
      cur /= 2;
    }
  }
  return x;
}
// After the tree over G lanes with V < G several lanes hold the same sum; one
// reports it.
template <int V, int G = 16>
__device__ __forceinline__ bool tree_owner(int lane) {
  constexpr int dup = V >= G ? 0 : (G / V - 1);
  return (lane & dup) == 0;
}

// ---------------------------------------------------------------------------
// Block-level helpers (first NT threads of the block, barrier `sync`)
// ---------------------------------------------------------------------------
// Warp 0: the histogram bin (counting from the top) holding the need-th
// largest element.  rx[0] = bin, rx[1] = count above it, rx[2] = count in it.
__device__ __forceinline__ void scan_bins_desc(const uint32_t* hist, uint32_t need, uint32_t* rx,
                                               int lane) {
  uint32_t v[8], sum = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    v[e] = hist[255 - 8 * lane - e];
    sum += v[e];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  uint32_t above = incl - sum;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if (above < need && need <= above + v[e]) {
      rx[0] = 255 - 8 * lane - e;
      rx[1] = above;
      rx[2] = v[e];
    }
    above += v[e];
  }
}

// Exact radix select over unique 64-bit keys: returns the smallest value
// 'thr' such that exactly 'need' keys are >= thr.  for_each(f) must call f on
// every key once (strided over the NT participating threads); sync() is the
// barrier of those threads.  Requires need <= number of keys.  Uses rx[0..7]
// (rx 8-byte aligned) and hist[256].
template <int NT, class ForEach, class Sync>
__device__ __forceinline__ uint64_t radix_threshold_desc(ForEach for_each, uint32_t need,
                                                         uint32_t* hist, uint32_t* rx, int tid,
                                                         Sync sync) {
  // the bytes every key shares need no histogram pass
  unsigned long long* mm = reinterpret_cast<unsigned long long*>(rx + 4);  // rx[4..7]: min, max
  if (tid == 0) {
    mm[0] = ~0ull;
    mm[1] = 0ull;
  }
  sync();
  unsigned long long lo = ~0ull, hi = 0ull;
  for_each([&](uint64_t key) {
    lo = key < lo ? key : lo;
    hi = key > hi ? key : hi;
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long l2 = __shfl_xor_sync(kFull, lo, o), h2 = __shfl_xor_sync(kFull, hi, o);
    lo = l2 < lo ? l2 : lo;
    hi = h2 > hi ? h2 : hi;
  }
  if ((tid & 31) == 0) {
    atomicMin(&mm[0], lo);
    atomicMax(&mm[1], hi);
  }
  sync();
  const unsigned long long kmin = mm[0], kmax = mm[1];
  sync();
  const int common = kmin == kmax ? 64 : __clzll((long long)(kmin ^ kmax));
  const int top = 56 - 8 * (common / 8);  // first byte that differs
  if (top < 0) return kmin;               // all keys equal (cannot happen: keys are unique)
  const uint64_t cmask = top >= 56 ? 0ull : ~((1ull << (top + 8)) - 1);
  uint64_t prefix = kmin & cmask, mask = cmask;
  for (int shift = top; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += NT) hist[b] = 0;
    sync();
    for_each([&](uint64_t key) {
      if ((key & mask) == prefix) atomicAdd(&hist[(uint32_t)(key >> shift) & 255u], 1u);
    });
    sync();
    if (tid < 32) scan_bins_desc(hist, need, rx, tid);
    sync();
    const uint32_t bin = rx[0], above = rx[1], inbin = rx[2];
    need -= above;
    prefix |= (uint64_t)bin << shift;
    mask |= 0xffull << shift;
    if (inbin == need) break;
  }
  return prefix;
}

// Bitonic sort, descending, of n = E * NT keys (n a power of two) held in
// registers, E consecutive keys per thread; buf (n keys of shared memory) is
// only the exchange area of strides that cross warps.  Strides below E stay
// in a thread, strides below 32 E use warp shuffles.
template <int E, int NT, class Sync>
__device__ __forceinline__ void bitonic_regs_desc(uint64_t (&v)[E], uint64_t* buf, int n, int tid,
                                                  Sync sync) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 32 * E) {
        // only threads that hold keys touch buf (n may be smaller than E * NT)
        const bool active = tid * E < n;
        sync();
        if (active)
#pragma unroll
          for (int e = 0; e < E; ++e) buf[tid * E + e] = v[e];
        sync();
        if (active)
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const int i = tid * E + e;
            const uint64_t w = buf[i ^ stride];
            const bool asc = (i & size) != 0, lower = (i & stride) == 0;
            const bool keep_max = lower != asc;
            v[e] = keep_max ? (v[e] > w ? v[e] : w) : (v[e] < w ? v[e] : w);
          }
      } else if (stride >= E) {
        const int ld = stride / E;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = tid * E + e;
          const uint64_t w = __shfl_xor_sync(kFull, v[e], ld);
          const bool asc = (i & size) != 0, lower = (i & stride) == 0;
          const bool keep_max = lower != asc;
          v[e] = keep_max ? (v[e] > w ? v[e] : w) : (v[e] < w ? v[e] : w);
        }
      } else {
        // in-thread strides 1, 2, 4: compile-time indices keep v in registers
        auto ce = [&](auto S_) {
          constexpr int S = decltype(S_)::value;
#pragma unroll
          for (int e = 0; e < E; ++e) {
            if constexpr (S < E) {
              if (e & S) continue;
              const int i = tid * E + e;
              const uint64_t x = v[e], y = v[e + S];
              const bool asc = (i & size) != 0;
              const bool swap = asc ? (x > y) : (x < y);
              v[e] = swap ? y : x;
              v[e + S] = swap ? x : y;
            }
          }
        };
        if (stride == 1) ce(std::integral_constant<int, 1>{});
        else if (stride == 2) ce(std::integral_constant<int, 2>{});
        else ce(std::integral_constant<int, 4>{});
      }
    }
  }
}

// Sorts buf[0..n) descending (n a power of two, n <= 8 * NT) with NT threads.
template <int NT, class Sync>
__device__ __forceinline__ void block_sort_desc(uint64_t* buf, int n, int tid, Sync sync) {
  auto run = [&](auto E_) {
    constexpr int E = decltype(E_)::value;
    uint64_t v[E];
    const bool active = tid * E < n;
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = active ? buf[tid * E + e] : 0ull;
    bitonic_regs_desc<E, NT>(v, buf, n, tid, sync);
    sync();
    if (active)
#pragma unroll
      for (int e = 0; e < E; ++e) buf[tid * E + e] = v[e];
    sync();
  };
  if (n <= NT) run(std::integral_constant<int, 1>{});
  else if (n <= 2 * NT) run(std::integral_constant<int, 2>{});
  else if (n <= 4 * NT) run(std::integral_constant<int, 4>{});
  else run(std::integral_constant<int, 8>{});
}

template <int NT, class Sync>
__device__ __forceinline__ uint32_t block_sum(uint32_t v, uint32_t* wsum, int tid, Sync sync) {
  const int lane = tid & 31, w = tid >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  if (lane == 0) wsum[w] = v;
  sync();
  uint32_t t = 0;
#pragma unroll 4
  for (int x = 0; x < NT / 32; ++x) t += wsum[x];
  sync();
  return t;
}

// Exclusive scan of v over the NT threads; *total gets the sum.
template <int NT, class Sync>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* wsum, uint32_t* total, int tid,
                                                    Sync sync) {
  constexpr int NW = NT / 32;
  const int lane = tid & 31, w = tid >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[w] = incl;
  sync();
  if (w == 0) {
    uint32_t s = lane < NW ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, s, o);
      if (lane >= o) s += y;
    }
    if (lane < NW) wsum[lane] = s;
  }
  sync();
  const uint32_t excl = (w ? wsum[w - 1] : 0) + incl - v;
  *total = wsum[NW - 1];
  sync();
  return excl;
}

// ---------------------------------------------------------------------------
// Candidate buffers of the scoring consumers
// ---------------------------------------------------------------------------
// Shrink one candidate buffer to at most k keys, all >= floor, that include
// every key of the buffer which can still be among the unit's k best:
// floor = max(local threshold, the unit's shared threshold gth), then, if
// more than k keys reach it, the k-th largest of them.  A threshold found by
// the radix select is a lower bound of the unit's k-th best (k keys of this
// piece reach it) and is published to gth.  All consumer threads call it.
// rx needs 10 words (8-byte aligned).
__device__ __forceinline__ void compact_candidates(uint64_t* cand, uint32_t* cnt, uint64_t* thr,
                                                   uint64_t* gth, uint64_t* fl, uint64_t* scratch,
                                                   uint32_t* hist, uint32_t* rx, int k, int ctid) {
  const int lane = ctid & 31;
  if (ctid == 0) {
    uint64_t f = *thr;
    const uint64_t g = __ldcg(reinterpret_cast<const unsigned long long*>(gth));
    *fl = g > f ? g : f;
    rx[3] = 0;
    rx[8] = 0;
    rx[9] = (*cnt <= (uint32_t)k && *fl == *thr) ? 1u : 0u;  // nothing to do
  }
  consumer_sync();
  if (rx[9]) {
    consumer_sync();
    return;
  }
  const uint64_t floor = *fl;
  const uint32_t n = *cnt;
  uint32_t c = 0;
  for (uint32_t i = ctid; i < n; i += kCT) c += cand[i] >= floor ? 1u : 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
  if (lane == 0 && c) atomicAdd(&rx[8], c);
  consumer_sync();
  const uint32_t nge = rx[8];
  uint64_t t = floor;
  if (nge > (uint32_t)k) {
    auto for_each = [&](auto f) {
      for (uint32_t i = ctid; i < n; i += kCT) {
        const uint64_t key = cand[i];
        if (key >= floor) f(key);
      }
    };
    t = radix_threshold_desc<kCT>(for_each, (uint32_t)k, hist, rx, ctid, consumer_sync);
  }
  for (uint32_t i0 = 0; i0 < n; i0 += kCT) {
    const uint32_t i = i0 + ctid;
    const uint64_t key = i < n ? cand[i] : 0;
    const bool keep = i < n && key >= t;
    const uint32_t m = __ballot_sync(kFull, keep);
    if (m) {
      uint32_t base = 0;
      if (lane == 0) base = atomicAdd(&rx[3], __popc(m));
      base = __shfl_sync(kFull, base, 0);
      const uint32_t dst = base + __popc(m & lanemask_lt());
      if (keep && dst < (uint32_t)k) scratch[dst] = key;
    }
  }
  consumer_sync();
  const uint32_t kept = rx[3] < (uint32_t)k ? rx[3] : (uint32_t)k;
  for (uint32_t i = ctid; i < kept; i += kCT) cand[i] = scratch[i];
  if (ctid == 0) {
    *cnt = kept;
    *thr = t;
    if (nge > (uint32_t)k) atomicMax(reinterpret_cast<unsigned long long*>(gth), (unsigned long long)t);
  }
  consumer_sync();
}

// Shared-memory layout of a scoring CTA.
struct ScoreSmem {
  int stages, stage_bytes;
  uint8_t* ring;
  uint64_t* full;
  uint64_t* empty;
  uint32_t* cnt;      // [8]
  uint64_t* thr;      // [8]
  uint32_t* hist;     // [256]
  uint32_t* rx;       // [10]
  uint64_t* fl;       // [1]
  uint64_t* cand;     // [P][cap]
  uint64_t* scratch;  // [k]
  template <class KF>
  __device__ void carve(uint8_t* smem, int P, int cap) {
    stages = KF::kStages;
    stage_bytes = KF::kStageBytes;
    ring = smem;
    full = reinterpret_cast<uint64_t*>(smem + KF::kStages * KF::kStageBytes);
    empty = full + KF::kStages;
    cnt = reinterpret_cast<uint32_t*>(empty + KF::kStages);
    thr = reinterpret_cast<uint64_t*>(cnt + 8);
    hist = reinterpret_cast<uint32_t*>(thr + 8);
    rx = hist + 256;
    fl = reinterpret_cast<uint64_t*>(rx + 10);
    cand = fl + 1;
    scratch = cand + (size_t)P * cap;
  }
};

// ---------------------------------------------------------------------------
// Per-lane scoring machinery of one consumer warp (16 warps x 8 keys = one tile)
// ---------------------------------------------------------------------------
// Lane layout of a consumer warp: groups of G lanes (G = 16: a half-warp
// scores 4 keys, lane j holds elements 8j .. 8j+7 of every query; G = 8: a
// quarter-warp scores 2 keys, lane j holds elements 16j .. 16j+15); after the
// tree over the group each lane keeps VL (token, position) results.  A warp
// scores 8 keys either way.
template <int PP, int G = 16>
struct ScorerLanes {
  static constexpr int KPG = G / 4;                 // keys per group: 8 keys per warp / (32 / G) groups
  static constexpr int V = KPG * PP;                // (token, position) pairs per lane
  static constexpr int VL = V >= G ? V / G : 1;     // values left per lane after the tree
  static constexpr int LPP = PP == 1 ? 0 : PP == 2 ? 1 : PP == 4 ? 2 : 3;

  int lane, j, X, px, tx, rowbase;
  bool owner;
  int rrow[VL], rpos[VL];
  uint32_t lead[VL], same[VL];

  // Slot (tau, p) of this lane scores token row tau ^ tx against position
  // p ^ px.  Result r is (row rrow[r], position rpos[r]); for insertion, lane
  // q < P leads position q: lead[r] = lanes reporting position q, same[r] =
  // lanes reporting this lane's position.
  __device__ __forceinline__ void init_lanes(int warp, int lane_) {
    lane = lane_;
    const int h = lane / G;
    j = lane & (G - 1);
    X = tree_perm<V, G>(lane);
    tx = X >> LPP;
    px = X & (PP - 1);
    owner = tree_owner<V, G>(lane);
    rowbase = warp * 8 + h * KPG;
#pragma unroll
    for (int r = 0; r < VL; ++r) {
      const int cmb = r ^ X;
      rrow[r] = warp * 8 + h * KPG + (cmb >> LPP);
      rpos[r] = cmb & (PP - 1);
      lead[r] = 0;
      same[r] = 0;
      for (int q = 0; q < PP; ++q) {
        const uint32_t m = __ballot_sync(kFull, owner && rpos[r] == q);
        if (lane == q) lead[r] = m;
        if (rpos[r] == q) same[r] = m;
      }
    }
  }

  // Inserts the tile's results that reach their position's threshold.
  // t: token of row 0; nt: rows in the tile; len: unit length.
  __device__ __forceinline__ void filter(const float (&acc)[V], int64_t t, int nt, int64_t len, int P,
                                         const uint64_t* thr, uint32_t* cnt, uint64_t* cand, int cap) {
    // full tiles whose tokens every position sees need no per-result tests
    const bool interior = nt == kTile && t + kTile <= len - (P - 1);
#pragma unroll
    for (int r = 0; r < VL; ++r) {
      const int p = rpos[r];
      const int64_t tok = t + rrow[r];
      float s = acc[r];
      if (s == 0.f) s = 0.f;  // +0 for a zero score
      const uint64_t key = sel_key(s, (uint32_t)tok);
      bool ok = owner && p < P;
      if (!interior) ok = ok && rrow[r] < nt && tok < len - (P - 1 - p);
      const bool pass = ok && key >= thr[p];
      const uint32_t mall = __ballot_sync(kFull, pass);
      if (mall) {
        uint32_t base = 0;
        if (lane < P) {
          const uint32_t n_here = __popc(mall & lead[r]);
          if (n_here) base = atomicAdd(&cnt[lane], n_here);
        }
        base = __shfl_sync(kFull, base, p);
        if (pass) {
          const uint32_t dst = base + __popc(mall & same[r] & lanemask_lt());
          if (dst < (uint32_t)cap) cand[(size_t)p * cap + dst] = key;
        }
      }
    }
  }
};

// bf16 keys: the canonical fp32 score (reading R1).
template <int PP>
struct Scorer : ScorerLanes<PP> {
  using B = ScorerLanes<PP>;
  using B::V; using B::VL; using B::j; using B::px; using B::tx; using B::rowbase;
  static constexpr int PH = PP >= 2 ? PP / 2 : 1;  // position pairs (packed fp32x2 FMA)
  int rowoff[4];
  float qf[PP][8];
  float2 qp[PH][8];

  __device__ __forceinline__ void init(int warp, int lane_) {
    B::init_lanes(warp, lane_);
#pragma unroll
    for (int tau = 0; tau < 4; ++tau) rowoff[tau] = (rowbase + (tau ^ tx)) * kKeyBytes + j * 16;
  }

  // This lane's chunk of unit i's queries, in slot order (fp32, exact).
  __device__ __forceinline__ void load_queries(const SelectArgs& a, int64_t i, int P) {
#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int pq = p ^ px;
      if (pq < P) {
        const uint4 v = *reinterpret_cast<const uint4*>(a.queries + (i * P + pq) * kDim + j * 8);
        qf[p][0] = bf_lo(v.x); qf[p][1] = bf_hi(v.x);
        qf[p][2] = bf_lo(v.y); qf[p][3] = bf_hi(v.y);
        qf[p][4] = bf_lo(v.z); qf[p][5] = bf_hi(v.z);
        qf[p][6] = bf_lo(v.w); qf[p][7] = bf_hi(v.w);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) qf[p][e] = 0.f;
      }
    }
#pragma unroll
    for (int m = 0; m < PH; ++m)
#pragma unroll
      for (int e = 0; e < 8; ++e) qp[m][e] = make_float2(qf[2 * m][e], PP >= 2 ? qf[(2 * m + 1) % PP][e] : 0.f);
  }

  // Scores a ring stage holding the tile that starts at token t; release() is
  // called once the stage is no longer read.
  template <class Release>
  __device__ __forceinline__ void score(const uint8_t* stage, int64_t t, float (&acc)[V], Release release) {
    score_rows(stage, acc, release, [&](int tau) { return rowoff[tau]; });
  }

  // Same for nt keys of unit u from token t in global memory: rows past the
  // end read the last row instead (their results are discarded by filter()).
  __device__ __forceinline__ void score_global(const SelectArgs& a, int u, int64_t t, int nt, float (&acc)[V]) {
    const uint8_t* tile = reinterpret_cast<const uint8_t*>(a.keys + ((int64_t)u * a.stride + t) * kDim);
    score_rows(tile, acc, [] {}, [&](int tau) {
      const int r = rowbase + (tau ^ tx);
      return (r < nt ? r : nt - 1) * kKeyBytes + j * 16;
    });
  }

  template <class Release, class Off>
  __device__ __forceinline__ void score_rows(const uint8_t* tile, float (&acc)[V], Release release, Off off) {
#pragma unroll
    for (int tau = 0; tau < 4; ++tau) {
      const uint4 kv = *reinterpret_cast<const uint4*>(tile + off(tau));
      const float kf[8] = {bf_lo(kv.x), bf_hi(kv.x), bf_lo(kv.y), bf_hi(kv.y),
                           bf_lo(kv.z), bf_hi(kv.z), bf_lo(kv.w), bf_hi(kv.w)};
      if constexpr (PP >= 2) {
        // positions 2m and 2m+1 at once; each lane of the pair is the
        // position's own FMA chain in element order
        float2 s2[PH];
#pragma unroll
        for (int m = 0; m < PH; ++m) s2[m] = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 kk = make_float2(kf[e], kf[e]);
#pragma unroll
          for (int m = 0; m < PH; ++m) s2[m] = __ffma2_rn(qp[m][e], kk, s2[m]);
        }
#pragma unroll
        for (int m = 0; m < PH; ++m) {
          acc[tau * PP + 2 * m] = s2[m].x;
          acc[tau * PP + 2 * m + 1] = s2[m].y;
        }
      } else {
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) s = __fmaf_rn(qf[0][e], kf[e], s);
        acc[tau] = s;
      }
    }
    release();
    tree16<V>(acc);
  }
};

// int8 keys (reading R12): exact int32 dot products of the codes (4-byte dot
// instructions, tree of integer sums), then (((float)dot * s_q) * s_k) / 128.
template <int PP>
struct ScorerI8 : ScorerLanes<PP, 8> {
  // Groups of 8 lanes: the integer dot products are exact, so their order is
  // free, and 8 lanes per key halve the tree's shuffles against 16.
  using B = ScorerLanes<PP, 8>;
  using B::V; using B::VL; using B::KPG; using B::j; using B::px; using B::tx; using B::rowbase; using B::rrow;
  using B::rpos;
  int qi[PP][4];    // this lane's 16 query codes per slot position
  float qs[VL];     // query scale of each result's position (fp16, read as fp32)

  __device__ __forceinline__ void init(int warp, int lane_) { B::init_lanes(warp, lane_); }

  __device__ __forceinline__ void load_queries(const SelectArgs& a, int64_t i, int P) {
#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int pq = p ^ px;
      if (pq < P) {
        const uint4 v = *reinterpret_cast<const uint4*>(a.q8 + (i * P + pq) * kDim + j * 16);
        qi[p][0] = (int)v.x;
        qi[p][1] = (int)v.y;
        qi[p][2] = (int)v.z;
        qi[p][3] = (int)v.w;
      } else {
        qi[p][0] = qi[p][1] = qi[p][2] = qi[p][3] = 0;
      }
    }
#pragma unroll
    for (int r = 0; r < VL; ++r)
      qs[r] = rpos[r] < P ? __half2float(__ushort_as_half(a.qscale[i * P + rpos[r]])) : 0.f;
  }

  template <class Release>
  __device__ __forceinline__ void score(const uint8_t* stage, int64_t t, float (&acc)[V], Release release) {
    const uint16_t* scales = reinterpret_cast<const uint16_t*>(stage + KeysInt8::kScaleOff) + (t & 7);
    score_rows(stage, scales, acc, release, [](int r) { return r; });
  }

  // nt keys of unit u from token t in global memory; rows past the end read
  // the last row (their results are discarded by filter()).
  __device__ __forceinline__ void score_global(const SelectArgs& a, int u, int64_t t, int nt, float (&acc)[V]) {
    const int64_t base = (int64_t)u * a.stride + t;
    score_rows(reinterpret_cast<const uint8_t*>(a.keys8 + base * kDim), a.kscale + base, acc, [] {},
               [nt](int r) { return r < nt ? r : nt - 1; });
  }

  template <class Release, class Clamp>
  __device__ __forceinline__ void score_rows(const uint8_t* codes, const uint16_t* scales, float (&acc)[V],
                                             Release release, Clamp clamp) {
    int32_t ai[V];
#pragma unroll
    for (int tau = 0; tau < KPG; ++tau) {
      const uint4 kv = *reinterpret_cast<const uint4*>(codes + clamp(rowbase + (tau ^ tx)) * kDim + j * 16);
#pragma unroll
      for (int p = 0; p < PP; ++p)
        ai[tau * PP + p] = __dp4a((int)kv.x, qi[p][0],
                                  __dp4a((int)kv.y, qi[p][1], __dp4a((int)kv.z, qi[p][2], __dp4a((int)kv.w, qi[p][3], 0))));
    }
    // the results' key scales, before the stage may be refilled
    float ks[VL];
#pragma unroll
    for (int r = 0; r < VL; ++r) ks[r] = __half2float(__ushort_as_half(scales[clamp(rrow[r])]));
    release();
    tree8<V>(ai);
#pragma unroll
    for (int r = 0; r < VL; ++r) acc[r] = ((((float)ai[r]) * qs[r]) * ks[r]) * 0.0078125f;
  }
};

// Producer side: streams keys [t, t + nt) of unit u into a ring stage and
// arms its barrier with the byte count (int8: the code rows, then the scales
// from token t - t % 8, rounded up to 16 bytes; the scale array of a unit is
// padded to a multiple of 8 tokens, so the copy stays inside it).
template <class KF>
__device__ __forceinline__ void issue_tile(const SelectArgs& a, uint8_t* stage, uint64_t* full, int u, int64_t t,
                                           int nt, uint64_t pol) {
  const int64_t row = (int64_t)u * a.stride + t;
  if constexpr (KF::kInt8) {
    const int d = (int)(t & 7);  // the scales start at token t - d (16-byte aligned)
    const uint32_t cb = (uint32_t)nt * kDim, sb = ((uint32_t)(nt + d) * 2u + 15u) & ~15u;
    mbar_arrive_expect_tx(full, cb + sb);
    bulk_g2s_hint(stage, a.keys8 + row * kDim, cb, full, pol);
    bulk_g2s_hint(stage + KeysInt8::kScaleOff, a.kscale + (row - d), sb, full, pol);
  } else {
    const uint32_t bytes = (uint32_t)nt * kKeyBytes;
    mbar_arrive_expect_tx(full, bytes);
    bulk_g2s_hint(stage, a.keys + row * kDim, bytes, full, pol);
  }
}

// ---------------------------------------------------------------------------
// Miss-row copy by 16-byte loads from the mapped host pool (zero copy), NT
// threads per CTA, batches of up to ROWS rows of one unit, each thread with up
// to U loads in flight.  Used by the gather kernel (every CTA of its launch)
// and by a score launch of a staged step in unit groups (the previous group's
// rows: its first CTAs copy them, its scoring CTAs help once they are done).
// ---------------------------------------------------------------------------
struct CopyScratch {      // shared memory of a copying CTA
  int64_t* src_off;       // [ROWS]
  int64_t* dst_off;       // [ROWS]
  int32_t* list;          // [NT] (helpers)
  uint32_t* word;         // [4]: rows of unmapped blocks, claimed batch, list count
};

// Rows [b0, b0 + nrow) of unit i's miss list (all threads; ends with a barrier).
template <int NT, int U>
__device__ __forceinline__ void copy_batch(const GatherArgs& a, int i, int64_t b0, int nrow, const CopyScratch& cs) {
  const int tid = threadIdx.x;
  const int cpr = a.row_elems / 8;  // 16-byte chunks per row
  if (tid < nrow) {
    const int64_t loc = b0 + tid - a.miss_off[i];
    const int u = a.units[i];
    const int32_t t = a.miss_tok[(int64_t)i * a.pk + loc];
    const int32_t s = a.miss_slot[(int64_t)i * a.pk + loc];
    const int64_t hr = host_row(a.rows, u, t);
    cs.src_off[tid] = hr < 0 ? -1 : hr * a.row_elems;
    cs.dst_off[tid] = ((int64_t)u * a.C + s) * a.row_elems;
    if (hr < 0) atomicAdd(&cs.word[0], 1u);
  }
  __syncthreads();
  const int total = nrow * cpr;
  for (int q0 = tid; q0 < total; q0 += NT * U) {
    uint4 v[U];
#pragma unroll
    for (int x = 0; x < U; ++x) {
      const int q = q0 + x * NT;
      if (q < total) {
        const int row = q / cpr, c = q - row * cpr;
        if (cs.src_off[row] >= 0) v[x] = *reinterpret_cast<const uint4*>(a.host_pool + cs.src_off[row] + c * 8);
      }
    }
#pragma unroll
    for (int x = 0; x < U; ++x) {
      const int q = q0 + x * NT;
      if (q < total) {
        const int row = q / cpr, c = q - row * cpr;
        if (cs.src_off[row] >= 0) *reinterpret_cast<uint4*>(a.hot + cs.dst_off[row] + c * 8) = v[x];
      }
    }
  }
  __syncthreads();
}

// Unit i's batches taken one at a time from its claim counter (shared with the
// other CTAs that copy or help); returns the rows this CTA copied.
template <int NT, int ROWS, int U>
__device__ __forceinline__ int64_t copy_claimed(const GatherArgs& a, int i, const CopyScratch& cs) {
  const int64_t r0 = a.miss_off[i], r1 = a.miss_off[i + 1];
  int64_t moved = 0;
  for (;;) {
    if (threadIdx.x == 0) cs.word[1] = (uint32_t)atomicAdd(&a.claim[i], 1);
    __syncthreads();
    const int64_t b0 = r0 + (int64_t)cs.word[1] * ROWS;
    __syncthreads();  // every thread has read the claim before the next one is written
    if (b0 >= r1) return moved;
    const int nrow = (int)((r1 - b0) < ROWS ? (r1 - b0) : ROWS);
    copy_batch<NT, U>(a, i, b0, nrow, cs);
    moved += nrow;
  }
}

// Adds a CTA's copied rows to the statistics (thread 0, after a barrier).
__device__ __forceinline__ void copy_stats(const GatherArgs& a, int64_t moved, const CopyScratch& cs, bool in_score) {
  if (threadIdx.x == 0 && a.stats) {
    const uint32_t bad = cs.word[0];
    moved -= bad;
    if (moved) {
      atomicAdd(&a.stats->rows_h2d, (unsigned long long)moved);
      atomicAdd(&a.stats->bytes_h2d, (unsigned long long)moved * a.row_elems * 2ull);
      if (in_score) atomicAdd(&a.stats->rows_h2d_in_score, (unsigned long long)moved);
    }
    if (bad) atomicAdd(&a.stats->block_errors, (unsigned long long)bad);
  }
}

// CTA `cta` of `ncta` copying CTAs.  Units are assigned to CTAs by their place in the
// list (i, i + ncta, ...), the same in every step: the rows one CTA reads then stay in the
// same few units' regions of the pool from step to step, and the GPU keeps those regions'
// address translations.  Taken in any order that changes between steps, the translations
// of a 38.7 GB pool are missed again each step and the same copy runs at half the rate
// (probe: 208 GB/s with a fixed unit-to-CTA assignment, 89-107 GB/s with rows or units
// claimed dynamically).  With claim counters (a.claim), a unit's batches are still taken
// in order by its CTA, but CTAs that help (copy_help) may take the last ones.  Without
// them and with fewer units than CTAs, each unit gets k = ncta / n CTAs, which take its
// batches in turn (again the same CTAs for the same unit in every step).
template <int NT, int ROWS, int U>
__device__ __forceinline__ void gather_rows_ldg(const GatherArgs& a, int cta, int ncta, const CopyScratch& cs,
                                                bool in_score = false) {
  static_assert(ROWS <= NT, "one thread per row of a batch fetches its addresses");
  const int tid = threadIdx.x;
  int64_t moved = 0;
  if (tid == 0) cs.word[0] = 0;
  __syncthreads();
  if (a.claim) {
    for (int i = cta; i < a.n; i += ncta) moved += copy_claimed<NT, ROWS, U>(a, i, cs);
  } else {
    const int k = a.n >= ncta || a.n <= 0 ? 1 : ncta / a.n;
    const int first = k == 1 ? cta : cta / k, sub = k == 1 ? 0 : cta % k;
    const int ustep = k == 1 ? ncta : a.n;
    for (int i = first; i < a.n; i += ustep)
      for (int64_t b0 = a.miss_off[i] + (int64_t)sub * ROWS; b0 < a.miss_off[i + 1]; b0 += (int64_t)k * ROWS) {
        const int64_t R_i = a.miss_off[i + 1];
        const int nrow = (int)((R_i - b0) < ROWS ? (R_i - b0) : ROWS);
        copy_batch<NT, U>(a, i, b0, nrow, cs);
        moved += nrow;
      }
  }
  __syncthreads();
  copy_stats(a, moved, cs, in_score);
}

// A CTA that has finished its own work takes the batches the copying CTAs have not yet
// claimed, scanning the units from the end of the list (the copying CTAs take theirs
// from the front).  When the copy keeps pace with the scoring, nothing is left.
template <int NT, int ROWS, int U>
__device__ __forceinline__ void copy_help(const GatherArgs& a, const CopyScratch& cs) {
  const int tid = threadIdx.x;
  int64_t moved = 0;
  if (tid == 0) cs.word[0] = 0;
  for (int base = 0; base < a.n; base += NT) {
    if (tid == 0) cs.word[2] = 0;
    __syncthreads();
    if (base + tid < a.n) {
      const int i = a.n - 1 - (base + tid);
      const int64_t rows = a.miss_off[i + 1] - a.miss_off[i];
      const int nb = (int)((rows + ROWS - 1) / ROWS);
      if (*reinterpret_cast<const volatile int32_t*>(&a.claim[i]) < nb) cs.list[atomicAdd(&cs.word[2], 1u)] = i;
    }
    __syncthreads();
    const int cnt = (int)cs.word[2];
    for (int e = 0; e < cnt; ++e) moved += copy_claimed<NT, ROWS, U>(a, cs.list[e], cs);
    __syncthreads();
  }
  copy_stats(a, moved, cs, true);
}

template <int PP, class KF>
struct ScorerFor {
  using type = Scorer<PP>;
};
template <int PP>
struct ScorerFor<PP, KeysInt8> {
  using type = ScorerI8<PP>;
};
// Start of a piece: counters cleared, thresholds set (consumer threads).
__device__ __forceinline__ void piece_begin(const ScoreSmem& sm, int P, const uint64_t* start_thr, int ctid) {
  if (ctid < P) {
    sm.cnt[ctid] = 0;
    sm.thr[ctid] = start_thr ? start_thr[ctid] : 0ull;
  }
  consumer_sync();
}

// Every kCheckTiles tiles: adopt the unit's shared thresholds and compact the
// buffers that could overflow within the next tiles.
__device__ __forceinline__ void piece_check(const ScoreSmem& sm, int P, int k, int cap, uint64_t* gth, int ctid) {
  consumer_sync();
  const uint32_t trigger = (uint32_t)(cap - kCheckTiles * kTile);
  bool need = false;
  for (int p = 0; p < P; ++p) need |= sm.cnt[p] > trigger;
  if (ctid < P) {
    const uint64_t g = __ldcg(reinterpret_cast<const unsigned long long*>(gth + ctid));
    if (g > sm.thr[ctid]) sm.thr[ctid] = g;
  }
  if (need) {
    for (int p = 0; p < P; ++p)
      if (sm.cnt[p] > trigger)
        compact_candidates(sm.cand + (size_t)p * cap, &sm.cnt[p], &sm.thr[p], gth + p, sm.fl, sm.scratch, sm.hist,
                           sm.rx, k, ctid);
  }
}

// End of a piece: at most k candidates per position, written to segment `seg`.
__device__ __forceinline__ void piece_end(const ScoreSmem& sm, int P, int k, int cap, uint64_t* gth, int64_t seg,
                                          uint64_t* seg_keys, int32_t* seg_cnt, int ctid) {
  consumer_sync();
  // at most k per position; keys under the shared threshold may stay (select drops them)
  for (int p = 0; p < P; ++p)
    if (sm.cnt[p] > (uint32_t)k)
      compact_candidates(sm.cand + (size_t)p * cap, &sm.cnt[p], &sm.thr[p], gth + p, sm.fl, sm.scratch, sm.hist,
                         sm.rx, k, ctid);
  for (int p = 0; p < P; ++p) {
    const uint32_t np = sm.cnt[p];
    uint64_t* dst = seg_keys + (seg * P + p) * (int64_t)k;
    for (uint32_t e = ctid; e < np; e += kCT) dst[e] = sm.cand[(size_t)p * cap + e];
    if (ctid == 0) seg_cnt[seg * P + p] = (int32_t)np;
  }
  consumer_sync();
}

// Candidates of (unit i, position p) over segments [seg0, seg0 + nseg).
// Segments may have been written by other CTAs of the same launch: read
// through L2.
__device__ __forceinline__ uint32_t candidate_count(const SelectArgs& a, int p, int64_t seg0, int nseg) {
  uint32_t n = 0;
  for (int c = 0; c < nseg; ++c) n += (uint32_t)__ldcg(&a.seg_cnt[(seg0 + c) * a.P + p]);
  return n;
}

// Whether the speculative threshold of (unit i, position p) was too high.  It
// is exact when at least min(k, visible) keys reached it: then every key of
// the top k did.
__device__ __forceinline__ bool spec_short(const SelectArgs& a, int i, int p, uint32_t n) {
  if (!a.tspec || a.tspec[(int64_t)i * a.P + p] == 0) return false;
  const int64_t vis = (a.off[i + 1] - a.off[i]) - (a.P - 1 - p);
  const uint32_t need = (uint32_t)(vis < a.k ? (vis > 0 ? vis : 0) : a.k);
  return n < need;
}

// For positions p0 .. p0+np-1 (warp w handles p0 + w; np <= NT / 32):
// seg_off[w * (nseg + 1) + c] = candidates of (., p0 + w) in segments
// seg0 .. seg0+c-1, c <= nseg; one load per lane per 32 segments.
template <int NT, class Sync>
__device__ __forceinline__ void segment_offsets(const SelectArgs& a, int p0, int np, int64_t seg0, int nseg,
                                                uint32_t* seg_off, int tid, Sync sync) {
  const int w = tid >> 5, lane = tid & 31;
  if (w < np) {
    const int p = p0 + w;
    uint32_t* so = seg_off + w * (nseg + 1);
    uint32_t carry = 0;
    for (int b = 0; b < nseg; b += 32) {
      const int c = b + lane;
      const uint32_t v = c < nseg ? (uint32_t)__ldcg(&a.seg_cnt[(seg0 + c) * a.P + p]) : 0u;
      uint32_t incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      if (c < nseg) so[c] = carry + incl - v;
      carry += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) so[nseg] = carry;
  }
  sync();
}

// Writes ranks [0, k) of (unit i, position p) from W[0 .. count) (winners in
// rank order, shared memory), padding after; four payload lookups in flight
// per thread.
template <int NT>
__device__ __forceinline__ void write_ranks(const SelectArgs& a, int i, int p, const uint64_t* W, int count,
                                            int tid) {
  const int k = a.k;
  const int64_t ob = ((int64_t)i * a.P + p) * k;
  const int32_t* cs = a.cache_slots ? a.cache_slots + (int64_t)a.units[i] * a.stride : nullptr;
  for (int r0 = tid; r0 < k; r0 += 4 * NT) {
    uint64_t key[4];
    int32_t slot[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = r0 + u * NT;
      key[u] = r < count ? W[r] : 0ull;
      slot[u] = (r < count && cs) ? cs[key_token(key[u])] : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = r0 + u * NT;
      if (r >= k) break;
      int32_t tok = -1, pay = KVO_PAD_PAYLOAD;
      float sc = __uint_as_float(0xff800000u);
      if (r < count) {
        tok = (int32_t)key_token(key[u]);
        sc = key_score(key[u]);
        pay = slot[u] >= 0 ? slot[u] : -(tok + 1);
      }
      a.out_tok[ob + r] = tok;
      if (a.out_score) a.out_score[ob + r] = sc;
      a.out_pay[ob + r] = pay;
      if (a.out_pay_user && a.out_pay_user != a.out_pay) a.out_pay_user[ob + r] = pay;
    }
  }
}

// State the next step's speculative threshold starts from: the k-th best key
// (0 when fewer than k tokens were visible) and this step's query norm.
__device__ __forceinline__ void write_spec(const SelectArgs& a, int i, int p, uint64_t kth) {
  if (!a.spec) return;
  const int u = a.units[i];
  a.spec[(int64_t)u * a.P + p] = kth;
  if (a.qn_prev && a.qn_cur) a.qn_prev[(int64_t)u * a.P + p] = a.qn_cur[(int64_t)i * a.P + p];
}

// ---------------------------------------------------------------------------
// Exact top-k of one (unit i, position p) over segments [seg0, seg0 + nseg)
// with NT threads.  Returns false when the speculative threshold of (i, p)
// was too high (then nothing is written).  Shared memory: keys (keycap u64;
// more candidates than that are read from global memory instead), sorted
// (kpad u64, kpad = k rounded up to a power of two), hist[256], rx[10]
// (8-byte aligned).
// ---------------------------------------------------------------------------
template <int NT, class Sync>
__device__ __forceinline__ bool select_body(const SelectArgs& a, int i, int p, int64_t seg0, int nseg,
                                            bool verify, uint64_t* keys, uint32_t keycap, uint64_t* sorted,
                                            uint32_t* hist, uint32_t* rx, int tid, Sync sync) {
  const int P = a.P, k = a.k;
  const int64_t s0 = a.off[i], s1 = a.off[i + 1];
  // segments may have been written by other CTAs of the same launch: read through L2
  auto seg_count = [&](int64_t seg) { return (uint32_t)__ldcg(&a.seg_cnt[seg * P + p]); };
  uint32_t n = 0;
  for (int c = 0; c < nseg; ++c) n += seg_count(seg0 + c);
  // A speculative threshold is exact when at least min(k, visible) keys
  // reached it: then every key of the top k did.
  if (verify && a.tspec && a.tspec[(int64_t)i * P + p] != 0) {
    const int64_t vis = (s1 - s0) - (P - 1 - p);
    const uint32_t need = (uint32_t)(vis < k ? (vis > 0 ? vis : 0) : k);
    if (n < need) return false;
  }
  const bool in_smem = n <= keycap;
  if (in_smem) {
    uint32_t base = 0;
    for (int c = 0; c < nseg; ++c) {
      const int64_t seg = seg0 + c;
      const uint32_t m = seg_count(seg);
      const uint64_t* src = a.seg_keys + (seg * P + p) * (int64_t)k;
      for (uint32_t e = tid; e < m; e += NT) keys[base + e] = __ldcg(src + e);
      base += m;
    }
    sync();
  }
  auto for_each = [&](auto f) {
    if (in_smem) {
      for (uint32_t e = tid; e < n; e += NT) f(keys[e]);
    } else {
      for (int c = 0; c < nseg; ++c) {
        const int64_t seg = seg0 + c;
        const uint32_t m = seg_count(seg);
        const uint64_t* src = a.seg_keys + (seg * P + p) * (int64_t)k;
        for (uint32_t e = tid; e < m; e += NT) f(__ldcg(src + e));
      }
    }
  };
  uint64_t thr = 0;
  if (n > (uint32_t)k) thr = radix_threshold_desc<NT>(for_each, (uint32_t)k, hist, rx, tid, sync);
  const uint32_t count = n < (uint32_t)k ? n : (uint32_t)k;
  int kpad = 1;
  while (kpad < k) kpad <<= 1;
  if (tid == 0) rx[9] = 0;
  sync();
  const int lane = tid & 31;
  // keys >= thr go to the sort buffer (uniform trip counts: full-warp ballots)
  // src is shared memory (from_global false) or a segment in global memory
  auto keep_from = [&](const uint64_t* src, uint32_t m, bool from_global) {
    for (uint32_t b = 0; b < m; b += NT) {
      const uint32_t e = b + tid;
      const uint64_t key = e < m ? (from_global ? __ldcg(src + e) : src[e]) : 0;
      const bool keep = e < m && key >= thr;
      const uint32_t msk = __ballot_sync(kFull, keep);
      if (msk) {
        uint32_t base = 0;
        if (lane == 0) base = atomicAdd(&rx[9], __popc(msk));
        base = __shfl_sync(kFull, base, 0);
        const uint32_t dst = base + __popc(msk & lanemask_lt());
        if (keep && dst < (uint32_t)kpad) sorted[dst] = key;
      }
    }
  };
  if (in_smem) {
    keep_from(keys, n, false);
  } else {
    for (int c = 0; c < nseg; ++c) {
      const int64_t seg = seg0 + c;
      keep_from(a.seg_keys + (seg * P + p) * (int64_t)k, seg_count(seg), true);
    }
  }
  sync();
  for (int e = count + tid; e < kpad; e += NT) sorted[e] = 0;
  sync();
  block_sort_desc<NT>(sorted, kpad, tid, sync);

  write_ranks<NT>(a, i, p, sorted, (int)count, tid);
  if (tid == 0) write_spec(a, i, p, count >= (uint32_t)k ? sorted[k - 1] : 0ull);
  sync();
  return true;
}

constexpr uint32_t kMaxBucket = 256;

// ---------------------------------------------------------------------------
// Exact top-k of one (unit i, position p) by a bucket sort, for candidate
// sets that fit shared memory: the key range [lo, hi] is cut into B buckets
// of equal width (numbered from the top), a histogram and its prefix give
// each bucket's first rank, the keys are scattered to their buckets, and a
// key's rank is its bucket's first rank plus the number of larger keys in the
// same bucket.  A few barriers instead of the radix passes and the bitonic
// network; each candidate's cache_slots entry is fetched with the candidates
// (one more batch of loads) and the outputs are written straight from the
// rank pass.  seg_off: segment_offsets() of (., p) in shared memory.  Returns
// false, having written nothing, when the candidates exceed what `region`
// holds or a bucket holds more than kMaxBucket keys (then the caller runs
// select_body).  region: `bytes` of shared memory (16-byte aligned); wsum:
// 32 words.
// ---------------------------------------------------------------------------
template <int NT, class Sync>
__device__ __forceinline__ bool bucket_select(const SelectArgs& a, int i, int p, int64_t seg0, int nseg,
                                              const uint32_t* seg_off, uint8_t* region, size_t bytes, int log2B,
                                              uint32_t* wsum, int tid, Sync sync) {
  const int P = a.P, k = a.k;
  const int B = 1 << log2B;
  uint32_t* cnt = reinterpret_cast<uint32_t*>(region);        // [B]
  uint32_t* pos = cnt + B;                                    // [B]
  unsigned long long* red = reinterpret_cast<unsigned long long*>(pos + B);  // [4]
  const size_t fixed = (size_t)8 * B + 32;
  const uint32_t keycap = bytes > fixed ? (uint32_t)((bytes - fixed) / 24) : 0u;
  uint64_t* K = reinterpret_cast<uint64_t*>(red + 4);         // [keycap] candidates
  uint64_t* S = K + keycap;                                   // [keycap] candidates by bucket
  int32_t* KC = reinterpret_cast<int32_t*>(S + keycap);       // [keycap] cache_slots of K
  int32_t* SC = KC + keycap;                                  // [keycap] cache_slots of S
  const uint32_t n = seg_off[nseg];
  if (n > keycap) return false;
  const int u = a.units[i];
  const int32_t* cs = a.cache_slots ? a.cache_slots + (int64_t)u * a.stride : nullptr;
  const int64_t ob = ((int64_t)i * P + p) * k;
  auto emit = [&](int r, uint64_t key, int32_t slot) {
    const int32_t tok = (int32_t)key_token(key);
    a.out_tok[ob + r] = tok;
    if (a.out_score) a.out_score[ob + r] = key_score(key);
    const int32_t pay = slot >= 0 ? slot : -(tok + 1);
    a.out_pay[ob + r] = pay;
    if (a.out_pay_user && a.out_pay_user != a.out_pay) a.out_pay_user[ob + r] = pay;
  };
  auto pad = [&](int r) {
    a.out_tok[ob + r] = -1;
    if (a.out_score) a.out_score[ob + r] = __uint_as_float(0xff800000u);
    a.out_pay[ob + r] = KVO_PAD_PAYLOAD;
    if (a.out_pay_user && a.out_pay_user != a.out_pay) a.out_pay_user[ob + r] = KVO_PAD_PAYLOAD;
  };
  if (n == 0) {
    for (int r = tid; r < k; r += NT) pad(r);
    if (tid == 0) write_spec(a, i, p, 0ull);
    sync();
    return true;
  }
  if (tid == 0) {
    red[0] = ~0ull;
    red[1] = 0ull;
    red[2] = 0ull;
  }
  for (int b = tid; b < B; b += NT) cnt[b] = 0;
  // candidates of every piece into K with their cache_slots entries (eight
  // of each in flight per thread), and the key range
  unsigned long long lo = ~0ull, hi = 0ull;
  for (uint32_t e0 = tid; e0 < n; e0 += 8 * NT) {
    uint64_t v[8];
    int32_t c[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      const uint32_t e = e0 + x * NT;
      v[x] = 0;
      if (e < n) {
        int lo_c = 0, hi_c = nseg - 1;  // last segment with seg_off <= e
        while (lo_c < hi_c) {
          const int mid = (lo_c + hi_c + 1) >> 1;
          if (seg_off[mid] <= e) lo_c = mid; else hi_c = mid - 1;
        }
        v[x] = __ldcg(a.seg_keys + ((seg0 + lo_c) * P + p) * (int64_t)k + (e - seg_off[lo_c]));
      }
    }
#pragma unroll
    for (int x = 0; x < 8; ++x) c[x] = (e0 + x * NT < n && cs) ? cs[key_token(v[x])] : -1;
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      const uint32_t e = e0 + x * NT;
      if (e < n) {
        K[e] = v[x];
        KC[e] = c[x];
        lo = v[x] < lo ? v[x] : lo;
        hi = v[x] > hi ? v[x] : hi;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long l2 = __shfl_xor_sync(kFull, lo, o), h2 = __shfl_xor_sync(kFull, hi, o);
    lo = l2 < lo ? l2 : lo;
    hi = h2 > hi ? h2 : hi;
  }
  sync();  // red initialised before the atomics
  if ((tid & 31) == 0) {
    atomicMin(&red[0], lo);
    atomicMax(&red[1], hi);
  }
  sync();
  // bucket = floor((x - lo) * B / (range + 1)) up to rounding, through one
  // precomputed multiplier (exact offsets when the range is below B)
  const uint64_t kmin = red[0], range = red[1] - red[0];
  const bool direct = range < (uint64_t)B;
  const uint64_t mul = direct ? 0ull : (range == ~0ull ? (uint64_t)B : (~0ull / (range + 1)) * (uint64_t)B);
  auto bucket = [&](uint64_t x) {
    const uint64_t d = x - kmin;
    return (uint32_t)(B - 1) - (uint32_t)(direct ? d : __umul64hi(d, mul));
  };
  for (uint32_t e = tid; e < n; e += NT) atomicAdd(&cnt[bucket(K[e])], 1u);
  sync();
  // first rank of every bucket (each thread owns B / NT consecutive buckets)
  constexpr int kMaxPer = 8;
  const int per = B / NT;  // B is a multiple of NT, at most kMaxPer * NT
  uint32_t loc = 0, mx = 0;
  for (int j = 0; j < per && j < kMaxPer; ++j) {
    const uint32_t c = cnt[tid * per + j];
    loc += c;
    mx = c > mx ? c : mx;
  }
  uint32_t total;
  uint32_t run = block_excl_scan<NT>(loc, wsum, &total, tid, sync);
  for (int j = 0; j < per && j < kMaxPer; ++j) {
    pos[tid * per + j] = run;
    run += cnt[tid * per + j];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint32_t m2 = __shfl_xor_sync(kFull, mx, o);
    mx = m2 > mx ? m2 : mx;
  }
  if ((tid & 31) == 0 && mx) atomicMax(&red[2], (unsigned long long)mx);
  sync();
  if (red[2] > kMaxBucket) {
    sync();  // nothing written: the caller may reuse the buffers at once
    return false;
  }
  // scatter (pos[b] ends as the end of bucket b)
  for (uint32_t e = tid; e < n; e += NT) {
    const uint64_t x = K[e];
    const uint32_t j = atomicAdd(&pos[bucket(x)], 1u);
    S[j] = x;
    SC[j] = KC[e];
  }
  sync();
  // rank within the bucket; winners written at their rank
  for (uint32_t j = tid; j < n; j += NT) {
    const uint64_t x = S[j];
    const uint32_t b = bucket(x);
    const uint32_t end = pos[b], beg = end - cnt[b];
    uint32_t r = beg;
    for (uint32_t t = beg; t < end; ++t) r += S[t] > x ? 1u : 0u;
    if (r < (uint32_t)k) {
      emit((int)r, x, SC[j]);
      if (r == (uint32_t)k - 1) write_spec(a, i, p, x);
    }
  }
  for (int r = (int)n + tid; r < k; r += NT) pad(r);
  if (tid == 0 && n < (uint32_t)k) write_spec(a, i, p, 0ull);
  sync();
  return true;
}

// ---------------------------------------------------------------------------
// plan (all NT threads of a CTA; warp_sums[32] and carry in shared memory):
// off[i] = sum of len[units[j]] for j < i (checked against T); the unit's
// shared thresholds zeroed; squared query norms and speculative start
// thresholds; with pbeg set, the piece table, counters and statuses of the
// fused step; the previous step's miss bytes to the host mirror.
// ---------------------------------------------------------------------------
template <int NT>
__device__ __forceinline__ void plan_body(const SelectArgs& a, int tid, int64_t* warp_sums, int64_t* carry_p) {
  int64_t& carry = *carry_p;
  const int lane = tid & 31, w = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < a.n; base += NT) {
    const int i = base + tid;
    const int64_t v = i < a.n ? (int64_t)a.len[a.units[i]] : 0;
    int64_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    if (w == 0) {
      int64_t s = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(kFull, s, o);
        if (lane >= o) s += y;
      }
      warp_sums[lane] = s;
    }
    __syncthreads();
    const int64_t excl = carry + (w ? warp_sums[w - 1] : 0) + incl - v;
    if (i < a.n) a.off[i] = excl;
    __syncthreads();
    if (tid == NT - 1) carry = excl + v;
    __syncthreads();
  }
  for (int e = tid; e < a.n * a.P; e += NT) {
    a.gthr[e] = 0;
    if (!a.tspec) continue;
    const int i = e / a.P, p = e - (e / a.P) * a.P;
    const int u = a.units[i];
    // squared query norm (fp32; only steers the speculative threshold)
    const uint4* q = reinterpret_cast<const uint4*>(a.queries + (int64_t)e * kDim);
    float s2 = 0.f;
#pragma unroll 8
    for (int c = 0; c < kDim / 8; ++c) {
      const uint4 v = q[c];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) s2 += bf_lo(w[x]) * bf_lo(w[x]) + bf_hi(w[x]) * bf_hi(w[x]);
    }
    if (a.qn_cur) a.qn_cur[e] = s2;
    uint64_t t = 0;
    if (a.spec && a.qn_prev && a.spec_scale > 0.f) {
      const uint64_t kth = a.spec[(int64_t)u * a.P + p];
      const float sk = key_score(kth);
      const float prev = a.qn_prev[(int64_t)u * a.P + p];
      const int64_t vis = (int64_t)a.len[u] - (a.P - 1 - p);
      if (kth != 0 && sk > 0.f && prev > 0.f && s2 > 0.f && vis > a.k) {
        const float ts = sk * sqrtf(s2 / prev) * a.spec_scale;
        if (ts > 0.f) t = (uint64_t)order_bits(ts) << 32;
      }
    }
    a.tspec[e] = t;
  }
  if (a.fb) {
    for (int i = tid; i < a.n; i += NT) a.fb[i] = 0;
    if (tid == 0) *a.fb_any = 0;
  }
  if (tid == 0) {
    a.off[a.n] = carry;
    if (carry != a.T) atomicOr(a.err, kErrPlan);
    if (a.bytes_prev && a.stats) {
      const unsigned long long total = a.stats->bytes_h2d;
      *reinterpret_cast<volatile unsigned long long*>(a.bytes_prev) = total - *a.bytes_seen;
      *a.bytes_seen = total;
    }
  }
  if (a.pbeg) {
    // pieces of the fused step: unit i owns pieces_of(i, len) of them
    __syncthreads();
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < a.n; base += NT) {
      const int i = base + tid;
      int64_t v = 0;
      if (i < a.n) v = pieces_of(i, a.len[a.units[i]], a.piece_tokens);
      int64_t incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) warp_sums[w] = incl;
      __syncthreads();
      if (w == 0) {
        int64_t s = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int64_t y = __shfl_up_sync(kFull, s, o);
          if (lane >= o) s += y;
        }
        warp_sums[lane] = s;
      }
      __syncthreads();
      const int64_t excl = carry + (w ? warp_sums[w - 1] : 0) + incl - v;
      if (i < a.n) a.pbeg[i] = excl;
      __syncthreads();
      if (tid == NT - 1) carry = excl + v;
      __syncthreads();
    }
    for (int i = tid; i < a.n; i += NT) {
      a.pdone[i] = 0;
      a.status_init[i] = KVO_ETIMEOUT;
    }
    if (tid < 4) a.ctr[tid] = 0ull;
    if (tid == 0) {
      a.pbeg[a.n] = carry;
      if (carry != a.n_pieces) atomicOr(a.err, kErrPlan);
    }
  }
}

// ---------------------------------------------------------------------------
// Residency update of one unit (listed index i) with NT threads.
//
// No sorting: the distinct misses come out in token order from a token
// bitmap (each thread owns a contiguous run of words; one block scan), and
// the LRU order is an explicit list of the unit's slots kept in (last_use,
// slot) order: victims are the first m entries not hit this step, and the
// step's touched slots (hits and filled misses, all with the new stamp) move
// to the end in slot order.  Every slot starts free with last_use 0, so the
// initial list 0..C-1 is in that order, and the update preserves it.
// Shared memory: bitmap [(C+31)/32] u32, M [P*k] i32, V [P*k] i32, wsum[32].
// ready(m) is called once by all NT threads as soon as the m miss rows and
// their slots (miss_tok, miss_slot) are written: before the LRU list and the
// remap when m > 0, at the end otherwise.  Returns the miss count (0 unless
// the status is OK).
// ---------------------------------------------------------------------------
template <int NT, class Sync, class Ready>
__device__ __forceinline__ uint32_t residency_body(const ResidencyArgs& a, int i, uint32_t* bitmap, int32_t* M,
                                                   int32_t* V, uint32_t* wsum, int tid, Sync sync,
                                                   int32_t* status_out, Ready ready) {
  constexpr int kB = 8;    // loads in flight per thread in the token-bitmap passes
  constexpr int kTB = 16;  // and in the top-k passes
  constexpr int kLB = 16;  // and in the LRU-list passes (one line per lane per load)
  constexpr int NW = NT / 32;
  const int lane = tid & 31, wid = tid >> 5;
  const int C = a.C, PK = a.P * a.k;
  const int nwords = (C + 31) >> 5;
  const int u = a.units[i];
  const int32_t* tok = a.tok + (int64_t)i * PK;
  const int32_t* pay = a.pay + (int64_t)i * PK;
  int32_t* out_slot = a.out_slot + (int64_t)i * PK;
  int32_t* cs = a.cache_slots + (int64_t)u * a.stride;
  int32_t* st = a.slot_token + (int64_t)u * C;
  uint32_t* lu = a.last_use + (int64_t)u * C;
  uint32_t* tbm = a.tok_bits + (int64_t)u * a.tok_words;

  // scalars in one round trip; the error word can change under a concurrent
  // launch, so it is read once and shared
  if (tid == 0) {
    wsum[0] = *((volatile uint32_t*)a.err);
    wsum[1] = a.stamp[u];
    wsum[2] = (uint32_t)a.order_par[u];
    wsum[3] = (uint32_t)a.len[u];
  }
  for (int w = tid; w < nwords; w += NT) bitmap[w] = 0;
  sync();
  int32_t status = wsum[0] != 0 ? KVO_ETIMEOUT : KVO_OK;
  const uint32_t stamp = wsum[1] + 1;
  const int par = (int)wsum[2];
  const int tw = (int)((wsum[3] + 31) >> 5);
  const int32_t* cur = a.order + ((int64_t)par * a.U + u) * C;
  int32_t* nxt = a.order + ((int64_t)(par ^ 1) * a.U + u) * C;
  sync();  // wsum is reused below
  uint32_t m = 0, hits = 0;

  if (status == KVO_OK) {
    // payload says hit (slot) or miss (token): mark hit slots and miss tokens
    for (int e0 = tid; e0 < PK; e0 += kTB * NT) {
      int32_t t[kTB], pv[kTB];
#pragma unroll
      for (int x = 0; x < kTB; ++x) {
        const int e = e0 + x * NT;
        t[x] = e < PK ? tok[e] : -1;
        pv[x] = e < PK ? pay[e] : -1;
      }
#pragma unroll
      for (int x = 0; x < kTB; ++x) {
        if (t[x] < 0) continue;
        if (pv[x] >= 0) {
          if (pv[x] < C) atomicOr(&bitmap[pv[x] >> 5], 1u << (pv[x] & 31));
        } else {
          atomicOr(&tbm[t[x] >> 5], 1u << (t[x] & 31));
        }
      }
    }
    __threadfence_block();
    sync();
    // distinct misses in token order; the bitmap words are cleared behind.
    // Warp w owns words [tb, te); a slice is 32 consecutive words, one per
    // lane, so every load is one coalesced line and emission follows token order.
    const int tpw = (tw + NW - 1) / NW;
    const int tb = min(tw, wid * tpw), te = min(tw, tb + tpw);
    uint32_t c = 0;
    for (int w = tb; w < te; w += 32 * kB) {
      uint32_t wv[kB];
#pragma unroll
      for (int x = 0; x < kB; ++x) wv[x] = w + x * 32 + lane < te ? __ldcg(&tbm[w + x * 32 + lane]) : 0u;
#pragma unroll
      for (int x = 0; x < kB; ++x) c += __popc(wv[x]);
    }
    uint32_t total;
    // the exclusive prefix of lane 0 is everything the lower warps hold
    uint32_t pos = __shfl_sync(kFull, block_excl_scan<NT>(c, wsum, &total, tid, sync), 0);
    m = total;
    if (__any_sync(kFull, c != 0)) {
      for (int w = tb; w < te; w += 32 * kB) {
        uint32_t wv[kB];
#pragma unroll
        for (int x = 0; x < kB; ++x) wv[x] = w + x * 32 + lane < te ? __ldcg(&tbm[w + x * 32 + lane]) : 0u;
#pragma unroll
        for (int x = 0; x < kB; ++x) {
          uint32_t bits = wv[x];
          if (__ballot_sync(kFull, bits != 0) == 0) continue;
          const uint32_t cnt = __popc(bits);
          uint32_t incl = cnt;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
          }
          uint32_t p = pos + incl - cnt;
          if (bits) tbm[w + x * 32 + lane] = 0;
          while (bits) {
            const int b = __ffs(bits) - 1;
            bits &= bits - 1;
            if (p < (uint32_t)PK) M[p] = (w + x * 32 + lane) * 32 + b;
            ++p;
          }
          pos += __shfl_sync(kFull, incl, 31);
        }
      }
    }
    uint32_t hc = 0;
    for (int w = tid; w < nwords; w += NT) hc += __popc(bitmap[w]);
    hits = block_sum<NT>(hc, wsum, tid, sync);
    if (hits + m > (uint32_t)C) status = KVO_ECAPACITY;
  }

  if (status == KVO_OK) {
    if (tid == 0) a.stamp[u] = stamp;
    for (int w = tid; w < nwords; w += NT) {
      uint32_t bits = bitmap[w];
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1;
        lu[w * 32 + b] = stamp;
      }
    }
    // warp w owns list entries [lb, le); a slice is 32 consecutive entries,
    // one per lane (coalesced loads), ranked in list order by ballots
    const int lpw = (C + NW - 1) / NW;
    const int lb = min(C, wid * lpw), le = min(C, lb + lpw);
    // slots outside [0, C) never come from a valid list; they count as touched
    auto hit = [&](int s) { return (unsigned)s >= (unsigned)C || ((bitmap[s >> 5] >> (s & 31)) & 1u) != 0; };
    auto count_untouched = [&]() {
      uint32_t c = 0;
      for (int j = lb; j < le; j += 32 * kLB) {
        int32_t v[kLB];
#pragma unroll
        for (int x = 0; x < kLB; ++x) v[x] = j + x * 32 + lane < le ? cur[j + x * 32 + lane] : 0;
#pragma unroll
        for (int x = 0; x < kLB; ++x) c += (j + x * 32 + lane < le && !hit(v[x])) ? 1u : 0u;
      }
      return c;
    };
    // One pass over this warp's range in list order: the untouched entry of
    // rank r is the r-th victim while r < m and otherwise keeps its order at
    // position r - m of the new list (victims are the first m untouched
    // entries, so this is the old list without the touched slots and victims).
    auto split_untouched = [&](uint32_t q0) {
      const uint32_t lt = (1u << lane) - 1u;
      for (int j = lb; j < le; j += 32 * kLB) {
        int32_t v[kLB];
#pragma unroll
        for (int x = 0; x < kLB; ++x) v[x] = j + x * 32 + lane < le ? cur[j + x * 32 + lane] : 0;
#pragma unroll
        for (int x = 0; x < kLB; ++x) {
          const bool un = j + x * 32 + lane < le && !hit(v[x]);
          const uint32_t bal = __ballot_sync(kFull, un);
          const uint32_t r = q0 + __popc(bal & lt);
          if (un) {
            if (r < m) V[r] = v[x];
            else if (r - m < (uint32_t)C) nxt[r - m] = v[x];
          }
          q0 += __popc(bal);
        }
      }
    };
    uint32_t untouched = 0;
    if (hits + m > 0) {
      const uint32_t q0 = __shfl_sync(kFull, block_excl_scan<NT>(count_untouched(), wsum, &untouched, tid, sync), 0);
      split_untouched(q0);
      sync();
    }
    if (m > 0) {
      // i-th miss (token order) takes the i-th victim
      for (uint32_t r0 = tid; r0 < m; r0 += 4 * NT) {
        int32_t old[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const uint32_t r = r0 + x * NT;
          old[x] = r < m ? st[V[r]] : -1;
        }
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const uint32_t r = r0 + x * NT;
          if (r >= m) break;
          const int s = V[r];
          const int32_t t = M[r];
          if (old[x] >= 0) cs[old[x]] = -1;
          st[s] = t;
          cs[t] = s;
          lu[s] = stamp;
          a.miss_tok[(int64_t)i * PK + r] = t;
          a.miss_slot[(int64_t)i * PK + r] = s;
        }
      }
      sync();
      ready(m);  // the miss rows and their slots are final
      for (uint32_t r = tid; r < m; r += NT) atomicOr(&bitmap[V[r] >> 5], 1u << (V[r] & 31));
    }
    sync();
    if (hits + m > 0) {
      // the touched slots (hits and victims) follow in slot order
      const uint32_t kept = untouched - m;
      const int wper = (nwords + NT - 1) / NT;
      const int v0 = tid * wper, v1 = min(nwords, v0 + wper);
      uint32_t tc = 0;
      for (int w = v0; w < v1; ++w) tc += __popc(bitmap[w]);
      uint32_t tt;
      uint32_t o = kept + block_excl_scan<NT>(tc, wsum, &tt, tid, sync);
      for (int w = v0; w < v1; ++w) {
        uint32_t bits = bitmap[w];
        while (bits) {
          const int b = __ffs(bits) - 1;
          bits &= bits - 1;
          if (o < (uint32_t)C) nxt[o++] = w * 32 + b;
        }
      }
      if (tid == 0) a.order_par[u] = par ^ 1;
    }
    __threadfence_block();
    sync();
    // remap logical top-k positions to physical slots: a hit keeps its slot
    // (victims are never hit), a miss takes the victim its rank among the
    // distinct misses (M, ascending) points to
    const int mm = (int)(m < (uint32_t)PK ? m : (uint32_t)PK);
    for (int e0 = tid; e0 < PK; e0 += kTB * NT) {
      int32_t t[kTB], pv[kTB];
#pragma unroll
      for (int x = 0; x < kTB; ++x) {
        const int e = e0 + x * NT;
        t[x] = e < PK ? tok[e] : -1;
        pv[x] = e < PK ? pay[e] : -1;
      }
#pragma unroll
      for (int x = 0; x < kTB; ++x) {
        const int e = e0 + x * NT;
        if (e >= PK) break;
        int32_t slot = -1;
        if (t[x] >= 0) {
          if (pv[x] >= 0) {
            slot = pv[x];
          } else {
            int lo = 0, hi = mm;  // first M[j] >= t
            while (lo < hi) {
              const int mid = (lo + hi) >> 1;
              if (M[mid] < t[x]) lo = mid + 1; else hi = mid;
            }
            slot = lo < mm && M[lo] == t[x] ? V[lo] : -1;
          }
        }
        out_slot[e] = slot;
      }
    }
  } else {
    m = 0;
    for (int e = tid; e < PK; e += NT) out_slot[e] = -1;
  }

  if (tid == 0) {
    a.status[i] = status;
    a.miss_cnt[i] = (int32_t)m;
    if (a.stats) {
      if (status == KVO_OK) {
        atomicAdd(&a.stats->unit_steps, 1ull);
        atomicAdd(&a.stats->hits, (unsigned long long)hits);
        atomicAdd(&a.stats->misses, (unsigned long long)m);
      } else if (status == KVO_ECAPACITY) {
        atomicAdd(&a.stats->capacity_errors, 1ull);
      }
    }
  }
  if (status_out) *status_out = status;
  sync();
  if (m == 0) ready(0u);
  return m;
}

}  // namespace dev
}  // namespace kvo
