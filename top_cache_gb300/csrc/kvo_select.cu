// Indexer scoring and the fused top-k ("Layerwise and Sparse KV Cache
// Offloading Design", section 4, Decode step 3; "FlashOffloading ... What does
// it mean?", the LIM paragraph: index and slot packed into one int32 so the
// winners already say hit or miss).
//
// Three kernels, all on the caller's stream:
//  plan_kernel   : flat token offsets of the listed units (one block).
//  score_kernel  : persistent, one CTA per SM.  The listed units' cached
//                  tokens form one flat range that is cut into G equal
//                  pieces; each CTA streams its piece's indexer keys through
//                  a bulk-copy ring in shared memory, scores every token
//                  against the P queries (CUDA-core fp32, the canonical
//                  order), and keeps, per (unit, position), the tokens that
//                  can still be in the top-k in a shared-memory candidate
//                  buffer filtered by a rising threshold.  At the end of each
//                  unit piece it writes at most k candidates per position.
//  select_kernel : one CTA per (unit, position): exact radix select of the k
//                  best candidates over the unit's pieces, bitonic sort into
//                  (score desc, token asc) order, payload packed from
//                  cache_slots for the winners.
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "kvo_internal.cuh"

namespace kvo {

namespace {

constexpr int kTile = 128;                  // tokens per ring stage
constexpr int kTileBytes = kTile * kKeyBytes;
constexpr int kStages = 3;
constexpr int kCW = 16;                     // consumer warps
constexpr int kCT = kCW * 32;               // consumer threads
constexpr int kScoreThreads = kCT + 32;     // + one producer warp
constexpr int kCheckTiles = 8;            // tiles between candidate-buffer checks
constexpr int kSmemMax = 222 * 1024;        // leaves room for a co-resident copy CTA
constexpr int kSmemFixed = kStages * kTileBytes + 2 * kStages * 8 + 8 * 4 + 8 * 8 + 256 * 4 + 10 * 4 + 8;
constexpr int kSelThreads = 512;
constexpr int kSelSmemKeys = 8192;          // candidates held in shared memory by select
constexpr int kMaxK = 4096;

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
template <int CUR, int V>
__device__ __forceinline__ void tree_level(float (&a)[V], int m) {
  if constexpr (CUR > 1) {
#pragma unroll
    for (int i = 0; i < CUR / 2; ++i) a[i] = a[i] + __shfl_xor_sync(kFull, a[i + CUR / 2], m);
  } else {
    a[0] = a[0] + __shfl_xor_sync(kFull, a[0], m);
  }
}

template <int V>
__device__ __forceinline__ void tree16(float (&a)[V]) {
  tree_level<V, V>(a, 8);
  tree_level<(V >= 2 ? V / 2 : 1), V>(a, 4);
  tree_level<(V >= 4 ? V / 4 : 1), V>(a, 2);
  tree_level<(V >= 8 ? V / 8 : 1), V>(a, 1);
}

// X_l: the lane's slot permutation (slot i holds pair i ^ X_l), which is also
// the pair held in slot 0 after tree16.
template <int V>
__device__ __forceinline__ int tree_perm(int lane) {
  int x = 0, cur = V;
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) {
    if (cur > 1) {
      if (lane & m) x += cur / 2;
      cur /= 2;
    }
  }
  return x;
}
// After tree16 with V < 16 several lanes hold the same sum; one reports it.
template <int V>
__device__ __forceinline__ bool tree_owner(int lane) {
  constexpr int dup = V >= 16 ? 0 : (16 / V - 1);
  return (lane & dup) == 0;
}

// Warp 0 of the block: find the histogram bin (counting from the top) that
// holds the need-th largest element.  rx[0] = bin, rx[1] = count above it,
// rx[2] = count in it.
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
// barrier of those threads.  Requires need <= number of keys.
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
template <int E, int NT>
__device__ __forceinline__ void bitonic_regs_desc(uint64_t (&v)[E], uint64_t* buf, int n, int tid) {
  const int lane = tid & 31;
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 32 * E) {
        // only threads that hold keys touch buf (n may be smaller than E * NT)
        const bool active = tid * E < n;
        __syncthreads();
        if (active)
#pragma unroll
          for (int e = 0; e < E; ++e) buf[tid * E + e] = v[e];
        __syncthreads();
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
  (void)lane;
}

// Sorts buf[0..n) descending (n a power of two, n <= 8 * NT) with all NT threads.
template <int NT>
__device__ __forceinline__ void block_sort_desc(uint64_t* buf, int n, int tid) {
  auto run = [&](auto E_) {
    constexpr int E = decltype(E_)::value;
    uint64_t v[E];
    const bool active = tid * E < n;
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = active ? buf[tid * E + e] : 0ull;
    bitonic_regs_desc<E, NT>(v, buf, n, tid);
    __syncthreads();
    if (active)
#pragma unroll
      for (int e = 0; e < E; ++e) buf[tid * E + e] = v[e];
    __syncthreads();
  };
  if (n <= NT) run(std::integral_constant<int, 1>{});
  else if (n <= 2 * NT) run(std::integral_constant<int, 2>{});
  else if (n <= 4 * NT) run(std::integral_constant<int, 4>{});
  else run(std::integral_constant<int, 8>{});
}

__device__ __forceinline__ void consumer_sync() { named_sync(1, kCT); }

// Shrink one candidate buffer to at most k keys, all >= floor, that include
// every key of the buffer which can still be among the unit's k best:
// floor = max(local threshold, the unit's shared threshold gth), then, if
// more than k keys reach it, the k-th largest of them.  A threshold found by
// the radix select is a lower bound of the unit's k-th best (k keys of this
// piece reach it) and is published to gth.  All consumer threads call it.
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
  }
  consumer_sync();
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

struct Piece {
  int i;          // index into the listed units
  int64_t t0, t1; // local token range
  int64_t len;    // unit length
};

// The pieces of CTA c's flat range, in order.  Returns false when done.
struct PieceIter {
  const int64_t* off;
  const int32_t* only;  // if set, pieces of units with only[i] == 0 are skipped
  int n;
  int64_t g0, g1;
  int i;
  __device__ void begin(const int64_t* o, int n_, int64_t a, int64_t b, const int32_t* only_ = nullptr) {
    off = o;
    only = only_;
    n = n_;
    g0 = a;
    g1 = b;
    i = (a < b) ? find_segment(o, n_, a) : n_;
  }
  __device__ bool next(Piece& pc) {
    while (i < n) {
      const int64_t s = off[i], e = off[i + 1];
      if (s >= g1) {
        i = n;
        return false;
      }
      const int cur = i++;
      const int64_t a = s > g0 ? s : g0, b = e < g1 ? e : g1;
      if (a < b && (!only || only[cur] != 0)) {
        pc.i = cur;
        pc.t0 = a - s;
        pc.t1 = b - s;
        pc.len = e - s;
        return true;
      }
    }
    return false;
  }
};

}  // namespace

// ---------------------------------------------------------------------------
// plan: off[i] = sum of len[units[j]] for j < i; check off[n] == T.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) plan_kernel(SelectArgs a) {
  __shared__ int64_t warp_sums[32];
  __shared__ int64_t carry;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < a.n; base += 1024) {
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
    if (tid == 1023) carry = excl + v;
    __syncthreads();
  }
  for (int e = tid; e < a.n * a.P; e += 1024) {
    a.gthr[e] = 0;
    if (!a.tspec) continue;
    const int i = e / a.P, p = e - (e / a.P) * a.P;
    const int u = a.units[i];
    // squared query norm (fp32; only steers the speculative threshold)
    const uint4* q = reinterpret_cast<const uint4*>(a.queries + (int64_t)e * kDim);
    float s2 = 0.f;
#pragma unroll 4
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
    for (int i = tid; i < a.n; i += 1024) a.fb[i] = 0;
    if (tid == 0) *a.fb_any = 0;
  }
  if (tid == 0) {
    a.off[a.n] = carry;
    if (carry != a.T) atomicOr(a.err, kErrPlan);
  }
}

// ---------------------------------------------------------------------------
// score: one persistent CTA per flat piece of the token range.
// ---------------------------------------------------------------------------
template <int PP>
__global__ void __launch_bounds__(kScoreThreads, 1) score_kernel(SelectArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kTileBytes);
  uint64_t* empty = full + kStages;
  uint32_t* cnt = reinterpret_cast<uint32_t*>(empty + kStages);  // [8]
  uint64_t* thr = reinterpret_cast<uint64_t*>(cnt + 8);           // [8]
  uint32_t* hist = reinterpret_cast<uint32_t*>(thr + 8);          // [256]
  uint32_t* rx = hist + 256;                                      // [10]
  uint64_t* fl = reinterpret_cast<uint64_t*>(rx + 10);            // [1]
  uint64_t* cand = fl + 1;                                        // [P][cap]
  uint64_t* scratch = cand + (size_t)a.P * a.cap;                 // [k]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  if (a.fallback && *reinterpret_cast<volatile uint32_t*>(a.fb_any) == 0) return;
  const int64_t g0 = cta_start(c, a.T, a.G), g1 = cta_start(c + 1, a.T, a.G);
  const int32_t* only = a.fallback ? a.fb : nullptr;  // rescoring pass: flagged units only
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (g0 >= g1) return;

  if (warp == kCW) {
    // ---------------- producer: stream every tile of every piece ----------
    if (lane == 0) {
      PieceIter it;
      it.begin(a.off, a.n, g0, g1, only);
      Piece pc;
      uint32_t seq = 0;
      while (it.next(pc)) {
        const int u = a.units[pc.i];
        const uint16_t* kb = a.keys + ((int64_t)u * a.stride) * kDim;
        for (int64_t t = pc.t0; t < pc.t1; t += kTile, ++seq) {
          const int stage = seq % kStages;
          const uint32_t round = seq / kStages;
          if (round > 0 && !mbar_wait(&empty[stage], (round - 1) & 1u, a.wait_ns))
            atomicOr(a.err, kErrTimeout);
          const int64_t nt = (pc.t1 - t) < kTile ? (pc.t1 - t) : kTile;
          const uint32_t bytes = (uint32_t)nt * kKeyBytes;
          mbar_arrive_expect_tx(&full[stage], bytes);
          bulk_g2s(ring + stage * kTileBytes, kb + t * kDim, bytes, &full[stage]);
        }
      }
    }
    return;
  }

  // ---------------- consumers ----------------------------------------------
  constexpr int V = 4 * PP;                 // (token, position) pairs per lane
  constexpr int VL = V >= 16 ? V / 16 : 1;  // values left per lane after the tree
  constexpr int LPP = PP == 1 ? 0 : PP == 2 ? 1 : PP == 4 ? 2 : 3;
  constexpr int PH = PP >= 2 ? PP / 2 : 1;  // position pairs (packed fp32x2 FMA)
  const int ctid = tid;                     // consumers are threads 0..kCT-1
  const int h = lane >> 4, j = lane & 15;
  // slot (tau, p) of this lane scores token row tau ^ tx against position p ^ px
  const int X = tree_perm<V>(lane);
  const int tx = X >> LPP, px = X & (PP - 1);
  const bool owner = tree_owner<V>(lane);
  const int P = a.P, k = a.k, cap = a.cap;
  const uint32_t trigger = (uint32_t)(cap - kCheckTiles * kTile);
  int rowoff[4];
#pragma unroll
  for (int tau = 0; tau < 4; ++tau) rowoff[tau] = (warp * 8 + h * 4 + (tau ^ tx)) * kKeyBytes + j * 16;
  // Result r of this lane is (row rrow[r], position rpos[r]).  For insertion,
  // lane q < P is the leader of position q: lead[r] = lanes reporting
  // position q; same[r] = lanes reporting this lane's position.
  int rrow[VL], rpos[VL];
  uint32_t lead[VL], same[VL];
#pragma unroll
  for (int r = 0; r < VL; ++r) {
    const int cmb = r ^ X;
    rrow[r] = warp * 8 + h * 4 + (cmb >> LPP);
    rpos[r] = cmb & (PP - 1);
    lead[r] = 0;
    same[r] = 0;
    for (int q = 0; q < PP; ++q) {
      const uint32_t m = __ballot_sync(kFull, owner && rpos[r] == q);
      if (lane == q) lead[r] = m;
      if (rpos[r] == q) same[r] = m;
    }
  }

  PieceIter it;
  it.begin(a.off, a.n, g0, g1, only);
  Piece pc;
  uint32_t seq = 0;
  while (it.next(pc)) {
    const int i = pc.i;
    uint64_t* gth = a.gthr + (int64_t)i * P;
    // this lane's chunk of the queries, in slot order (fp32, exact); with
    // several positions, slots 2m and 2m+1 are packed for fp32x2 FMAs
    float qf[PP][8];
#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int pq = p ^ px;
      if (pq < P) {
        const uint4 v = *reinterpret_cast<const uint4*>(a.queries + ((int64_t)i * P + pq) * kDim + j * 8);
        qf[p][0] = bf_lo(v.x); qf[p][1] = bf_hi(v.x);
        qf[p][2] = bf_lo(v.y); qf[p][3] = bf_hi(v.y);
        qf[p][4] = bf_lo(v.z); qf[p][5] = bf_hi(v.z);
        qf[p][6] = bf_lo(v.w); qf[p][7] = bf_hi(v.w);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) qf[p][e] = 0.f;
      }
    }
    float2 qp[PH][8];
#pragma unroll
    for (int m = 0; m < PH; ++m)
#pragma unroll
      for (int e = 0; e < 8; ++e) qp[m][e] = make_float2(qf[2 * m][e], PP >= 2 ? qf[(2 * m + 1) % PP][e] : 0.f);
    if (ctid < P) {
      cnt[ctid] = 0;
      thr[ctid] = (!a.fallback && a.tspec) ? a.tspec[(int64_t)i * P + ctid] : 0ull;
    }
    consumer_sync();
    // tokens before this index are visible to every position
    const int64_t all_visible = pc.len - (P - 1);

    int ti = 0;
    for (int64_t t = pc.t0; t < pc.t1; t += kTile, ++seq, ++ti) {
      const int stage = seq % kStages;
      const uint32_t round = seq / kStages;
      if (!mbar_wait(&full[stage], round & 1u, a.wait_ns) && lane == 0) atomicOr(a.err, kErrTimeout);
      const int nt = (int)((pc.t1 - t) < kTile ? (pc.t1 - t) : kTile);
      const uint8_t* tile = ring + stage * kTileBytes;

      float acc[V];
#pragma unroll
      for (int tau = 0; tau < 4; ++tau) {
        const uint4 kv = *reinterpret_cast<const uint4*>(tile + rowoff[tau]);
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
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      tree16<V>(acc);

      // full tiles whose tokens every position sees need no per-result tests
      const bool interior = nt == kTile && t + kTile <= all_visible;
#pragma unroll
      for (int r = 0; r < VL; ++r) {
        const int p = rpos[r];
        const int64_t tok = t + rrow[r];
        float s = acc[r];
        if (s == 0.f) s = 0.f;  // +0 for a zero score
        const uint64_t key = sel_key(s, (uint32_t)tok);
        bool ok = owner && p < P;
        if (!interior) ok = ok && rrow[r] < nt && tok < pc.len - (P - 1 - p);
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
      // every kCheckTiles tiles: adopt the unit's shared thresholds and
      // compact the buffers that could overflow within the next tiles
      if (t + kTile < pc.t1 && (ti + 1) % kCheckTiles == 0) {
        consumer_sync();
        bool need = false;
        for (int p = 0; p < P; ++p) need |= cnt[p] > trigger;
        if (ctid < P) {
          const uint64_t g = __ldcg(reinterpret_cast<const unsigned long long*>(gth + ctid));
          if (g > thr[ctid]) thr[ctid] = g;
        }
        if (need) {
          for (int p = 0; p < P; ++p)
            if (cnt[p] > trigger)
              compact_candidates(cand + (size_t)p * cap, &cnt[p], &thr[p], gth + p, fl, scratch, hist,
                                 rx, k, ctid);
        }
      }
    }

    // piece done: at most k candidates per position, all above the shared threshold
    consumer_sync();
    for (int p = 0; p < P; ++p)
      compact_candidates(cand + (size_t)p * cap, &cnt[p], &thr[p], gth + p, fl, scratch, hist, rx, k,
                         ctid);
    const int64_t seg = (int64_t)c + i;
    for (int p = 0; p < P; ++p) {
      const uint32_t np = cnt[p];
      uint64_t* dst = a.seg_keys + (seg * P + p) * (int64_t)k;
      for (uint32_t e = ctid; e < np; e += kCT) dst[e] = cand[(size_t)p * cap + e];
      if (ctid == 0) a.seg_cnt[seg * P + p] = (int32_t)np;
    }
    consumer_sync();
  }
}

// ---------------------------------------------------------------------------
// select: exact top-k of one (unit, position) over its pieces' candidates.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSelThreads) select_kernel(SelectArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* keys = reinterpret_cast<uint64_t*>(smem);          // [kSelSmemKeys]
  uint64_t* sorted = keys + kSelSmemKeys;                       // [kpad]
  __shared__ uint32_t hist[256];
  __shared__ __align__(8) uint32_t rx[10];

  const int tid = threadIdx.x;
  const int P = a.P, k = a.k;
  const int i = blockIdx.x / P, p = blockIdx.x % P;
  if (a.fallback && a.fb[i] == 0) return;  // rescoring pass: only flagged units
  if (a.fallback && p == 0 && threadIdx.x == 0 && a.stats) atomicAdd(&a.stats->rescored, 1ull);
  const int64_t s0 = a.off[i], s1 = a.off[i + 1];
  int c0 = 0, c1 = -1;
  if (s1 > s0) {
    c0 = cta_of(s0, a.T, a.G);
    c1 = cta_of(s1 - 1, a.T, a.G);
  }
  uint32_t n = 0;
  for (int c = c0; c <= c1; ++c) n += (uint32_t)a.seg_cnt[((int64_t)c + i) * P + p];
  // A speculative threshold is exact when at least min(k, visible) keys
  // reached it: then every key of the top k did.  Otherwise the unit is
  // rescored without speculation.
  if (!a.fallback && a.tspec && a.tspec[(int64_t)i * P + p] != 0) {
    const int64_t vis = (s1 - s0) - (P - 1 - p);
    const uint32_t need = (uint32_t)(vis < k ? (vis > 0 ? vis : 0) : k);
    if (n < need) {
      if (tid == 0) {
        a.fb[i] = 1;
        atomicExch(a.fb_any, 1u);
      }
      return;
    }
  }
  const bool in_smem = n <= (uint32_t)kSelSmemKeys;
  auto sync = [] { __syncthreads(); };

  if (in_smem) {
    uint32_t base = 0;
    for (int c = c0; c <= c1; ++c) {
      const int64_t seg = (int64_t)c + i;
      const uint32_t m = (uint32_t)a.seg_cnt[seg * P + p];
      const uint64_t* src = a.seg_keys + (seg * P + p) * (int64_t)k;
      for (uint32_t e = tid; e < m; e += kSelThreads) keys[base + e] = src[e];
      base += m;
    }
    __syncthreads();
  }
  auto for_each = [&](auto f) {
    if (in_smem) {
      for (uint32_t e = tid; e < n; e += kSelThreads) f(keys[e]);
    } else {
      for (int c = c0; c <= c1; ++c) {
        const int64_t seg = (int64_t)c + i;
        const uint32_t m = (uint32_t)a.seg_cnt[seg * P + p];
        const uint64_t* src = a.seg_keys + (seg * P + p) * (int64_t)k;
        for (uint32_t e = tid; e < m; e += kSelThreads) f(src[e]);
      }
    }
  };
  uint64_t thr = 0;
  if (n > (uint32_t)k) thr = radix_threshold_desc<kSelThreads>(for_each, (uint32_t)k, hist, rx, tid, sync);
  const uint32_t count = n < (uint32_t)k ? n : (uint32_t)k;
  int kpad = 1;
  while (kpad < k) kpad <<= 1;
  if (tid == 0) rx[9] = 0;
  __syncthreads();
  const int lane = tid & 31;
  // keys >= thr go to the sort buffer (uniform trip counts: full-warp ballots)
  auto keep_from = [&](const uint64_t* src, uint32_t m) {
    for (uint32_t b = 0; b < m; b += kSelThreads) {
      const uint32_t e = b + tid;
      const uint64_t key = e < m ? src[e] : 0;
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
    keep_from(keys, n);
  } else {
    for (int c = c0; c <= c1; ++c) {
      const int64_t seg = (int64_t)c + i;
      keep_from(a.seg_keys + (seg * P + p) * (int64_t)k, (uint32_t)a.seg_cnt[seg * P + p]);
    }
  }
  __syncthreads();
  for (int e = count + tid; e < kpad; e += kSelThreads) sorted[e] = 0;
  __syncthreads();
  block_sort_desc<kSelThreads>(sorted, kpad, tid);

  const int u = a.units[i];
  const int64_t obase = ((int64_t)i * P + p) * k;
  for (int r = tid; r < k; r += kSelThreads) {
    int32_t tok = -1, pay = KVO_PAD_PAYLOAD;
    float sc = __uint_as_float(0xff800000u);
    if (r < (int)count) {
      const uint64_t key = sorted[r];
      tok = (int32_t)key_token(key);
      sc = key_score(key);
      const int32_t cs = a.cache_slots ? a.cache_slots[(int64_t)u * a.stride + tok] : -1;
      pay = cs >= 0 ? cs : -(tok + 1);
    }
    a.out_tok[obase + r] = tok;
    if (a.out_score) a.out_score[obase + r] = sc;
    a.out_pay[obase + r] = pay;
    if (a.out_pay_user && a.out_pay_user != a.out_pay) a.out_pay_user[obase + r] = pay;
  }
  if (a.spec && tid == 0) {
    a.spec[(int64_t)u * P + p] = count >= (uint32_t)k ? sorted[k - 1] : 0ull;
    if (a.qn_prev && a.qn_cur) a.qn_prev[(int64_t)u * P + p] = a.qn_cur[(int64_t)i * P + p];
  }
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
int score_cap_for(int P, int k) {
  const long avail = (long)kSmemMax - kSmemFixed - (long)k * 8 - 256;
  if (avail <= 0) return 0;
  long cap = avail / ((long)P * 8);
  long target = 3L * k;
  if (target < k + 2L * kCheckTiles * kTile) target = k + 2L * kCheckTiles * kTile;
  if (cap > target) cap = target;
  cap &= ~63L;
  if (cap < (long)k + (long)kCheckTiles * kTile) return 0;
  return (int)cap;
}

static size_t score_smem(const SelectArgs& a) {
  return (size_t)kSmemFixed + (size_t)a.P * a.cap * 8 + (size_t)a.k * 8;
}

cudaError_t launch_plan(const SelectArgs& a, cudaStream_t s) {
  plan_kernel<<<1, 1024, 0, s>>>(a);
  return cudaGetLastError();
}

template <int PP>
static cudaError_t launch_score_pp(const SelectArgs& a, cudaStream_t s) {
  const size_t smem = score_smem(a);
  cudaError_t e = cudaFuncSetAttribute(score_kernel<PP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  score_kernel<PP><<<a.G, kScoreThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_score(const SelectArgs& a, cudaStream_t s) {
  if (a.P <= 1) return launch_score_pp<1>(a, s);
  if (a.P <= 2) return launch_score_pp<2>(a, s);
  if (a.P <= 4) return launch_score_pp<4>(a, s);
  return launch_score_pp<8>(a, s);
}

cudaError_t launch_select(const SelectArgs& a, cudaStream_t s) {
  if (a.k > kMaxK) return cudaErrorInvalidValue;
  int kpad = 1;
  while (kpad < a.k) kpad <<= 1;
  const size_t smem = (size_t)kSelSmemKeys * 8 + (size_t)kpad * 8;
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  select_kernel<<<a.n * a.P, kSelThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvo
