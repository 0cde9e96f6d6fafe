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
//  select_kernel : one CTA per (unit, position): exact top-k of the unit's
//                  candidates in (score desc, token asc) order by a bucket
//                  sort, or by radix select and a bitonic sort when they
//                  crowd one bucket; payload packed from cache_slots for the
//                  winners.
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "kvo_device.cuh"
#include "kvo_internal.cuh"

namespace kvo {

using namespace dev;

namespace {

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
  plan_body<1024>(a, threadIdx.x, warp_sums, &carry);
}

// The copying part of a score launch (the previous unit group's miss rows), in
// separate functions so that their registers (12 loads in flight per thread) do
// not constrain the scoring code's.  Scratch: the start of the CTA's dynamic
// shared memory (unused by a copying CTA; a scoring CTA's key ring once it has
// scored).
__device__ __forceinline__ CopyScratch copy_scratch(uint8_t* smem) {
  int64_t* src = reinterpret_cast<int64_t*>(smem);
  int64_t* dst = src + kScoreGatherRows;
  int32_t* list = reinterpret_cast<int32_t*>(dst + kScoreGatherRows);
  return CopyScratch{src, dst, list, reinterpret_cast<uint32_t*>(list + kScoreThreads)};
}
__device__ __noinline__ void score_launch_copy(const GatherArgs& g, int cta, int ncta, uint8_t* smem) {
  gather_rows_ldg<kScoreThreads, kScoreGatherRows, 12>(g, cta, ncta, copy_scratch(smem), true);
}
// Every thread of a scoring CTA calls it after its part of the scoring (the
// producer warp and the consumer warps from different places): the barrier
// below is where the key ring becomes free (every tile issued has been used).
__device__ __noinline__ void score_launch_help(const GatherArgs& g, uint8_t* smem) {
  __syncthreads();
  copy_help<kScoreThreads, kScoreGatherRows, 12>(g, copy_scratch(smem));
}

// ---------------------------------------------------------------------------
// score: one persistent CTA per flat piece of the token range (after the
// CTAs, if any, that copy the previous unit group's miss rows).
// ---------------------------------------------------------------------------
template <int PP, class KF>
__global__ void __launch_bounds__(kScoreThreads, 1) score_kernel(SelectArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  ScoreSmem sm;
  sm.carve<KF>(smem, a.P, a.cap);

  if ((int)blockIdx.x < a.gather_ctas) {
    // the previous unit group's miss rows, copied while this group is scored
    score_launch_copy(a.prev, (int)blockIdx.x, a.gather_ctas, smem);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = (int)blockIdx.x - a.gather_ctas;
  if (a.fallback && *reinterpret_cast<volatile uint32_t*>(a.fb_any) == 0) return;
  const int64_t g0 = cta_start(c, a.T, a.G), g1 = cta_start(c + 1, a.T, a.G);
  const int32_t* only = a.fallback ? a.fb : nullptr;  // rescoring pass: flagged units only
  if (tid == 0) {
    for (int s = 0; s < KF::kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kCW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // scoring CTAs of a launch that also copies the previous group's rows take the rows
  // its copying CTAs have not yet claimed once their own scoring is done
  // (the condition is read from the kernel parameters where it is used, so that no
  // register holds it across the scoring loop)
  if (g0 >= g1) {
    if (a.gather_ctas > 0 && a.prev.claim) score_launch_help(a.prev, smem);
    return;
  }

  if (warp == kCW) {
    // ---------------- producer: stream every tile of every piece ----------
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();  // keys are read once per step
      PieceIter it;
      it.begin(a.off, a.n, g0, g1, only);
      Piece pc;
      uint32_t seq = 0;
      while (it.next(pc)) {
        const int u = a.units[pc.i];
        for (int64_t t = pc.t0; t < pc.t1; t += kTile, ++seq) {
          const int stage = seq % KF::kStages;
          const uint32_t round = seq / KF::kStages;
          if (round > 0 && !mbar_wait(&sm.empty[stage], (round - 1) & 1u, a.wait_ns))
            atomicOr(a.err, kErrTimeout);
          const int nt = (int)((pc.t1 - t) < kTile ? (pc.t1 - t) : kTile);
          issue_tile<KF>(a, sm.ring + stage * KF::kStageBytes, &sm.full[stage], u, t, nt, pol);
        }
      }
    }
    if (a.gather_ctas > 0 && a.prev.claim) score_launch_help(a.prev, smem);
    return;
  }

  // ---------------- consumers ----------------------------------------------
  const int ctid = tid;  // consumers are threads 0..kCT-1
  const int P = a.P, k = a.k, cap = a.cap;
  typename ScorerFor<PP, KF>::type sc;
  sc.init(warp, lane);
  constexpr int V = ScorerFor<PP, KF>::type::V;

  PieceIter it;
  it.begin(a.off, a.n, g0, g1, only);
  Piece pc;
  uint32_t seq = 0;
  while (it.next(pc)) {
    const int i = pc.i;
    uint64_t* gth = a.gthr + (int64_t)i * P;
    sc.load_queries(a, i, P);
    piece_begin(sm, P, (!a.fallback && a.tspec) ? a.tspec + (int64_t)i * P : nullptr, ctid);
    int ti = 0;
    for (int64_t t = pc.t0; t < pc.t1; t += kTile, ++seq, ++ti) {
      const int stage = seq % KF::kStages;
      const uint32_t round = seq / KF::kStages;
      if (!mbar_wait(&sm.full[stage], round & 1u, a.wait_ns) && lane == 0) atomicOr(a.err, kErrTimeout);
      const int nt = (int)((pc.t1 - t) < kTile ? (pc.t1 - t) : kTile);
      float acc[V];
      sc.score(sm.ring + stage * KF::kStageBytes, t, acc, [&] {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[stage]);
      });
      sc.filter(acc, t, nt, pc.len, P, sm.thr, sm.cnt, sm.cand, cap);
      if (t + kTile < pc.t1 && (ti + 1) % kCheckTiles == 0) piece_check(sm, P, k, cap, gth, ctid);
    }
    piece_end(sm, P, k, cap, gth, (int64_t)c + i, a.seg_keys, a.seg_cnt, ctid);
  }
  if (a.gather_ctas > 0 && a.prev.claim) score_launch_help(a.prev, smem);
}

// int8 indexer: rotation and quantization of n keys (one warp per key).
__global__ void __launch_bounds__(256) quant_keys_kernel(const uint16_t* src, int64_t n, int8_t* codes,
                                                         uint16_t* scales) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t r = w0; r < n; r += nw) warp_quant128(src + r * kDim, codes + r * kDim, scales + r, lane);
}

// ---------------------------------------------------------------------------
// select: exact top-k of one (unit, position) over its pieces' candidates.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSelThreads) select_kernel(SelectArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  // bucket sort over all kSelSmemBytes, or the fallback's keys [kSelSmemKeys]
  // and sorted [kpad] over the same bytes
  uint64_t* base = reinterpret_cast<uint64_t*>(smem);
  __shared__ uint32_t hist[256];
  __shared__ __align__(8) uint32_t rx[10];
  __shared__ uint32_t seg_off[kSelMaxSegs + 1];

  const int tid = threadIdx.x;
  const int P = a.P;
  const int i = blockIdx.x / P, p = blockIdx.x % P;
  if (a.fallback && a.fb[i] == 0) return;  // rescoring pass: only flagged units
  if (a.fallback && p == 0 && threadIdx.x == 0 && a.stats) atomicAdd(&a.stats->rescored, 1ull);
  const int64_t s0 = a.off[i], s1 = a.off[i + 1];
  int c0 = 0, c1 = -1;
  if (s1 > s0) {
    c0 = cta_of(s0, a.T, a.G);
    c1 = cta_of(s1 - 1, a.T, a.G);
  }
  const int64_t seg0 = (int64_t)c0 + i;
  const int nseg = c1 - c0 + 1;
  auto sync = [] { __syncthreads(); };
  const bool few = nseg <= kSelMaxSegs;
  if (few) segment_offsets<kSelThreads>(a, p, 1, seg0, nseg, seg_off, tid, sync);
  const uint32_t n = few ? seg_off[nseg] : candidate_count(a, p, seg0, nseg);
  // a speculative threshold that was too high sends the unit to the rescoring pass
  if (!a.fallback && spec_short(a, i, p, n)) {
    if (tid == 0) {
      a.fb[i] = 1;
      atomicExch(a.fb_any, 1u);
    }
    return;
  }
  if (!few || !bucket_select<kSelThreads>(a, i, p, seg0, nseg, seg_off, smem, kSelSmemBytes, kSelLog2B, hist, tid,
                                          sync))
    select_body<kSelThreads>(a, i, p, seg0, nseg, false, base, kSelSmemKeys, base + kSelSmemKeys, hist, rx, tid,
                             sync);
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
int score_cap_for(int P, int k, bool int8) {
  const long fixed = int8 ? smem_fixed<KeysInt8>() : smem_fixed<KeysBf16>();
  const long avail = (long)kSmemMax - fixed - (long)k * 8 - 256;
  if (avail <= 0) return 0;
  long cap = avail / ((long)P * 8);
  long target = 3L * k;
  if (target < k + 2L * kCheckTiles * kTile) target = k + 2L * kCheckTiles * kTile;
  if (cap > target) cap = target;
  cap &= ~63L;
  if (cap < (long)k + (long)kCheckTiles * kTile) return 0;
  return (int)cap;
}

template <class KF>
static size_t score_smem(const SelectArgs& a) {
  return (size_t)smem_fixed<KF>() + (size_t)a.P * a.cap * 8 + (size_t)a.k * 8;
}

cudaError_t launch_quant_keys(const uint16_t* src, int64_t n, int8_t* codes, uint16_t* scales, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 7) / 8;
  if (blocks > 4096) blocks = 4096;
  quant_keys_kernel<<<(int)blocks, 256, 0, s>>>(src, n, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_plan(const SelectArgs& a, cudaStream_t s) {
  plan_kernel<<<1, 1024, 0, s>>>(a);
  return cudaGetLastError();
}

template <int PP, class KF>
static cudaError_t launch_score_pp(const SelectArgs& a, cudaStream_t s) {
  const size_t smem = score_smem<KF>(a);
  cudaError_t e = cudaFuncSetAttribute(score_kernel<PP, KF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  score_kernel<PP, KF><<<a.G + a.gather_ctas, kScoreThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <class KF>
static cudaError_t launch_score_kf(const SelectArgs& a, cudaStream_t s) {
  if (a.P <= 1) return launch_score_pp<1, KF>(a, s);
  if (a.P <= 2) return launch_score_pp<2, KF>(a, s);
  if (a.P <= 4) return launch_score_pp<4, KF>(a, s);
  return launch_score_pp<8, KF>(a, s);
}

cudaError_t launch_score(const SelectArgs& a, cudaStream_t s) {
  return a.keys8 ? launch_score_kf<KeysInt8>(a, s) : launch_score_kf<KeysBf16>(a, s);
}

cudaError_t launch_select(const SelectArgs& a, cudaStream_t s) {
  if (a.k > kMaxK) return cudaErrorInvalidValue;
  int kpad = 1;
  while (kpad < a.k) kpad <<= 1;
  const size_t smem = kSelSmemBytes;
  if ((size_t)kSelSmemKeys * 8 + (size_t)kpad * 8 > smem) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  select_kernel<<<a.n * a.P, kSelThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvo
