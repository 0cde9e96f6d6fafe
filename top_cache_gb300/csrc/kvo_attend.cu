// Sparse attention over the hot buffer on the 5th-generation tensor cores:
// decode step 7 of "Layerwise and Sparse KV Cache Offloading Design"
// (section 4, "Decode step": the attention operator reads the resident rows).
//
// Reading R13 of the oracle (the pages name an SFA/MLA sparse-attention model
// but give no formula): absorbed latent attention.  A hot row is 576 bf16 =
// latent (512, which is also the value) | rope key (64); the query of a head
// has the same split.  For unit u, position p and head h, over the slots of
// that position's top-k list (pads, slot < 0, skipped):
//   s_i = scale * q_h . row_i,   out_h = sum_i softmax(s)_i * row_i[0:512],
//   lse_h = log sum_i exp(s_i).
//
// A cluster of two CTAs per (unit, position, group of 128 heads); CTA c of
// the pair owns value columns 256c..256c+255 (slabs 4c..4c+3 of a row) and
// rows 64c..64c+63 of every 128-row block.  The scores are split by slab: CTA
// c computes the partial S over its own four value slabs, plus the rope slab
// on the blocks whose index has its parity, so each row slab is copied and
// multiplied once per pair.  Per block:
//   - each CTA sends its partial scores of the partner's rows into the
//     partner's shared memory and adds the partner's partial scores of its
//     own rows (distributed shared memory: st.async, whose bytes count down
//     the receiver's expect-tx barrier, so no arrival travels with them);
//   - the two agree on each head's block maximum the same way;
//   - each writes P (bf16) of its 64 rows into both CTAs' P tile, and each
//     computes O[:, own 256 columns] += P V over all 128 rows.
// Issuing a tcgen05.mma from one thread costs about a hundred cycles whatever
// N is up to 128, so every MMA is as wide as the operands allow: S MMAs have
// N = 128, P V is eight MMAs of N = 256.  S is freed as soon as the softmax
// has read it (P lives in shared memory), so the next block's S overlaps the
// softmax of this one.
//   warps 0-3  copy the rope query slab, then this CTA's slabs of every
//              block with 16-byte cp.async into the 128-byte-swizzled
//              K-major layout; completion is counted by each ring entry's
//              mbarrier (cp.async.mbarrier.arrive.noinc), so they never
//              wait for their own copies.  Ring: nine 16 KB entries, the
//              value slabs of even blocks in 0-3, of odd blocks in 4-7 (side
//              by side: the N = 256 operand of P V), the rope slab in 8;
//   warps 4-7  put this CTA's four query slabs into TMEM, then run the
//              online softmax, one head (TMEM lane) per thread: the running
//              maximum moves only when a score passes it by more than 2^8 (O
//              is then rescaled in TMEM); P is rounded to bf16 and l sums the
//              rounded weights, so out is their exact weighted mean; at the
//              end the pair adds its two l, and O / l in bf16 and lse;
//   warp 8     holds 512 TMEM columns; lane 0 issues every tcgen05.mma:
//              S(j) (A: query slabs in TMEM, the rope one in shared memory),
//              then P V of block j-1 (A: P tile, B: value slabs).
// Every mbarrier wait is bounded: on expiry the CTA sets kErrTimeout in the
// error word and stops; both CTAs always meet at the final cluster barrier,
// after which no access to the partner's shared memory is made.
#include <cuda_bf16.h>

#include "kvo_internal.cuh"

namespace kvo {
namespace {

constexpr int kRow = 576;                 // elements per hot row
constexpr int kVal = 512;                 // value (latent) elements
constexpr int kM = 128;                   // heads per CTA pair: M of the MMAs
constexpr int kBlk = 128;                 // rows per block: N of S, K of P V
constexpr int kOwnRows = kBlk / 2;        // rows of a block whose softmax this CTA runs
constexpr int kVSlabs = 4;                // value slabs of one CTA
constexpr int kRopeSlab = 8;              // slab of the rope key
constexpr int kRing = 2 * kVSlabs + 1;    // value slabs of two blocks + the rope slab
constexpr int kHalfCols = kVal / 2;       // value columns per CTA
constexpr int kAttThreads = 288;
constexpr int kProducers = 128;           // warps 0-3: copies
constexpr int kSoftWarp0 = 4;             // warps 4-7: softmax
constexpr int kMmaWarp = 8;               // TMEM allocation and MMA issue
constexpr int kSoftThreads = 128;
constexpr int kRowStep = kProducers / 8;  // rows of an entry between one copy thread's chunks
constexpr uint32_t kQSlab = kM * 128;     // one slab of the query tile
constexpr uint32_t kEntry = kBlk * 128;   // one slab of a row block
constexpr uint32_t kPSlab = kM * 128;     // 64 rows of P (K-major, 128-byte swizzled)
constexpr uint32_t kQOff = 0;                               // rope query slab
constexpr uint32_t kROff = kQOff + kQSlab;                  // ring
constexpr uint32_t kPOff = kROff + kRing * kEntry;          // P tile: two slabs
constexpr uint32_t kXSOff = kPOff + 2 * kPSlab;             // partner's partial scores of own rows
constexpr uint32_t kXSBytes = kM * kOwnRows * 4;           // partial scores of 64 rows of 128 heads
constexpr uint32_t kXMOff = kXSOff + kXSBytes;              // partner's block maxima [2][128], then its l
constexpr uint32_t kBarOff = kXMOff + 2 * kM * 4;
constexpr uint32_t kFetchOff = kBarOff + 256;        // fetching variant: claim-mask barriers [2], masks [2][2][4]
constexpr uint32_t kAttSmem = kFetchOff + 128 + 1024;  // barriers, flags, masks, 1 KB alignment slack
constexpr int kWriterWarp = 9;                        // fetching variant: writes filled rows to the hot buffer
constexpr int kAttThreadsFetch = kAttThreads + 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;    // O: 256 fp32 columns
constexpr uint32_t kColS = 256;  // S: 128 fp32 columns (this CTA's partial, then read out)
constexpr uint32_t kColQ = 384;  // query slabs 4c + i: 128 columns of bf16 pairs (32 per slab)
constexpr float kRescaleLog2 = 8.f;
static_assert(kAttSmem <= 232448, "shared memory of one CTA");
static_assert(kROff % 1024 == 0 && kPOff % 1024 == 0, "128-byte-swizzled tiles sit on 1 KB boundaries");
static_assert(kBlk % kRowStep == 0 && kSoftWarp0 % 4 == 0, "copy rows; softmax warps start a TMEM lane quadrant");
static_assert(kSoftThreads == kM, "one softmax thread per head");

// Shared-memory matrix descriptor, 128-byte swizzle (start, leading and stride
// byte offsets in 16-byte units; descriptor version 1).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: bf16 A and B, fp32 D, M and N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int c = 0; c < 32; ++c) v[c] = __uint_as_float(r[c]);
}
// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Wait for every cp.async this thread has issued.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// The barrier counts one arrival once every cp.async this thread has issued
// so far has landed (its pending count is not raised: the arrival is one of
// those it was initialised for).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// 2^x with the hardware approximation (relative error near 2^-22, far below
// the bf16 rounding of the weights); 2^-inf = 0, tiny results flush to zero.
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint4 ld_shared_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Source of one part of a miss row in this call (epoch e, e2 = 2e): 0 = the hot
// buffer (another CTA has written it: 2e + 1), 1 = the host pool, claimed by this
// CTA (which then writes it to the hot buffer), 2 = the host pool, claimed by
// another CTA that has not finished writing it (the same bytes, read again).
__device__ __forceinline__ int claim_part(uint32_t* w, uint32_t e2) {
  if (ld_acquire_gpu(w) == e2 + 1u) return 0;
  return atomicMax(w, e2) < e2 ? 1 : 2;
}
// The order of the (unit, position) pairs of the fetching variant.  Rounds of G
// units: round r runs position 0 of units rG.. (their miss rows are fetched
// and written by these pairs), then positions 1..P-1 of the previous round's
// units, whose shared miss rows are by then mostly in the hot buffer.  Pair b
// of n*P -> (list index i, position p).
__device__ __forceinline__ void pair_order(int b, int n, int P, int G, int& i, int& p) {
  i = 0;
  p = 0;
  if (P == 1 || G <= 0) {
    i = b / P;
    p = b % P;
    return;
  }
  const int ng = (n + G - 1) / G;
  int base = 0;
  for (int r = 0; r <= ng; ++r) {
    if (r < ng) {
      const int g = min(G, n - r * G);
      if (b < base + g) {
        i = r * G + (b - base);
        return;
      }
      base += g;
    }
    if (r >= 1) {
      const int g = min(G, n - (r - 1) * G);
      if (b < base + (P - 1) * g) {
        const int x = b - base;
        p = 1 + x / g;
        i = (r - 1) * G + x % g;
        return;
      }
      base += (P - 1) * g;
    }
  }
}
// 16-byte chunk c (0..7) of row r in a 128-byte-swizzled slab (1 KB aligned).
__device__ __forceinline__ uint32_t swz(uint32_t slab, int r, int c) {
  return slab + (uint32_t)r * 128u + ((uint32_t)(c ^ (r & 7)) << 4);
}

// ---- the CTA pair: distributed shared memory and cluster-scope barriers ----
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_local_v4(uint32_t addr, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}
__device__ __forceinline__ float4 ld_local_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
               : "memory");
  return v;
}
// Stores into the partner's shared memory whose bytes count down the
// partner's barrier `peer_bar` (expect-tx) once they have landed.
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t x, uint32_t y, uint32_t z, uint32_t w,
                                            uint32_t peer_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
               "r"(x), "r"(y), "r"(z), "r"(w), "r"(peer_bar)
               : "memory");
}
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t peer_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr),
               "r"(__float_as_uint(v)), "r"(peer_bar)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on a barrier that the partner arrives on (acquire at cluster scope).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 31u) == 0 && global_ns() - t0 > limit_ns) return false;
  }
}
// MMA completion signalled to the same barrier in both CTAs of the pair.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}
// Every thread of both CTAs.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <bool kFetch>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFetch ? kAttThreadsFetch : kAttThreads, 1)
    attend_kernel(AttendArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;  // the same in both CTAs
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* q_full = bars;            // copies and softmax: query slabs in place
  uint64_t* e_full = bars + 1;        // [kRing] copies: entry in place
  uint64_t* e_free = e_full + kRing;  // [kRing] MMA: the entry's last reader done
  uint64_t* s_full = e_free + kRing;  // MMA: partial S of a block ready
  uint64_t* s_free = s_full + 1;      // softmax: S read out
  uint64_t* xs_full = s_free + 1;     // partner: its partial scores of own rows written (expect-tx)
  uint64_t* xm_full = xs_full + 1;    // partner: its block maxima (at the end its l) written (expect-tx)
  uint64_t* p_full = xm_full + 1;     // own softmax threads and the partner's P stores: the P tile complete
  uint64_t* p_free = p_full + 1;      // both CTAs' MMA: P V of a block done
  uint64_t* o_final = p_free + 1;     // MMA: the last P V done
  uint64_t* fin = o_final + 1;        // MMA: everything issued is done
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(fin + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  uint64_t* m_ready = reinterpret_cast<uint64_t*>(smem + kFetchOff);     // [2] copies: a block's claim masks set
  uint32_t* cmask = reinterpret_cast<uint32_t*>(smem + kFetchOff + 16);  // [block & 1][value, rope][4 words]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int b = blockIdx.x;
  const int half = b & 1;  // the rank in the cluster
  const uint32_t peer = (uint32_t)(half ^ 1);
  b >>= 1;
  const int HG = a.H / kM;
  const int hg = b % HG;
  b /= HG;
  int p = b % a.P, i = b / a.P;
  if (kFetch) pair_order(b, a.n, a.P, a.group, i, p);
  const int u = a.units[i];
  const int64_t list = ((int64_t)i * a.P + p) * a.k;
  const int64_t qrow0 = ((int64_t)i * a.P + p) * a.H + (int64_t)hg * kM;
  const int nb = (a.k + kBlk - 1) / kBlk;
  auto own_rope = [&](int j) { return (j & 1) == half; };
  auto fail = [&]() {
    atomicOr(a.err, kErrTimeout);
    *abort_flag = 1u;
  };

  if (tid == 0) {
    mbar_init(q_full, kProducers + kSoftThreads);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&e_full[s], kProducers);
      mbar_init(&e_free[s], kFetch ? 2 : 1);  // fetching: the writer warp has read the entry too
    }
    if (kFetch) {
      mbar_init(&m_ready[0], kProducers / 32);
      mbar_init(&m_ready[1], kProducers / 32);
      for (int w = 0; w < 16; ++w) cmask[w] = 0u;
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, kSoftThreads);
    // The exchange barriers complete when the partner's bytes have landed and
    // one local arrival has announced how many (for the next phase, right
    // after the current one is seen complete, before the partner can send).
    mbar_init(xs_full, 1);
    mbar_init(xm_full, 1);
    mbar_init(p_full, kSoftThreads + 1);  // this CTA's softmax threads + the partner's half of P
    mbar_init(p_free, 2);                 // this CTA's P V and the partner's
    mbar_init(o_final, 1);
    mbar_init(fin, 1);
    mbar_arrive_expect_tx(xs_full, kXSBytes);
    mbar_arrive_expect_tx(xm_full, kM * 4);
    mbar_arrive_expect_tx(p_full, kPSlab);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32((const void*)tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_before();
  cluster_sync();  // both CTAs' barriers exist before either arrives on the other's
  tc_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < kProducers / 32) {
    // ---- copies: the rope query slab, then this CTA's slabs of every block ----
    const uint8_t* qsrc = reinterpret_cast<const uint8_t*>(a.q) + qrow0 * (kRow * 2);
    for (int idx = tid; idx < kM * 8; idx += kProducers) {
      const int r = idx >> 3, c = idx & 7;
      cp_async16(swz(sb + kQOff, r, c), qsrc + (size_t)r * (kRow * 2) + kRopeSlab * 128 + c * 16);
    }
    cp_async_arrive_noinc(q_full);
    const uint8_t* ubase = reinterpret_cast<const uint8_t*>(a.hot) + (size_t)u * a.C * (kRow * 2);
    const uint8_t* hbase = reinterpret_cast<const uint8_t*>(a.host_pool);
    // this thread copies chunk csub of rows rsub + kRowStep m of every entry;
    // the slots (and, fetching, the payloads) of the next block's rows are read a block ahead
    const int rsub = tid >> 3, csub = tid & 7;
    constexpr int kRowsPT = kBlk / kRowStep;
    int32_t rs[kRowsPT], rs_next[kRowsPT], py_next[kRowsPT];
    int64_t hrow[kRowsPT];  // fetching: host-pool row of a miss row
    auto load_rows = [&](int j) {
#pragma unroll
      for (int m = 0; m < kRowsPT; ++m) {
        const int r = j * kBlk + rsub + kRowStep * m;
        const bool in = j < nb && r < a.k;
        rs_next[m] = in ? __ldg(a.slots + list + r) : -1;
        if (kFetch) py_next[m] = in ? __ldg(a.pay + list + r) : INT32_MIN;
      }
    };
    // host: bit m set = row m's part comes from the host pool
    auto issue = [&](int slab, int slot, uint32_t host) {
      const uint32_t dst = sb + kROff + (uint32_t)slot * kEntry;
#pragma unroll
      for (int m = 0; m < kRowsPT; ++m) {
        const uint8_t* src = (kFetch && ((host >> m) & 1u)) ? hbase + hrow[m] * (kRow * 2)
                                                             : ubase + (size_t)rs[m] * (kRow * 2);
        cp_async16(swz(dst, rsub + kRowStep * m, csub), src + slab * 128 + csub * 16);
      }
      cp_async_arrive_noinc(&e_full[slot]);  // counts once this thread's copies have landed
    };
    unsigned long long dup_bytes = 0;
    load_rows(0);
    // A block's value slabs reuse the slots of block j-2's, freed by its P V;
    // the rope slot is reused every other block (the blocks of this CTA's parity).
    for (int j = 0; j < nb; ++j) {
      if (__any_sync(kFull, *abort_flag != 0u)) break;  // warp-uniform: shuffles follow
      const int vb = kVSlabs * (j & 1);
      bool ok = true;
      if (j >= 2) {
        const uint32_t par = (uint32_t)((j >> 1) - 1) & 1u;
#pragma unroll
        for (int v = 0; v < kVSlabs; ++v) ok = ok && __all_sync(kFull, mbar_wait(&e_free[vb + v], par, a.wait_ns));
        if (own_rope(j)) ok = ok && __all_sync(kFull, mbar_wait(&e_free[kRing - 1], par, a.wait_ns));
      }
      if (!ok) {
        fail();
        break;
      }
      uint32_t host_v = 0u, host_r = 0u;
#pragma unroll
      for (int m = 0; m < kRowsPT; ++m) {
        const int32_t slot = rs_next[m];
        const bool valid = slot >= 0 && slot < a.C;
        rs[m] = valid ? slot : 0;  // a pad reads a valid row; the softmax drops it
        if (kFetch) {
          // a miss row of the step: its parts come from the host pool unless
          // another CTA of this call has already written them to the hot buffer
          const int32_t pay = py_next[m];
          hrow[m] = -1;
          int tv = 0, tr = 0;
          if (valid && pay < 0 && pay != INT32_MIN) {
            hrow[m] = host_row(a.hrows, u, (int64_t)(-(pay + 1)));
            if (hrow[m] >= 0 && csub == 0) {  // one lane of the row's eight claims for them
              uint32_t* w = a.claim + ((size_t)u * a.C + (size_t)slot) * 3;
              const uint32_t e2 = 2u * a.epoch;
              tv = claim_part(w + half, e2);
              if (own_rope(j)) tr = claim_part(w + 2, e2);
            }
          }
          tv = __shfl_sync(kFull, tv, lane & ~7);
          tr = __shfl_sync(kFull, tr, lane & ~7);
          if (tv) host_v |= 1u << m;
          if (tr) host_r |= 1u << m;
          const int r = rsub + kRowStep * m;
          if (csub == 0) {
            if (tv == 1) atomicOr(&cmask[((j & 1) * 2 + 0) * 4 + (r >> 5)], 1u << (r & 31));
            if (tr == 1) atomicOr(&cmask[((j & 1) * 2 + 1) * 4 + (r >> 5)], 1u << (r & 31));
            dup_bytes += (tv == 2 ? 512u : 0u) + (tr == 2 ? 128u : 0u);
          }
        }
      }
      load_rows(j + 1);
      if (kFetch) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&m_ready[j & 1]);  // this warp's claims of block j are in the masks
      }
      if (own_rope(j)) issue(kRopeSlab, kRing - 1, host_r);
#pragma unroll
      for (int v = 0; v < kVSlabs; ++v) issue(kVSlabs * half + v, vb + v, host_v);
    }
    if (kFetch && dup_bytes && a.stats) atomicAdd(&a.stats->fetch_dup_bytes, dup_bytes);
    cp_async_wait_all();
  } else if (warp == kMmaWarp) {
    // ---- MMA issue (one thread) ----
    if (lane == 0) {
      constexpr uint32_t kIdQK = idesc_bf16(kM, kBlk, false);
      constexpr uint32_t kIdPV = idesc_bf16(kM, kHalfCols, true);
      bool ok = mbar_wait(q_full, 0, a.wait_ns);
      fence_proxy_async_smem();  // the tensor cores read what cp.async wrote (acquired through the barrier)
      // ring slot s: kd0 + s * (kEntry >> 4) (the start address field, in 16-byte units)
      const uint64_t kd0 = sdesc(sb + kROff, 16, 1024);
      auto kd = [&](int s) { return kd0 + (uint64_t)((uint32_t)s * (kEntry >> 4)); };
      const uint64_t qd_rope = sdesc(sb + kQOff, 16, 1024);
      // P tile: K step kk is in slab kk / 4 at byte 32 (kk % 4) of each row
      uint64_t pd[kBlk / 16];
#pragma unroll
      for (int kk = 0; kk < kBlk / 16; ++kk)
        pd[kk] = sdesc(sb + kPOff + (uint32_t)(kk >> 2) * kPSlab, 16, 1024) + (uint32_t)((kk & 3) * 2);
      // O += P V for block jj; V: the block's four value slabs side by side, the
      // four 64-column chunks of one N = 256 MN-major operand (chunk stride one
      // entry, 8-row groups 1 KB apart)
      auto issue_pv = [&](int jj) -> bool {
        if (!mbar_wait_cluster(p_full, jj & 1, a.wait_ns)) return false;
        if (jj + 1 < nb) mbar_arrive_expect_tx(p_full, kPSlab);  // the partner's half of the next P
        fence_proxy_async_smem();  // P was written with ordinary and asynchronous stores
        tc_after();
        const int vb = kVSlabs * (jj & 1);
        const uint64_t vdesc = sdesc(sb + kROff + (uint32_t)vb * kEntry, kEntry, 1024);
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk)
          mma_ss(tmem + kColO, pd[kk], vdesc + ((uint32_t)kk * 16u * 128u >> 4), kIdPV, (jj > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int v = 0; v < kVSlabs; ++v) mma_commit(&e_free[vb + v]);
        mma_commit_pair(p_free);  // both CTAs learn that this P tile and these slots are free
        return true;
      };
      const uint32_t dS = tmem + kColS;
      for (int j = 0; ok && j < nb; ++j) {
        // S(j) overwrites S(j-1) once the softmax has read it out
        if (j >= 1 && !mbar_wait(s_free, (j - 1) & 1, a.wait_ns)) {
          ok = false;
          break;
        }
        tc_after();
        const uint32_t par = (uint32_t)(j >> 1) & 1u;
        uint32_t acc = 0u;
        if (own_rope(j)) {
          if (*abort_flag || !mbar_wait(&e_full[kRing - 1], par, a.wait_ns)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();
          tc_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(dS, qd_rope + (uint32_t)(kk * 2), kd(kRing - 1) + (uint32_t)(kk * 2), kIdQK, (kk > 0) ? 1u : 0u);
          mma_commit(&e_free[kRing - 1]);
          acc = 1u;
        }
        const int vb = kVSlabs * (j & 1);
#pragma unroll
        for (int v = 0; v < kVSlabs; ++v) {
          if (*abort_flag || !mbar_wait(&e_full[vb + v], par, a.wait_ns)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();
          tc_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(dS, tmem + kColQ + 32u * (uint32_t)v + 8u * (uint32_t)kk, kd(vb + v) + (uint32_t)(kk * 2), kIdQK,
                   (acc || v > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
        mma_commit(s_full);
        if (j >= 1 && !issue_pv(j - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && !issue_pv(nb - 1)) ok = false;
      if (ok) mma_commit(o_final);
      if (!ok) fail();
      // Everything issued above is complete before TMEM is freed.  The tensor
      // pipe waits on nothing outside this CTA, so this wait is not cut short
      // by a small caller's limit: it is bounded by 2 s at least.
      mma_commit(fin);
      if (!mbar_wait(fin, 0, a.wait_ns > 2000000000ull ? a.wait_ns : 2000000000ull)) fail();
    }
    __syncwarp();
  } else if (kFetch && warp == kWriterWarp) {
    // ---- fetching: the rows this CTA claimed go to their hot slots ----
    // Once a block's entries have landed, each claimed row part is read from
    // the ring (un-swizzled) and stored to the row's hot slot; then its claim
    // word says written (release, after a fence), and the entries are freed.
    uint8_t* hot_u = reinterpret_cast<uint8_t*>(a.hot_w) + (size_t)u * a.C * (kRow * 2);
    const uint32_t done = 2u * a.epoch + 1u;
    unsigned long long bytes = 0, rows = 0;
    for (int j = 0; j < nb; ++j) {
      if (__any_sync(kFull, *abort_flag != 0u)) break;
      const uint32_t par = (uint32_t)(j >> 1) & 1u;
      const int vb = kVSlabs * (j & 1);
      const bool rope = own_rope(j);
      bool ok = __all_sync(kFull, mbar_wait(&m_ready[j & 1], par, a.wait_ns));
#pragma unroll
      for (int v = 0; v < kVSlabs; ++v) ok = ok && __all_sync(kFull, mbar_wait(&e_full[vb + v], par, a.wait_ns));
      if (rope) ok = ok && __all_sync(kFull, mbar_wait(&e_full[kRing - 1], par, a.wait_ns));
      if (!ok) {
        fail();
        break;
      }
      uint32_t* mk = cmask + (j & 1) * 8;
      uint32_t mv[4], mr[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        mv[w] = mk[w];
        mr[w] = mk[4 + w];
      }
      __syncwarp();
      // cleared for block j + 2, whose claims start after this warp frees block j's entries
      if (lane < 8) mk[lane] = 0u;
      const int32_t* bslots = a.slots + list + (int64_t)j * kBlk;
#pragma unroll 1
      for (int w = 0; w < 4; ++w) {
        uint32_t bits = mv[w];
        while (bits) {  // value part: lane -> slab lane / 8, chunk lane % 8
          const int r = 32 * w + __ffs(bits) - 1;
          bits &= bits - 1u;
          const int32_t slot = __ldg(bslots + r);
          const int v = lane >> 3, c = lane & 7;
          const uint4 x = ld_shared_u4(swz(sb + kROff + (uint32_t)(vb + v) * kEntry, r, c));
          *reinterpret_cast<uint4*>(hot_u + (size_t)slot * (kRow * 2) + half * 512 + v * 128 + c * 16) = x;
        }
        bits = mr[w];
        while (bits) {  // rope part: lanes 0-7, one chunk each
          const int r = 32 * w + __ffs(bits) - 1;
          bits &= bits - 1u;
          if (lane < 8) {
            const int32_t slot = __ldg(bslots + r);
            const uint4 x = ld_shared_u4(swz(sb + kROff + (uint32_t)(kRing - 1) * kEntry, r, lane));
            *reinterpret_cast<uint4*>(hot_u + (size_t)slot * (kRow * 2) + kRopeSlab * 128 + lane * 16) = x;
          }
        }
      }
      __threadfence();
      __syncwarp();
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        if ((mv[w] >> lane) & 1u) {
          const int32_t slot = __ldg(bslots + 32 * w + lane);
          st_release_gpu(a.claim + ((size_t)u * a.C + (size_t)slot) * 3 + half, done);
        }
        if ((mr[w] >> lane) & 1u) {
          const int32_t slot = __ldg(bslots + 32 * w + lane);
          st_release_gpu(a.claim + ((size_t)u * a.C + (size_t)slot) * 3 + 2, done);
        }
        bytes += (unsigned long long)__popc(mv[w]) * 512u + (unsigned long long)__popc(mr[w]) * 128u;
        if (half == 0) rows += (unsigned long long)__popc(mv[w]);
      }
      __syncwarp();
      if (lane == 0) {  // the entries may be refilled once the MMAs are done with them too
#pragma unroll
        for (int v = 0; v < kVSlabs; ++v) mbar_arrive(&e_free[vb + v]);
        if (rope) mbar_arrive(&e_free[kRing - 1]);
      }
    }
    if (lane == 0 && a.stats && bytes) {
      atomicAdd(&a.stats->bytes_h2d, bytes);
      if (rows) atomicAdd(&a.stats->rows_h2d, rows);
    }
  } else if (warp >= kSoftWarp0 && warp < kSoftWarp0 + kSoftThreads / 32) {
    // ---- online softmax: head hd (TMEM lane hd), rows 64 half.. of each block ----
    const int hd = tid - kSoftWarp0 * 32;
    const uint32_t lane_addr = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t sS = tmem + lane_addr + kColS;
    {  // this CTA's query slabs 4 half + i into TMEM: column 32i + x holds elements 64(4 half + i) + 2x, + 2x + 1
      const uint4* qv = reinterpret_cast<const uint4*>(a.q + (size_t)(qrow0 + hd) * kRow) + 32 * half;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const uint4 x = __ldg(qv + 4 * c + q4);
          w[4 * q4] = x.x;
          w[4 * q4 + 1] = x.y;
          w[4 * q4 + 2] = x.z;
          w[4 * q4 + 3] = x.w;
        }
        tmem_st16(tmem + lane_addr + kColQ + 16u * (uint32_t)c, w);
      }
      tmem_wait_st();
      tc_before();
      mbar_arrive(q_full);
    }
    // the partner's shared memory: where this thread's partial scores of its
    // rows, block maxima and P go, and its barriers
    const uint32_t xs_peer = peer_addr(sb + kXSOff, peer), xm_peer = peer_addr(sb + kXMOff, peer);
    const uint32_t p_peer = peer_addr(sb + kPOff, peer);
    const uint32_t xs_full_peer = peer_addr(smem_u32(xs_full), peer), xm_full_peer = peer_addr(smem_u32(xm_full), peer);
    const uint32_t p_full_peer = peer_addr(smem_u32(p_full), peer);
    // partial scores of head hd, rows 4c..4c+3 of the 64: 16-byte cell
    // (c, hd), so that a warp's stores fill consecutive banks
    auto xs_off = [&](int c) { return ((uint32_t)c * kM + (uint32_t)hd) * 16u; };
    // P of head hd, rows 64 half + 8c..: 16-byte chunk c of the head's row in slab `half`
    const uint32_t p_row = (uint32_t)half * kPSlab + (uint32_t)hd * 128u;
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    // slots of rows 64 half + 32c + lane of the next block (validity masks)
    int32_t sn[2];
    auto load_valid = [&](int j) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int r = j * kBlk + kOwnRows * half + 32 * c + lane;
        sn[c] = j < nb && r < a.k ? __ldg(a.slots + list + r) : -1;
      }
    };
    load_valid(0);
    for (int j = 0; j < nb; ++j) {
      // every decision below is warp-uniform; the waits are bounded, so a warp
      // that stops leaves the others and the partner to time out
      bool f = __any_sync(kFull, *abort_flag != 0u);
      if (!f) f = !__all_sync(kFull, mbar_wait(s_full, j & 1, a.wait_ns));
      if (f) {
        ok = false;
        break;
      }
      tc_after();
      uint32_t vm[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) vm[c] = __ballot_sync(kFull, sn[c] >= 0 && sn[c] < a.C);
      load_valid(j + 1);
      // the partner's rows' partial scores to its memory, then own rows' to
      // registers.  The partner's buffer is free: the partner sent its block
      // maximum of the last block after reading what this CTA wrote for it,
      // and that maximum has arrived (the last iteration waited for it).
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float ps[32];
        tmem_ld32(sS + (uint32_t)(kOwnRows * (int)peer) + 32u * (uint32_t)h2, ps);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_async_v4(xs_peer + xs_off(8 * h2 + c), __float_as_uint(ps[4 * c]), __float_as_uint(ps[4 * c + 1]),
                      __float_as_uint(ps[4 * c + 2]), __float_as_uint(ps[4 * c + 3]), xs_full_peer);
      }
      float t[kOwnRows];
      tmem_ld32(sS + (uint32_t)(kOwnRows * half), *reinterpret_cast<float(*)[32]>(&t[0]));
      tmem_ld32(sS + (uint32_t)(kOwnRows * half) + 32u, *reinterpret_cast<float(*)[32]>(&t[32]));
      tmem_wait_ld();
      tc_before();
      mbar_arrive(s_free);  // S is read out: the next block's S may start
      if (!__all_sync(kFull, mbar_wait_cluster(xs_full, j & 1, a.wait_ns))) {
        ok = false;
        break;
      }
      if (hd == 0 && j + 1 < nb) mbar_arrive_expect_tx(xs_full, kXSBytes);
#pragma unroll
      for (int c = 0; c < kOwnRows / 4; ++c) {
        const float4 x = ld_local_f4(sb + kXSOff + xs_off(c));
        t[4 * c] += x.x;
        t[4 * c + 1] += x.y;
        t[4 * c + 2] += x.z;
        t[4 * c + 3] += x.w;
      }
      // log2-scaled scores, -inf for dropped rows, and their maximum
      float mx = -INFINITY;
      if ((vm[0] & vm[1]) == kFull) {  // every row listed (the masks are the same in all lanes)
#pragma unroll
        for (int r = 0; r < kOwnRows; ++r) {
          t[r] *= sl2;
          mx = fmaxf(mx, t[r]);
        }
      } else {
#pragma unroll
        for (int r = 0; r < kOwnRows; ++r) {
          t[r] = ((vm[r >> 5] >> (r & 31)) & 1u) ? t[r] * sl2 : -INFINITY;
          mx = fmaxf(mx, t[r]);
        }
      }
      st_async_f32(xm_peer + (uint32_t)(((j & 1) * kM + hd) * 4), mx, xm_full_peer);
      if (!__all_sync(kFull, mbar_wait_cluster(xm_full, j & 1, a.wait_ns))) {
        ok = false;
        break;
      }
      if (hd == 0) mbar_arrive_expect_tx(xm_full, kM * 4);  // the next block's maxima, or at the end the l
      mx = fmaxf(mx, reinterpret_cast<const float*>(smem + kXMOff)[(j & 1) * kM + hd]);
      // Both CTAs hold the same maxima and running maximum, so they take the
      // same decisions.  The running maximum moves only when a score passes it
      // by more than 2^8 (always on the first block with a listed row); O is
      // then rescaled, once the last P V is done.
      bool pv_seen = j == 0;
      if (__any_sync(kFull, mx > m_run + kRescaleLog2)) {
        const float m_new = fmaxf(m_run, mx);
        const float fac = m_new == -INFINITY ? 1.f : exp2f(m_run - m_new);
        l_run *= fac;
        if (j > 0) {
          if (!__all_sync(kFull, mbar_wait_cluster(p_free, (j - 1) & 1, a.wait_ns))) {
            ok = false;
            break;
          }
          pv_seen = true;
          tc_after();
#pragma unroll 1
          for (int c0 = 0; c0 < kHalfCols; c0 += 16) {
            uint32_t w[16];
            tmem_ld16(tmem + lane_addr + kColO + (uint32_t)c0, w);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 16; ++c) w[c] = __float_as_uint(__uint_as_float(w[c]) * fac);
            tmem_st16(tmem + lane_addr + kColO + (uint32_t)c0, w);
          }
          tmem_wait_st();
        }
        m_run = m_new;
      }
      // the P tiles are free once both CTAs' P V of the last block is done
      if (!pv_seen && !__all_sync(kFull, mbar_wait_cluster(p_free, (j - 1) & 1, a.wait_ns))) {
        ok = false;
        break;
      }
      const float mu = m_run == -INFINITY ? 0.f : m_run;
      // P of the 64 rows (bf16) into both CTAs' P tile; l sums the rounded weights
      float ls = 0.f;
#pragma unroll
      for (int c = 0; c < kOwnRows / 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(ex2_ftz(t[8 * c + 2 * e] - mu), ex2_ftz(t[8 * c + 2 * e + 1] - mu));
          ls += __low2float(b2) + __high2float(b2);
          w[e] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        const uint32_t off = p_row + ((uint32_t)(c ^ (hd & 7)) << 4);
        st_local_v4(sb + kPOff + off, w[0], w[1], w[2], w[3]);
        st_async_v4(p_peer + off, w[0], w[1], w[2], w[3], p_full_peer);
      }
      l_run += ls;
      mbar_arrive(p_full);
    }
    if (ok) ok = __all_sync(kFull, mbar_wait(o_final, 0, a.wait_ns));
    tc_after();
    // l of the whole row: this CTA's rows and the partner's
    st_async_f32(xm_peer + (uint32_t)(((nb & 1) * kM + hd) * 4), l_run, xm_full_peer);
    const bool lx = __all_sync(kFull, mbar_wait_cluster(xm_full, nb & 1, a.wait_ns));
    if (ok && lx) {
      const float l = l_run + reinterpret_cast<const float*>(smem + kXMOff)[(nb & 1) * kM + hd];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint16_t* orow = a.out + (size_t)(qrow0 + hd) * kVal + (size_t)half * kHalfCols;
#pragma unroll 1
      for (int c0 = 0; c0 < kHalfCols; c0 += 32) {
        float o[32];
        tmem_ld32(tmem + lane_addr + kColO + (uint32_t)c0, o);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(o[2 * c] * inv, o[2 * c + 1] * inv);
          w[c] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) dst[q4] = make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
      }
      if (half == 0 && a.lse)
        a.lse[qrow0 + hd] = l > 0.f ? (m_run + log2f(l)) * 0.6931471805599453f : -INFINITY;
    } else {
      fail();
    }
  }
  tc_before();
  cluster_sync();  // no access to the partner's shared memory after this
  if (*abort_flag) {
    // A pair that stopped early may leave an asynchronous store of the
    // partner's into this CTA's shared memory in flight (it was issued before
    // the partner reached the barrier): give it time to land before exiting.
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 20000u) {
    }
  }
  if (warp == kMmaWarp) {
    tc_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

}  // namespace

size_t attend_smem_bytes() { return kAttSmem; }

cudaError_t launch_attend(const AttendArgs& a, cudaStream_t s) {
  if (a.n <= 0) return cudaSuccess;
  const int64_t grid = (int64_t)a.n * a.P * (a.H / kM) * 2;
  if (a.pay) {
    cudaError_t e = cudaFuncSetAttribute(attend_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAttSmem);
    if (e != cudaSuccess) return e;
    attend_kernel<true><<<(unsigned)grid, kAttThreadsFetch, kAttSmem, s>>>(a);
  } else {
    cudaError_t e = cudaFuncSetAttribute(attend_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAttSmem);
    if (e != cudaSuccess) return e;
    attend_kernel<false><<<(unsigned)grid, kAttThreads, kAttSmem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace kvo
