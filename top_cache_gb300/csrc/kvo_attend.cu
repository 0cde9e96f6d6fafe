// Sparse attention over the hot buffer on the 5th-generation tensor cores:
// decode step 7 of "Layerwise and Sparse KV Cache Offloading Design"
// (section 4, "Decode step": sparse attention consumes the resident K/V).
//
// Reading R13 of the oracle (the pages name an SFA/MLA sparse-attention model
// but give no formula): absorbed latent attention.  A hot row is 576 bf16 =
// latent (512, which is also the value) | rope key (64); the query of a head
// has the same split.  For unit u, position p and head h, over the slots of
// that position's top-k list (pads, slot < 0, skipped):
//   s_i = scale * q_h . row_i,   out_h = sum_i softmax(s)_i * row_i[0:512],
//   lse_h = log sum_i exp(s_i).
//
// One CTA per (unit, position, group of 128 heads, half of the 512 value
// columns); 512 threads.  The list is cut into blocks of 128 rows.  Issuing a
// tcgen05.mma from one thread costs about a hundred cycles whatever N is up to
// 128, so every MMA is made as wide as the operands allow: S MMAs have N = 128
// (a block), and one block's P V is eight MMAs of N = 256 (this CTA's value
// columns).  The query tile (128 x 576 bf16) stays on chip: the four
// 64-column slabs that match this CTA's value slabs in TMEM (the A operand of
// their S MMAs: issuing an MMA with A in TMEM is cheaper), the other five in
// shared memory.  That leaves room for a ring of nine 16 KB entries, one per
// slab of a block (entry t always holds slab t of the current block), this
// CTA's four value slabs last and side by side, so that they form the N = 256
// operand of P V, while the next block's other five slabs stream in:
//   warps 0-3  copy those five query slabs, then every slab of every block with
//              16-byte cp.async into the 128-byte-swizzled K-major layout the
//              MMA reads (four warps: the rate at which cp.async goes out
//              grows with the warps issuing it);
//   warp 4     holds 512 TMEM columns; lane 0 issues every tcgen05.mma:
//              S = Q K^T (M 128, N 128, K 64 per slab) into the S buffer;
//              once P is ready, O += P V (M 128, N 256, K 128), P read from
//              TMEM, before the next block's S (S is single-buffered);
//   warps 8-15 put the other four into TMEM, then run the online softmax: a
//              head (TMEM lane) per thread pair, warp 8+q taking the first 64
//              rows of a block and warp 12+q the other 64 for heads 32q..;
//              each reads its scores once, the pair agrees on the block
//              maximum through TMEM and a named barrier, the running maximum
//              moves only when it grows by more than 2^8 (O is then rescaled
//              in TMEM), P is rounded to bf16 and written back over the first
//              64 columns of S, and l sums the rounded weights so that out is
//              their exact weighted mean; at the end O / l in bf16 and lse.
// A ring entry is freed by the MMAs that read it last: the S MMAs for the five
// slabs only the scores use, the P V MMAs for the value slabs.
// Every mbarrier wait is bounded: on expiry the CTA sets kErrTimeout in the
// error word, stops, waits for its own copies and MMAs and frees its TMEM.
#include <cuda_bf16.h>

#include "kvo_internal.cuh"

namespace kvo {
namespace {

constexpr int kRow = 576;                 // elements per hot row
constexpr int kVal = 512;                 // value (latent) elements
constexpr int kM = 128;                   // heads per CTA: M of the MMAs
constexpr int kBlk = 128;                 // rows per block: N of S, K of P V
constexpr int kSlabs = kRow / 64;         // 128-byte slabs of a row
constexpr int kVSlabs = 4;                // value slabs of this CTA's half
constexpr int kRing = kSlabs;             // ring entries: entry t holds slab t of a block
constexpr int kQTmemSlabs = kVSlabs;      // query slabs in TMEM: this CTA's value slabs (entries 5..8)
constexpr int kHalfCols = kVal / 2;       // value columns per CTA
constexpr int kAttThreads = 512;
constexpr int kProducers = 128;           // warps 0-3: copies
constexpr int kMmaWarp = 4;               // TMEM allocation and MMA issue
constexpr int kSoftWarp0 = 8;             // warps 8-15: softmax
constexpr int kSoftThreads = 256;
constexpr int kRowStep = kProducers / 8;  // rows of an entry between one copy thread's chunks
constexpr uint32_t kQSlab = kM * 128;     // one slab of the query tile
constexpr uint32_t kEntry = kBlk * 128;   // one slab of a row block
constexpr uint32_t kQOff = 0;             // the query slabs of entries 0..4, in entry order
constexpr uint32_t kROff = (kSlabs - kQTmemSlabs) * kQSlab;
constexpr uint32_t kBarOff = kROff + kRing * kEntry;
constexpr uint32_t kAttSmem = kBarOff + 256 + 1024;  // barriers, flags, 1 KB alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;    // O: 256 fp32 columns
constexpr uint32_t kColS = 256;  // S: 128 fp32 columns; P (bf16 pairs) over its first 64
constexpr uint32_t kColQ = 384;  // query slabs 4 half + i: 128 columns of bf16 pairs (32 per slab)
constexpr float kRescaleLog2 = 8.f;
static_assert(kAttSmem <= 232448, "shared memory of one CTA");
static_assert(kBlk % kRowStep == 0 && kSoftWarp0 % 4 == 0, "copy rows; softmax warps start a TMEM lane quadrant");
static_assert(kRing == kSlabs, "entry t of the ring holds slab t of the current block");
static_assert(kColQ + kQTmemSlabs * 32 <= kTmemCols, "TMEM columns");
static_assert(kQTmemSlabs == 4, "the softmax warps load four query slabs, two per warp pair member");

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
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
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
// Two consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st2(uint32_t taddr, uint32_t x, uint32_t y) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(taddr), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void tmem_ld2(uint32_t taddr, uint32_t& x, uint32_t& y) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];" : "=r"(x), "=r"(y) : "r"(taddr) : "memory");
}
// Barrier `id` (1..15) over `threads` threads (whole warps).
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
// 16-byte chunk c (0..7) of row r in a 128-byte-swizzled slab (1 KB aligned).
__device__ __forceinline__ uint32_t swz(uint32_t slab, int r, int c) {
  return slab + (uint32_t)r * 128u + ((uint32_t)(c ^ (r & 7)) << 4);
}

// Slab of the row that entry t (0..8) of a block carries: first the five the
// scores alone use (the other half's value slabs, the rope key), then this
// CTA's value slabs in column order.
__device__ __forceinline__ int slab_of(int t, int half) {
  return t < 4 ? 4 * (1 - half) + t : t == 4 ? 8 : 4 * half + (t - 5);
}

__global__ void __launch_bounds__(kAttThreads, 1) attend_kernel(AttendArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* q_full = bars;            // copies and softmax warps: query tile in place
  uint64_t* e_full = bars + 1;        // [kRing] copies: entry in place
  uint64_t* e_free = e_full + kRing;  // [kRing] MMA: the entry's last reader done
  uint64_t* s_full = e_free + kRing;  // MMA: S of a block ready
  uint64_t* p_full = s_full + 1;      // softmax: P of a block in TMEM
  uint64_t* pv_done = p_full + 1;     // MMA: one more block's P V done
  uint64_t* o_final = pv_done + 1;    // MMA: the last P V done
  uint64_t* fin = o_final + 1;        // MMA: everything issued is done
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(fin + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int b = blockIdx.x;
  const int half = b & 1;
  b >>= 1;
  const int HG = a.H / kM;
  const int hg = b % HG;
  b /= HG;
  const int p = b % a.P;
  const int i = b / a.P;
  const int u = a.units[i];
  const int64_t list = ((int64_t)i * a.P + p) * a.k;
  const int64_t qrow0 = ((int64_t)i * a.P + p) * a.H + (int64_t)hg * kM;
  const int nb = (a.k + kBlk - 1) / kBlk;
  const int ne = nb * kSlabs;  // ring entries over the whole list
  auto fail = [&]() {
    atomicOr(a.err, kErrTimeout);
    *abort_flag = 1u;
  };

  if (tid == 0) {
    mbar_init(q_full, kProducers + kSoftThreads);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&e_full[s], kProducers);
      mbar_init(&e_free[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, kSoftThreads);
    mbar_init(pv_done, 1);
    mbar_init(o_final, 1);
    mbar_init(fin, 1);
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
  __syncthreads();
  tc_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= kSoftWarp0) {
    // the softmax warps put this CTA's value slabs 4 half + i (i < 4) of
    // their head's query into TMEM, the A operand of those slabs' S MMAs:
    // column 32i + x of lane h holds elements 64(4 half + i) + 2x and + 2x + 1
    // of head h.  Warps 8+q and 12+q (lanes 32q..) take i = 0-1 and 2-3.
    const int ch = (warp - kSoftWarp0) >> 2;
    const uint4* qv =
        reinterpret_cast<const uint4*>(a.q + (size_t)(qrow0 + 32 * (warp & 3) + lane) * kRow) + 32 * half + 16 * ch;
    const uint32_t qa = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + kColQ + 64u * (uint32_t)ch;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t w[16];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint4 x = __ldg(qv + 4 * c + q4);
        w[4 * q4] = x.x;
        w[4 * q4 + 1] = x.y;
        w[4 * q4 + 2] = x.z;
        w[4 * q4 + 3] = x.w;
      }
      tmem_st16(qa + 16u * (uint32_t)c, w);
    }
    tmem_wait_st();
    tc_before();
    mbar_arrive(q_full);
  }
  if (warp < kProducers / 32) {
    // ---- copies: the query slabs of entries 0..4, then every slab of every block ----
    const uint8_t* qsrc = reinterpret_cast<const uint8_t*>(a.q) + qrow0 * (kRow * 2);
    constexpr int kQChunks = (kSlabs - kQTmemSlabs) * 8;
    for (int idx = tid; idx < kM * kQChunks; idx += kProducers) {
      const int r = idx / kQChunks, g = idx - r * kQChunks;  // 16-byte chunk g of the smem part
      cp_async16(swz(sb + kQOff + (uint32_t)(g >> 3) * kQSlab, r, g & 7),
                 qsrc + (size_t)r * (kRow * 2) + slab_of(g >> 3, half) * 128 + (g & 7) * 16);
    }
    cp_async_arrive_noinc(q_full);
    const uint8_t* ubase = reinterpret_cast<const uint8_t*>(a.hot) + (size_t)u * a.C * (kRow * 2);
    // this thread copies chunk csub of rows rsub + kRowStep m of every entry
    const int rsub = tid >> 3, csub = tid & 7;
    // slots of this thread's rows of the current block (rs) and of the next
    // (rs_next, loaded a block ahead so that a block's first copies do not
    // wait for them)
    int32_t rs[kBlk / kRowStep], rs_next[kBlk / kRowStep];
    auto load_rows = [&](int j, int32_t (&dst)[kBlk / kRowStep]) {
#pragma unroll
      for (int m = 0; m < kBlk / kRowStep; ++m) {
        const int r = j * kBlk + rsub + kRowStep * m;
        dst[m] = j < nb && r < a.k ? __ldg(a.slots + list + r) : -1;
      }
    };
    load_rows(0, rs_next);
    int rs_block = -1;
    auto issue = [&](int e) {
      const int j = e / kSlabs, t = e - j * kSlabs;
      if (j != rs_block) {  // blocks are issued in order: rs_next holds block j
#pragma unroll
        for (int m = 0; m < kBlk / kRowStep; ++m)  // a pad reads a valid row; the softmax drops it
          rs[m] = rs_next[m] < 0 || rs_next[m] >= a.C ? 0 : rs_next[m];
        rs_block = j;
        load_rows(j + 1, rs_next);
      }
      const uint32_t dst = sb + kROff + (uint32_t)(e % kRing) * kEntry;
      const int s = slab_of(t, half);
#pragma unroll
      for (int m = 0; m < kBlk / kRowStep; ++m)
        cp_async16(swz(dst, rsub + kRowStep * m, csub), ubase + (size_t)rs[m] * (kRow * 2) + s * 128 + csub * 16);
      cp_async_arrive_noinc(&e_full[e % kRing]);  // counts once this thread's copies have landed
    };
    // Entries go out in order, each as soon as its ring slot is free; a
    // block's first entry only once the previous block has landed (its last
    // entry's barrier has completed): the value slabs of a block are on the
    // critical path (their slots free up only when the last block's P V is
    // done), and the next block's slabs would share the copy bandwidth with
    // them.  Completion is tracked by the entry's barrier itself, so the
    // warps never wait for their own copies and keep the ring full.
    for (int e = 0; e < ne; ++e) {
      if (__any_sync(kFull, *abort_flag != 0u)) break;  // warp-uniform: shuffles follow
      const int j = e / kSlabs, t = e - j * kSlabs;
      bool ok = true;
      if (t == 0 && j > 0)
        ok = __all_sync(kFull, mbar_wait(&e_full[kSlabs - 1], (j - 1) & 1, a.wait_ns));
      if (ok && e >= kRing)
        ok = __all_sync(kFull, mbar_wait(&e_free[t], ((e / kRing) - 1) & 1, a.wait_ns));
      if (!ok) {
        fail();
        break;
      }
      issue(e);
    }
    cp_async_wait_all();
  } else if (warp == kMmaWarp) {
    // ---- MMA issue (one thread) ----
    if (lane == 0) {
      constexpr uint32_t kIdQK = idesc_bf16(kM, kBlk, false);
      constexpr uint32_t kIdPV = idesc_bf16(kM, kHalfCols, true);
      bool ok = mbar_wait(q_full, 0, a.wait_ns);
      fence_proxy_async_smem();  // the tensor cores read what cp.async wrote (acquired through the barrier)
      // entry t always sits in ring slot t: the descriptors are fixed
      uint64_t kd[kSlabs], qd[kSlabs];
      uint32_t qa[kSlabs];
#pragma unroll
      for (int t = 0; t < kSlabs; ++t) {
        const int tq = t - (kSlabs - kQTmemSlabs);  // >= 0: the query slab is in TMEM
        kd[t] = sdesc(sb + kROff + (uint32_t)t * kEntry, 16, 1024);
        qd[t] = sdesc(sb + kQOff + (uint32_t)(tq < 0 ? t : 0) * kQSlab, 16, 1024);
        qa[t] = tmem + kColQ + 32u * (uint32_t)(tq < 0 ? 0 : tq);
      }
      // V: the four value slabs of a block in slots kSlabs-kVSlabs.. are the
      // four 64-column chunks of one N = 256 MN-major operand (chunk stride:
      // one ring entry; 8-row groups 1 KB apart)
      const uint64_t vdesc = sdesc(sb + kROff + (uint32_t)(kSlabs - kVSlabs) * kEntry, kEntry, 1024);
      int pv_next = 0;  // first block whose P V is not issued yet
      // O += P V for block jj; the value slabs' entries are freed once done
      auto issue_pv = [&](int jj) -> bool {
        if (!mbar_wait(&p_full[0], jj & 1, a.wait_ns)) return false;
        tc_after();
        const uint32_t pa = tmem + kColS;  // P: first 64 columns of S
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk)
          mma_ts(tmem + kColO, pa + 8u * (uint32_t)kk, vdesc + ((uint32_t)kk * 16u * 128u >> 4), kIdPV,
                 (jj > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int v = 0; v < kVSlabs; ++v) mma_commit(&e_free[kSlabs - kVSlabs + v]);
        mma_commit(pv_done);
        return true;
      };
      auto flush_pv = [&](int upto) -> bool {  // P V of blocks pv_next..upto, in order
        for (; pv_next <= upto; ++pv_next)
          if (!issue_pv(pv_next)) return false;
        return true;
      };
      for (int j = 0; ok && j < nb; ++j) {
        // S holds P of block j-1 until its P V is issued (the tensor pipe runs
        // MMAs in order, so P is read before this block's S overwrites it);
        // the same P V frees the value slots this block's entries 5..8 reuse
        if (j >= 1 && !flush_pv(j - 1)) {
          ok = false;
          break;
        }
        const uint32_t dS = tmem + kColS;
#pragma unroll
        for (int t = 0; t < kSlabs; ++t) {
          const int e = j * kSlabs + t;
          if (*abort_flag || !mbar_wait(&e_full[t], (e / kRing) & 1, a.wait_ns)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();  // as for the query slabs
          tc_after();
          if (t >= kSlabs - kQTmemSlabs) {  // A: the query slab in TMEM (8 columns per K step)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(dS, qa[t] + 8u * (uint32_t)kk, kd[t] + (uint32_t)(kk * 2), kIdQK, (t > 0 || kk > 0) ? 1u : 0u);
          } else {  // A: from shared memory
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(dS, qd[t] + (uint32_t)(kk * 2), kd[t] + (uint32_t)(kk * 2), kIdQK, (t > 0 || kk > 0) ? 1u : 0u);
          }
          if (t < kSlabs - kVSlabs) mma_commit(&e_free[t]);  // only the scores read this slab
        }
        if (!ok) break;
        mma_commit(&s_full[0]);
      }
      if (ok && !flush_pv(nb - 1)) ok = false;
      if (ok) mma_commit(o_final);
      if (!ok) fail();
      mma_commit(fin);  // everything issued above is complete before TMEM is freed
      if (!mbar_wait(fin, 0, a.wait_ns)) fail();
    }
    __syncwarp();
  } else if (warp >= kSoftWarp0) {
    // ---- online softmax: warps 8+q and 12+q share the heads (TMEM lanes)
    // 32q..32q+31, one thread per head and half (ch) of each block's rows ----
    const int q = warp & 3, ch = (warp - kSoftWarp0) >> 2;
    const int h = 32 * q + lane;
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    const uint32_t sS = tmem + lane_addr + kColS;
    // exchange slots: the last two S columns of each half, read by their
    // owner before the exchange and written by no MMA until P is consumed
    const uint32_t x_mine = sS + 64u * (uint32_t)ch + 62u, x_peer = sS + 64u * (uint32_t)(1 - ch) + 62u;
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    // slots of this half's rows 64ch + 32c + lane of the next block (validity masks)
    int32_t sn[2];
    auto load_valid = [&](int j) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int r = j * kBlk + 64 * ch + 32 * c + lane;
        sn[c] = j < nb && r < a.k ? __ldg(a.slots + list + r) : -1;
      }
    };
    // the partner warps pass (stop flag, value) through TMEM and a named
    // barrier, so that they take every decision (stop, rescale) together;
    // every exchange is reached by both (a stop is taken only after one)
    uint32_t peer_stop, peer_val;
    auto exchange = [&](bool stop_mine, float val) {
      tmem_st2(x_mine, stop_mine ? 1u : 0u, __float_as_uint(val));
      tmem_wait_st();
      tc_before();
      named_bar_sync(1 + q, 64);
      tc_after();
      tmem_ld2(x_peer, peer_stop, peer_val);
      tmem_wait_ld();
    };
    load_valid(0);
    for (int j = 0; j < nb; ++j) {
      bool stop = __any_sync(kFull, *abort_flag != 0u);
      if (!stop) stop = !__all_sync(kFull, mbar_wait(&s_full[0], j & 1, a.wait_ns));
      tc_after();
      uint32_t vm[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) vm[c] = __ballot_sync(kFull, sn[c] >= 0 && sn[c] < a.C);
      load_valid(j + 1);
      // this half's 64 scores, log2-scaled, -inf for dropped rows
      float t[64];
      tmem_ld32(sS + 64u * (uint32_t)ch, *reinterpret_cast<float(*)[32]>(&t[0]));
      tmem_ld32(sS + 64u * (uint32_t)ch + 32u, *reinterpret_cast<float(*)[32]>(&t[32]));
      tmem_wait_ld();
      float mx = -INFINITY;
      if ((vm[0] & vm[1]) == kFull) {  // every row listed (the masks are the same in all lanes)
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          t[i] *= sl2;
          mx = fmaxf(mx, t[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          t[i] = ((vm[i >> 5] >> (i & 31)) & 1u) ? t[i] * sl2 : -INFINITY;
          mx = fmaxf(mx, t[i]);
        }
      }
      exchange(stop, mx);
      if (__any_sync(kFull, stop || peer_stop != 0u)) {  // warp-uniform, and the same in both partners
        ok = false;
        break;
      }
      mx = fmaxf(mx, __uint_as_float(peer_val));
      // the maximum moves only when a score passes it by more than 2^8 (always
      // on the first block with a listed row); O is then rescaled in TMEM
      if (__any_sync(kFull, mx > m_run + kRescaleLog2)) {
        const float m_new = fmaxf(m_run, mx);
        const float f = m_new == -INFINITY ? 1.f : exp2f(m_run - m_new);
        l_run *= f;
        if (j > 0) {  // O holds P V of blocks 0..j-1
          if (!__all_sync(kFull, mbar_wait(pv_done, (j - 1) & 1, a.wait_ns))) {
            fail();  // the partner learns of it at the next exchange
          } else {
            tc_after();
#pragma unroll 1
            for (int c0 = 0; c0 < kHalfCols / 2; c0 += 32) {
              const uint32_t oa = tmem + lane_addr + kColO + (uint32_t)(kHalfCols / 2 * ch + c0);
              float o[32];
              tmem_ld32(oa, o);
              tmem_wait_ld();
              uint32_t w[32];
#pragma unroll
              for (int c = 0; c < 32; ++c) w[c] = __float_as_uint(o[c] * f);
              tmem_st32(oa, w);
            }
            tmem_wait_st();
          }
        }
        m_run = m_new;
      }
      const float mu = m_run == -INFINITY ? 0.f : m_run;
      // P rounded to bf16 over columns 32ch.. of S (every thread has read its
      // scores: the exchange came after); l sums the rounded weights
      float ls = 0.f;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(ex2_ftz(t[32 * c + 2 * e] - mu), ex2_ftz(t[32 * c + 2 * e + 1] - mu));
          ls += __low2float(b2) + __high2float(b2);
          w[e] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        tmem_st16(sS + 32u * (uint32_t)ch + 16u * (uint32_t)c, w);
      }
      tmem_wait_st();
      l_run += ls;
      tc_before();
      mbar_arrive(&p_full[0]);
    }
    if (ok) ok = __all_sync(kFull, mbar_wait(o_final, 0, a.wait_ns));
    tc_after();
    // l of the whole row: both halves' sums (no MMA touches S any more)
    exchange(!ok, l_run);
    if (ok && peer_stop == 0u) {
      const float l = l_run + __uint_as_float(peer_val);
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint16_t* orow = a.out + (size_t)(qrow0 + h) * kVal + (size_t)half * kHalfCols + (size_t)(kHalfCols / 2) * ch;
#pragma unroll 1
      for (int c0 = 0; c0 < kHalfCols / 2; c0 += 32) {
        float o[32];
        tmem_ld32(tmem + lane_addr + kColO + (uint32_t)(kHalfCols / 2 * ch + c0), o);
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
      if (half == 0 && ch == 0 && a.lse)
        a.lse[qrow0 + h] = l > 0.f ? (m_run + log2f(l)) * 0.6931471805599453f : -INFINITY;
    } else {
      fail();
    }
  }
  tc_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

}  // namespace

size_t attend_smem_bytes() { return kAttSmem; }

cudaError_t launch_attend(const AttendArgs& a, cudaStream_t s) {
  if (a.n <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAttSmem);
  if (e != cudaSuccess) return e;
  const int64_t grid = (int64_t)a.n * a.P * (a.H / kM) * 2;
  attend_kernel<<<(unsigned)grid, kAttThreads, kAttSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvo
