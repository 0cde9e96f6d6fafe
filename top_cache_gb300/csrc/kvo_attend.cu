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
// columns); 256 threads:
//   warps 0-1  copy the query tile once, then 32-row blocks of the hot rows
//              named by the list, with 16-byte cp.async into the 128-byte
//              swizzled layout the MMA reads (two stages);
//   warp 2     holds 512 TMEM columns; lane 0 issues every tcgen05.mma:
//              S = Q K^T (M 128, N 32, K 576, both operands K-major in shared
//              memory) into one of two S buffers, then O += P V (M 128, N 256,
//              K 32) with P read from TMEM and V (the same rows) MN-major;
//   warps 4-7  online softmax, one head (TMEM lane) per thread: S from TMEM,
//              exp2 against a running maximum that moves only when it grows by
//              more than 2^8 (O is then rescaled in TMEM), P rounded to bf16
//              and written back to TMEM, l summed from the rounded weights so
//              that out is their exact weighted mean; at the end O / l in bf16
//              and lse.
// Every mbarrier wait is bounded: on expiry the CTA sets kErrTimeout in the
// error word, stops, waits for its own copies and MMAs and frees its TMEM.
#include <cuda_bf16.h>

#include "kvo_internal.cuh"

namespace kvo {
namespace {

constexpr int kRow = 576;                 // elements per hot row
constexpr int kVal = 512;                 // value (latent) elements
constexpr int kM = 128;                   // heads per CTA: M of both MMAs
constexpr int kBlk = 16;                  // rows per block: N of S, K of P V
constexpr int kStages = 4;                // row blocks in flight
constexpr int kSlabs = kRow / 64;         // 128-byte slabs of a row
constexpr int kHalfCols = kVal / 2;       // value columns per CTA: N of P V
constexpr int kAttThreads = 256;
constexpr int kProducers = 64;            // warps 0-1
constexpr uint32_t kQSlab = kM * 128;     // one slab of the query tile
constexpr uint32_t kKSlab = kBlk * 128;   // one slab of a row block
constexpr uint32_t kKStage = kSlabs * kKSlab;
constexpr uint32_t kQOff = 0;
constexpr uint32_t kKOff = kSlabs * kQSlab;
constexpr uint32_t kBarOff = kKOff + kStages * kKStage;
constexpr uint32_t kAttSmem = kBarOff + 256 + 1024;  // barriers, flags, 1 KB alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;    // O: 256 fp32 columns
constexpr uint32_t kColS = 256;  // S[2]: kBlk fp32 columns each
constexpr uint32_t kColP = 256 + 2 * kBlk;  // P[2]: kBlk / 2 columns of bf16 pairs each
constexpr float kRescaleLog2 = 8.f;
static_assert(kAttSmem <= 232448, "shared memory of one CTA");
static_assert(kBlk == 16, "the softmax moves one 16-column S tile and one 8-column P tile per block");
static_assert(kStages - 2 <= 2, "cp_async_wait_n covers up to kStages - 2 younger groups");

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
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int c = 0; c < 16; ++c) v[c] = __uint_as_float(r[c]);
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
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
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// wait until at most n committed groups are pending (n clamped to 0..2)
__device__ __forceinline__ void cp_async_wait_n(int n) {
  if (n <= 0) cp_async_wait<0>();
  else if (n == 1) cp_async_wait<1>();
  else cp_async_wait<2>();
}
// 16-byte chunk c (0..7) of row r in a 128-byte-swizzled slab (1 KB aligned).
__device__ __forceinline__ uint32_t swz(uint32_t slab, int r, int c) {
  return slab + (uint32_t)r * 128u + ((uint32_t)(c ^ (r & 7)) << 4);
}

__global__ void __launch_bounds__(kAttThreads, 1) attend_kernel(AttendArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* q_full = bars;                       // producers: query tile in place
  uint64_t* k_full = bars + 1;                   // [kStages] producers: row block in place
  uint64_t* k_empty = k_full + kStages;          // [kStages] MMA: block's P V done, stage free
  uint64_t* s_full = k_empty + kStages;          // [2] MMA: S of a block ready
  uint64_t* s_empty = s_full + 2;                // [2] softmax: S read
  uint64_t* p_full = s_empty + 2;                // [2] softmax: P of a block in TMEM
  uint64_t* pv_done = p_full + 2;                // MMA: one more P V done
  uint64_t* o_final = pv_done + 1;               // MMA: the last P V done
  uint64_t* fin = o_final + 1;                   // MMA: everything issued is done
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
  auto fail = [&]() {
    atomicOr(a.err, kErrTimeout);
    *abort_flag = 1u;
  };

  if (tid == 0) {
    mbar_init(q_full, kProducers);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], kProducers);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], 128);
      mbar_init(&p_full[s], 128);
    }
    mbar_init(pv_done, 1);
    mbar_init(o_final, 1);
    mbar_init(fin, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 2) {
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

  if (warp < 2) {
    // ---- copies: query tile, then row blocks (kBlk / 2 rows per warp) ----
    const uint8_t* qsrc = reinterpret_cast<const uint8_t*>(a.q) + qrow0 * (kRow * 2);
    for (int idx = tid; idx < kM * 72; idx += kProducers) {
      const int r = idx / 72, g = idx - r * 72;
      cp_async16(swz(sb + kQOff + (uint32_t)(g >> 3) * kQSlab, r, g & 7), qsrc + (size_t)r * (kRow * 2) + g * 16);
    }
    cp_async_commit();
    const uint8_t* ubase = reinterpret_cast<const uint8_t*>(a.hot) + (size_t)u * a.C * (kRow * 2);
    // slot of row (lane & 15) of this warp's 16 rows of block j; loaded one
    // block ahead so that its latency overlaps the wait for the previous block
    auto load_slot = [&](int j) -> int32_t {
      const int r = j * kBlk + warp * (kBlk / 2) + (lane % (kBlk / 2));
      return j < nb && r < a.k ? __ldg(a.slots + list + r) : -1;
    };
    auto gather = [&](int j, int32_t slot) {
      const uint32_t st = sb + kKOff + (uint32_t)(j % kStages) * kKStage;
      const int r0 = warp * (kBlk / 2);
      if (slot < 0 || slot >= a.C) slot = 0;  // a pad reads a valid row; the softmax drops it
#pragma unroll 4
      for (int x = 0; x < kBlk / 2; ++x) {
        const uint8_t* src = ubase + (size_t)__shfl_sync(kFull, slot, x) * (kRow * 2);
        const int row = r0 + x;
        for (int g = lane; g < 72; g += 32) cp_async16(swz(st + (uint32_t)(g >> 3) * kKSlab, row, g & 7), src + g * 16);
      }
      cp_async_commit();
    };
    gather(0, load_slot(0));
    int32_t slot_next = load_slot(1);
    // Block j is announced as soon as its copies have landed; only then does
    // the warp wait for the stage of block j+1 (freed by the P V of block
    // j+1-kStages, which the MMA issues after it has seen block j+2-kStages)
    // and start copying block j+1.
    for (int j = 0; j < nb; ++j) {
      cp_async_wait<0>();
      fence_proxy_async_smem();  // the tensor cores read what cp.async wrote
      if (j == 0) mbar_arrive(q_full);
      mbar_arrive(&k_full[j % kStages]);
      if (j + 1 >= nb) break;
      if (__any_sync(kFull, *abort_flag != 0u)) break;  // warp-uniform: shuffles follow
      // stage of block j+1 last held block j+1-kStages
      const int jn = j + 1;
      const bool ok = __all_sync(kFull, jn < kStages || mbar_wait(&k_empty[jn % kStages], ((jn / kStages) - 1) & 1, a.wait_ns));
      if (!ok) {
        fail();
        break;
      }
      gather(j + 1, slot_next);
      slot_next = load_slot(j + 2);
    }
    cp_async_wait<0>();
  } else if (warp == 2) {
    // ---- MMA issue (one thread) ----
    if (lane == 0) {
      constexpr uint32_t kIdQK = idesc_bf16(kM, kBlk, false);
      constexpr uint32_t kIdPV = idesc_bf16(kM, kHalfCols, true);
      bool ok = mbar_wait(q_full, 0, a.wait_ns);
      const uint64_t qdesc = sdesc(sb + kQOff, 16, 1024);
      auto issue_pv = [&](int jj) -> bool {
        const int sp = jj & 1;
        if (!mbar_wait(&p_full[sp], (jj >> 1) & 1, a.wait_ns)) return false;
        tc_after();
        // V = this CTA's 4 value slabs of the block: MN-major, 64 columns per
        // slab (leading offset = slab stride), 8-row groups 1 KB apart
        const uint32_t vb = sb + kKOff + (uint32_t)(jj % kStages) * kKStage + (uint32_t)half * 4u * kKSlab;
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk)
          mma_ts(tmem + kColO, tmem + kColP + (uint32_t)sp * (kBlk / 2) + (uint32_t)kk * 8u,
                 sdesc(vb + (uint32_t)kk * 16u * 128u, kKSlab, 1024), kIdPV, (jj > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&k_empty[jj % kStages]);
        mma_commit(pv_done);
        return true;
      };
      for (int j = 0; ok && j < nb; ++j) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        const int st = j & 1;
        if (!mbar_wait(&k_full[j % kStages], (j / kStages) & 1, a.wait_ns) ||
            (j >= 2 && !mbar_wait(&s_empty[st], ((j - 2) >> 1) & 1, a.wait_ns))) {
          ok = false;
          break;
        }
        tc_after();
        // base descriptors once per block; the 36 K-steps add compile-time
        // offsets to the start-address field (shared addresses stay below
        // 2^18, so the 14-bit field never carries)
        const uint64_t kdesc = sdesc(sb + kKOff + (uint32_t)(j % kStages) * kKStage, 16, 1024);
        const uint32_t dS = tmem + kColS + (uint32_t)st * kBlk;
        mma_ss(dS, qdesc, kdesc, kIdQK, 0u);
#pragma unroll
        for (int kk = 1; kk < kRow / 16; ++kk) {
          const uint32_t c = (uint32_t)(kk & 3) * 32u;
          mma_ss(dS, qdesc + (((uint32_t)(kk >> 2) * kQSlab + c) >> 4),
                 kdesc + (((uint32_t)(kk >> 2) * kKSlab + c) >> 4), kIdQK, 1u);
        }
        mma_commit(&s_full[st]);
        if (j >= 1 && !issue_pv(j - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && nb > 0 && !issue_pv(nb - 1)) ok = false;
      if (ok) mma_commit(o_final);
      if (!ok) fail();
      mma_commit(fin);  // everything issued above is complete before TMEM is freed
      if (!mbar_wait(fin, 0, a.wait_ns)) fail();
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---- online softmax, one head per thread ----
    const int h = tid - 128;
    const uint32_t lane_addr = (uint32_t)(32 * (warp & 3)) << 16;
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    // slot of row `lane` of the next block, loaded a block ahead (validity mask)
    int32_t sl_next = lane < kBlk && lane < a.k ? __ldg(a.slots + list + lane) : -1;
    for (int j = 0; j < nb; ++j) {
      if (__any_sync(kFull, *abort_flag != 0u)) {  // warp-uniform: TMEM access is warp-wide
        ok = false;
        break;
      }
      const int st = j & 1;
      ok = __all_sync(kFull, mbar_wait(&s_full[st], (j >> 1) & 1, a.wait_ns));
      if (!ok) break;
      tc_after();
      float v[kBlk];
      tmem_ld16(tmem + lane_addr + kColS + (uint32_t)st * kBlk, v);
      tmem_wait_ld();
      tc_before();
      mbar_arrive(&s_empty[st]);
      const int32_t sl = sl_next;
      sl_next = lane < kBlk && (j + 1) * kBlk + lane < a.k ? __ldg(a.slots + list + (j + 1) * kBlk + lane) : -1;
      const uint32_t vm = __ballot_sync(kFull, sl >= 0 && sl < a.C);
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kBlk; ++c) {
        v[c] = ((vm >> c) & 1u) ? v[c] * sl2 : -INFINITY;
        mx = fmaxf(mx, v[c]);
      }
      if (__any_sync(kFull, mx > m_run + kRescaleLog2)) {
        // the warp moves its maxima together (TMEM access is warp-wide)
        const float m_new = fmaxf(m_run, mx);
        const float f = m_new == -INFINITY ? 1.f : exp2f(m_run - m_new);
        l_run *= f;
        if (j > 0) {  // O holds P V of blocks 0..j-1
          ok = __all_sync(kFull, mbar_wait(pv_done, (j - 1) & 1, a.wait_ns));
          if (!ok) break;
          tc_after();
#pragma unroll 1
          for (int c0 = 0; c0 < kHalfCols; c0 += 32) {
            float o[32];
            tmem_ld32(tmem + lane_addr + kColO + (uint32_t)c0, o);
            tmem_wait_ld();
            uint32_t w[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) w[c] = __float_as_uint(o[c] * f);
            tmem_st32(tmem + lane_addr + kColO + (uint32_t)c0, w);
          }
          tmem_wait_st();
        }
        m_run = m_new;
      }
      const float mu = m_run == -INFINITY ? 0.f : m_run;
      uint32_t pk[kBlk / 2];
      float ls = 0.f;
#pragma unroll
      for (int c = 0; c < kBlk / 2; ++c) {
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(exp2f(v[2 * c] - mu), exp2f(v[2 * c + 1] - mu));
        ls += __low2float(b2) + __high2float(b2);
        pk[c] = *reinterpret_cast<const uint32_t*>(&b2);
      }
      l_run += ls;
      tmem_st8(tmem + lane_addr + kColP + (uint32_t)st * (kBlk / 2), pk);
      tmem_wait_st();
      tc_before();
      mbar_arrive(&p_full[st]);
    }
    if (ok) ok = __all_sync(kFull, mbar_wait(o_final, 0, a.wait_ns));
    if (ok) {
      tc_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      uint16_t* orow = a.out + (size_t)(qrow0 + h) * kVal + (size_t)half * kHalfCols;
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
        a.lse[qrow0 + h] = l_run > 0.f ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
    } else {
      fail();
    }
  }
  tc_before();
  __syncthreads();
  if (warp == 2) {
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
