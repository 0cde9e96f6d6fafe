// Residency update, miss-row fill and new-token append.
//
// "Layerwise and Sparse KV Cache Offloading Design", section 4 "Sparse Decode
// Offload", Decode step: (2) each new token's K/V row lands at its own logical
// index of the host pool, (4) a per-layer LRU table tells hits from misses,
// gives each miss a hot slot and picks the slots to evict, (5) only missed
// rows cross host -> device, (6) the top-k's logical positions become hot
// slots.  "FlashOffloading ... What does it mean?", decode paragraphs: the
// shelf has a fixed size, the four MTP3 positions' miss lists become one
// list without repeats before any load, cache_slots gives a token's slot or -1.
//
//  residency_kernel : one CTA per unit; merge + dedup of the P lists, LRU
//                     victims in (last_use, slot) order, reverse-index
//                     updates, remap; the last CTA to finish writes the
//                     prefix sums of the per-unit miss counts.
//  gather_ldg_kernel / gather_bulk_kernel : persistent copy of every miss row
//                     from the mapped pinned host pool into the hot buffers.
//  append_kernel    : one CTA per unit; new rows to the host pool, new keys
//                     to the indexer cache, len += n.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvo_device.cuh"
#include "kvo_internal.cuh"

namespace kvo {

namespace {

constexpr int kResThreads = 1024;
constexpr int kGatherThreads = 256;
constexpr int kGatherRows = 32;     // rows per batch (LDG gather)
constexpr int kBulkDepth = 4;       // rows in flight per warp (bulk gather)

}  // namespace

// ---------------------------------------------------------------------------
// residency: merge/dedup, LRU, reverse index, remap (one CTA per unit)
//
// No sorting: the distinct misses come out in token order from a token
// bitmap (each thread owns a contiguous run of words; one block scan), and
// the LRU order is an explicit list of the unit's slots kept in (last_use,
// slot) order: victims are the first m entries not hit this step, and the
// step's touched slots (hits and filled misses, all with the new stamp) move
// to the end in slot order.  Every slot starts free with last_use 0, so the
// initial list 0..C-1 is in that order, and the update preserves it.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kResThreads) residency_kernel(ResidencyArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int PK = a.P * a.k;
  const int nwords_pad = (((a.C + 31) >> 5) + 3) & ~3;
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem);        // [nwords_pad] hit, then touched slots
  int32_t* M = reinterpret_cast<int32_t*>(bitmap + nwords_pad);  // [PK] distinct misses, ascending
  int32_t* V = M + PK;                                          // [PK] victims in LRU order
  __shared__ uint32_t wsum[32];
  __shared__ uint32_t sc[8];
  const int tid = threadIdx.x;
  auto sync = [] { __syncthreads(); };
  dev::residency_body<kResThreads>(a, blockIdx.x, bitmap, M, V, wsum, tid, sync, nullptr, [](uint32_t) {});

  // the last CTA writes the prefix sums of the miss counts
  __threadfence();
  __syncthreads();
  if (tid == 0) sc[2] = (atomicAdd(a.done_ctr, 1u) == (uint32_t)(a.n - 1)) ? 1u : 0u;
  __syncthreads();
  if (sc[2]) {
    __threadfence();
    int64_t carry = 0;
    for (int base = 0; base < a.n; base += kResThreads) {
      const int e = base + tid;
      const uint32_t v = e < a.n ? (uint32_t)__ldcg(&a.miss_cnt[e]) : 0u;
      uint32_t total;
      const uint32_t pos = dev::block_excl_scan<kResThreads>(v, wsum, &total, tid, sync);
      if (e < a.n) a.miss_off[e] = carry + pos;
      carry += total;
    }
    if (tid == 0) {
      a.miss_off[a.n] = carry;
      *a.done_ctr = 0;
    }
  }
}

// ---------------------------------------------------------------------------
// gather, 16-byte loads from the mapped host pool (zero copy)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kGatherThreads) gather_ldg_kernel(GatherArgs a) {
  __shared__ int64_t src_off[kGatherRows];
  __shared__ int64_t dst_off[kGatherRows];
  __shared__ uint32_t word[4];
  const dev::CopyScratch cs{src_off, dst_off, nullptr, word};
  dev::gather_rows_ldg<kGatherThreads, kGatherRows, 8>(a, (int)blockIdx.x, (int)gridDim.x, cs);
}

// ---------------------------------------------------------------------------
// gather, bulk async copies host -> shared -> hot (one elected lane per warp,
// kBulkDepth rows in flight per warp)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kGatherThreads) gather_bulk_kernel(GatherArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kWarps = kGatherThreads / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t row_bytes = (uint32_t)a.row_elems * 2u;
  const uint32_t slot_bytes = (row_bytes + 127u) & ~127u;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // [kWarps][kBulkDepth]
  uint8_t* stage = smem + 128 * ((kWarps * kBulkDepth * 8 + 127) / 128);
  uint64_t* mybar = bars + warp * kBulkDepth;
  uint8_t* mybuf = stage + (size_t)warp * kBulkDepth * slot_bytes;
  if (lane == 0) {
    for (int d = 0; d < kBulkDepth; ++d) mbar_init(&mybar[d], 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (lane != 0) return;
  const int64_t R = a.miss_off[a.n];
  const int64_t gw = (int64_t)blockIdx.x * kWarps + warp;
  const int64_t nw = (int64_t)gridDim.x * kWarps;
  // rows handled by this warp: r = gw + q * nw, q = 0, 1, ...
  const int64_t nq = R > gw ? (R - gw + nw - 1) / nw : 0;
  // a row of an unmapped block (paged pool) is copied onto itself from the hot
  // buffer, which leaves it as it was; *bad reports it
  auto addr = [&](int64_t q, const uint16_t** src, uint16_t** dst, bool* bad) {
    const int64_t r = gw + q * nw;
    const int i = find_segment(a.miss_off, a.n, r);
    const int64_t loc = r - a.miss_off[i];
    const int u = a.units[i];
    const int32_t t = a.miss_tok[(int64_t)i * a.pk + loc];
    const int32_t s = a.miss_slot[(int64_t)i * a.pk + loc];
    const int64_t hr = host_row(a.rows, u, t);
    *dst = a.hot + ((int64_t)u * a.C + s) * a.row_elems;
    *src = hr < 0 ? *dst : a.host_pool + hr * a.row_elems;
    *bad = hr < 0;
  };
  bool timed_out = false;
  unsigned long long n_bad = 0;
  const int64_t pro = nq < kBulkDepth ? nq : kBulkDepth;
  for (int64_t q = 0; q < pro; ++q) {
    const uint16_t* src;
    uint16_t* dst;
    bool bad;
    addr(q, &src, &dst, &bad);
    mbar_arrive_expect_tx(&mybar[q], row_bytes);
    bulk_g2s(mybuf + q * slot_bytes, src, row_bytes, &mybar[q]);
  }
  for (int64_t q = 0; q < nq; ++q) {
    const int d = (int)(q % kBulkDepth);
    const uint32_t parity = (uint32_t)((q / kBulkDepth) & 1);
    if (!mbar_wait(&mybar[d], parity, a.wait_ns)) timed_out = true;
    const uint16_t* src;
    uint16_t* dst;
    bool bad;
    addr(q, &src, &dst, &bad);
    n_bad += bad ? 1u : 0u;
    bulk_s2g(dst, mybuf + d * slot_bytes, row_bytes);
    bulk_commit();
    if (q + kBulkDepth < nq) {
      bulk_wait_read_all();  // staging slot d is free again
      addr(q + kBulkDepth, &src, &dst, &bad);
      mbar_arrive_expect_tx(&mybar[d], row_bytes);
      bulk_g2s(mybuf + d * slot_bytes, src, row_bytes, &mybar[d]);
    }
  }
  bulk_wait_all();
  if (timed_out) atomicOr(a.err, kErrTimeout);
  if (nq && a.stats) {
    if ((unsigned long long)nq > n_bad) {
      atomicAdd(&a.stats->rows_h2d, (unsigned long long)nq - n_bad);
      atomicAdd(&a.stats->bytes_h2d, ((unsigned long long)nq - n_bad) * row_bytes);
    }
    if (n_bad) atomicAdd(&a.stats->block_errors, n_bad);
  }
}

// ---------------------------------------------------------------------------
// append: one CTA per listed unit
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) append_kernel(AppendArgs a) {
  __shared__ int32_t base;
  __shared__ unsigned int bad;  // rows of unmapped blocks (paged pool), not written
  const int i = blockIdx.x, tid = threadIdx.x;
  const int u = a.units[i];
  if (tid == 0) {
    base = a.len[u];
    bad = 0;
  }
  __syncthreads();
  const int cpr = a.row_elems / 8;
  const int64_t nrow_chunks = (int64_t)a.n_tok * cpr;
  const uint4* src = reinterpret_cast<const uint4*>(a.rows + (int64_t)i * a.n_tok * a.row_elems);
  for (int64_t q = tid; q < nrow_chunks; q += blockDim.x) {
    const int64_t tj = q / cpr, c = q - tj * cpr;
    const int64_t hr = host_row(a.hrows, u, base + tj);
    if (hr >= 0)
      *reinterpret_cast<uint4*>(a.host_pool + hr * a.row_elems + c * 8) = src[q];
    else if (c == 0)
      atomicAdd(&bad, 1u);
  }
  if (a.idx8) {
    // int8 indexer: each new key rotated and quantized by one warp
    const int w = tid >> 5, nw = blockDim.x >> 5;
    for (int tj = w; tj < a.n_tok; tj += nw) {
      const int64_t dst = (int64_t)u * a.stride + base + tj;
      dev::warp_quant128(a.keys + ((int64_t)i * a.n_tok + tj) * kDim, a.idx8 + dst * kDim, a.idxs + dst, tid & 31);
    }
  } else {
    const int64_t nkey_chunks = (int64_t)a.n_tok * (kDim / 8);
    const uint4* ksrc = reinterpret_cast<const uint4*>(a.keys + (int64_t)i * a.n_tok * kDim);
    for (int64_t q = tid; q < nkey_chunks; q += blockDim.x) {
      const int64_t tj = q / (kDim / 8), c = q - tj * (kDim / 8);
      *reinterpret_cast<uint4*>(a.idx + ((int64_t)u * a.stride + base + tj) * kDim + c * 8) = ksrc[q];
    }
  }
  __syncthreads();
  if (tid == 0) {
    a.len[u] = base + a.n_tok;
    if (a.stats) {
      const unsigned long long ok = (unsigned long long)a.n_tok - bad;
      if (bad) atomicAdd(&a.stats->block_errors, (unsigned long long)bad);
      atomicAdd(&a.stats->rows_d2h, ok);
      atomicAdd(&a.stats->bytes_d2h, ok * a.row_elems * 2ull);
    }
  }
}

// reset: one CTA per listed unit; residency cleared, length cut back.
__global__ void __launch_bounds__(256) reset_kernel(ResetArgs a) {
  const int i = blockIdx.x, u = a.units[i];
  int32_t* cs = a.cache_slots + (int64_t)u * a.stride;
  const int32_t len = a.len[u];
  for (int32_t t = threadIdx.x; t < len; t += blockDim.x) cs[t] = -1;
  for (int s = threadIdx.x; s < a.C; s += blockDim.x) {
    a.slot_token[(int64_t)u * a.C + s] = -1;
    a.last_use[(int64_t)u * a.C + s] = 0;
    a.order[(int64_t)u * a.C + s] = s;
  }
  if (threadIdx.x == 0) a.order_par[u] = 0;
  for (int p = threadIdx.x; p < a.P; p += blockDim.x) {
    a.spec[(int64_t)u * a.P + p] = 0;
    a.qn_prev[(int64_t)u * a.P + p] = 0.f;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    a.stamp[u] = 0;
    a.len[u] = a.keep;
  }
}

__global__ void order_init_kernel(int32_t* order, int32_t* par, int U, int C) {
  const size_t n = (size_t)U * C;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n; e += (size_t)gridDim.x * blockDim.x)
    order[e] = (int32_t)(e % (size_t)C);
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < (size_t)U; e += (size_t)gridDim.x * blockDim.x)
    par[e] = 0;
}

__global__ void set_len_kernel(int32_t* len, int32_t unit, int32_t value) { len[unit] = value; }

__global__ void fill_i32_kernel(int32_t* p, int32_t v, size_t n) {
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n; e += (size_t)gridDim.x * blockDim.x)
    p[e] = v;
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
size_t residency_smem(int C, int P, int k) {
  const int nwords = (C + 31) / 32;
  const int nwords_pad = (nwords + 3) & ~3;
  return (size_t)nwords_pad * 4 + (size_t)P * k * 4 * 2;
}

cudaError_t launch_residency(const ResidencyArgs& a, cudaStream_t s) {
  const size_t smem = residency_smem(a.C, a.P, a.k);
  cudaError_t e = cudaFuncSetAttribute(residency_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  residency_kernel<<<a.n, kResThreads, smem, s>>>(a);
  return cudaGetLastError();
}

// A deferred fill completed without the attention call: CTA i copies the
// miss_cnt[i] rows of listed unit i, 16 bytes per thread and step.
__global__ void __launch_bounds__(256) flush_fill_kernel(GatherArgs a) {
  const int i = blockIdx.x;
  const int64_t u = a.units[i];
  const int64_t m = a.miss_cnt[i];
  const int chunks = a.row_elems / 8;
  unsigned long long rows = 0, bad = 0;
  for (int64_t e = threadIdx.x; e < m * chunks; e += blockDim.x) {
    const int64_t r = e / chunks;
    const int c = (int)(e % chunks);
    const int32_t t = a.miss_tok[(int64_t)i * a.pk + r];
    const int32_t s = a.miss_slot[(int64_t)i * a.pk + r];
    const int64_t hr = host_row(a.rows, u, t);
    if (hr < 0) {  // unmapped block: the hot row stays as it was
      bad += c == 0;
      continue;
    }
    const uint4 x = *reinterpret_cast<const uint4*>(a.host_pool + hr * a.row_elems + c * 8);
    *reinterpret_cast<uint4*>(a.hot + (u * a.C + s) * a.row_elems + c * 8) = x;
    rows += c == 0;
  }
  if (a.stats && rows) {
    atomicAdd(&a.stats->rows_h2d, rows);
    atomicAdd(&a.stats->bytes_h2d, rows * (unsigned long long)a.row_elems * 2u);
  }
  if (a.stats && bad) atomicAdd(&a.stats->block_errors, bad);
}

cudaError_t launch_flush_fill(const GatherArgs& a, cudaStream_t s) {
  if (a.n <= 0) return cudaSuccess;
  flush_fill_kernel<<<a.n, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gather(const GatherArgs& a, int n_sm, cudaStream_t s) {
  if (a.mode == KVO_GATHER_BULK) {
    const uint32_t slot_bytes = ((uint32_t)a.row_elems * 2u + 127u) & ~127u;
    const size_t smem = 128 * ((kGatherThreads / 32 * kBulkDepth * 8 + 127) / 128) +
                        (size_t)(kGatherThreads / 32) * kBulkDepth * slot_bytes;
    cudaError_t e = cudaFuncSetAttribute(gather_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    gather_bulk_kernel<<<n_sm, kGatherThreads, smem, s>>>(a);
  } else {
    gather_ldg_kernel<<<n_sm, kGatherThreads, 0, s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
  append_kernel<<<a.n, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_reset(const ResetArgs& a, cudaStream_t s) {
  reset_kernel<<<a.n, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_order_init(int32_t* order, int32_t* par, int U, int C, cudaStream_t s) {
  order_init_kernel<<<1024, 256, 0, s>>>(order, par, U, C);
  return cudaGetLastError();
}

cudaError_t launch_set_len(int32_t* len, int32_t unit, int32_t value, cudaStream_t s) {
  set_len_kernel<<<1, 1, 0, s>>>(len, unit, value);
  return cudaGetLastError();
}

cudaError_t launch_fill_i32(int32_t* p, int32_t v, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  size_t blocks = (n + 255) / 256;
  if (blocks > 65535) blocks = 65535;
  fill_i32_kernel<<<(unsigned)blocks, 256, 0, s>>>(p, v, n);
  return cudaGetLastError();
}

}  // namespace kvo
