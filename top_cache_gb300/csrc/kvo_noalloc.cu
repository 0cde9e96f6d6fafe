// kvo_select_noalloc: the scoring and fused top-k of kvo_select for callers
// that must not allocate memory.
//
// Some callers cannot call cudaMalloc or any allocating routine at the point
// where they select: an operator or plugin hosted by a framework that owns all
// device memory and forbids its extensions to allocate, or a latency-critical
// decode loop that cannot afford an allocation, the fragmentation it causes, or
// the device synchronisation that freeing memory can bring.  This entry point
// takes the same inputs and outputs as kvo_select but no workspace: its scratch
// is a file-scope device array of fixed size (kNoallocScratchBytes), part of
// the library image, so every GPU that loads the library holds it until the
// process exits (under lazy module loading, from the first call on that
// device).  An accepted call allocates nothing on the host or the device: the
// per-unit lengths travel to the GPU inside a kernel parameter.
//
// Sharing rules: every call uses the same array, and the array keeps the last
// call's contents.  Whatever must start at zero is cleared by the call itself
// on its stream.  Two calls whose work overlaps on the GPU (different streams
// without ordering, or different host threads) race on the array and give
// undefined results; order them on one stream or synchronise between them.
//
// The first call on a device resolves the array's device address for that
// device (cudaGetSymbolAddress, with that device current), once per device;
// make that first call before any stream capture.  The address is kept for
// the life of the process: a cudaDeviceReset on that device ends the module
// instance it points into, so calls after a reset are not supported (as for
// every other resource of this library on that device).
//
// Completion status: the kernels record an expired bounded wait (bit 1) or a
// failed internal consistency check (bit 2) in an error word.  A caller that
// passes `status` (a device word of its own) gets that word there, cleared at
// the start of the call; nonzero means the outputs are not valid.  Without
// `status` the word lives in the fixed array and cannot be observed.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kvo_internal.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = (size_t)16 << 20;  // 16 MiB
constexpr int kNoallocMaxUnits = 64;
constexpr int kNoallocMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

struct NoallocLengths {
  int32_t n;
  int32_t len[kNoallocMaxUnits];
};

// Writes the identity unit list and the lengths, and clears the error word.
__global__ void noalloc_setup_kernel(NoallocLengths p, int32_t* units, int32_t* len, uint32_t* err) {
  for (int i = threadIdx.x; i < p.n; i += blockDim.x) {
    units[i] = i;
    len[i] = p.len[i];
  }
  if (threadIdx.x == 0) *err = 0;
}

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoallocMaxDevices] = {};

int noalloc_fail(int code, const char* msg) {
  kvo::set_last_error(msg);
  return code;
}

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

extern "C" {

int kvo_select_noalloc(const void* keys, int64_t unit_stride, const int32_t* cache_slots,
                       const int64_t* lengths, int32_t n_units, int32_t n_pos, int32_t k,
                       const void* queries, int32_t* tokens, float* scores, int32_t* payload,
                       uint32_t* status, void* stream) {
  if (!keys || !lengths || !queries || !tokens) return noalloc_fail(KVO_EINVAL, "NULL argument");
  if (n_units < 1 || n_pos < 1 || n_pos > 8 || k < 1 || k > 4096)
    return noalloc_fail(KVO_EINVAL, "size out of range");
  if (n_units > kNoallocMaxUnits)
    return noalloc_fail(KVO_ERANGE, "n_units above the fixed scratch limit of 64 units");
  if (unit_stride < 1 || unit_stride >= (int64_t)1 << 31)
    return noalloc_fail(KVO_EINVAL, "unit_stride out of range");
  if ((reinterpret_cast<uintptr_t>(keys) & 15u) || (reinterpret_cast<uintptr_t>(queries) & 15u))
    return noalloc_fail(KVO_EINVAL, "keys/queries not 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(status) & 3u) return noalloc_fail(KVO_EINVAL, "status not 4-byte aligned");
  const int cap = kvo::score_cap_for(n_pos, k, false);
  if (cap == 0) return noalloc_fail(KVO_EINVAL, "k too large for n_pos");
  int dev = 0, n_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoallocMaxDevices)
    return noalloc_fail(KVO_ECUDA, "no usable current device");
  if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return noalloc_fail(KVO_ECUDA, "device query failed");

  // scratch layout (same parts as kvo_select's workspace)
  const size_t n = (size_t)n_units, PK = (size_t)n_pos * k, segs = (size_t)n_sm + n;
  const size_t need = up256(n * 4) * 2 + up256((n + 1) * 8) + up256(n * n_pos * 8) +
                      up256(segs * PK * 8) + up256(segs * n_pos * 4) + up256(n * PK * 4) + up256(4);
  if (need > kNoallocScratchBytes)
    return noalloc_fail(KVO_ERANGE, "n_units * n_pos * k needs more than the 16 MiB fixed scratch");

  NoallocLengths lens{};
  lens.n = n_units;
  int64_t T = 0;
  for (int32_t i = 0; i < n_units; ++i) {
    if (lengths[i] < 0 || lengths[i] > unit_stride) return noalloc_fail(KVO_EINVAL, "length out of range");
    lens.len[i] = (int32_t)lengths[i];
    T += lengths[i];
  }

  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) return kvo::set_cuda_error(e, "cudaGetSymbolAddress of the fixed scratch");
      if (!p) return noalloc_fail(KVO_ECUDA, "cudaGetSymbolAddress of the fixed scratch returned NULL");
      g_noalloc_ptr[dev] = p;
    }
    base = g_noalloc_ptr[dev];
  }

  uint8_t* w = static_cast<uint8_t*>(base);
  int32_t* d_units = reinterpret_cast<int32_t*>(w); w += up256(n * 4);
  int32_t* d_len = reinterpret_cast<int32_t*>(w); w += up256(n * 4);
  int64_t* d_off = reinterpret_cast<int64_t*>(w); w += up256((n + 1) * 8);
  uint64_t* d_gthr = reinterpret_cast<uint64_t*>(w); w += up256(n * n_pos * 8);
  uint64_t* d_seg_keys = reinterpret_cast<uint64_t*>(w); w += up256(segs * PK * 8);
  int32_t* d_seg_cnt = reinterpret_cast<int32_t*>(w); w += up256(segs * n_pos * 4);
  int32_t* d_pay = reinterpret_cast<int32_t*>(w); w += up256(n * PK * 4);
  uint32_t* d_err = status ? status : reinterpret_cast<uint32_t*>(w);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  noalloc_setup_kernel<<<1, 64, 0, s>>>(lens, d_units, d_len, d_err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return kvo::set_cuda_error(e, "no-allocation select set-up launch");

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
  int64_t g = (T + 4095) / 4096;
  sa.G = (int)(g < 1 ? 1 : (g > n_sm ? n_sm : g));
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
  if (e != cudaSuccess) return kvo::set_cuda_error(e, "no-allocation select launch");
  return KVO_OK;
}

}  // extern "C"
