// The fused decode step for bf16 indexer keys, and the host entry points of
// the fused launch (the int8 instantiation is compiled in kvo_fused_i8.cu).
#include "kvo_fused.cuh"

namespace kvo {

cudaError_t launch_fused_i8(const FusedArgs& a, int grid, cudaStream_t s);

namespace {
// Self-test of the bounded waits every kernel relies on: one thread waits on a
// global flag that nothing sets (spin_until, as the fused step's cross-CTA
// waits) and then on an mbarrier phase that cannot complete (mbar_wait, as the
// copy and MMA pipelines), each limited to limit_ns.  Both must give up.
// out[0] / out[1]: 1 when the flag / mbarrier wait expired; out[2]: ns waited.
__global__ void wait_selftest_kernel(const uint32_t* flag, uint64_t limit_ns, unsigned long long* out) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 2);  // two arrivals complete the phase; only one ever comes
  fence_mbar_init();
  const uint64_t t0 = global_ns();
  const bool a = spin_until([&] { return ld_volatile_u32(flag) != 0u; }, limit_ns);
  mbar_arrive(&bar);
  const bool b = mbar_wait(&bar, 0, limit_ns);
  out[0] = a ? 0ull : 1ull;
  out[1] = b ? 0ull : 1ull;
  out[2] = global_ns() - t0;
  mbar_inval(&bar);
}
}  // namespace

cudaError_t run_wait_selftest(uint64_t limit_ns, unsigned long long* host_out) {
  uint32_t* flag = nullptr;
  unsigned long long* out = nullptr;
  cudaError_t e = cudaMalloc(&flag, 4);
  if (e == cudaSuccess) e = cudaMalloc(&out, 3 * sizeof(unsigned long long));
  if (e == cudaSuccess) e = cudaMemset(flag, 0, 4);
  if (e == cudaSuccess) {
    wait_selftest_kernel<<<1, 32>>>(flag, limit_ns, out);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(host_out, out, 3 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
  if (flag) cudaFree(flag);
  if (out) cudaFree(out);
  return e;
}

size_t fused_smem_bytes(int P, int k, int cap, bool int8) {
  const size_t fixed = int8 ? dev::smem_fixed<dev::KeysInt8>() : dev::smem_fixed<dev::KeysBf16>();
  return fixed + (size_t)P * cap * 8 + (size_t)k * 8 + kFusedExtra;
}

int fused_chunk_rows() { return kChunkRows; }

cudaError_t launch_fused(const FusedArgs& a, int grid, cudaStream_t s) {
  if (a.s.keys8) return launch_fused_i8(a, grid, s);
  return launch_fused_kf<dev::KeysBf16>(a, grid, s);
}

}  // namespace kvo
