// The fused decode step for bf16 indexer keys, and the host entry points of
// the fused launch (the int8 instantiation is compiled in kvo_fused_i8.cu).
#include "kvo_fused.cuh"

namespace kvo {

cudaError_t launch_fused_i8(const FusedArgs& a, int grid, cudaStream_t s);

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
