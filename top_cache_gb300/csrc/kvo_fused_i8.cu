// The fused decode step for int8 indexer keys (reading R12 of the oracle;
// "FlashOffloading ... What does it mean?", the LIM C8 paragraph): the same
// kernel as kvo_fused.cu, scoring int8 code rows with their fp16 scales.
#include "kvo_fused.cuh"

namespace kvo {

cudaError_t launch_fused_i8(const FusedArgs& a, int grid, cudaStream_t s) {
  return launch_fused_kf<dev::KeysInt8>(a, grid, s);
}

}  // namespace kvo
