// tcgen05 gather attention over an int8 pool with side-tensor scales (head dim 256, GQA <= 16).
#include "gather_umma.cuh"

namespace qkv {
cudaError_t launch_umma_int8_side(const GatherArgs& a, cudaStream_t stream) {
  return umma::launch<QKV_INT8_SIDE>(a, stream);
}
}  // namespace qkv
