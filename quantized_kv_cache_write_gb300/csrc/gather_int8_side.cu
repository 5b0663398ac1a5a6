// Gather-attention instantiation for the QKV_INT8_SIDE slot-pool layout (one translation unit per
// layout so the four kernels compile in parallel).
#include "gather_attn.cuh"

namespace qkv {
cudaError_t launch_gather_int8_side(const GatherArgs& a, cudaStream_t stream) {
  return gather::launch<QKV_INT8_SIDE>(a, stream);
}
cudaError_t gather_ctas_per_sm_int8_side(int* n) { return gather::resident_ctas_per_sm<QKV_INT8_SIDE>(n); }
}  // namespace qkv
