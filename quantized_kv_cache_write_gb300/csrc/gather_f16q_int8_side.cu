// Gather-attention instantiation for the QKV_INT8_SIDE layout with an IEEE-half query (the
// FP16-activation contract); one translation unit per layout so the kernels compile in parallel.
#include "gather_attn.cuh"

namespace qkv {
cudaError_t launch_gather_f16q_int8_side(const GatherArgs& a, cudaStream_t stream) {
  return gather::launch_f16q<QKV_INT8_SIDE>(a, stream);
}
}  // namespace qkv
