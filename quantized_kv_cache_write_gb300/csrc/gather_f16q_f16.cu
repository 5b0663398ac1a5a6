// Gather-attention instantiation for the QKV_F16 layout with an IEEE-half query (the
// FP16-activation contract); one translation unit per layout so the kernels compile in parallel.
#include "gather_attn.cuh"

namespace qkv {
cudaError_t launch_gather_f16q_f16(const GatherArgs& a, cudaStream_t stream) {
  return gather::launch_f16q<QKV_F16>(a, stream);
}
}  // namespace qkv
