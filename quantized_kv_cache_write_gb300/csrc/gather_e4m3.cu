// Gather-attention instantiation for the QKV_E4M3 slot-pool layout (one translation unit per
// layout so the four kernels compile in parallel).
#include "gather_attn.cuh"

namespace qkv {
cudaError_t launch_gather_e4m3(const GatherArgs& a, cudaStream_t stream) {
  return gather::launch<QKV_E4M3>(a, stream);
}
}  // namespace qkv
