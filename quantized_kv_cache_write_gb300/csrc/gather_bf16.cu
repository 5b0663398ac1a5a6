// Gather-attention instantiation for the QKV_BF16 slot-pool layout (one translation unit per
// layout so the four kernels compile in parallel).
#include "gather_attn.cuh"

namespace qkv {
cudaError_t launch_gather_bf16(const GatherArgs& a, cudaStream_t stream) {
  return gather::launch<QKV_BF16>(a, stream);
}
}  // namespace qkv
