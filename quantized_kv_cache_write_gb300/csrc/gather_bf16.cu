// Gather-attention instantiation for the QKV_BF16 slot-pool layout (one translation unit per
// layout so the four kernels compile in parallel).
#include "gather_attn.cuh"

namespace qkv {
cudaError_t launch_gather_bf16(const GatherArgs& a, cudaStream_t stream) {
  return gather::launch<QKV_BF16>(a, stream);
}
cudaError_t gather_ctas_per_sm_bf16(int* n) { return gather::resident_ctas_per_sm<QKV_BF16>(n); }
}  // namespace qkv
