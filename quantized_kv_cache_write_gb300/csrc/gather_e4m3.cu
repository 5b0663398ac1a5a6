// Gather-attention instantiation for the QKV_E4M3 slot-pool layout (one translation unit per
// layout so the four kernels compile in parallel).
#include "gather_attn.cuh"

namespace qkv {
cudaError_t launch_gather_e4m3(const GatherArgs& a, cudaStream_t stream) {
  return gather::launch<QKV_E4M3>(a, stream);
}
cudaError_t gather_ctas_per_sm_e4m3(int* n) { return gather::resident_ctas_per_sm<QKV_E4M3>(n); }
}  // namespace qkv
