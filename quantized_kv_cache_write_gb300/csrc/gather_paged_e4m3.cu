// Gather-attention instantiation for the QKV_E4M3 layout over a paged pool (block table +
// logical positions); one translation unit per layout so the kernels compile in parallel.
#include "gather_attn.cuh"

namespace qkv {
cudaError_t launch_gather_paged_e4m3(const GatherArgs& a, cudaStream_t stream) {
  return gather::launch<QKV_E4M3, true>(a, stream);
}
}  // namespace qkv
