// Gather-attention instantiation for the QKV_INT8_INLINE layout over a paged pool (block table +
// logical positions); one translation unit per layout so the kernels compile in parallel.
#include "gather_attn.cuh"

namespace qkv {
cudaError_t launch_gather_paged_int8_inline(const GatherArgs& a, cudaStream_t stream) {
  return gather::launch<QKV_INT8_INLINE, true>(a, stream);
}
}  // namespace qkv
