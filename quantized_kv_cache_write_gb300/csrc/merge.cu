// Split-K merge: lse = log sum_s exp(lse_s), o = v_scale_post * sum_s exp(lse_s - lse) * o_s.
//
// Pages: "[Perf][SM70][FP8] Hoist QSA E4M3 KV scales" §Changes (split-K applies the V scale
// once after the merge); "[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache"
// §Implementation scope (the split-K workspace).
//
// One warp per (row, query head); each lane owns 8 of the output columns (head_dim 256: all
// 32 lanes, 128: 16), so every partial row is read as one coalesced line. Bandwidth-trivial
// next to the gather.
#include "qkv_internal.cuh"

namespace qkv {
namespace {

constexpr int kMergeThreads = 256;

__global__ void __launch_bounds__(kMergeThreads)
    splitk_merge_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part, int64_t rows,
                        int num_q_heads, int head_dim, int num_splits, float v_scale_post,
                        float* __restrict__ out, float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int64_t item = (static_cast<int64_t>(blockIdx.x) * kMergeThreads + threadIdx.x) >> 5;
  if (item >= rows * num_q_heads) return;
  const int64_t r = item / num_q_heads;
  const int g = static_cast<int>(item - r * num_q_heads);

  if (8 * lane >= head_dim) return;  // head_dim 128: lanes 16..31 have no columns
  const int col4[2] = {2 * lane, 2 * lane + 1};  // lane owns columns 8 lane .. 8 lane + 7
  merge_head<2, 4>(o_part + (r * num_splits * num_q_heads + g) * head_dim, lse_part + r * num_splits * num_q_heads + g,
                   num_q_heads, num_splits, head_dim, v_scale_post, col4, out + item * head_dim,
                   (lse != nullptr && lane == 0) ? lse + item : nullptr);
}

}  // namespace

cudaError_t launch_splitk_merge(const float* o_part, const float* lse_part, int64_t rows, int num_q_heads,
                                int head_dim, int num_splits, float v_scale_post, float* out, float* lse,
                                cudaStream_t stream) {
  const int64_t warps = rows * num_q_heads;
  const unsigned blocks = static_cast<unsigned>((warps * 32 + kMergeThreads - 1) / kMergeThreads);
  splitk_merge_kernel<<<blocks, kMergeThreads, 0, stream>>>(o_part, lse_part, rows, num_q_heads, head_dim,
                                                             num_splits, v_scale_post, out, lse);
  return cudaGetLastError();
}

}  // namespace qkv
