// Split-K merge: lse = log sum_s exp(lse_s), o = v_scale_post * sum_s exp(lse_s - lse) * o_s.
//
// Pages: "[Perf][SM70][FP8] Hoist QSA E4M3 KV scales" §Changes (split-K applies the V scale
// once after the merge); "[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache"
// §Implementation scope (the split-K workspace).
//
// One warp per (row, query head); each lane owns 8 of the 256 output columns, so every
// partial row is read as one coalesced 1 KB line. Bandwidth-trivial next to the gather.
#include "qkv_internal.cuh"

namespace qkv {
namespace {

constexpr int kMergeThreads = 256;

__global__ void __launch_bounds__(kMergeThreads)
    splitk_merge_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part, int64_t rows,
                        int num_q_heads, int num_splits, float v_scale_post, float* __restrict__ out,
                        float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int64_t item = (static_cast<int64_t>(blockIdx.x) * kMergeThreads + threadIdx.x) >> 5;
  if (item >= rows * num_q_heads) return;
  const int64_t r = item / num_q_heads;
  const int g = static_cast<int>(item - r * num_q_heads);

  const float* lp = lse_part + r * num_splits * num_q_heads + g;
  float m = -INFINITY;
  for (int s = 0; s < num_splits; ++s) m = fmaxf(m, lp[static_cast<int64_t>(s) * num_q_heads]);

  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  float* dst = out + item * kHeadDim + lane * 8;
  if (m == -INFINITY) {
    reinterpret_cast<float4*>(dst)[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    reinterpret_cast<float4*>(dst)[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lse != nullptr && lane == 0) lse[item] = -INFINITY;
    return;
  }
  float wsum = 0.f;
  for (int s = 0; s < num_splits; ++s) {
    const float ls = lp[static_cast<int64_t>(s) * num_q_heads];
    if (ls == -INFINITY) continue;
    const float w = expf(ls - m);
    wsum += w;
    const float4* src =
        reinterpret_cast<const float4*>(o_part + ((r * num_splits + s) * num_q_heads + g) * kHeadDim + lane * 8);
    const float4 a = src[0], b = src[1];
    acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
    acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
  }
  const float f = v_scale_post / wsum;
  reinterpret_cast<float4*>(dst)[0] = make_float4(acc[0] * f, acc[1] * f, acc[2] * f, acc[3] * f);
  reinterpret_cast<float4*>(dst)[1] = make_float4(acc[4] * f, acc[5] * f, acc[6] * f, acc[7] * f);
  if (lse != nullptr && lane == 0) lse[item] = m + logf(wsum);
}

}  // namespace

cudaError_t launch_splitk_merge(const float* o_part, const float* lse_part, int64_t rows, int num_q_heads,
                                int num_splits, float v_scale_post, float* out, float* lse,
                                cudaStream_t stream) {
  const int64_t warps = rows * num_q_heads;
  const unsigned blocks = static_cast<unsigned>((warps * 32 + kMergeThreads - 1) / kMergeThreads);
  splitk_merge_kernel<<<blocks, kMergeThreads, 0, stream>>>(o_part, lse_part, rows, num_q_heads, num_splits,
                                                             v_scale_post, out, lse);
  return cudaGetLastError();
}

}  // namespace qkv
