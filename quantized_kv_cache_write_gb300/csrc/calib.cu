// Calibration statistics of one K or V tensor: an exact magnitude histogram of its 16-bit
// values (bf16, or IEEE half for the FP16-activation contract), accumulated over any number of
// calls, then the statistics read from it.
//
// Pages: "Qwen3.8 Flash Next NVFP4 QSA FP8 E4M3 KV Scales" §Calibration (scale = max
// envelope / 448; max-abs, p99.9, p99.99 and saturation per tensor); "[Model][SM70][FP8] Add
// calibrated E4M3 QSA KV cache" §Why calibrated scale is part of this contract (at a given
// scale, nonzero elements below E4M3's smallest subnormal 2^-9 and in the subnormal band
// below 2^-6) and §Implementation scope (per-layer, per-tensor statistics).
//
// A bf16 or half magnitude is 15 bits, so 32768 bins of (bits & 0x7FFF) hold the tensor's
// magnitudes exactly, and every statistic is an exact function of the histogram: order
// statistics by prefix sums, and the scaled-magnitude counts by classifying each bin's value
// (the fp32 IEEE division each of its elements would get; the classes are runs of bins).
//
// histogram: a persistent grid (one 1024-thread CTA per SM, or more for huge inputs), each
// CTA with a private 128 KB shared-memory histogram fed by 16 B streaming loads and shared
// atomics; at the end each CTA adds its non-zero bins into the caller's uint64 histogram.
// HBM-bound: 2 bytes read per element.
// stats: one CTA of 32 warps, each reading a 1024-bin range in coalesced rows; the class
// edges and the rank bins are then located by a few warps at once.
#include <atomic>

#include "qkv_internal.cuh"

namespace qkv {
namespace {

constexpr int kBins = QKV_CALIB_BINS;
constexpr int kHistThreads = 1024;
// magnitude bits of +inf (above: NaN): bf16 0x7F80, IEEE half 0x7C00
template <bool F16>
__device__ __forceinline__ uint32_t first_nonfinite() { return F16 ? 0x7C00u : 0x7F80u; }
constexpr int64_t kMaxPerCta = int64_t(1) << 31;  // keeps every shared count below 2^32

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void count8(uint32_t* sh, const uint4& r) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    atomicAdd(sh + (w[j] & 0x7FFFu), 1u);
    atomicAdd(sh + ((w[j] >> 16) & 0x7FFFu), 1u);
  }
}

__global__ void __launch_bounds__(kHistThreads, 1)
    calib_hist_kernel(const uint16_t* __restrict__ x, int64_t n, unsigned long long* __restrict__ hist) {
  extern __shared__ uint32_t sh[];  // [kBins]
  for (int b = threadIdx.x; b < kBins; b += kHistThreads) sh[b] = 0u;
  __syncthreads();
  const int64_t nvec = n / 8;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kHistThreads;
  int64_t i = static_cast<int64_t>(blockIdx.x) * kHistThreads + threadIdx.x;
  for (; i + 3 * stride < nvec; i += 4 * stride) {  // four 16 B loads in flight per thread
    uint4 r[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) r[u] = ld_stream16(xv + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) count8(sh, r[u]);
  }
  for (; i < nvec; i += stride) count8(sh, ld_stream16(xv + i));
  for (int64_t j = nvec * 8 + static_cast<int64_t>(blockIdx.x) * kHistThreads + threadIdx.x; j < n; j += stride)
    atomicAdd(sh + (x[j] & 0x7FFFu), 1u);
  __syncthreads();
  for (int b = threadIdx.x; b < kBins; b += kHistThreads) {
    const uint32_t c = sh[b];
    if (c != 0u) atomicAdd(hist + b, static_cast<unsigned long long>(c));
  }
}

// the value of a magnitude bin (bf16, or IEEE half when F16), exactly
template <bool F16>
__device__ __forceinline__ float bin_value(uint32_t b) {
  return F16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(b))) : __uint_as_float(b << 16);
}

__device__ __forceinline__ unsigned long long warp_sum(unsigned long long v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Inclusive scan over the 32 lanes of a warp.
__device__ __forceinline__ unsigned long long warp_scan(unsigned long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long u = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += u;
  }
  return v;
}

constexpr int kStatsWarps = 32;                    // one CTA of 32 warps
constexpr int kWarpBins = kBins / kStatsWarps;     // warp w owns bins [1024 w, 1024 w + 1024)
static_assert(kWarpBins == 32 * 32, "a warp's range is 32 rows of 32 bins");

// sum of hist[b] over b in [from, to), both inside one warp range (a whole warp calls it)
__device__ __forceinline__ unsigned long long range_sum(const unsigned long long* __restrict__ hist, uint32_t from,
                                                        uint32_t to) {
  const uint32_t lane = threadIdx.x & 31;
  unsigned long long s = 0;
#pragma unroll
  for (uint32_t j = 0; j < 32; ++j) {  // at most 1024 bins: every load in flight at once
    const uint32_t b = from + 32 * j + lane;
    if (b < to) s += hist[b];
  }
  return warp_sum(s);
}

// The first bin b in [0, limit) for which the monotone predicate holds (false ... false
// true ... true over b), or `limit` if none: three radix-32 rounds over the 15 bin bits, one
// candidate per lane. The whole warp calls it and every lane gets the answer.
template <class Pred>
__device__ __forceinline__ uint32_t first_true(uint32_t limit, Pred pred) {
  const uint32_t lane = threadIdx.x & 31;
  uint32_t ans = 0;
#pragma unroll
  for (int level = 10; level >= 0; level -= 5) {
    const uint32_t b = ans + ((lane + 1) << level) - 1;
    const bool before = b < limit && !pred(b);  // the answer lies past b
    ans += static_cast<uint32_t>(__popc(__ballot_sync(0xffffffffu, before))) << level;
  }
  return ans;
}

// Nearest-rank bin: the smallest b with PS(b + 1) >= r (PS(x) = sum of hist[0, x)), for
// 1 <= r <= N, given the exclusive prefix `excl` of the warp range w that holds it. Rows of 32
// bins are summed first, then the row that holds the rank is scanned. The whole warp calls it.
__device__ __forceinline__ uint32_t rank_bin(const unsigned long long* __restrict__ hist, uint32_t w,
                                             unsigned long long excl, unsigned long long r) {
  const uint32_t lane = threadIdx.x & 31, base = w * kWarpBins;
  unsigned long long mine = 0;  // lane j: the sum of row j (its 32 loads in flight at once)
#pragma unroll
  for (int k = 0; k < 32; ++k) mine += hist[base + 32 * lane + k];
  const unsigned long long rows_incl = excl + warp_scan(mine);
  const uint32_t row = __popc(__ballot_sync(0xffffffffu, rows_incl < r));  // rows wholly below the rank
  const unsigned long long row_excl = __shfl_sync(0xffffffffu, rows_incl - mine, row & 31);
  const unsigned long long in_row = row_excl + warp_scan(hist[base + 32 * (row & 31) + lane]);
  const uint32_t k = __popc(__ballot_sync(0xffffffffu, in_row < r));
  return base + 32 * row + k;
}

// One CTA of 32 warps; warp w owns the 1024 bins [1024 w, 1024 w + 1024) and reads them row
// by row (lane l: bins 1024 w + 32 j + l), so every load is one coalesced 256 B row.
//   1. per-warp sums of the finite and non-finite bins and the highest finite bin with a count;
//   2. warp 0: prefix over the warps, N, amax, the scale, the nearest ranks, and three bin
//      thresholds. A bin's scaled magnitude fl(value / scale) does not decrease with the bin
//      (values rise with the bits, and a correctly rounded division is monotone), so each
//      class is a contiguous run of bins and its count is a difference of prefix sums;
//   3. five warps at once: the prefix sums at the three thresholds and the two rank bins.
template <bool F16>
__global__ void __launch_bounds__(kStatsWarps * 32) calib_stats_kernel(const unsigned long long* __restrict__ hist,
                                                                       float scale_in,
                                                                       qkv_calib_summary* __restrict__ out) {
  const uint32_t kFirstNonfinite = first_nonfinite<F16>();
  __shared__ unsigned long long s_fin[kStatsWarps], s_nonfin[kStatsWarps], s_excl[kStatsWarps];
  __shared__ uint32_t s_top[kStatsWarps];
  __shared__ unsigned long long s_N, s_nonfinite, s_rank[2], s_ps[3];
  __shared__ uint32_t s_thr[3], s_rank_w[2];
  __shared__ float s_amax, s_scale, s_p[2];
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  {  // 1. (16 loads in flight per thread)
    unsigned long long fin = 0, nonfin = 0;
    uint32_t top = 0;  // 1 + the highest finite bin with a count
#pragma unroll 16
    for (int j = 0; j < 32; ++j) {
      const uint32_t b = warp * kWarpBins + 32 * j + lane;
      const unsigned long long c = hist[b];
      if (b < kFirstNonfinite) {
        fin += c;
        if (c != 0ull) top = b + 1;
      } else {
        nonfin += c;
      }
    }
    fin = warp_sum(fin);
    nonfin = warp_sum(nonfin);
    top = __reduce_max_sync(0xffffffffu, top);
    if (lane == 0) {
      s_fin[warp] = fin;
      s_nonfin[warp] = nonfin;
      s_top[warp] = top;
    }
  }
  __syncthreads();

  if (warp == 0) {  // 2.
    const unsigned long long fin = s_fin[lane], incl = warp_scan(fin);
    s_excl[lane] = incl - fin;
    const unsigned long long N = __shfl_sync(0xffffffffu, incl, 31);
    const unsigned long long nonfinite = warp_sum(s_nonfin[lane]);
    const uint32_t top = __reduce_max_sync(0xffffffffu, s_top[lane]);
    const float amax = top ? bin_value<F16>(top - 1u) : 0.f;
    const float scale = scale_in > 0.f ? scale_in : __fdiv_rn(amax, 448.0f);
    // nearest ranks ceil(q N), q = 999/1000 and 9999/10000, in exact integer arithmetic
    const unsigned long long r[2] = {(999ull * N + 999ull) / 1000ull, (9999ull * N + 9999ull) / 10000ull};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t w = __popc(__ballot_sync(0xffffffffu, incl < r[i]));  // warp ranges wholly below the rank
      if (lane == 0) {
        s_rank[i] = r[i];
        s_rank_w[i] = w;
      }
    }
    uint32_t thr[3] = {0u, 0u, 0u};
    if (scale > 0.f) {  // a zero scale (an all-zero tensor) leaves the classes at 0
      const float kSub = 0.001953125f, kNorm = 0.015625f, kSat = 464.0f;  // 2^-9, 2^-6, (448 + 480) / 2
      auto y = [&](uint32_t b) { return __fdiv_rn(bin_value<F16>(b), scale); };
      thr[0] = first_true(kFirstNonfinite, [&](uint32_t b) { return y(b) >= kSub; });
      thr[1] = first_true(kFirstNonfinite, [&](uint32_t b) { return y(b) >= kNorm; });
      thr[2] = first_true(kFirstNonfinite, [&](uint32_t b) { return y(b) > kSat; });
    }
    if (lane == 0) {
      s_N = N;
      s_nonfinite = nonfinite;
      s_amax = amax;
      s_scale = scale;
      s_thr[0] = thr[0];
      s_thr[1] = thr[1];
      s_thr[2] = thr[2];
      s_p[0] = s_p[1] = 0.f;
    }
  }
  __syncthreads();

  // 3. (warps 1-3: PS(threshold); warps 4-5: the rank bins; N = 0 leaves both percentiles 0)
  if (warp >= 1 && warp <= 3) {
    const uint32_t B = s_thr[warp - 1];  // <= kFirstNonfinite < kBins
    const uint32_t w = B / kWarpBins;
    const unsigned long long ps = s_excl[w] + range_sum(hist, w * kWarpBins, B);
    if (lane == 0) s_ps[warp - 1] = ps;
  } else if ((warp == 4 || warp == 5) && s_N > 0ull) {
    const int i = warp - 4;
    const uint32_t b = rank_bin(hist, s_rank_w[i], s_excl[s_rank_w[i]], s_rank[i]);
    if (lane == 0) s_p[i] = bin_value<F16>(b);
  }
  __syncthreads();

  if (threadIdx.x == 0) {
    const unsigned long long N = s_N, zeros = hist[0];
    const bool classes = s_scale > 0.f;
    out->count = N;
    out->zeros = zeros;
    out->nonfinite = s_nonfinite;
    // below 2^-9: bins [1, thr0) (bin 0 holds the zeros, which count in no class)
    out->below_subnormal = classes ? s_ps[0] - zeros : 0ull;
    out->subnormal = classes ? s_ps[1] - s_ps[0] : 0ull;
    out->saturated = classes ? N - s_ps[2] : 0ull;
    out->amax = s_amax;
    out->p99_9 = s_p[0];
    out->p99_99 = s_p[1];
    out->scale = s_scale;
  }
}

// Per-device caches below are atomic: host threads may race on a device's first call, and
// both then store the same value.
int sm_count_cached() {
  static std::atomic<int> count[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int c = count[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    count[dev].store(c, std::memory_order_relaxed);
  }
  return c;
}

}  // namespace

cudaError_t launch_calib_histogram(const void* x, int64_t n, uint64_t* hist, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  static std::atomic<bool> attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  constexpr int smem = kBins * sizeof(uint32_t);
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(calib_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(true, std::memory_order_release);
  }
  const int sms = sm_count_cached();
  if (sms <= 0) return cudaErrorInvalidDevice;
  // a CTA never counts more than kMaxPerCta elements, so its shared uint32 bins cannot wrap
  const int64_t need = (n + kMaxPerCta - 1) / kMaxPerCta;
  const int64_t grid = need > sms ? need : sms;
  calib_hist_kernel<<<static_cast<unsigned>(grid), kHistThreads, smem, stream>>>(
      static_cast<const uint16_t*>(x), n, reinterpret_cast<unsigned long long*>(hist));
  return cudaGetLastError();
}

cudaError_t launch_calib_stats(const uint64_t* hist, bool f16, float scale, qkv_calib_summary* stats,
                               cudaStream_t stream) {
  auto kern = f16 ? calib_stats_kernel<true> : calib_stats_kernel<false>;
  kern<<<1, 1024, 0, stream>>>(reinterpret_cast<const unsigned long long*>(hist), scale, stats);
  return cudaGetLastError();
}

}  // namespace qkv
