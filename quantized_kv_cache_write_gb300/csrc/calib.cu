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
// (one fp32 IEEE division per bin, the same division an element would get).
//
// histogram: a persistent grid (one 1024-thread CTA per SM, or more for huge inputs), each
// CTA with a private 128 KB shared-memory histogram fed by 16 B streaming loads and shared
// atomics; at the end each CTA adds its non-zero bins into the caller's uint64 histogram.
// HBM-bound: 2 bytes read per element.
// stats: one CTA of 1024 threads, 32 consecutive bins per thread.
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

// Inclusive block-wide sum scan of one uint64 per thread (1024 threads); `total` gets the sum.
__device__ __forceinline__ unsigned long long block_scan(unsigned long long v, unsigned long long* sw,
                                                         unsigned long long& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long u = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += u;
  }
  if (lane == 31) sw[warp] = v;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = sw[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned long long u = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += u;
    }
    sw[lane] = w;
  }
  __syncthreads();
  const unsigned long long before = warp > 0 ? sw[warp - 1] : 0ull;
  total = sw[31];
  __syncthreads();  // sw is reused by the next scan
  return v + before;
}

// the value of a magnitude bin (bf16, or IEEE half when F16), exactly
template <bool F16>
__device__ __forceinline__ float bin_value(uint32_t b) {
  return F16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(b))) : __uint_as_float(b << 16);
}

template <bool F16>
__global__ void __launch_bounds__(1024) calib_stats_kernel(const unsigned long long* __restrict__ hist, float scale_in,
                                                           qkv_calib_summary* __restrict__ out) {
  const uint32_t kFirstNonfinite = first_nonfinite<F16>();
  __shared__ unsigned long long sw[32];
  __shared__ float s_p[2];
  __shared__ uint32_t s_top;
  const uint32_t t = threadIdx.x, b0 = 32u * t;
  if (t == 0) {
    s_p[0] = s_p[1] = 0.f;
    s_top = 0u;
  }
  // three passes over the thread's 32 bins, each re-reading them (256 KB in all, from L2)
  unsigned long long fin = 0, nonfin = 0;
  uint32_t top = 0;  // 1 + the highest finite bin with a count
#pragma unroll 4
  for (int j = 0; j < 32; ++j) {
    const unsigned long long c = hist[b0 + j];
    if (b0 + j < kFirstNonfinite) {
      fin += c;
      if (c != 0ull) top = b0 + j + 1;
    } else {
      nonfin += c;
    }
  }
  unsigned long long N = 0, nonfinite = 0;
  const unsigned long long incl = block_scan(fin, sw, N);
  block_scan(nonfin, sw, nonfinite);
  atomicMax(&s_top, top);
  // nearest ranks ceil(q N), q = 999/1000 and 9999/10000, in exact integer arithmetic
  const unsigned long long r999 = (999ull * N + 999ull) / 1000ull;
  const unsigned long long r9999 = (9999ull * N + 9999ull) / 10000ull;
  {
    unsigned long long run = incl - fin;
#pragma unroll 4
    for (int j = 0; j < 32 && b0 + j < kFirstNonfinite; ++j) {
      const unsigned long long c = hist[b0 + j];
      const unsigned long long prev = run;
      run += c;
      if (c != 0ull && prev < r999 && run >= r999) s_p[0] = bin_value<F16>(b0 + j);
      if (c != 0ull && prev < r9999 && run >= r9999) s_p[1] = bin_value<F16>(b0 + j);
    }
  }
  __syncthreads();
  const float amax = s_top ? bin_value<F16>(s_top - 1u) : 0.f;
  const float scale = scale_in > 0.f ? scale_in : __fdiv_rn(amax, 448.0f);
  // scaled-magnitude classes; a zero scale (an all-zero tensor) leaves them at 0
  unsigned long long below = 0, sub = 0, sat = 0;
  if (scale > 0.f) {
    const float kSub = 0.001953125f, kNorm = 0.015625f, kSat = 464.0f;  // 2^-9, 2^-6, (448 + 480) / 2
#pragma unroll 4
    for (int j = 0; j < 32 && b0 + j < kFirstNonfinite; ++j) {
      const uint32_t b = b0 + j;
      const unsigned long long c = hist[b];
      if (c == 0ull) continue;
      const float y = __fdiv_rn(bin_value<F16>(b), scale);
      if (b != 0u && y < kSub) below += c;
      if (y >= kSub && y < kNorm) sub += c;
      if (y > kSat) sat += c;
    }
  }
  unsigned long long tb, ts, tt;
  block_scan(below, sw, tb);
  block_scan(sub, sw, ts);
  block_scan(sat, sw, tt);
  if (t == 0) {
    out->count = N;
    out->zeros = hist[0];
    out->nonfinite = nonfinite;
    out->below_subnormal = tb;
    out->subnormal = ts;
    out->saturated = tt;
    out->amax = amax;
    out->p99_9 = s_p[0];
    out->p99_99 = s_p[1];
    out->scale = scale;
  }
}

int sm_count_cached() {
  static int count[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (count[dev] == 0) {
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    count[dev] = c;
  }
  return count[dev];
}

}  // namespace

cudaError_t launch_calib_histogram(const void* x, int64_t n, uint64_t* hist, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  constexpr int smem = kBins * sizeof(uint32_t);
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(calib_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
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
