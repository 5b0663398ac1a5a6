// Quantize-on-write kernels: int8 per-(token, head) absmax/127 (side or inline scale
// layout) and FP8 E4M3 with calibrated per-layer scales, plus the amax/448 calibration
// reduction. New tokens are bf16, or IEEE half for the FP16-activation contract of
// "[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache" §Purpose (exact widening either way).
//
// Pages: "int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next QSA path" §The finding
// worth upstreaming (per-(token,head) scale, 260 B inline record vs side tensor);
// "Qwen3.8 Flash Next NVFP4 QSA FP8 E4M3 KV Scales" §Calibration (stored = e4m3fn(x/scale),
// scale = max envelope / 448).
//
// One warp owns one (token, head) row of K or V, or both rows when the write is large: 32 lanes
// x 8 values = a 256-wide head vector, read as one coalesced line (head_dim 128: lanes 16..31
// idle); the absmax is a 5-step shuffle reduction; the codes leave as one coalesced line.
// Every code is the one the IEEE quotient fl(x / scale) rounds to (round-to-nearest-even), so
// the stored bytes equal a plain fp32 reference bit for bit; int8 takes the division itself
// only where a bracket of two multiplications cannot decide (see bracket_lo / bracket_hi).
#include <atomic>

#include "qkv_internal.cuh"

namespace qkv {
namespace {

constexpr int kWriteThreads = 256;

struct HeadVec {
  float x[8];
};

// Eight consecutive 16-bit activations (bf16, or IEEE half when F16), loaded raw (streaming:
// the new tokens are consumed once) and widened exactly to fp32.
__device__ __forceinline__ uint4 load_raw8(const uint16_t* src) {
  uint4 raw;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(raw.x), "=r"(raw.y), "=r"(raw.z), "=r"(raw.w)
               : "l"(src));
  return raw;
}

template <bool F16>
__device__ __forceinline__ HeadVec widen8(const uint4& raw) {
  HeadVec h;
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (F16) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      h.x[2 * i] = f.x;
      h.x[2 * i + 1] = f.y;
    } else {
      h.x[2 * i] = bf16lo(w[i]);
      h.x[2 * i + 1] = bf16hi(w[i]);
    }
  }
  return h;
}

// int8 codes without a division per value. With r = fl(1 / s), the exact products
// x fl(r (1 -+ 2^-20)) lie below and above the IEEE quotient fl(x / s): the roundings of r and
// of r (1 -+ 2^-20) each move a value by at most 2^-24 of itself, so both products differ from
// x / s by more than 2^-22 of it, on opposite sides, and fl(x / s) by at most 2^-24. Rounding to
// an integer is monotonic, so where both products round to the same integer, fl(x / s) rounds to
// it as well; otherwise (x / s within about 2^-20 of a half-integer, a few values in 10^4) the
// division decides. This holds while r is a finite normal float: scales in [2^-100, 2^100];
// other scales always divide. (E4M3 keeps its division: a bracket there takes two conversions
// per pair instead of one, which measured slower than the divisions.)
constexpr float kBracket = 9.5367431640625e-07f;  // 2^-20
__device__ __forceinline__ bool bracket_ok(float s) { return s >= 7.8886090522101181e-31f && s <= 1.2676506002282294e30f; }
__device__ __forceinline__ float bracket_lo(float s) { return __fmul_rn(__frcp_rn(s), 1.0f - kBracket); }
__device__ __forceinline__ float bracket_hi(float s) { return __fmul_rn(__frcp_rn(s), 1.0f + kBracket); }
// RN(y + 1.5 2^23) holds rint(y), ties to even, in its low mantissa bits for |y| < 2^22; its low
// byte is the code's two's complement byte
constexpr float kRintMagic = 12582912.0f;

__device__ __forceinline__ float warp_max(float a) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
  return a;
}

// Large writes pair a token head's K and V rows in one warp (two row loads in flight per
// lane, one slot load for both); small ones give each row its own warp, twice the warps to
// spread a latency-bound launch over. Measured on one GB300 (int8 side / E4M3): 262144 tokens
// 143 -> 117 / 113 -> 91 us paired; 2048 tokens 7-9 / 7 us either way.
constexpr int64_t kPairedMinUnits = 16384;  // (token, head) units from which rows are paired

// The (token t, head h) of a unit. 32-bit division whenever the index fits, which it does at
// any realistic size (64-bit division is several times longer).
__device__ __forceinline__ void decode_unit(int64_t unit, int num_heads, int64_t& t, int& h) {
  if (unit <= 0xFFFFFFFFll) {
    const uint32_t t32 = static_cast<uint32_t>(unit) / static_cast<uint32_t>(num_heads);
    t = t32;
    h = static_cast<int>(static_cast<uint32_t>(unit) - t32 * static_cast<uint32_t>(num_heads));
  } else {
    t = unit / num_heads;
    h = static_cast<int>(unit - t * num_heads);
  }
}

// Whether a token's slot is written: false when it is skipped (-1) or out of range (flagged by
// lane 0 of the warp that `flags`, one per token).
__device__ __forceinline__ bool slot_ok(int64_t slot, int64_t num_slots, uint32_t* dev_status, int lane, bool flags) {
  if (slot == -1) return false;
  if (slot < -1 || slot >= num_slots) {
    if (lane == 0 && flags && dev_status != nullptr) atomicOr(dev_status, QKV_DEV_BAD_SLOT);
    return false;
  }
  return true;
}

// The slot of token t in a paged pool: -1 when its position is -1 (skipped); -2 (flagged, then
// skipped) for a position outside [-1, max_blocks * block_size), a sequence outside
// [0, num_seqs) or an unallocated block (id < 0); a slot past the pool is flagged by the caller.
__device__ __forceinline__ int64_t paged_slot(const WritePaging& pg, int64_t t, int64_t num_slots) {
  const int seq = __ldg(pg.token_seq + t), pos = __ldg(pg.token_pos + t);  // both loads in flight
  if (pos == -1) return -1;
  if (pos < -1 || static_cast<int64_t>(pos) >= static_cast<int64_t>(pg.max_blocks) * pg.block_size || seq < 0 ||
      seq >= pg.num_seqs)
    return -2;
  const int b = pos / pg.block_size;
  const int blk = __ldg(pg.block_table + static_cast<int64_t>(seq) * pg.max_blocks + b);
  if (blk < 0) return -2;
  return static_cast<int64_t>(blk) * pg.block_size + (pos - b * pg.block_size);
}

// The warp's rows: one row (K or V: kv) of a (token, head) unit, or both rows of a unit when
// paired. Every row and the slot are loaded before any is used, so the loads are in flight
// together (a skipped token's rows are still in bounds: t < num_tokens). Returns false for a
// warp past the end, a skipped token or a bad slot; the result is warp-uniform.
template <bool kPaired, bool kPaged>
__device__ __forceinline__ bool warp_rows(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int head_dim,
                                          int64_t num_tokens, int num_heads, int64_t token_stride,
                                          const int64_t* __restrict__ slot_mapping, const WritePaging& pg,
                                          int64_t num_slots, uint32_t* dev_status, int lane, bool act,
                                          uint4 (&raw)[2], int& kv, int64_t& rec) {
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * kWriteThreads + threadIdx.x) >> 5;
  const int64_t unit = kPaired ? wid : wid >> 1;
  if (unit >= num_tokens * num_heads) return false;
  kv = kPaired ? 0 : static_cast<int>(wid & 1);
  int64_t t;
  int h;
  decode_unit(unit, num_heads, t, h);
  const int64_t off = t * token_stride + static_cast<int64_t>(h) * head_dim + lane * 8;
  raw[0] = act ? load_raw8((kv ? v : k) + off) : make_uint4(0, 0, 0, 0);
  if (kPaired) raw[1] = act ? load_raw8(v + off) : make_uint4(0, 0, 0, 0);
  const int64_t slot = kPaged ? paged_slot(pg, t, num_slots) : slot_mapping[t];
  if (!slot_ok(slot, num_slots, dev_status, lane, kv == 0 && h == 0)) return false;
  rec = slot * num_heads + h;
  return true;
}

// int8 codes and scale of one head row into record `rec` of `cache` (and `scale_out`, side layout).
template <bool kInline>
__device__ __forceinline__ void store_int8_row(const HeadVec& hv, int lane, bool act, int head_dim, int64_t rec,
                                               uint8_t* __restrict__ cache, float* __restrict__ scale_out) {
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(hv.x[i]));
  a = warp_max(a);
  const float scale = __fdiv_rn(a, 127.0f);
  uint32_t word[2] = {0u, 0u};
  if (scale > 0.f) {
    // |x| <= amax and scale = fl(amax / 127) keep |x / scale| below 127.5, so the clamp never
    // acts on a finite value (a NaN value fails the bracket test and takes the clamped division)
    const bool br = bracket_ok(scale);
    const float rlo = bracket_lo(scale), rhi = bracket_hi(scale);
    uint32_t c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float lo = __fmaf_rn(hv.x[i], rlo, kRintMagic), hi = __fmaf_rn(hv.x[i], rhi, kRintMagic);
      c[i] = (br && lo == hi) ? __float_as_uint(lo)
                              : static_cast<uint32_t>(max(-127, min(127, __float2int_rn(__fdiv_rn(hv.x[i], scale)))));
    }
    // low bytes of c[4w .. 4w + 3] into word w, c[4w] lowest: two byte permutes per pair, one
    // to join the pairs
#pragma unroll
    for (int w = 0; w < 2; ++w)
      word[w] = __byte_perm(__byte_perm(c[4 * w], c[4 * w + 1], 0x0040), __byte_perm(c[4 * w + 2], c[4 * w + 3], 0x0040),
                            0x5410);
  }
  if (kInline) {
    uint8_t* base = cache + rec * (head_dim + 4);  // head_dim codes, then the fp32 scale
    uint32_t* dst = reinterpret_cast<uint32_t*>(base + lane * 8);  // records are 4 B aligned
    if (act) {
      dst[0] = word[0];
      dst[1] = word[1];
    }
    if (lane == 0) *reinterpret_cast<float*>(base + head_dim) = scale;
  } else {
    if (act) *reinterpret_cast<uint2*>(cache + rec * head_dim + lane * 8) = make_uint2(word[0], word[1]);
    if (lane == 0) scale_out[rec] = scale;
  }
}

// E4M3 codes of one head row (lanes that own dims only) into record `rec` of `cache`.
__device__ __forceinline__ void store_e4m3_row(const HeadVec& hv, int lane, int head_dim, int64_t rec, float s,
                                               uint8_t* __restrict__ cache) {
  uint32_t p[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 y = make_float2(__fdiv_rn(hv.x[2 * j], s), __fdiv_rn(hv.x[2 * j + 1], s));
    // .x lands in the low byte; round to nearest even, saturate to +-448, sign kept.
    p[j] = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
  }
  // code pairs 2w, 2w + 1 into word w (low halves), one byte permute each
  *reinterpret_cast<uint2*>(cache + rec * head_dim + lane * 8) =
      make_uint2(__byte_perm(p[0], p[1], 0x5410), __byte_perm(p[2], p[3], 0x5410));
}

template <bool kInline, bool F16, bool kPaired, bool kPaged>
__global__ void __launch_bounds__(kWriteThreads)
    write_int8_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int head_dim,
                      int64_t num_tokens, int num_heads, int64_t token_stride,
                      const int64_t* __restrict__ slot_mapping, const WritePaging pg, uint8_t* __restrict__ k_cache,
                      uint8_t* __restrict__ v_cache, float* __restrict__ k_scale,
                      float* __restrict__ v_scale, int64_t num_slots, uint32_t* dev_status) {
  const int lane = threadIdx.x & 31;
  const bool act = 8 * lane < head_dim;  // lane owns head dims 8 lane .. 8 lane + 7 (128: lanes 0..15)
  uint4 raw[2];
  int kv;
  int64_t rec;
  if (!warp_rows<kPaired, kPaged>(k, v, head_dim, num_tokens, num_heads, token_stride, slot_mapping, pg, num_slots,
                                  dev_status, lane, act, raw, kv, rec))
    return;
  store_int8_row<kInline>(widen8<F16>(raw[0]), lane, act, head_dim, rec, kv ? v_cache : k_cache,
                          kv ? v_scale : k_scale);
  if (kPaired) store_int8_row<kInline>(widen8<F16>(raw[1]), lane, act, head_dim, rec, v_cache, v_scale);
}

template <bool F16, bool kPaired, bool kPaged>
__global__ void __launch_bounds__(kWriteThreads)
    write_e4m3_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int head_dim,
                      int64_t num_tokens, int num_heads, int64_t token_stride,
                      const int64_t* __restrict__ slot_mapping, const WritePaging pg, uint8_t* __restrict__ k_cache,
                      uint8_t* __restrict__ v_cache, float k_scale, float v_scale, int64_t num_slots,
                      uint32_t* dev_status) {
  const int lane = threadIdx.x & 31;
  const bool act = 8 * lane < head_dim;  // head_dim 128: lanes 16..31 own no dims (no shuffles follow)
  uint4 raw[2];
  int kv;
  int64_t rec;
  if (!warp_rows<kPaired, kPaged>(k, v, head_dim, num_tokens, num_heads, token_stride, slot_mapping, pg, num_slots,
                                  dev_status, lane, act, raw, kv, rec) ||
      !act)
    return;
  store_e4m3_row(widen8<F16>(raw[0]), lane, head_dim, rec, kv ? v_scale : k_scale, kv ? v_cache : k_cache);
  if (kPaired) store_e4m3_row(widen8<F16>(raw[1]), lane, head_dim, rec, v_scale, v_cache);
}

// max |x| over n bf16 values, as fp32 bits (non-negative floats order like their bits). A
// grid-stride loop with four 16 B loads in flight per thread.
__device__ __forceinline__ uint32_t absmax8(uint32_t m, const uint4& r) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) m = max(m, max((w[j] & 0x7FFFu) << 16, w[j] & 0x7FFF0000u));
  return m;
}

__global__ void __launch_bounds__(256)
    absmax_bf16_kernel(const uint16_t* __restrict__ x, int64_t n, uint32_t* __restrict__ amax_bits) {
  uint32_t m = 0;
  const int64_t nvec = n / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < nvec; i += 4 * stride) {
    uint4 r[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) r[u] = __ldg(xv + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) m = absmax8(m, r[u]);
  }
  for (; i < nvec; i += stride) m = absmax8(m, __ldg(xv + i));
  for (int64_t j = nvec * 8 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < n; j += stride)
    m = max(m, static_cast<uint32_t>(x[j] & 0x7FFFu) << 16);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
  __shared__ uint32_t red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) m = max(m, red[w]);
    atomicMax(amax_bits, m);
  }
}

__global__ void e4m3_scale_kernel(const uint32_t* __restrict__ amax_bits, float* __restrict__ scale_out) {
  scale_out[0] = __fdiv_rn(__uint_as_float(amax_bits[0]), 448.0f);
}

bool write_paired(int64_t num_tokens, int num_heads) { return num_tokens * num_heads >= kPairedMinUnits; }

unsigned write_blocks(int64_t num_tokens, int num_heads) {
  const int64_t warps = num_tokens * num_heads * (write_paired(num_tokens, num_heads) ? 1 : 2);
  return static_cast<unsigned>((warps * 32 + kWriteThreads - 1) / kWriteThreads);
}

template <bool kInline, bool F16, bool kPaired, bool kPaged>
void launch_int8(unsigned blocks, const uint16_t* k, const uint16_t* v, int head_dim, int64_t num_tokens,
                 int num_heads, int64_t token_stride, const int64_t* slot_mapping, const WritePaging& pg,
                 uint8_t* kc, uint8_t* vc, float* ks, float* vs, int64_t num_slots, uint32_t* dev_status,
                 cudaStream_t stream) {
  write_int8_kernel<kInline, F16, kPaired, kPaged><<<blocks, kWriteThreads, 0, stream>>>(
      k, v, head_dim, num_tokens, num_heads, token_stride, slot_mapping, pg, kc, vc, ks, vs, num_slots, dev_status);
}

template <bool kInline, bool F16>
void launch_int8(bool paired, bool paged, unsigned blocks, const uint16_t* k, const uint16_t* v, int head_dim,
                 int64_t num_tokens, int num_heads, int64_t token_stride, const int64_t* slot_mapping,
                 const WritePaging& pg, uint8_t* kc, uint8_t* vc, float* ks, float* vs, int64_t num_slots,
                 uint32_t* dev_status, cudaStream_t stream) {
  auto kern = paired ? (paged ? launch_int8<kInline, F16, true, true> : launch_int8<kInline, F16, true, false>)
                     : (paged ? launch_int8<kInline, F16, false, true> : launch_int8<kInline, F16, false, false>);
  kern(blocks, k, v, head_dim, num_tokens, num_heads, token_stride, slot_mapping, pg, kc, vc, ks, vs, num_slots,
       dev_status, stream);
}

template <bool F16, bool kPaired, bool kPaged>
void launch_e4m3(unsigned blocks, const uint16_t* k, const uint16_t* v, int head_dim, int64_t num_tokens,
                 int num_heads, int64_t token_stride, const int64_t* slot_mapping, const WritePaging& pg,
                 uint8_t* kc, uint8_t* vc, float ks, float vs, int64_t num_slots, uint32_t* dev_status,
                 cudaStream_t stream) {
  write_e4m3_kernel<F16, kPaired, kPaged><<<blocks, kWriteThreads, 0, stream>>>(
      k, v, head_dim, num_tokens, num_heads, token_stride, slot_mapping, pg, kc, vc, ks, vs, num_slots, dev_status);
}

}  // namespace

cudaError_t launch_write_int8(const void* k, const void* v, bool f16, int head_dim, int64_t num_tokens, int num_heads,
                              int64_t token_stride, const int64_t* slot_mapping, const WritePaging* paging,
                              bool inline_layout, void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                              int64_t num_slots, uint32_t* dev_status, cudaStream_t stream) {
  const unsigned blocks = write_blocks(num_tokens, num_heads);
  const bool pr = write_paired(num_tokens, num_heads), pgd = paging != nullptr;
  const WritePaging pg = pgd ? *paging : WritePaging{nullptr, nullptr, nullptr, 0, 0, 1};
  auto kk = static_cast<const uint16_t*>(k);
  auto vv = static_cast<const uint16_t*>(v);
  auto kc = static_cast<uint8_t*>(k_cache);
  auto vc = static_cast<uint8_t*>(v_cache);
  float* ks = inline_layout ? nullptr : k_scale;
  float* vs = inline_layout ? nullptr : v_scale;
  auto kern = inline_layout ? (f16 ? launch_int8<true, true> : launch_int8<true, false>)
                            : (f16 ? launch_int8<false, true> : launch_int8<false, false>);
  kern(pr, pgd, blocks, kk, vv, head_dim, num_tokens, num_heads, token_stride, slot_mapping, pg, kc, vc, ks, vs,
       num_slots, dev_status, stream);
  return cudaGetLastError();
}

cudaError_t launch_write_e4m3(const void* k, const void* v, bool f16, int head_dim, int64_t num_tokens, int num_heads,
                              int64_t token_stride, const int64_t* slot_mapping, const WritePaging* paging,
                              void* k_cache, void* v_cache, float k_scale, float v_scale, int64_t num_slots,
                              uint32_t* dev_status, cudaStream_t stream) {
  const bool pr = write_paired(num_tokens, num_heads), pgd = paging != nullptr;
  const WritePaging pg = pgd ? *paging : WritePaging{nullptr, nullptr, nullptr, 0, 0, 1};
  auto kern = f16 ? (pr ? (pgd ? launch_e4m3<true, true, true> : launch_e4m3<true, true, false>)
                        : (pgd ? launch_e4m3<true, false, true> : launch_e4m3<true, false, false>))
                  : (pr ? (pgd ? launch_e4m3<false, true, true> : launch_e4m3<false, true, false>)
                        : (pgd ? launch_e4m3<false, false, true> : launch_e4m3<false, false, false>));
  kern(write_blocks(num_tokens, num_heads), static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v), head_dim,
       num_tokens, num_heads, token_stride, slot_mapping, pg, static_cast<uint8_t*>(k_cache),
       static_cast<uint8_t*>(v_cache), k_scale, v_scale, num_slots, dev_status, stream);
  return cudaGetLastError();
}

cudaError_t launch_e4m3_calibrate(const void* x, int64_t n, uint32_t* amax_bits, float* scale_out,
                                  cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  if (n > 0) {
    // one wave of 256-thread blocks (8 per SM); each thread then keeps four loads in flight
    static std::atomic<int> sm_count[64] = {};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int sms = sm_count[dev].load(std::memory_order_relaxed);
    if (sms == 0) {
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      sm_count[dev].store(sms, std::memory_order_relaxed);
    }
    int64_t want = (n / 8 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    const unsigned blocks = static_cast<unsigned>(want < 1 ? 1 : (want > cap ? cap : want));
    absmax_bf16_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint16_t*>(x), n, amax_bits);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  e4m3_scale_kernel<<<1, 1, 0, stream>>>(amax_bits, scale_out);
  return cudaGetLastError();
}

}  // namespace qkv
