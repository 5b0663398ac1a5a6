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
// One warp owns one (token, head, tensor): 32 lanes x 8 values = a 256-wide head vector, read
// as one coalesced line (head_dim 128: lanes 16..31 idle); the absmax is a 5-step shuffle
// reduction; the codes leave as one coalesced line. Division is IEEE (__fdiv_rn) and rounding is
// round-to-nearest-even so the stored bytes equal a plain fp32 reference bit for bit.
#include "qkv_internal.cuh"

namespace qkv {
namespace {

constexpr int kWriteThreads = 256;

struct HeadVec {
  float x[8];
};

// Eight consecutive 16-bit activations (bf16, or IEEE half when F16), widened exactly to fp32.
template <bool F16>
__device__ __forceinline__ HeadVec load_head8(const uint16_t* src) {
  // Streaming read: the new tokens are consumed once.
  uint4 raw;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(raw.x), "=r"(raw.y), "=r"(raw.z), "=r"(raw.w)
               : "l"(src));
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

__device__ __forceinline__ float warp_max(float a) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
  return a;
}

// Decode the warp's work item: (token, head, is_v). Returns false when the token is skipped.
__device__ __forceinline__ bool decode_item(int64_t item, int num_heads, const int64_t* slot_mapping,
                                            int64_t num_slots, uint32_t* dev_status, int lane,
                                            int64_t& t, int& h, int& is_v, int64_t& slot) {
  is_v = static_cast<int>(item & 1);
  const int64_t th = item >> 1;
  t = th / num_heads;
  h = static_cast<int>(th - t * num_heads);
  slot = slot_mapping[t];
  if (slot == -1) return false;
  if (slot < -1 || slot >= num_slots) {
    if (lane == 0 && is_v == 0 && h == 0 && dev_status != nullptr) atomicOr(dev_status, QKV_DEV_BAD_SLOT);
    return false;
  }
  return true;
}

template <bool kInline, bool F16>
__global__ void __launch_bounds__(kWriteThreads)
    write_int8_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int head_dim,
                      int64_t num_tokens, int num_heads, int64_t token_stride,
                      const int64_t* __restrict__ slot_mapping, uint8_t* __restrict__ k_cache,
                      uint8_t* __restrict__ v_cache, float* __restrict__ k_scale,
                      float* __restrict__ v_scale, int64_t num_slots, uint32_t* dev_status) {
  const int lane = threadIdx.x & 31;
  const int64_t item = (static_cast<int64_t>(blockIdx.x) * kWriteThreads + threadIdx.x) >> 5;
  if (item >= num_tokens * num_heads * 2) return;
  int64_t t, slot;
  int h, is_v;
  if (!decode_item(item, num_heads, slot_mapping, num_slots, dev_status, lane, t, h, is_v, slot)) return;

  const bool act = 8 * lane < head_dim;  // lane owns head dims 8 lane .. 8 lane + 7
  const uint16_t* src = (is_v ? v : k) + t * token_stride + static_cast<int64_t>(h) * head_dim + lane * 8;
  const HeadVec hv = act ? load_head8<F16>(src) : HeadVec{};
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(hv.x[i]));
  a = warp_max(a);
  const float scale = __fdiv_rn(a, 127.0f);

  uint32_t word[2] = {0u, 0u};
  if (scale > 0.f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int c = __float2int_rn(__fdiv_rn(hv.x[i], scale));
      c = max(-127, min(127, c));
      word[i >> 2] |= (static_cast<uint32_t>(c) & 0xFFu) << (8 * (i & 3));
    }
  }
  const int64_t rec = slot * num_heads + h;
  uint8_t* cache = is_v ? v_cache : k_cache;
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
    if (lane == 0) (is_v ? v_scale : k_scale)[rec] = scale;
  }
}

template <bool F16>
__global__ void __launch_bounds__(kWriteThreads)
    write_e4m3_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int head_dim,
                      int64_t num_tokens, int num_heads, int64_t token_stride,
                      const int64_t* __restrict__ slot_mapping, uint8_t* __restrict__ k_cache,
                      uint8_t* __restrict__ v_cache, float k_scale, float v_scale, int64_t num_slots,
                      uint32_t* dev_status) {
  const int lane = threadIdx.x & 31;
  const int64_t item = (static_cast<int64_t>(blockIdx.x) * kWriteThreads + threadIdx.x) >> 5;
  if (item >= num_tokens * num_heads * 2) return;
  int64_t t, slot;
  int h, is_v;
  if (!decode_item(item, num_heads, slot_mapping, num_slots, dev_status, lane, t, h, is_v, slot)) return;

  if (8 * lane >= head_dim) return;  // head_dim 128: lanes 16..31 own no dims (no shuffles follow)
  const uint16_t* src = (is_v ? v : k) + t * token_stride + static_cast<int64_t>(h) * head_dim + lane * 8;
  const HeadVec hv = load_head8<F16>(src);
  const float s = is_v ? v_scale : k_scale;
  uint32_t word[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const float2 y = make_float2(__fdiv_rn(hv.x[i], s), __fdiv_rn(hv.x[i + 1], s));
    // .x lands in the low byte; round to nearest even, saturate to +-448, sign kept.
    const uint32_t p = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
    word[i >> 2] |= (p & 0xFFFFu) << (8 * (i & 3));
  }
  uint8_t* cache = is_v ? v_cache : k_cache;
  *reinterpret_cast<uint2*>(cache + (slot * num_heads + h) * head_dim + lane * 8) = make_uint2(word[0], word[1]);
}

// max |x| over n bf16 values, as fp32 bits (non-negative floats order like their bits).
__global__ void __launch_bounds__(256)
    absmax_bf16_kernel(const uint16_t* __restrict__ x, int64_t n, uint32_t* __restrict__ amax_bits) {
  uint32_t m = 0;
  const int64_t nvec = n / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    const uint4 r = __ldg(xv + i);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      m = max(m, (w[j] & 0x7FFFu) << 16);
      m = max(m, w[j] & 0x7FFF0000u);
    }
  }
  for (int64_t i = nvec * 8 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    m = max(m, static_cast<uint32_t>(x[i] & 0x7FFFu) << 16);
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

unsigned write_blocks(int64_t num_tokens, int num_heads) {
  const int64_t warps = num_tokens * num_heads * 2;
  return static_cast<unsigned>((warps * 32 + kWriteThreads - 1) / kWriteThreads);
}

}  // namespace

cudaError_t launch_write_int8(const void* k, const void* v, bool f16, int head_dim, int64_t num_tokens, int num_heads,
                              int64_t token_stride, const int64_t* slot_mapping, bool inline_layout,
                              void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                              int64_t num_slots, uint32_t* dev_status, cudaStream_t stream) {
  const unsigned blocks = write_blocks(num_tokens, num_heads);
  auto kk = static_cast<const uint16_t*>(k);
  auto vv = static_cast<const uint16_t*>(v);
  auto kc = static_cast<uint8_t*>(k_cache);
  auto vc = static_cast<uint8_t*>(v_cache);
  float* ks = inline_layout ? nullptr : k_scale;
  float* vs = inline_layout ? nullptr : v_scale;
  auto kern = inline_layout ? (f16 ? write_int8_kernel<true, true> : write_int8_kernel<true, false>)
                            : (f16 ? write_int8_kernel<false, true> : write_int8_kernel<false, false>);
  kern<<<blocks, kWriteThreads, 0, stream>>>(kk, vv, head_dim, num_tokens, num_heads, token_stride, slot_mapping, kc,
                                             vc, ks, vs, num_slots, dev_status);
  return cudaGetLastError();
}

cudaError_t launch_write_e4m3(const void* k, const void* v, bool f16, int head_dim, int64_t num_tokens, int num_heads,
                              int64_t token_stride, const int64_t* slot_mapping, void* k_cache,
                              void* v_cache, float k_scale, float v_scale, int64_t num_slots,
                              uint32_t* dev_status, cudaStream_t stream) {
  auto kern = f16 ? write_e4m3_kernel<true> : write_e4m3_kernel<false>;
  kern<<<write_blocks(num_tokens, num_heads), kWriteThreads, 0, stream>>>(
      static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v), head_dim, num_tokens, num_heads, token_stride,
      slot_mapping, static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), k_scale, v_scale, num_slots,
      dev_status);
  return cudaGetLastError();
}

cudaError_t launch_e4m3_calibrate(const void* x, int64_t n, uint32_t* amax_bits, float* scale_out,
                                  cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  if (n > 0) {
    int64_t want = (n / 8 + 255) / 256;
    const int64_t cap = 152 * 8;
    const unsigned blocks = static_cast<unsigned>(want < 1 ? 1 : (want > cap ? cap : want));
    absmax_bf16_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint16_t*>(x), n, amax_bits);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  e4m3_scale_kernel<<<1, 1, 0, stream>>>(amax_bits, scale_out);
  return cudaGetLastError();
}

}  // namespace qkv
