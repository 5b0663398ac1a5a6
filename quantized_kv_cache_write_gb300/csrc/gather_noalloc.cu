// qsa_gather_attn_splitk_noalloc: the split-K gather decode plus its merge, with the split
// partials kept in a fixed static device buffer instead of caller-provided workspace.
//
// Who needs this: a caller that owns only its inputs and outputs and may not allocate
// device memory itself -- for example a plugin running inside a host engine that hands it
// pre-allocated tensors and forbids allocation during serving, because cudaMalloc can
// synchronise the whole device and fragments a memory pool the host manages. Such a caller
// cannot provide the [rows, P, Hq, head_dim] partial buffers that qsa_gather_attn needs for
// num_splits > 1; this entry point supplies them from the static array below.
//
// The array costs every GPU that loads libqkv.so kQkvNoallocScratchBytes of device memory
// until the process exits. All calls share it: two calls that overlap on the GPU (different
// streams, or different host threads) race on it and corrupt each other's results.
#include <mutex>

#include "qkv_internal.cuh"

namespace {

constexpr size_t kScratchBytes = QKV_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of g_noalloc_scratch per device. In host code the symbol's name is only a
// host-side stand-in, never a device address, so the address is looked up once per device
// with cudaGetSymbolAddress while that device is current.
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" qkv_status qsa_gather_attn_splitk_noalloc(
    const void* q, int64_t rows, int num_q_heads, int num_kv_heads, int head_dim, qkv_format fmt,
    const void* k_cache, const void* v_cache, const float* k_scale_tok, const float* v_scale_tok,
    float k_scale_layer, float v_scale_layer, int64_t num_slots, const int32_t* topk_idx, int topk,
    float softmax_scale, int num_splits, float* out, float* lse, uint32_t* dev_status, void* stream) {
  if (num_splits == 1)  // nothing to keep between kernels: the plain call needs no workspace
    return qsa_gather_attn(q, rows, num_q_heads, num_kv_heads, head_dim, fmt, k_cache, v_cache, k_scale_tok,
                           v_scale_tok, k_scale_layer, v_scale_layer, num_slots, topk_idx, topk, softmax_scale, 1,
                           out, lse, nullptr, nullptr, dev_status, stream);
  if (rows < 0 || num_q_heads < 1 || num_splits < 1 || !qkv::head_dim_ok(head_dim)) return QKV_ERR_ARG;
  if (rows == 0) return QKV_OK;
  if (out == nullptr || (reinterpret_cast<uintptr_t>(out) & 15) != 0) return QKV_ERR_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3) != 0) return QKV_ERR_ALIGN;

  // Partials layout inside the scratch: o_part [rows, P, Hq, head_dim] fp32, then lse_part
  // [rows, P, Hq] fp32 starting on a 256 B boundary. Sizes beyond the array are refused. Each
  // factor is bounded by division before it multiplies, so the product cannot wrap.
  const uint64_t cap = kScratchBytes;
  if (static_cast<uint64_t>(rows) > cap) return QKV_ERR_ARG;
  const uint64_t rp_cap = cap / static_cast<uint64_t>(rows);
  if (static_cast<uint64_t>(num_splits) > rp_cap) return QKV_ERR_ARG;
  const uint64_t rp = static_cast<uint64_t>(rows) * static_cast<uint64_t>(num_splits);  // <= cap
  if (static_cast<uint64_t>(num_q_heads) > cap / rp) return QKV_ERR_ARG;
  const uint64_t parts = rp * static_cast<uint64_t>(num_q_heads);  // <= cap
  const uint64_t o_bytes = parts * static_cast<uint64_t>(head_dim) * sizeof(float);
  const uint64_t lse_off = (o_bytes + 255) & ~uint64_t(255);
  if (lse_off + parts * sizeof(float) > kScratchBytes) return QKV_ERR_ARG;

  void* base = nullptr;
  if (scratch_for_current_device(&base) != cudaSuccess) return QKV_ERR_CUDA;
  float* o_part = static_cast<float*>(base);
  float* lse_part = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + lse_off);

  // Every partial (row, split, head) is written by the gather -- empty splits as 0 / -inf --
  // before the merge reads it, so the shared array needs no clearing between calls.
  qkv_status st = qsa_gather_attn(q, rows, num_q_heads, num_kv_heads, head_dim, fmt, k_cache, v_cache,
                                  k_scale_tok, v_scale_tok, k_scale_layer, v_scale_layer, num_slots, topk_idx,
                                  topk, softmax_scale, num_splits, nullptr, nullptr, o_part, lse_part, dev_status,
                                  stream);
  if (st != QKV_OK) return st;
  return qsa_splitk_merge(o_part, lse_part, rows, num_q_heads, head_dim, num_splits,
                          fmt == QKV_E4M3 ? v_scale_layer : 1.0f, out, lse, stream);
}
