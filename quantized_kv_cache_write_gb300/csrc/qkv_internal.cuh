// Internal device helpers and launcher declarations for libqkv.so (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qkv.h"

namespace qkv {

constexpr int kHeadDim = 256;       // the pages' head dim (256 B of int8 per head)
constexpr int kHeadDimSmall = 128;  // the other head dim the kernels take
__host__ __device__ constexpr bool head_dim_ok(int d) { return d == kHeadDim || d == kHeadDimSmall; }
constexpr int kMaxGroup = 128;  // GQA group; above 16 the gather runs one CTA per 16 query heads

// Paged addressing of the writes: token t sits at logical position token_pos[t] of sequence
// token_seq[t], and its slot is block_table[seq, pos / block_size] * block_size + pos %
// block_size (the gather's paged addressing, for the tokens being written).
struct WritePaging {
  const int32_t* token_seq;
  const int32_t* token_pos;
  const int32_t* block_table;
  int64_t num_seqs;
  int max_blocks;
  int block_size;
};

// ------------------------------------------------------------------ launchers
// paging == nullptr: slot ids in slot_mapping; else slot_mapping is unused
cudaError_t launch_write_int8(const void* k, const void* v, bool f16, int head_dim, int64_t num_tokens, int num_heads,
                              int64_t token_stride, const int64_t* slot_mapping, const WritePaging* paging,
                              bool inline_layout, void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                              int64_t num_slots, uint32_t* dev_status, cudaStream_t stream);
cudaError_t launch_write_e4m3(const void* k, const void* v, bool f16, int head_dim, int64_t num_tokens, int num_heads,
                              int64_t token_stride, const int64_t* slot_mapping, const WritePaging* paging,
                              void* k_cache, void* v_cache, float k_scale, float v_scale, int64_t num_slots,
                              uint32_t* dev_status, cudaStream_t stream);
cudaError_t launch_e4m3_calibrate(const void* x, int64_t n, uint32_t* amax_bits, float* scale_out,
                                  cudaStream_t stream);
cudaError_t launch_calib_histogram(const void* x, int64_t n, uint64_t* hist, cudaStream_t stream);
cudaError_t launch_calib_stats(const uint64_t* hist, bool f16, float scale, qkv_calib_summary* stats,
                               cudaStream_t stream);
cudaError_t launch_splitk_merge(const float* o_part, const float* lse_part, int64_t rows,
                                int num_q_heads, int head_dim, int num_splits, float v_scale_post, float* out,
                                float* lse, cudaStream_t stream);

// Arguments of one gather-attention launch (already validated on the host).
struct GatherArgs {
  const __nv_bfloat16* q;  // bf16, or IEEE half bits for the fp16-query launchers
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const float* k_scale_tok;
  const float* v_scale_tok;
  float k_scale_layer;
  float v_scale_layer;
  int64_t num_slots;
  const int32_t* topk_idx;
  const int32_t* topk_len = nullptr;  // varlen: valid entries per row [rows], or null (all topk)
  int64_t rows;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;  // 256 or 128
  int topk;
  int num_splits;
  float softmax_scale;
  float* out;       // [rows, Hq, D] when num_splits == 1
  float* lse;       // [rows, Hq] or null
  float* o_part;    // [rows, P, Hq, D] when num_splits > 1
  float* lse_part;  // [rows, P, Hq]
  uint32_t* dev_status;
  // fused split-K merge (num_splits > 1 only): arrival counters [rows, Hkv, ceil(G / 16)], zero
  // on entry and left zero; the last split CTA of a (row, KV head, head chunk) merges into
  // out / lse. Null = no merge.
  uint32_t* counters = nullptr;
  // paged pools only (the paged launchers): topk_idx then holds logical positions
  const int32_t* block_table = nullptr;  // [num_seqs, max_blocks]
  const int32_t* row_seq = nullptr;      // [rows]
  int64_t num_seqs = 0;
  int max_blocks = 0;
  int block_size = 0;
  // persistent grid: [2] counters (next item, CTAs finished), zero on entry and left zero; the
  // launch then sizes its grid to the CTAs that stay resident. Null = one CTA per item.
  uint32_t* sched = nullptr;
  // slot-range shard: the pool holds global slots [slot_lo, slot_lo + num_slots) at local ids
  // 0 .. num_slots - 1; an entry outside that range is another shard's and is skipped (not
  // flagged). Off: entries are local slot ids, as always.
  int64_t slot_lo = 0;
  bool shard = false;
};

cudaError_t launch_gather_bf16(const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_gather_int8_side(const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_gather_int8_inline(const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_gather_e4m3(const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_gather_paged_bf16(const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_gather_paged_int8_side(const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_gather_paged_int8_inline(const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_gather_paged_e4m3(const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_gather_f16q_int8_side(const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_gather_f16q_int8_inline(const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_gather_f16q_e4m3(const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_gather_f16q_f16(const GatherArgs& a, cudaStream_t stream);
// tensor-core (tcgen05) gather: persistent, one CTA per SM; int8 side scales, head dim 256,
// GQA group <= 16, slot ids, bf16 query
cudaError_t launch_umma_int8_side(const GatherArgs& a, cudaStream_t stream);
cudaError_t gather_ctas_per_sm_bf16(int* n);
cudaError_t gather_ctas_per_sm_int8_side(int* n);
cudaError_t gather_ctas_per_sm_int8_inline(int* n);
cudaError_t gather_ctas_per_sm_e4m3(int* n);

// ------------------------------------------------------------------ device helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; src_bytes < 16 zero-fills the rest (0 reads nothing).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];\n" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;\n" ::"r"(addr), "r"(v));
}

__device__ __forceinline__ void sts_u8(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u8 [%0], %1;\n" ::"r"(addr), "r"(v));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Two 16 x 16 byte matrices, transposed: lanes 0-15 give the row addresses (16 B each) of
// matrix 0, lanes 16-31 those of matrix 1. Lane (g, c) = (lane / 4, lane % 4) receives in r0
// the bytes of rows 4c .. 4c + 3 (row 4c in the low byte) at column g of matrix 0, in r1 the
// same rows at column g + 8; r2, r3 likewise for matrix 1.
__device__ __forceinline__ void ldmatrix_x2_trans_b8(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                     uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, fp32 accumulate. Register-only, so not volatile:
// the compiler may interleave independent MMAs.
__device__ __forceinline__ void mma_f16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ tensor memory (TMEM)
// Allocate `ncols` TMEM columns (a power of two >= 32) for this CTA; one full warp executes
// it, and the base address lands in shared memory at `smem_dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_dst), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_alloc_permit() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// 32 consecutive 32-bit columns of the calling thread's own TMEM lane (shape 32x32b: lane =
// the warp's quarter base + lane id). The values are valid only after tmem_wait_ld on them.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]), "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]), "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]), "=f"(v[31])
               : "r"(taddr));
}
// Wait for this thread's outstanding TMEM loads; naming the destination registers keeps their
// uses after the wait.
__device__ __forceinline__ void tmem_wait_ld(float (&v)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]), "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15]), "+f"(v[16]), "+f"(v[17]), "+f"(v[18]), "+f"(v[19]), "+f"(v[20]), "+f"(v[21]), "+f"(v[22]), "+f"(v[23]), "+f"(v[24]), "+f"(v[25]), "+f"(v[26]), "+f"(v[27]), "+f"(v[28]), "+f"(v[29]), "+f"(v[30]), "+f"(v[31]) : : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n" ::"r"(taddr),
               "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// ------------------------------------------------------------------ packed fp32 pairs
// Two fp32 values in one 64-bit register pair; the .f32x2 arithmetic rounds each lane as the
// scalar op would (round to nearest, subnormals kept).
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};\n" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;\n" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// Scale two consecutive floats in place.
__device__ __forceinline__ void f2scale(float* v, uint64_t s) {
  float a, b;
  f2unpack(f2mul(f2pack(v[0], v[1]), s), a, b);
  v[0] = a;
  v[1] = b;
}

// Split-K merge of one (row, query head) over the NV float4 column groups col4[0..NV):
//   lse = log sum_s exp(lse_s),  o = v_scale_post * sum_s exp(lse_s - lse) o_s,
// with empty splits (lse_s = -inf) skipped and an all-empty row giving o = 0, lse = -inf.
// o_head = o_part at (row, split 0, head): splits are Hq * head_dim floats apart; lp = lse_part
// at (row, split 0, head): splits are Hq floats apart. Partials are read through L2
// (ld.global.cg) because in the fused gather other CTAs of the same launch wrote them. The
// loads of U splits are issued together (U * NV 16 B loads in flight per thread); the sums
// still run over s = 0, 1, ... in order, so a column's result does not depend on which thread
// or kernel merges it, nor on U.
template <int NV, int U>
__device__ __forceinline__ void merge_head(const float* o_head, const float* lp, int Hq, int P, int head_dim,
                                           float v_scale_post,
                                           const int (&col4)[NV], float* out_head, float* lse_out) {
  float m = -INFINITY;
#pragma unroll 4
  for (int s = 0; s < P; ++s) m = fmaxf(m, __ldcg(lp + static_cast<int64_t>(s) * Hq));
  float4* dst = reinterpret_cast<float4*>(out_head);
  if (m == -INFINITY) {
#pragma unroll
    for (int v = 0; v < NV; ++v) dst[col4[v]] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lse_out != nullptr) *lse_out = -INFINITY;
    return;
  }
  float acc[4 * NV];
#pragma unroll
  for (int i = 0; i < 4 * NV; ++i) acc[i] = 0.f;
  float wsum = 0.f;
  const int64_t sstride = static_cast<int64_t>(Hq) * head_dim;
  for (int s0 = 0; s0 < P; s0 += U) {
    float4 x[U][NV];
    float ls[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool in = s0 + u < P;
      ls[u] = in ? __ldcg(lp + static_cast<int64_t>(s0 + u) * Hq) : -INFINITY;
      const float4* src = reinterpret_cast<const float4*>(o_head + (in ? s0 + u : s0) * sstride);
#pragma unroll
      for (int v = 0; v < NV; ++v) x[u][v] = __ldcg(src + col4[v]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (ls[u] == -INFINITY) continue;
      const float w = expf(ls[u] - m);
      wsum += w;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        acc[4 * v] += w * x[u][v].x;
        acc[4 * v + 1] += w * x[u][v].y;
        acc[4 * v + 2] += w * x[u][v].z;
        acc[4 * v + 3] += w * x[u][v].w;
      }
    }
  }
  const float f = v_scale_post / wsum;
#pragma unroll
  for (int v = 0; v < NV; ++v)
    dst[col4[v]] = make_float4(acc[4 * v] * f, acc[4 * v + 1] * f, acc[4 * v + 2] * f, acc[4 * v + 3] * f);
  if (lse_out != nullptr) *lse_out = m + logf(wsum);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Two int8 codes sitting in bytes 0 and 2 of `x` (bytes 1, 3 ignored) -> exact fp16x2.
// (b ^ 0x80) placed under the fp16 exponent of 1024 gives 1024 + 128 + b; subtracting 1152
// leaves b exactly (every integer below 2048 is an fp16 value).
__device__ __forceinline__ uint32_t i8pair_to_f16x2(uint32_t x) {
  uint32_t y = (x & 0x00FF00FFu) ^ 0x64806480u;
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(y), "r"(0x64806480u));
  return r;
}

// Two E4M3 bytes (low byte -> low half) -> exact fp16x2 (native conversion).
__device__ __forceinline__ uint32_t e4m3pair_to_f16x2(uint32_t x16) {
  uint32_t r;
  unsigned short s = static_cast<unsigned short>(x16 & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(s));
  return r;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf162(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace qkv
