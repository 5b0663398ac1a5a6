// extern "C" entry points of libqkv.so: host-side validation, then one launch each on the
// caller's stream. Nothing here allocates, frees or synchronises. The declarations, with
// argument meaning, layout, ownership and error behaviour, are in qkv.h.
#include <cmath>
#include <cstdint>

#include "qkv_internal.cuh"

namespace {

using qkv::kMaxGroup;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool finite_positive(float s) { return std::isfinite(s) && s > 0.f; }
qkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? QKV_OK : QKV_ERR_CUDA; }

// Shared checks of the two write calls' token inputs.
qkv_status check_write_inputs(const void* k, const void* v, int64_t num_tokens, int num_kv_heads,
                              int head_dim, int64_t token_stride, const int64_t* slot_mapping,
                              const void* k_cache, const void* v_cache, int64_t num_slots,
                              const qkv::WritePaging* pg = nullptr) {
  if (num_tokens < 0 || num_slots < 0 || num_kv_heads < 1) return QKV_ERR_ARG;
  if (!qkv::head_dim_ok(head_dim)) return QKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return QKV_OK;
  // one warp per head row: 2 T H warps of 32 threads must fit a grid of 2^31 - 1 blocks of 256
  if (num_tokens > (int64_t(1) << 32) / num_kv_heads) return QKV_ERR_ARG;
  if (!k || !v || !k_cache || !v_cache) return QKV_ERR_ARG;
  if (pg == nullptr ? !slot_mapping : (!pg->token_seq || !pg->token_pos || !pg->block_table)) return QKV_ERR_ARG;
  if (token_stride < static_cast<int64_t>(num_kv_heads) * head_dim) return QKV_ERR_ARG;
  if (token_stride % 8 != 0 || !aligned(k, 16) || !aligned(v, 16)) return QKV_ERR_ALIGN;
  if (pg == nullptr) {
    if (!aligned(slot_mapping, 8)) return QKV_ERR_ALIGN;
  } else {
    if (pg->block_size < 1 || pg->max_blocks < 1 || pg->num_seqs < 1) return QKV_ERR_ARG;
    if (static_cast<int64_t>(pg->max_blocks) * pg->block_size > INT32_MAX) return QKV_ERR_ARG;
    if (!aligned(pg->token_seq, 4) || !aligned(pg->token_pos, 4) || !aligned(pg->block_table, 4))
      return QKV_ERR_ALIGN;
  }
  return QKV_OK;
}

}  // namespace

extern "C" {

const char* qkv_status_str(qkv_status s) {
  switch (s) {
    case QKV_OK: return "ok";
    case QKV_ERR_ARG: return "invalid argument";
    case QKV_ERR_SCALE: return "per-layer scale is not finite and positive";
    case QKV_ERR_UNSUPPORTED: return "unsupported head_dim or GQA group";
    case QKV_ERR_ALIGN: return "pointer or stride misaligned";
    case QKV_ERR_CUDA: return "CUDA launch failed";
  }
  return "unknown status";
}

}  // extern "C"

namespace {

qkv_status write_int8_impl(const void* k, const void* v, bool f16, int64_t num_tokens, int num_kv_heads,
                           int head_dim, int64_t token_stride, const int64_t* slot_mapping, qkv_format layout,
                           void* k_cache, void* v_cache, float* k_scale, float* v_scale, int64_t num_slots,
                           uint32_t* dev_status, void* stream, const qkv::WritePaging* pg = nullptr) {
  qkv_status st = check_write_inputs(k, v, num_tokens, num_kv_heads, head_dim, token_stride, slot_mapping,
                                     k_cache, v_cache, num_slots, pg);
  if (st != QKV_OK) return st;
  if (layout != QKV_INT8_SIDE && layout != QKV_INT8_INLINE) return QKV_ERR_ARG;
  const bool inl = layout == QKV_INT8_INLINE;
  if (inl && (k_scale || v_scale)) return QKV_ERR_ARG;
  if (num_tokens == 0) return QKV_OK;
  if (!inl && (!k_scale || !v_scale)) return QKV_ERR_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return QKV_ERR_ALIGN;
  if (!inl && (!aligned(k_scale, 4) || !aligned(v_scale, 4))) return QKV_ERR_ALIGN;
  if (dev_status && !aligned(dev_status, 4)) return QKV_ERR_ALIGN;
  return cuda_status(qkv::launch_write_int8(k, v, f16, head_dim, num_tokens, num_kv_heads, token_stride, slot_mapping, pg,
                                            inl, k_cache, v_cache, k_scale, v_scale, num_slots, dev_status,
                                            static_cast<cudaStream_t>(stream)));
}

qkv_status write_e4m3_impl(const void* k, const void* v, bool f16, int64_t num_tokens, int num_kv_heads,
                           int head_dim, int64_t token_stride, const int64_t* slot_mapping, void* k_cache,
                           void* v_cache, float k_scale, float v_scale, int64_t num_slots, uint32_t* dev_status,
                           void* stream, const qkv::WritePaging* pg = nullptr) {
  qkv_status st = check_write_inputs(k, v, num_tokens, num_kv_heads, head_dim, token_stride, slot_mapping,
                                     k_cache, v_cache, num_slots, pg);
  if (st != QKV_OK) return st;
  if (!finite_positive(k_scale) || !finite_positive(v_scale)) return QKV_ERR_SCALE;
  if (num_tokens == 0) return QKV_OK;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return QKV_ERR_ALIGN;
  if (dev_status && !aligned(dev_status, 4)) return QKV_ERR_ALIGN;
  return cuda_status(qkv::launch_write_e4m3(k, v, f16, head_dim, num_tokens, num_kv_heads, token_stride, slot_mapping, pg,
                                            k_cache, v_cache, k_scale, v_scale, num_slots, dev_status,
                                            static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

qkv_status qkv_write_int8(const void* k, const void* v, int64_t num_tokens, int num_kv_heads, int head_dim,
                          int64_t token_stride, const int64_t* slot_mapping, qkv_format layout, void* k_cache,
                          void* v_cache, float* k_scale, float* v_scale, int64_t num_slots, uint32_t* dev_status,
                          void* stream) {
  return write_int8_impl(k, v, false, num_tokens, num_kv_heads, head_dim, token_stride, slot_mapping, layout,
                         k_cache, v_cache, k_scale, v_scale, num_slots, dev_status, stream);
}

qkv_status qkv_write_int8_f16(const void* k, const void* v, int64_t num_tokens, int num_kv_heads, int head_dim,
                              int64_t token_stride, const int64_t* slot_mapping, qkv_format layout, void* k_cache,
                              void* v_cache, float* k_scale, float* v_scale, int64_t num_slots,
                              uint32_t* dev_status, void* stream) {
  return write_int8_impl(k, v, true, num_tokens, num_kv_heads, head_dim, token_stride, slot_mapping, layout,
                         k_cache, v_cache, k_scale, v_scale, num_slots, dev_status, stream);
}

qkv_status qkv_write_e4m3(const void* k, const void* v, int64_t num_tokens, int num_kv_heads, int head_dim,
                          int64_t token_stride, const int64_t* slot_mapping, void* k_cache, void* v_cache,
                          float k_scale, float v_scale, int64_t num_slots, uint32_t* dev_status, void* stream) {
  return write_e4m3_impl(k, v, false, num_tokens, num_kv_heads, head_dim, token_stride, slot_mapping, k_cache,
                         v_cache, k_scale, v_scale, num_slots, dev_status, stream);
}

qkv_status qkv_write_e4m3_f16(const void* k, const void* v, int64_t num_tokens, int num_kv_heads, int head_dim,
                              int64_t token_stride, const int64_t* slot_mapping, void* k_cache, void* v_cache,
                              float k_scale, float v_scale, int64_t num_slots, uint32_t* dev_status,
                              void* stream) {
  return write_e4m3_impl(k, v, true, num_tokens, num_kv_heads, head_dim, token_stride, slot_mapping, k_cache,
                         v_cache, k_scale, v_scale, num_slots, dev_status, stream);
}

qkv_status qkv_write_ex(const qkv_write_desc* d, void* stream) {
  if (d == nullptr || d->size != sizeof(qkv_write_desc)) return QKV_ERR_ARG;
  const bool paged = d->slot_mapping == nullptr;
  if (!paged && (d->token_seq || d->token_pos || d->block_table)) return QKV_ERR_ARG;  // one addressing only
  const qkv::WritePaging pg{d->token_seq, d->token_pos, d->block_table, d->num_seqs, d->max_blocks, d->block_size};
  const qkv::WritePaging* pp = paged ? &pg : nullptr;
  if (d->act_fp16 != 0 && d->act_fp16 != 1) return QKV_ERR_ARG;
  const bool f16 = d->act_fp16 == 1;
  if (d->fmt == QKV_INT8_SIDE || d->fmt == QKV_INT8_INLINE)
    return write_int8_impl(d->k, d->v, f16, d->num_tokens, d->num_kv_heads, d->head_dim, d->token_stride,
                           d->slot_mapping, d->fmt, d->k_cache, d->v_cache, d->k_scale, d->v_scale, d->num_slots,
                           d->dev_status, stream, pp);
  if (d->fmt == QKV_E4M3) {
    if (d->k_scale || d->v_scale) return QKV_ERR_ARG;  // per-token scale tensors belong to the int8 side layout
    return write_e4m3_impl(d->k, d->v, f16, d->num_tokens, d->num_kv_heads, d->head_dim, d->token_stride,
                           d->slot_mapping, d->k_cache, d->v_cache, d->k_scale_layer, d->v_scale_layer,
                           d->num_slots, d->dev_status, stream, pp);
  }
  return QKV_ERR_ARG;
}

qkv_status qkv_e4m3_calibrate(const void* x, int64_t n, uint32_t* amax_bits, float* scale_out, void* stream) {
  if (n < 0 || !amax_bits || !scale_out || (n > 0 && !x)) return QKV_ERR_ARG;
  if (n > 0 && !aligned(x, 16)) return QKV_ERR_ALIGN;
  if (!aligned(amax_bits, 4) || !aligned(scale_out, 4)) return QKV_ERR_ALIGN;
  return cuda_status(qkv::launch_e4m3_calibrate(x, n, amax_bits, scale_out, static_cast<cudaStream_t>(stream)));
}

qkv_status qkv_calib_histogram(const void* x, int64_t n, uint64_t* hist, void* stream) {
  if (n < 0 || n > (int64_t(1) << 40) || !hist || (n > 0 && !x)) return QKV_ERR_ARG;
  if ((n > 0 && !aligned(x, 16)) || !aligned(hist, 8)) return QKV_ERR_ALIGN;
  if (n == 0) return QKV_OK;
  return cuda_status(qkv::launch_calib_histogram(x, n, hist, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {
qkv_status calib_stats_impl(const uint64_t* hist, bool f16, float scale, qkv_calib_summary* stats, void* stream) {
  if (!hist || !stats) return QKV_ERR_ARG;
  if (!(scale == 0.f || finite_positive(scale))) return QKV_ERR_SCALE;
  if (!aligned(hist, 8) || !aligned(stats, 8)) return QKV_ERR_ALIGN;
  return cuda_status(qkv::launch_calib_stats(hist, f16, scale, stats, static_cast<cudaStream_t>(stream)));
}
}  // namespace

extern "C" {

qkv_status qkv_calib_stats(const uint64_t* hist, float scale, qkv_calib_summary* stats, void* stream) {
  return calib_stats_impl(hist, false, scale, stats, stream);
}

qkv_status qkv_calib_stats_f16(const uint64_t* hist, float scale, qkv_calib_summary* stats, void* stream) {
  return calib_stats_impl(hist, true, scale, stats, stream);
}

}  // extern "C"

namespace {

// Paged-pool arguments of qsa_gather_attn_paged (absent for qsa_gather_attn).
struct Paging {
  const int32_t* block_table;
  const int32_t* row_seq;
  int64_t num_seqs;
  int max_blocks;
  int block_size;
};

qkv_status gather_impl(const void* q, int64_t rows, int num_q_heads, int num_kv_heads, int head_dim,
                       qkv_format fmt, const void* k_cache, const void* v_cache, const float* k_scale_tok,
                       const float* v_scale_tok, float k_scale_layer, float v_scale_layer, int64_t num_slots,
                       const int32_t* topk_idx, int topk, float softmax_scale, int num_splits, float* out,
                       float* lse, float* o_part, float* lse_part, uint32_t* dev_status, void* stream,
                       const Paging* pg, uint32_t* counters = nullptr, bool q_f16 = false,
                       const int32_t* topk_len = nullptr, int engine = QSA_ENGINE_DEFAULT,
                       uint32_t* sched = nullptr, bool shard = false, int64_t slot_lo = 0) {
  if (rows < 0 || topk < 0 || num_splits < 1 || num_slots < 0) return QKV_ERR_ARG;
  // a 16-bit pool is multiplied in its own type, so it needs a query of that type
  if ((fmt == QKV_F16 && !q_f16) || (fmt == QKV_BF16 && q_f16)) return QKV_ERR_ARG;
  if (q_f16 && pg != nullptr) return QKV_ERR_ARG;
  if (pg != nullptr) {
    if (pg->num_seqs < 1 || pg->max_blocks < 1 || pg->block_size < 1) return QKV_ERR_ARG;
    if (static_cast<int64_t>(pg->max_blocks) * pg->block_size > INT32_MAX) return QKV_ERR_ARG;
    if (pg->num_seqs * pg->max_blocks > INT32_MAX) return QKV_ERR_ARG;
  }
  if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0) return QKV_ERR_ARG;
  if (!qkv::head_dim_ok(head_dim) || num_q_heads / num_kv_heads > kMaxGroup) return QKV_ERR_UNSUPPORTED;
  if (fmt != QKV_BF16 && fmt != QKV_INT8_SIDE && fmt != QKV_INT8_INLINE && fmt != QKV_E4M3 && fmt != QKV_F16)
    return QKV_ERR_ARG;
  if (!std::isfinite(softmax_scale)) return QKV_ERR_ARG;
  if (fmt == QKV_E4M3 && (!finite_positive(k_scale_layer) || !finite_positive(v_scale_layer)))
    return QKV_ERR_SCALE;
  const bool side = fmt == QKV_INT8_SIDE;
  if (side != (k_scale_tok != nullptr) || side != (v_scale_tok != nullptr)) return QKV_ERR_ARG;
  if (num_splits == 1) {
    if (!out || o_part || lse_part || counters) return QKV_ERR_ARG;
  } else if (counters != nullptr) {  // fused merge: partials and the merged output
    if (!out || !o_part || !lse_part) return QKV_ERR_ARG;
    if (!aligned(counters, 4)) return QKV_ERR_ALIGN;
  } else {
    if (out || lse || !o_part || !lse_part) return QKV_ERR_ARG;
  }
  if (static_cast<int64_t>(topk) + num_splits > INT32_MAX) return QKV_ERR_ARG;
  const int64_t head_chunks = (num_q_heads / num_kv_heads + 15) / 16;  // CTAs per (row, KV head, split)
  if (rows * num_kv_heads * head_chunks * static_cast<int64_t>(num_splits) > INT32_MAX) return QKV_ERR_ARG;
  // the kernels number records (slot * H + head) in 32 bits
  if (num_slots * num_kv_heads > INT32_MAX) return QKV_ERR_UNSUPPORTED;
  if (rows == 0) return QKV_OK;
  if (!q || !k_cache || !v_cache || (topk > 0 && !topk_idx)) return QKV_ERR_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16)) return QKV_ERR_ALIGN;
  if (topk_idx && !aligned(topk_idx, 4)) return QKV_ERR_ALIGN;
  if (topk_len && !aligned(topk_len, 4)) return QKV_ERR_ALIGN;
  if (side && (!aligned(k_scale_tok, 4) || !aligned(v_scale_tok, 4))) return QKV_ERR_ALIGN;
  if ((out && !aligned(out, 16)) || (o_part && !aligned(o_part, 16))) return QKV_ERR_ALIGN;
  if ((lse && !aligned(lse, 4)) || (lse_part && !aligned(lse_part, 4))) return QKV_ERR_ALIGN;
  if (dev_status && !aligned(dev_status, 4)) return QKV_ERR_ALIGN;
  if (engine == QSA_ENGINE_PERSISTENT) {
    if (sched == nullptr) return QKV_ERR_ARG;
    if (!aligned(sched, 4)) return QKV_ERR_ALIGN;
  }
  if (shard && (slot_lo < 0 || slot_lo > INT32_MAX || pg != nullptr)) return QKV_ERR_ARG;
  if (pg != nullptr) {
    if (!pg->block_table || !pg->row_seq) return QKV_ERR_ARG;
    if (!aligned(pg->block_table, 4) || !aligned(pg->row_seq, 4)) return QKV_ERR_ALIGN;
  }

  qkv::GatherArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k_cache = static_cast<const uint8_t*>(k_cache);
  a.v_cache = static_cast<const uint8_t*>(v_cache);
  a.k_scale_tok = k_scale_tok;
  a.v_scale_tok = v_scale_tok;
  a.k_scale_layer = k_scale_layer;
  a.v_scale_layer = v_scale_layer;
  a.num_slots = num_slots;
  a.topk_idx = topk_idx;
  a.topk_len = topk_len;
  a.rows = rows;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.topk = topk;
  a.num_splits = num_splits;
  a.softmax_scale = softmax_scale;
  a.out = out;
  a.lse = lse;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.dev_status = dev_status;
  a.counters = num_splits > 1 ? counters : nullptr;
  a.sched = engine == QSA_ENGINE_PERSISTENT ? sched : nullptr;
  a.shard = shard;
  a.slot_lo = shard ? slot_lo : 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (pg != nullptr) {
    a.block_table = pg->block_table;
    a.row_seq = pg->row_seq;
    a.num_seqs = pg->num_seqs;
    a.max_blocks = pg->max_blocks;
    a.block_size = pg->block_size;
    if (engine == QSA_ENGINE_TCGEN05) return QKV_ERR_UNSUPPORTED;
    switch (fmt) {
      case QKV_BF16: return cuda_status(qkv::launch_gather_paged_bf16(a, s));
      case QKV_INT8_SIDE: return cuda_status(qkv::launch_gather_paged_int8_side(a, s));
      case QKV_INT8_INLINE: return cuda_status(qkv::launch_gather_paged_int8_inline(a, s));
      case QKV_E4M3: return cuda_status(qkv::launch_gather_paged_e4m3(a, s));
    }
    return QKV_ERR_ARG;
  }
  if (q_f16) {
    if (engine == QSA_ENGINE_TCGEN05) return QKV_ERR_UNSUPPORTED;
    switch (fmt) {
      case QKV_INT8_SIDE: return cuda_status(qkv::launch_gather_f16q_int8_side(a, s));
      case QKV_INT8_INLINE: return cuda_status(qkv::launch_gather_f16q_int8_inline(a, s));
      case QKV_E4M3: return cuda_status(qkv::launch_gather_f16q_e4m3(a, s));
      case QKV_F16: return cuda_status(qkv::launch_gather_f16q_f16(a, s));
      default: return QKV_ERR_ARG;
    }
  }
  if (engine == QSA_ENGINE_TCGEN05) {
    if (fmt != QKV_INT8_SIDE || head_dim != 256 || num_q_heads / num_kv_heads > 16 || a.counters != nullptr ||
        shard)
      return QKV_ERR_UNSUPPORTED;
    return cuda_status(qkv::launch_umma_int8_side(a, s));
  }
  switch (fmt) {
    case QKV_BF16: return cuda_status(qkv::launch_gather_bf16(a, s));
    case QKV_INT8_SIDE: return cuda_status(qkv::launch_gather_int8_side(a, s));
    case QKV_INT8_INLINE: return cuda_status(qkv::launch_gather_int8_inline(a, s));
    case QKV_E4M3: return cuda_status(qkv::launch_gather_e4m3(a, s));
  }
  return QKV_ERR_ARG;
}

}  // namespace

extern "C" {

qkv_status qsa_gather_attn(const void* q, int64_t rows, int num_q_heads, int num_kv_heads, int head_dim,
                           qkv_format fmt, const void* k_cache, const void* v_cache, const float* k_scale_tok,
                           const float* v_scale_tok, float k_scale_layer, float v_scale_layer, int64_t num_slots,
                           const int32_t* topk_idx, int topk, float softmax_scale, int num_splits, float* out,
                           float* lse, float* o_part, float* lse_part, uint32_t* dev_status, void* stream) {
  return gather_impl(q, rows, num_q_heads, num_kv_heads, head_dim, fmt, k_cache, v_cache, k_scale_tok, v_scale_tok,
                     k_scale_layer, v_scale_layer, num_slots, topk_idx, topk, softmax_scale, num_splits, out, lse,
                     o_part, lse_part, dev_status, stream, nullptr);
}

qkv_status qsa_gather_attn_varlen(const void* q, int64_t rows, int num_q_heads, int num_kv_heads, int head_dim,
                                  qkv_format fmt, const void* k_cache, const void* v_cache,
                                  const float* k_scale_tok, const float* v_scale_tok, float k_scale_layer,
                                  float v_scale_layer, int64_t num_slots, const int32_t* topk_idx, int topk,
                                  const int32_t* topk_len, float softmax_scale, int num_splits, float* out,
                                  float* lse, float* o_part, float* lse_part, uint32_t* dev_status, void* stream) {
  if (rows > 0 && topk_len == nullptr) return QKV_ERR_ARG;
  return gather_impl(q, rows, num_q_heads, num_kv_heads, head_dim, fmt, k_cache, v_cache, k_scale_tok, v_scale_tok,
                     k_scale_layer, v_scale_layer, num_slots, topk_idx, topk, softmax_scale, num_splits, out, lse,
                     o_part, lse_part, dev_status, stream, nullptr, nullptr, false, topk_len);
}

qkv_status qsa_gather_attn_f16(const void* q, int64_t rows, int num_q_heads, int num_kv_heads, int head_dim,
                               qkv_format fmt, const void* k_cache, const void* v_cache, const float* k_scale_tok,
                               const float* v_scale_tok, float k_scale_layer, float v_scale_layer,
                               int64_t num_slots, const int32_t* topk_idx, int topk, float softmax_scale,
                               int num_splits, float* out, float* lse, float* o_part, float* lse_part,
                               uint32_t* dev_status, void* stream) {
  return gather_impl(q, rows, num_q_heads, num_kv_heads, head_dim, fmt, k_cache, v_cache, k_scale_tok, v_scale_tok,
                     k_scale_layer, v_scale_layer, num_slots, topk_idx, topk, softmax_scale, num_splits, out, lse,
                     o_part, lse_part, dev_status, stream, nullptr, nullptr, true);
}

qkv_status qsa_gather_attn_paged(const void* q, int64_t rows, int num_q_heads, int num_kv_heads, int head_dim,
                                 qkv_format fmt, const void* k_cache, const void* v_cache,
                                 const float* k_scale_tok, const float* v_scale_tok, float k_scale_layer,
                                 float v_scale_layer, int64_t num_slots, const int32_t* block_table,
                                 int64_t num_seqs, int max_blocks, int block_size, const int32_t* row_seq,
                                 const int32_t* topk_pos, int topk, float softmax_scale, int num_splits,
                                 float* out, float* lse, float* o_part, float* lse_part, uint32_t* dev_status,
                                 void* stream) {
  const Paging pg{block_table, row_seq, num_seqs, max_blocks, block_size};
  return gather_impl(q, rows, num_q_heads, num_kv_heads, head_dim, fmt, k_cache, v_cache, k_scale_tok, v_scale_tok,
                     k_scale_layer, v_scale_layer, num_slots, topk_pos, topk, softmax_scale, num_splits, out, lse,
                     o_part, lse_part, dev_status, stream, &pg);
}

qkv_status qsa_gather_attn_splitk_fused(const void* q, int64_t rows, int num_q_heads, int num_kv_heads,
                                        int head_dim, qkv_format fmt, const void* k_cache, const void* v_cache,
                                        const float* k_scale_tok, const float* v_scale_tok, float k_scale_layer,
                                        float v_scale_layer, int64_t num_slots, const int32_t* topk_idx, int topk,
                                        float softmax_scale, int num_splits, float* out, float* lse,
                                        float* o_part, float* lse_part, uint32_t* counters, uint32_t* dev_status,
                                        void* stream) {
  if (num_splits == 1)  // unsplit: the kernel writes out / lse itself; no workspace is touched
    return gather_impl(q, rows, num_q_heads, num_kv_heads, head_dim, fmt, k_cache, v_cache, k_scale_tok,
                       v_scale_tok, k_scale_layer, v_scale_layer, num_slots, topk_idx, topk, softmax_scale, 1, out,
                       lse, nullptr, nullptr, dev_status, stream, nullptr);
  if (num_splits > 1 && counters == nullptr) return QKV_ERR_ARG;
  return gather_impl(q, rows, num_q_heads, num_kv_heads, head_dim, fmt, k_cache, v_cache, k_scale_tok, v_scale_tok,
                     k_scale_layer, v_scale_layer, num_slots, topk_idx, topk, softmax_scale, num_splits, out, lse,
                     o_part, lse_part, dev_status, stream, nullptr, counters);
}

qkv_status qsa_suggest_num_splits(qkv_format fmt, int64_t rows, int num_q_heads, int num_kv_heads, int topk,
                                  int* num_splits) {
  if (!num_splits || rows < 0 || topk < 0) return QKV_ERR_ARG;
  if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0) return QKV_ERR_ARG;
  if (num_q_heads / num_kv_heads > kMaxGroup) return QKV_ERR_UNSUPPORTED;
  int per_sm = 0;
  cudaError_t e = cudaErrorInvalidValue;
  switch (fmt) {
    case QKV_BF16:
    case QKV_F16: e = qkv::gather_ctas_per_sm_bf16(&per_sm); break;  // the same 16-bit ring
    case QKV_INT8_SIDE: e = qkv::gather_ctas_per_sm_int8_side(&per_sm); break;
    case QKV_INT8_INLINE: e = qkv::gather_ctas_per_sm_int8_inline(&per_sm); break;
    case QKV_E4M3: e = qkv::gather_ctas_per_sm_e4m3(&per_sm); break;
    default: return QKV_ERR_ARG;
  }
  if (e != cudaSuccess) return QKV_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return QKV_ERR_CUDA;
  const int64_t units = rows * num_kv_heads * ((num_q_heads / num_kv_heads + 15) / 16);  // CTAs per split
  // one wave at up to two CTAs per SM: on the long-context and split-K workloads fewer, longer
  // CTAs per SM beat a third resident CTA (its prologue, epilogue and merge contend)
  const int64_t slots = static_cast<int64_t>(sms) * (per_sm < 1 ? 1 : (per_sm > 2 ? 2 : per_sm));
  int64_t p = units > 0 ? slots / units : 1;
  const int64_t cap = (static_cast<int64_t>(topk) + 127) / 128;  // at least 128 keys (8 tiles) per split
  if (p > cap) p = cap;
  if (p < 1) p = 1;
  *num_splits = static_cast<int>(p);
  return QKV_OK;
}

qkv_status qsa_gather_attn_ex(const qsa_gather_desc* d, void* stream) {
  if (d == nullptr || d->size != sizeof(qsa_gather_desc)) return QKV_ERR_ARG;
  if (d->q_fp16 != 0 && d->q_fp16 != 1) return QKV_ERR_ARG;
  if (d->engine != QSA_ENGINE_DEFAULT && d->engine != QSA_ENGINE_TCGEN05 && d->engine != QSA_ENGINE_PERSISTENT)
    return QKV_ERR_ARG;
  if (d->shard != 0 && d->shard != 1) return QKV_ERR_ARG;
  const bool paged = d->block_table != nullptr;
  if (!paged && d->row_seq != nullptr) return QKV_ERR_ARG;
  const Paging pg{d->block_table, d->row_seq, d->num_seqs, d->max_blocks, d->block_size};
  uint32_t* counters = d->num_splits > 1 ? d->counters : nullptr;  // an unsplit call merges nothing
  return gather_impl(d->q, d->rows, d->num_q_heads, d->num_kv_heads, d->head_dim, d->fmt, d->k_cache, d->v_cache,
                     d->k_scale_tok, d->v_scale_tok, d->k_scale_layer, d->v_scale_layer, d->num_slots, d->topk_idx,
                     d->topk, d->softmax_scale, d->num_splits, d->out, d->lse, d->o_part, d->lse_part, d->dev_status,
                     stream, paged ? &pg : nullptr, counters, d->q_fp16 != 0, d->topk_len, d->engine, d->sched,
                     d->shard != 0, d->slot_lo);
}

qkv_status qsa_splitk_merge(const float* o_part, const float* lse_part, int64_t rows, int num_q_heads,
                            int head_dim, int num_splits, float v_scale_post, float* out, float* lse,
                            void* stream) {
  if (rows < 0 || num_q_heads < 1 || num_splits < 1) return QKV_ERR_ARG;
  if (!qkv::head_dim_ok(head_dim)) return QKV_ERR_UNSUPPORTED;
  if (!std::isfinite(v_scale_post)) return QKV_ERR_ARG;
  if (rows == 0) return QKV_OK;
  if (rows > (int64_t(1) << 32) / num_q_heads) return QKV_ERR_ARG;  // one warp per (row, head): one grid
  if (!o_part || !lse_part || !out) return QKV_ERR_ARG;
  if (!aligned(o_part, 16) || !aligned(out, 16) || !aligned(lse_part, 4) || (lse && !aligned(lse, 4)))
    return QKV_ERR_ALIGN;
  return cuda_status(qkv::launch_splitk_merge(o_part, lse_part, rows, num_q_heads, head_dim, num_splits, v_scale_post,
                                              out, lse, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
