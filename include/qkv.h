/*
 * qkv.h -- C ABI of libqkv.so: quantize-on-write into a KV slot pool and the top-k
 * gather decode attention over it, hand-written for sm_103a (GB300).
 *
 * Pages cited (by title):
 *   [INT8-PR]  "int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next QSA path"
 *   [INT8-KV]  "SuperPUPS/Qwen3.8-Flash-Next-INT8KV" (INT8 KV build, int8_per_token_head)
 *   [E4M3-PR]  "[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache"
 *   [HOIST-PR] "[Perf][SM70][FP8] Hoist QSA E4M3 KV scales"
 *   [SCALES]   "Qwen3.8 Flash Next NVFP4 QSA FP8 E4M3 KV Scales" (model card)
 *
 * Conventions shared by every call
 *   - All tensor arguments are DEVICE pointers owned by the caller; the library never
 *     allocates, frees or synchronises. Work is enqueued on `stream` (a cudaStream_t passed
 *     as void*; NULL = the legacy default stream) and the call returns before it runs.
 *   - Arguments are validated on the host before any launch; an invalid call returns an
 *     error status and enqueues nothing. A launch failure returns QKV_ERR_CUDA.
 *   - Data-dependent problems found on the device (an out-of-range slot or index) are never
 *     trapped: the offending entry is skipped and a bit is OR-ed into the optional
 *     caller-provided device word `dev_status` (may be NULL).
 *   - head_dim must be 256 (256 B of int8 data per head, [INT8-PR §The finding worth
 *     upstreaming]) or 128 (the other common head size; all layouts and entry points).
 *     num_q_heads / num_kv_heads (the GQA group) must be 1..128 (groups above 16 run as one
 *     CTA per 16 query heads, each gathering the row's slots).
 *   - Pool layouts, S = num_slots, H = num_kv_heads, D = head_dim:
 *       QKV_BF16        K, V: bf16 [S, H, D]
 *       QKV_INT8_SIDE   K, V: int8 [S, H, D]; k_scale, v_scale: fp32 [S, H] (side tensors)
 *       QKV_INT8_INLINE K, V: bytes [S, H, D + 4]: D int8 codes then the fp32 scale,
 *                       little-endian (the 260 B record of [INT8-PR]; 132 B for D = 128)
 *       QKV_E4M3        K, V: E4M3 bytes [S, H, D]; one fp32 K and one fp32 V scale per layer
 *       QKV_F16         K, V: IEEE half [S, H, D] (the unquantised cache of the FP16-activation
 *                       contract; gathered with an fp16 query only: qsa_gather_attn_f16, or
 *                       qsa_gather_attn_ex with q_fp16 set)
 *   - Activations (q and new K/V tokens) are bf16; the *_f16 entry points take IEEE half
 *     instead, for the FP16-activation contract of [E4M3-PR §Purpose]. Widening is exact either way.
 */
#ifndef QKV_H
#define QKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QKV_OK = 0,
  QKV_ERR_ARG = 1,         /* null pointer, negative size, bad enum, unsupported shape mix */
  QKV_ERR_SCALE = 2,       /* a per-layer scale that is not finite or is <= 0 */
  QKV_ERR_UNSUPPORTED = 3, /* head_dim not 256 or 128, or GQA group outside 1..128 */
  QKV_ERR_ALIGN = 4,       /* a base pointer or stride breaks the required alignment */
  QKV_ERR_CUDA = 5         /* a kernel launch or attribute call failed */
} qkv_status;

typedef enum {
  QKV_BF16 = 0,
  QKV_INT8_SIDE = 1,
  QKV_INT8_INLINE = 2,
  QKV_E4M3 = 3,
  QKV_F16 = 4 /* unquantised IEEE-half pool; only with an fp16 query (qsa_gather_attn_f16) */
} qkv_format;

/* Bits OR-ed into *dev_status by the kernels. */
#define QKV_DEV_BAD_SLOT 1u  /* a write's slot is invalid (a slot_mapping entry >= num_slots or
                                 < -1, or a bad paged entry, see qkv_write_ex): token skipped */
#define QKV_DEV_BAD_INDEX 2u /* top-k entry >= num_slots or < -1: treated as padding (-1) */
#define QKV_DEV_TIMEOUT 4u   /* a gather CTA's bounded wait for its own copies or tensor-core
                                work ran out (not expected on a healthy GPU): the CTA stopped
                                early, its outputs are incomplete; the kernel returns instead of
                                hanging. Only the tcgen05 engine waits. A test can make it happen:
                                QKV_TEST_TCGEN05_DROP_HANDOFF=<block> in the environment drops
                                that block's hand-off inside each CTA (never set it otherwise) */

/*
 * qkv_write_int8 -- quantize new K/V tokens to int8 with one absmax scale per (token, head)
 * and store them at their slots.            [INT8-PR §The finding worth upstreaming; INT8-KV]
 *
 *   For each token t, KV head h, tensor X in {K, V}:
 *     amax = max_d |x_d| (bf16 widened to fp32), scale = amax / 127 (fp32 IEEE division),
 *     c_d = clamp(rint(x_d / scale), -127, 127) with ties to even; amax == 0 stores scale 0
 *     and zero codes. Codes and scale go to slot slot_mapping[t]; -1 skips the token.
 *
 *   num_tokens * num_kv_heads at most 2^32 (one launch), else QKV_ERR_ARG.
 *   k, v          bf16 [num_tokens, num_kv_heads, head_dim]; token t starts at element
 *                 t * token_stride (token_stride >= num_kv_heads*head_dim, a multiple of 8);
 *                 base pointers 16-byte aligned. Every token's rows are read, a skipped
 *                 token's too (its slot is loaded alongside them, not before).
 *   slot_mapping  int64 [num_tokens]. Slots must be distinct (duplicates race).
 *   layout        QKV_INT8_SIDE: k_cache/v_cache int8 [S,H,D] (16 B-aligned) and
 *                 k_scale/v_scale fp32 [S,H];
 *                 QKV_INT8_INLINE: k_cache/v_cache bytes [S,H,D+4] (16 B-aligned base; the
 *                 records themselves sit on 4 B boundaries), scale pointers must be NULL.
 *   num_slots     S; slots outside [0, S) set QKV_DEV_BAD_SLOT and are skipped.
 * Stored bytes are bit-identical to the CPU oracle's.
 */
qkv_status qkv_write_int8(const void* k, const void* v, int64_t num_tokens, int num_kv_heads,
                          int head_dim, int64_t token_stride, const int64_t* slot_mapping,
                          qkv_format layout, void* k_cache, void* v_cache, float* k_scale,
                          float* v_scale, int64_t num_slots, uint32_t* dev_status,
                          void* stream);

/*
 * qkv_write_e4m3 -- quantize new K/V tokens to FP8 E4M3 with calibrated per-layer scales.
 *                                 [SCALES §Calibration; E4M3-PR §Implementation scope]
 *   stored = e4m3fn(x / scale): the fp32 IEEE quotient rounded to the nearest E4M3 value,
 *   ties to even, magnitudes above 448 saturated to 448, sign kept (-0 -> 0x80).
 *   k_scale, v_scale must be finite and > 0, else QKV_ERR_SCALE (the fail-closed gate of
 *   [E4M3-PR §Non-obvious design decisions]; 1.0 is a legal value).
 *   k, v, token_stride, slot_mapping, num_slots, dev_status as for qkv_write_int8;
 *   k_cache, v_cache: E4M3 bytes [S, H, D], 16 B-aligned.
 */
qkv_status qkv_write_e4m3(const void* k, const void* v, int64_t num_tokens, int num_kv_heads,
                          int head_dim, int64_t token_stride, const int64_t* slot_mapping,
                          void* k_cache, void* v_cache, float k_scale, float v_scale,
                          int64_t num_slots, uint32_t* dev_status, void* stream);

/*
 * qkv_write_int8_f16, qkv_write_e4m3_f16 -- the same writes from IEEE-half tokens (k, v fp16
 * [num_tokens, num_kv_heads, head_dim]) for the FP16-activation contract [E4M3-PR §Purpose].
 * Each half widens exactly to fp32, so the arithmetic, the stored bytes and every other
 * argument are those of qkv_write_int8 / qkv_write_e4m3.
 */
qkv_status qkv_write_int8_f16(const void* k, const void* v, int64_t num_tokens, int num_kv_heads,
                              int head_dim, int64_t token_stride, const int64_t* slot_mapping,
                              qkv_format layout, void* k_cache, void* v_cache, float* k_scale,
                              float* v_scale, int64_t num_slots, uint32_t* dev_status,
                              void* stream);
qkv_status qkv_write_e4m3_f16(const void* k, const void* v, int64_t num_tokens, int num_kv_heads,
                              int head_dim, int64_t token_stride, const int64_t* slot_mapping,
                              void* k_cache, void* v_cache, float k_scale, float v_scale,
                              int64_t num_slots, uint32_t* dev_status, void* stream);

/*
 * qkv_write_ex -- the writes with every option through one descriptor: the format (int8 side,
 * int8 inline or E4M3), bf16 or IEEE-half tokens, and the slot addressing: slot ids
 * (slot_mapping, as qkv_write_int8 / qkv_write_e4m3) or a paged pool, where token t sits at
 * logical position token_pos[t] of sequence token_seq[t] and its slot is
 *     block_table[seq, pos / block_size] * block_size + pos % block_size
 * (the addressing qsa_gather_attn_paged reads; [E4M3-PR §Implementation scope]: the KV cache
 * is paged storage). Arithmetic and stored bytes are those of qkv_write_int8 / qkv_write_e4m3.
 *   size           sizeof(qkv_write_desc), for the layout check (else QKV_ERR_ARG).
 *   fmt            QKV_INT8_SIDE (k_scale, v_scale fp32 [S, H]), QKV_INT8_INLINE (scale
 *                  pointers NULL) or QKV_E4M3 (k_scale_layer, v_scale_layer finite and > 0,
 *                  else QKV_ERR_SCALE; scale pointers NULL); anything else QKV_ERR_ARG.
 *   act_fp16       0: k, v bf16; 1: IEEE half.
 *   slot_mapping   int64 [num_tokens] slot ids, -1 = skip; NULL selects paged addressing, and
 *                  then token_seq, token_pos (int32 [num_tokens]) and block_table (int32
 *                  [num_seqs, max_blocks], < 0 = unallocated) are required (4 B-aligned),
 *                  with block_size >= 1, max_blocks >= 1, num_seqs >= 1 and
 *                  max_blocks * block_size < 2^31. Giving both addressings is QKV_ERR_ARG.
 *                  A position of -1 skips the token. A position outside [-1, max_blocks *
 *                  block_size), a sequence outside [0, num_seqs), an unallocated block or a
 *                  slot outside [0, S) set QKV_DEV_BAD_SLOT and skip the token.
 *   the rest       as for qkv_write_int8 / qkv_write_e4m3.
 */
typedef struct {
  size_t size;
  qkv_format fmt;
  int act_fp16;
  const void* k;
  const void* v;
  int64_t num_tokens;
  int num_kv_heads;
  int head_dim;
  int64_t token_stride;
  const int64_t* slot_mapping;
  const int32_t* token_seq;
  const int32_t* token_pos;
  const int32_t* block_table;
  int64_t num_seqs;
  int max_blocks;
  int block_size;
  void* k_cache;
  void* v_cache;
  float* k_scale;
  float* v_scale;
  float k_scale_layer;
  float v_scale_layer;
  int64_t num_slots;
  uint32_t* dev_status;
} qkv_write_desc;

qkv_status qkv_write_ex(const qkv_write_desc* desc, void* stream);

/*
 * qkv_e4m3_calibrate -- per-tensor calibrated E4M3 scale = (max |x|) / 448 over n bf16
 * values, computed on the device.                             [SCALES §Calibration]
 *   x          bf16 [n], 16 B-aligned.
 *   amax_bits  device uint32 [1]: scratch that receives the fp32 bits of max|x| (the call
 *              clears it first with a memset on `stream`).
 *   scale_out  device fp32 [1]: amax / 448 (fp32 IEEE division). 0 when every x is 0.
 */
qkv_status qkv_e4m3_calibrate(const void* x, int64_t n, uint32_t* amax_bits, float* scale_out,
                              void* stream);

/*
 * Calibration statistics of one K or V tensor (one layer's K, say), computed on the device.
 *                       [SCALES §Calibration: scale = max envelope / 448, and max-abs,
 *                        p99.9, p99.99 and saturation per tensor; E4M3-PR §Why calibrated
 *                        scale is part of this contract: nonzero elements below E4M3's
 *                        smallest subnormal 2^-9 and in the subnormal band below 2^-6]
 *
 * qkv_calib_histogram adds the counts of the 16-bit magnitudes (bits & 0x7FFF) of x to hist.
 * Calls accumulate, so one histogram can cover a tensor seen over many steps; zero hist
 * before the first call. A bf16 magnitude has 15 bits, so the histogram is exact.
 *   x      bf16 (or IEEE half) [n], 16 B-aligned (n may be 0; n <= 2^40).
 *   hist   uint64 [QKV_CALIB_BINS], 8 B-aligned, owned by the caller.
 *
 * qkv_calib_stats reads a histogram and writes one qkv_calib_summary record (device memory):
 *   count            finite elements; zeros: elements equal to +-0; nonfinite: inf / NaN
 *                    elements (they take part in nothing else)
 *   amax             max |x| over the finite elements
 *   p99_9, p99_99    nearest-rank percentiles of |x| over the finite elements: with the
 *                    magnitudes sorted ascending, element ceil(q count), q = 999/1000 and
 *                    9999/10000 as exact fractions (0 when count is 0)
 *   scale            the scale the counts below refer to: `scale` when it is > 0, or, when
 *                    `scale` is 0, the calibrated amax / 448 (fp32 IEEE division)
 *   With y = |x| / scale (fp32 IEEE division) for each finite element:
 *   below_subnormal  nonzero elements with y < 2^-9
 *   subnormal        elements with 2^-9 <= y < 2^-6
 *   saturated        elements with y > 464: the ones the saturating encoder clips, whose
 *                    nearest value on the E4M3 grid continued past 448 would be above 448
 *                    (so at the calibrated scale it is always 0)
 *   A scale of 0 (an all-zero tensor) leaves those three counts at 0.
 *   scale  0 or finite and > 0, else QKV_ERR_SCALE.
 */
#define QKV_CALIB_BINS 32768
typedef struct {
  uint64_t count;
  uint64_t zeros;
  uint64_t nonfinite;
  uint64_t below_subnormal;
  uint64_t subnormal;
  uint64_t saturated;
  float amax;
  float p99_9;
  float p99_99;
  float scale;
} qkv_calib_summary;

qkv_status qkv_calib_histogram(const void* x, int64_t n, uint64_t* hist, void* stream);
qkv_status qkv_calib_stats(const uint64_t* hist, float scale, qkv_calib_summary* stats, void* stream);
/* The same for a histogram of IEEE-half values (the histogram call counts 15-bit magnitudes of
 * either type; only the bins' values differ). */
qkv_status qkv_calib_stats_f16(const uint64_t* hist, float scale, qkv_calib_summary* stats, void* stream);

/*
 * qsa_gather_attn -- top-k gather decode attention over a quantized slot pool.
 *                       [INT8-PR §The finding worth upstreaming; HOIST-PR §Changes]
 *   For row r, query head g (KV head g / G, G = num_q_heads / num_kv_heads) and the valid
 *   entries j of topk_idx[r, :] (-1 = padding):
 *     s_j = softmax_scale * q[r,g,:] . K_j,   o = sum_j softmax(s)_j V_j,
 *     lse = log sum_j exp(s_j)  (natural log; a row with no valid entry gives o = 0,
 *     lse = -inf). K_j / V_j are the dequantized slots: int8 c * per-(slot,head) scale,
 *     E4M3 dec(c) * per-layer scale, or bf16 values.
 *   Scale hoisting: the K scale multiplies the dot product, not each element (per slot for
 *   int8, folded into the softmax factor for E4M3); the int8 V scale multiplies p_j; the
 *   E4M3 V scale is applied once after normalisation -- or, when num_splits > 1, left to
 *   qsa_splitk_merge (pass v_scale_layer as its v_scale_post).
 *
 *   q             bf16 [rows, num_q_heads, head_dim], contiguous, 16 B-aligned.
 *   fmt           pool layout (see above); QKV_F16 is QKV_ERR_ARG here (qsa_gather_attn_f16).
 *                 k_cache / v_cache base pointers 16 B-aligned. S * num_kv_heads must stay
 *                 <= 2^31 - 1 (else QKV_ERR_UNSUPPORTED).
 *   k_scale_tok, v_scale_tok  fp32 [S, H] for QKV_INT8_SIDE, else must be NULL.
 *   k_scale_layer, v_scale_layer  per-layer scales for QKV_E4M3 (finite, > 0, else
 *                 QKV_ERR_SCALE); ignored for the other formats.
 *   topk_idx      int32 [rows, topk] slot ids, -1 = padding; entries outside [-1, S) set
 *                 QKV_DEV_BAD_INDEX and are treated as padding. Duplicates count twice.
 *   softmax_scale finite.
 *   num_splits    P >= 1. Split s covers index columns [s*c, min(topk, (s+1)*c)),
 *                 c = ceil(topk / P) ([E4M3-PR §Implementation scope]: split-K workspace).
 *   P == 1: out fp32 [rows, num_q_heads, head_dim] and optional lse fp32 [rows, num_q_heads]
 *           (NULL to skip); o_part / lse_part must be NULL.
 *   P > 1:  o_part fp32 [rows, P, num_q_heads, head_dim] and lse_part fp32
 *           [rows, P, num_q_heads] receive the normalised per-split partials (E4M3: without
 *           the V scale); out / lse must be NULL; follow with qsa_splitk_merge.
 */
qkv_status qsa_gather_attn(const void* q, int64_t rows, int num_q_heads, int num_kv_heads,
                           int head_dim, qkv_format fmt, const void* k_cache,
                           const void* v_cache, const float* k_scale_tok,
                           const float* v_scale_tok, float k_scale_layer, float v_scale_layer,
                           int64_t num_slots, const int32_t* topk_idx, int topk,
                           float softmax_scale, int num_splits, float* out, float* lse,
                           float* o_part, float* lse_part, uint32_t* dev_status, void* stream);

/*
 * qsa_gather_attn_varlen -- qsa_gather_attn for rows of different lengths: row r's valid
 * entries are topk_idx[r, 0 .. topk_len[r]); the entries past that length are never read (they
 * may hold anything). A batch that mixes long and short rows (the pages route such mixed
 * catch-up / decode batches across kernels, [E4M3-PR §Implementation scope]) then costs only
 * its valid entries. Inside the length, -1 is still padding.
 *   topk_len  int32 [rows], each in [0, topk]; a value outside is flagged with
 *             QKV_DEV_BAD_INDEX and clamped. NULL is QKV_ERR_ARG (use qsa_gather_attn).
 *   The split partition stays over the full width topk (split s covers columns
 *   [s c, (s + 1) c), c = ceil(topk / P)), so a short row's trailing splits are empty
 *   (o = 0, lse = -inf). Everything else as qsa_gather_attn; the result equals qsa_gather_attn
 *   on topk_idx with the entries past each row's length set to -1.
 */
qkv_status qsa_gather_attn_varlen(const void* q, int64_t rows, int num_q_heads, int num_kv_heads,
                                  int head_dim, qkv_format fmt, const void* k_cache,
                                  const void* v_cache, const float* k_scale_tok,
                                  const float* v_scale_tok, float k_scale_layer,
                                  float v_scale_layer, int64_t num_slots, const int32_t* topk_idx,
                                  int topk, const int32_t* topk_len, float softmax_scale,
                                  int num_splits, float* out, float* lse, float* o_part,
                                  float* lse_part, uint32_t* dev_status, void* stream);

/*
 * qsa_gather_attn_f16 -- qsa_gather_attn with an IEEE-half query, for the FP16-activation
 * contract [E4M3-PR §Purpose]. q fp16 [rows, num_q_heads, head_dim]; fmt one of
 * QKV_INT8_SIDE, QKV_INT8_INLINE, QKV_E4M3 or QKV_F16 (a half pool); QKV_BF16 is
 * QKV_ERR_ARG (a bf16 pool takes a bf16 query). Everything else -- splits, outputs, errors --
 * as qsa_gather_attn.
 */
qkv_status qsa_gather_attn_f16(const void* q, int64_t rows, int num_q_heads, int num_kv_heads,
                               int head_dim, qkv_format fmt, const void* k_cache,
                               const void* v_cache, const float* k_scale_tok,
                               const float* v_scale_tok, float k_scale_layer, float v_scale_layer,
                               int64_t num_slots, const int32_t* topk_idx, int topk,
                               float softmax_scale, int num_splits, float* out, float* lse,
                               float* o_part, float* lse_part, uint32_t* dev_status, void* stream);

/*
 * qsa_splitk_merge -- merge split-K partials.      [HOIST-PR §Changes: the V scale is
 *                                                    applied once after the merge]
 *   lse = log sum_s exp(lse_s), o = v_scale_post * sum_s exp(lse_s - lse) o_s.
 *   Rows whose splits are all empty (lse_s = -inf) give o = 0, lse = -inf.
 *   o_part fp32 [rows, P, num_q_heads, head_dim], lse_part fp32 [rows, P, num_q_heads],
 *   out fp32 [rows, num_q_heads, head_dim], lse fp32 [rows, num_q_heads] or NULL.
 *   v_scale_post finite (1.0 for the non-E4M3 formats). head_dim 256 or 128.
 *   rows * num_q_heads at most 2^32 (one launch), else QKV_ERR_ARG.
 */
qkv_status qsa_splitk_merge(const float* o_part, const float* lse_part, int64_t rows,
                            int num_q_heads, int head_dim, int num_splits, float v_scale_post,
                            float* out, float* lse, void* stream);

/*
 * qsa_gather_attn_splitk_fused -- qsa_gather_attn with num_splits > 1 and the split-K merge
 * fused into the same launch.     [E4M3-PR §Implementation scope: split-K workspace and merge;
 *                                  HOIST-PR §Changes: the V scale is applied after the merge]
 *   Every split CTA of a (row, KV head) writes its partial to o_part / lse_part exactly as
 *   qsa_gather_attn does, then increments the counter of its (row, KV head, chunk of 16 query
 *   heads). The CTA that brings the counter to num_splits merges the num_splits partials of
 *   those heads into out / lse (E4M3: times v_scale_layer) and resets the counter to 0. No CTA
 *   waits for another. The result is bit-identical to qsa_gather_attn followed by
 *   qsa_splitk_merge on the same partials; it saves the second launch and its gap.
 *
 *   Arguments as qsa_gather_attn, plus:
 *   out        fp32 [rows, num_q_heads, head_dim] (16 B-aligned) and lse fp32
 *              [rows, num_q_heads] or NULL: the merged result.
 *   o_part, lse_part  the split workspace, laid out as for qsa_gather_attn; left holding the
 *              partials.
 *   counters   uint32 [rows, num_kv_heads, ceil(G / 16)] (G = num_q_heads / num_kv_heads),
 *              4 B-aligned, owned by the caller. They must all be 0 before the first call;
 *              every call leaves them 0 again.
 *   num_splits == 1 runs the unsplit kernel (o_part, lse_part and counters are not touched and
 *   may be NULL). num_splits > 1 with counters NULL is QKV_ERR_ARG.
 *   Calls that overlap on the GPU must not share counters or workspace.
 */
qkv_status qsa_gather_attn_splitk_fused(const void* q, int64_t rows, int num_q_heads, int num_kv_heads,
                                        int head_dim, qkv_format fmt, const void* k_cache,
                                        const void* v_cache, const float* k_scale_tok,
                                        const float* v_scale_tok, float k_scale_layer,
                                        float v_scale_layer, int64_t num_slots,
                                        const int32_t* topk_idx, int topk, float softmax_scale,
                                        int num_splits, float* out, float* lse, float* o_part,
                                        float* lse_part, uint32_t* counters, uint32_t* dev_status,
                                        void* stream);

/*
 * qsa_suggest_num_splits -- a split count for a gather launch of this shape on the current
 * device: enough splits to fill one wave of resident CTAs, so that a launch with few rows
 * still spreads over every SM.       [E4M3-PR §Implementation scope: split-K workspace; the
 *                                     pages tune the partition per route, P256 / P1024]
 *   P = floor(SMs * C / (rows * num_kv_heads * ceil(G / 16))), at most ceil(topk / 128) (at
 *   least 8 tiles of 16 keys per split) and at least 1, where C is the occupancy of the
 *   layout's gather kernel (CTAs per SM) capped at 2. Any P gives the same result up to
 *   rounding.
 *   Host-only (queries the device, launches nothing). Errors as qsa_gather_attn's shape checks;
 *   a failed device query is QKV_ERR_CUDA.
 */
qkv_status qsa_suggest_num_splits(qkv_format fmt, int64_t rows, int num_q_heads, int num_kv_heads,
                                  int topk, int* num_splits);

/*
 * qsa_gather_attn_splitk_noalloc -- qsa_gather_attn with num_splits > 1 followed by
 * qsa_splitk_merge, for callers that cannot allocate device memory. The pages have no
 * counterpart: this is a packaging of the two calls above, not a step of the method.
 *
 *   Some callers own only their inputs and outputs -- e.g. a plugin inside a host engine
 *   that receives pre-allocated tensors and may not call cudaMalloc while serving (an
 *   allocation can synchronise the device and fragments the host's memory pool). They
 *   cannot supply the o_part / lse_part workspace of a split call. This entry point keeps
 *   the partials in a file-scope static device array of QKV_NOALLOC_SCRATCH_BYTES instead,
 *   and calls no cudaMalloc, cudaFree or other allocating routine.
 *
 *   Arguments are those of qsa_gather_attn, minus o_part / lse_part; out fp32
 *   [rows, num_q_heads, head_dim] (16 B-aligned) and optional lse fp32 [rows, num_q_heads]
 *   receive the merged result (E4M3: v_scale_layer applied after the merge). num_splits == 1
 *   is forwarded to qsa_gather_attn unchanged.
 *   Limit: rows * num_splits * num_q_heads * (head_dim + 1) * 4 bytes (lse part rounded up to
 *   256 B) must fit in QKV_NOALLOC_SCRATCH_BYTES (16 MiB: e.g. 64 rows x 8 splits x 16 heads,
 *   or 40 rows x 16 splits x 16 heads); larger calls return QKV_ERR_ARG and launch nothing.
 *   Set-up: the first call on each device looks up the array's device address with
 *   cudaGetSymbolAddress while that device is current; make that first call before any
 *   stream capture. The cached address belongs to the device's current context: do not keep
 *   using the library across cudaDeviceReset (or any other teardown of the primary context),
 *   since the next call would reuse the old address. The array is held by every GPU that loads
 *   the library until the process exits. All calls share it and it keeps the last call's partials (every partial is
 *   rewritten before it is read, so nothing needs clearing): calls that overlap on the GPU --
 *   on different streams or from different host threads -- race and corrupt each other.
 */
#define QKV_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
qkv_status qsa_gather_attn_splitk_noalloc(const void* q, int64_t rows, int num_q_heads, int num_kv_heads,
                                          int head_dim, qkv_format fmt, const void* k_cache,
                                          const void* v_cache, const float* k_scale_tok,
                                          const float* v_scale_tok, float k_scale_layer,
                                          float v_scale_layer, int64_t num_slots,
                                          const int32_t* topk_idx, int topk, float softmax_scale,
                                          int num_splits, float* out, float* lse,
                                          uint32_t* dev_status, void* stream);

/*
 * qsa_gather_attn_paged -- qsa_gather_attn over a paged pool: rows give logical token
 * positions in their sequence, and the kernel maps them to slots through a block table.
 *                       [E4M3-PR §Implementation scope: the KV reads run over paged
 *                        ("page4") storage; the block-table interface is the usual
 *                        vLLM-style one, not defined on the pages]
 *   For row r with sequence s = row_seq[r] and entry p = topk_pos[r, j]:
 *     slot = block_table[s * max_blocks + p / block_size] * block_size + p % block_size,
 *   then exactly as qsa_gather_attn with that slot. p = -1 is padding. These are flagged
 *   with QKV_DEV_BAD_INDEX and treated as padding: p < -1 or p >= max_blocks * block_size,
 *   a block id < 0 (unallocated), and a slot >= num_slots. A row whose s lies outside
 *   [0, num_seqs) is flagged once and is empty (o = 0, lse = -inf).
 *   block_table  int32 [num_seqs, max_blocks], block ids in units of block_size slots.
 *   row_seq      int32 [rows].
 *   topk_pos     int32 [rows, topk].
 *   block_size   >= 1; max_blocks >= 1; num_seqs >= 1; max_blocks * block_size < 2^31.
 *   Everything else -- formats, scales, splits, outputs, errors -- as qsa_gather_attn. The
 *   result equals qsa_gather_attn on the translated slot ids, bit for bit.
 */
qkv_status qsa_gather_attn_paged(const void* q, int64_t rows, int num_q_heads, int num_kv_heads,
                                 int head_dim, qkv_format fmt, const void* k_cache,
                                 const void* v_cache, const float* k_scale_tok,
                                 const float* v_scale_tok, float k_scale_layer, float v_scale_layer,
                                 int64_t num_slots, const int32_t* block_table, int64_t num_seqs,
                                 int max_blocks, int block_size, const int32_t* row_seq,
                                 const int32_t* topk_pos, int topk, float softmax_scale,
                                 int num_splits, float* out, float* lse, float* o_part,
                                 float* lse_part, uint32_t* dev_status, void* stream);

/*
 * qsa_gather_attn_ex -- one entry point for every combination of the gather's options: the
 * plain call's arguments plus, each optional, per-row lengths (varlen), a paged pool (block
 * table), the fused split-K merge (arrival counters) and an IEEE-half query. The operations
 * are those of qsa_gather_attn, qsa_gather_attn_varlen, qsa_gather_attn_paged,
 * qsa_gather_attn_splitk_fused and qsa_gather_attn_f16 [INT8-PR §The finding worth
 * upstreaming; HOIST-PR §Changes; E4M3-PR §Implementation scope, §Purpose], and the same
 * arguments mean the same things, with the same errors.
 *   size        sizeof(qsa_gather_desc), for the layout check (else QKV_ERR_ARG).
 *   q_fp16      0: bf16 query; 1: IEEE-half query (formats as for qsa_gather_attn_f16).
 *   topk_len    NULL, or int32 [rows] valid entries per row (qsa_gather_attn_varlen).
 *   block_table NULL, or a paged pool (qsa_gather_attn_paged: num_seqs, max_blocks,
 *               block_size, row_seq); topk_idx then holds positions. Paged pools take a bf16
 *               query (q_fp16 = 1 with a block table is QKV_ERR_ARG).
 *   counters    NULL, or the fused merge's arrival counters (qsa_gather_attn_splitk_fused);
 *               with num_splits > 1, out (and optionally lse) then receive the merged result
 *               and o_part / lse_part are the workspace.
 *   engine      QSA_ENGINE_DEFAULT, or QSA_ENGINE_TCGEN05: the same gather with q.K^T on the
 *               fifth-generation tensor cores (tcgen05.mma, K dequantised into tensor memory)
 *               in a warp-specialised CTA. It computes the same result to the same tolerance
 *               and is slower on GB300 (the tensor-memory MMA issue rate bounds it); only
 *               QKV_INT8_SIDE, head_dim 256, G <= 16, a bf16 query, no block table and no
 *               counters, else QKV_ERR_UNSUPPORTED. QSA_ENGINE_PERSISTENT: the default
 *               kernels on a persistent grid -- as many CTAs as stay resident, each taking
 *               the next free work item (row, KV head, 16-head chunk, split) from the counter
 *               sched[0] until none is left; no CTA waits for another. Any combination of the
 *               options above. Any other value is QKV_ERR_ARG.
 *   sched       QSA_ENGINE_PERSISTENT only (ignored otherwise): uint32 [2] on the device,
 *               zero before the first call (cudaMemset); every launch leaves it zero again.
 *               One launch at a time per sched buffer. NULL with that engine: QKV_ERR_ARG;
 *               not 4-byte aligned: QKV_ERR_ALIGN.
 *   shard       0, or 1: this pool is one shard of a pool split by slot range. It holds the
 *               global slots [slot_lo, slot_lo + num_slots) at local ids 0 .. num_slots - 1;
 *               topk_idx holds global slot ids, and an entry outside the shard's range is
 *               another shard's: skipped, not flagged (entries below -1 are still flagged).
 *               The output (out / lse, or the partials) is this shard's normalised partial and
 *               its lse: qsa_splitk_merge over the shards' partials gives the attention over the
 *               whole pool (the E4M3 V scale is applied inside each shard's unsplit output, so
 *               the cross-shard merge takes v_scale_post = 1). Not with a block table or the
 *               tcgen05 engine (QKV_ERR_ARG / QKV_ERR_UNSUPPORTED); any other value: QKV_ERR_ARG.
 *   slot_lo     shard only: the first global slot id of this shard, 0 <= slot_lo <= 2^31 - 1.
 */
#define QSA_ENGINE_DEFAULT 0
#define QSA_ENGINE_TCGEN05 1
#define QSA_ENGINE_PERSISTENT 2

typedef struct {
  size_t size;
  const void* q;
  int q_fp16;
  int64_t rows;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  qkv_format fmt;
  const void* k_cache;
  const void* v_cache;
  const float* k_scale_tok;
  const float* v_scale_tok;
  float k_scale_layer;
  float v_scale_layer;
  int64_t num_slots;
  const int32_t* topk_idx;
  int topk;
  float softmax_scale;
  int num_splits;
  float* out;
  float* lse;
  float* o_part;
  float* lse_part;
  uint32_t* dev_status;
  const int32_t* topk_len;
  const int32_t* block_table;
  int64_t num_seqs;
  int max_blocks;
  int block_size;
  const int32_t* row_seq;
  uint32_t* counters;
  int engine;
  uint32_t* sched;
  int shard;
  int64_t slot_lo;
} qsa_gather_desc;

qkv_status qsa_gather_attn_ex(const qsa_gather_desc* desc, void* stream);

/* Static, human-readable name of a status code. Never NULL. */
const char* qkv_status_str(qkv_status s);

#ifdef __cplusplus
}
#endif

#endif /* QKV_H */
