// Top-k gather decode attention over a quantized slot pool (sm_103a).
//
// Pages: "int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next QSA path" §The finding
// worth upstreaming (each query row gathers its top-k scattered slots; side-tensor vs
// inline 260 B scales); "[Perf][SM70][FP8] Hoist QSA E4M3 KV scales" §Changes (K scale in
// the post-dot softmax factor, V scale once after normalised accumulation or after the
// split-K merge); "[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache" §Implementation
// scope (split-K workspace).
//
// Work decomposition: one CTA (4 warps) per (query row, KV head, K-split). The split's
// index columns are staged in shared memory in chunks of kIdxCap, padding (-1) and bad
// entries are dropped by a block-wide stream compaction, and the surviving slots are
// streamed in tiles of kTile = 64 keys through a kStages-deep cp.async pipeline (16 B
// copies; the 256 B / 512 B rows land XOR-swizzled so every fragment read below is
// bank-conflict free).
//
// Per tile:
//   q.K^T  warp w owns keys [16w, 16w+16): mma.sync m16n8k16 with M = the GQA group (16
//          query heads, padded), N = 8 keys, K = 16 head dims. The query fragments stay in
//          registers for the whole CTA; the key codes are dequantised straight into the B
//          fragments (int8 -> fp16 by an exponent splice, E4M3 -> fp16 by the native cvt,
//          bf16 as stored), so no dequantised copy is ever written back to shared memory.
//          The head-dim order inside a fragment is permuted to match how a code word
//          unpacks; the query fragments use the same permutation, so the dot product is
//          unchanged.
//   softmax  logits are scaled by the hoisted K scale (per slot for int8, folded into the
//          per-head factor for E4M3), a cross-warp max exchange gives the tile max, and
//          p = exp2(s - m) goes to shared memory as a hi + lo pair (fp16 for int8/E4M3, bf16
//          for the bf16 layout), so p keeps ~22 (~17) bits: with outlier tokens a row can be
//          a near-even mix of two large V rows of opposite sign, and single-fp16 p then loses
//          ~1e-3 of the result to cancellation. int8 p also carries the slot's V scale and a
//          power of two that keeps every value a normal fp16.
//   p.V    warp w owns head dims [64w, 64w+64): A = p (ldmatrix), B = V codes dequantised
//          in registers, fp32 accumulators rescaled on a new max.
// The E4M3 V scale (and the power-of-two pre-scale) is applied once at the end; split
// partials are written normalised, without the E4M3 V scale.
#pragma once

#include "qkv_internal.cuh"

namespace qkv {
namespace gather {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kTile = 64;
constexpr int kIdxCap = 1024;
constexpr int kIdxPerThread = kIdxCap / kThreads;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kPShift = 14;  // p * 2^14 keeps p >= 2^-28 a normal fp16

template <int FMT>
struct Fmt;
template <>
struct Fmt<QKV_INT8_SIDE> {
  static constexpr int kRowBytes = 256, kGlobalRow = 256, kChunks = 16, kStages = 3, kMinBlocks = 2;
  static constexpr bool kInt8 = true, kSide = true, kInline = false, kE4m3 = false, kBf16 = false;
};
template <>
struct Fmt<QKV_INT8_INLINE> {
  // 17 aligned 16 B chunks cover any 260 B record that starts on a 4 B boundary.
  static constexpr int kRowBytes = 272, kGlobalRow = kInlineRecord, kChunks = 17, kStages = 3, kMinBlocks = 2;
  static constexpr bool kInt8 = true, kSide = false, kInline = true, kE4m3 = false, kBf16 = false;
};
template <>
struct Fmt<QKV_E4M3> {
  static constexpr int kRowBytes = 256, kGlobalRow = 256, kChunks = 16, kStages = 3, kMinBlocks = 2;
  static constexpr bool kInt8 = false, kSide = false, kInline = false, kE4m3 = true, kBf16 = false;
};
template <>
struct Fmt<QKV_BF16> {
  static constexpr int kRowBytes = 512, kGlobalRow = 512, kChunks = 32, kStages = 3, kMinBlocks = 1;
  static constexpr bool kInt8 = false, kSide = false, kInline = false, kE4m3 = false, kBf16 = true;
};

template <int FMT>
struct Smem {
  using F = Fmt<FMT>;
  static constexpr size_t kKV = size_t(F::kStages) * kTile * F::kRowBytes;  // one of K / V
  static constexpr size_t kScale = F::kSide ? size_t(F::kStages) * kTile * 4 : 0;
  static constexpr size_t kK = 0;
  static constexpr size_t kV = kK + kKV;
  static constexpr size_t kKs = kV + kKV;
  static constexpr size_t kVs = kKs + kScale;
  static constexpr size_t kIdx = kVs + kScale;
  static constexpr size_t kP = kIdx + kIdxCap * 4;
  static constexpr size_t kPBytes = 2 * 16 * kTile * 2;  // hi and lo halves of p
  static constexpr size_t kRed = kP + kPBytes;  // [kWarps][16] floats
  static constexpr size_t kVmax = kRed + kWarps * 16 * 4;
  static constexpr size_t kCnt = kVmax + kWarps * 4;
  static constexpr size_t kTotal = kCnt + (kWarps + 4) * 4;
};

// Shared-memory 16 B chunk position of chunk j of tile row `row`.
template <int FMT>
__device__ __forceinline__ int swz_k(int j, int row) {
  if (Fmt<FMT>::kInline) return j;
  if (Fmt<FMT>::kBf16) return j ^ (row & 1);
  return j ^ ((row & 1) << 2);
}
template <int FMT>
__device__ __forceinline__ int swz_v(int j, int row) {
  if (Fmt<FMT>::kInline) return j;
  return j ^ (row & 6);
}

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// Stage index columns [cs, ce) of row r into sIdx, dropping -1 and out-of-range entries
// (the latter also flag QKV_DEV_BAD_INDEX). Order is kept. Returns the number kept.
__device__ __forceinline__ int stage_indices(const GatherArgs& a, int64_t r, int cs, int ce, int32_t* sIdx,
                                             int* sCnt, int tid, int lane, int warp) {
  const int n = ce - cs;
  const int32_t* src = a.topk_idx + r * a.topk + cs;
  int vals[kIdxPerThread];
  int cnt = 0;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kIdxPerThread; ++i) {
    const int j = tid * kIdxPerThread + i;
    int v = (j < n) ? __ldg(src + j) : -1;
    if (v < -1 || static_cast<int64_t>(v) >= a.num_slots) {
      bad = true;
      v = -1;
    }
    vals[i] = v;
    cnt += (v >= 0);
  }
  if (bad && a.dev_status != nullptr) atomicOr(a.dev_status, QKV_DEV_BAD_INDEX);
  int x = cnt;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) sCnt[warp] = x;
  __syncthreads();
  int base = x - cnt, total = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int cw = sCnt[w];
    base += (w < warp) ? cw : 0;
    total += cw;
  }
#pragma unroll
  for (int i = 0; i < kIdxPerThread; ++i)
    if (vals[i] >= 0) sIdx[base++] = vals[i];
  __syncthreads();
  return total;
}

// Issue the cp.async copies of one tile (K rows, V rows, side scales) into stage `st`.
template <int FMT>
__device__ __forceinline__ void issue_tile(const GatherArgs& a, int h, const int32_t* sIdx, int tile_base,
                                           int nvalid, uint8_t* smem, int st, int tid) {
  using F = Fmt<FMT>;
  using L = Smem<FMT>;
  const int kk = tid >> 1, half = tid & 1;
  const int key = tile_base + kk;
  const bool valid = key < nvalid;
  const int64_t slot = valid ? sIdx[key] : 0;
  const int64_t rec = slot * a.num_kv_heads + h;
  const uint32_t dK = smem_u32(smem + L::kK + (size_t(st) * kTile + kk) * F::kRowBytes);
  const uint32_t dV = smem_u32(smem + L::kV + (size_t(st) * kTile + kk) * F::kRowBytes);
  if (F::kInline) {
    const int64_t off = rec * F::kGlobalRow;
    const int64_t al = off & ~int64_t(15);
    const int delta = static_cast<int>(off - al);
    const uint8_t* gK = a.k_cache + al;
    const uint8_t* gV = a.v_cache + al;
    constexpr int kFirst = (F::kChunks + 1) / 2;  // 9 chunks for half 0, 8 for half 1
    const int j0 = half ? kFirst : 0, j1 = half ? F::kChunks : kFirst;
    for (int j = j0; j < j1; ++j) {
      // the last chunk copies only the record's own bytes (never past the pool's end)
      const int nb = valid ? (j == F::kChunks - 1 ? delta + 4 : 16) : 0;
      cp_async16(dK + j * 16, gK + j * 16, nb);
      cp_async16(dV + j * 16, gV + j * 16, nb);
    }
  } else {
    const uint8_t* gK = a.k_cache + rec * F::kGlobalRow;
    const uint8_t* gV = a.v_cache + rec * F::kGlobalRow;
    const int nb = valid ? 16 : 0;
    constexpr int kHalf = F::kChunks / 2;
#pragma unroll
    for (int i = 0; i < kHalf; ++i) {
      const int j = half * kHalf + i;
      cp_async16(dK + swz_k<FMT>(j, kk) * 16, gK + j * 16, nb);
      cp_async16(dV + swz_v<FMT>(j, kk) * 16, gV + j * 16, nb);
    }
    if (F::kSide) {
      const float* gs = half ? a.v_scale_tok : a.k_scale_tok;
      const size_t so = half ? L::kVs : L::kKs;
      cp_async4(smem_u32(smem + so + (size_t(st) * kTile + kk) * 4), gs + rec, valid ? 4 : 0);
    }
  }
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, Fmt<FMT>::kMinBlocks) gather_attn_kernel(const GatherArgs a) {
  using F = Fmt<FMT>;
  using L = Smem<FMT>;
  extern __shared__ __align__(1024) uint8_t smem[];
  int32_t* sIdx = reinterpret_cast<int32_t*>(smem + L::kIdx);
  float* sRed = reinterpret_cast<float*>(smem + L::kRed);
  float* sVmax = reinterpret_cast<float*>(smem + L::kVmax);
  int* sCnt = reinterpret_cast<int*>(smem + L::kCnt);
  const uint32_t sP = smem_u32(smem + L::kP);
  const uint32_t sPlo = sP + 16 * kTile * 2;  // low halves of p

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = lane & 3, hn = lane >> 2;
  const int h0 = hn, h1 = hn + 8;
  const int P = a.num_splits, H = a.num_kv_heads, Hq = a.num_q_heads, G = Hq / H;
  const int64_t bid = blockIdx.x;
  const int split = static_cast<int>(bid % P);
  const int64_t rh = bid / P;
  const int h = static_cast<int>(rh % H);
  const int64_t r = rh / H;
  const int per_split = (a.topk + P - 1) / P;
  const int col0 = min(a.topk, split * per_split);
  const int col1 = min(a.topk, col0 + per_split);

  // ---------------- query fragments (registers for the whole CTA)
  uint32_t qf[16][4];
  float fac0, fac1;  // log2-domain logit factor of heads h0, h1
  {
    const __nv_bfloat16* qb = a.q + (r * Hq + static_cast<int64_t>(h) * G) * kHeadDim;
    uint32_t w0[4][8], w1[4][8];
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
      uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0, y0 = x0, y1 = x0;
      if (h0 < G) {
        const uint4* p = reinterpret_cast<const uint4*>(qb + h0 * kHeadDim + 64 * blk + 16 * c);
        x0 = __ldg(p);
        x1 = __ldg(p + 1);
      }
      if (h1 < G) {
        const uint4* p = reinterpret_cast<const uint4*>(qb + h1 * kHeadDim + 64 * blk + 16 * c);
        y0 = __ldg(p);
        y1 = __ldg(p + 1);
      }
      w0[blk][0] = x0.x; w0[blk][1] = x0.y; w0[blk][2] = x0.z; w0[blk][3] = x0.w;
      w0[blk][4] = x1.x; w0[blk][5] = x1.y; w0[blk][6] = x1.z; w0[blk][7] = x1.w;
      w1[blk][0] = y0.x; w1[blk][1] = y0.y; w1[blk][2] = y0.z; w1[blk][3] = y0.w;
      w1[blk][4] = y1.x; w1[blk][5] = y1.y; w1[blk][6] = y1.z; w1[blk][7] = y1.w;
    }
    float base = a.softmax_scale * kLog2e;
    if (F::kE4m3) base *= a.k_scale_layer;
    if (F::kBf16) {
#pragma unroll
      for (int blk = 0; blk < 4; ++blk)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          qf[blk * 4 + ks][0] = w0[blk][2 * ks];
          qf[blk * 4 + ks][1] = w1[blk][2 * ks];
          qf[blk * 4 + ks][2] = w0[blk][2 * ks + 1];
          qf[blk * 4 + ks][3] = w1[blk][2 * ks + 1];
        }
      fac0 = base;
      fac1 = base;
    } else {
      // fp16 operands: scale each head by a power of two so its largest |q| lands in
      // [2^14, 2^15) -- inside fp16's normal range whatever the bf16 magnitudes are.
      uint32_t m0 = 0, m1 = 0;
#pragma unroll
      for (int blk = 0; blk < 4; ++blk)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          m0 = max(m0, max((w0[blk][i] & 0x7FFFu) << 16, w0[blk][i] & 0x7FFF0000u));
          m1 = max(m1, max((w1[blk][i] & 0x7FFFu) << 16, w1[blk][i] & 0x7FFF0000u));
        }
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) {
        m0 = max(m0, __shfl_xor_sync(0xffffffffu, m0, off));
        m1 = max(m1, __shfl_xor_sync(0xffffffffu, m1, off));
      }
      const int e0 = static_cast<int>(m0 >> 23) - 127, e1 = static_cast<int>(m1 >> 23) - 127;
      const int sg0 = m0 ? max(-64, min(64, 14 - e0)) : 0;
      const int sg1 = m1 ? max(-64, min(64, 14 - e1)) : 0;
      const float u0 = pow2f(sg0), u1 = pow2f(sg1);
#pragma unroll
      for (int blk = 0; blk < 4; ++blk)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint32_t a0 = w0[blk][2 * ks], a1 = w0[blk][2 * ks + 1];
          const uint32_t b0 = w1[blk][2 * ks], b1 = w1[blk][2 * ks + 1];
          uint32_t* f = qf[blk * 4 + ks];
          if (F::kInt8) {
            // int8 B fragments hold head dims (+0, +2) and (+1, +3)
            f[0] = pack_half2(bf16lo(a0) * u0, bf16lo(a1) * u0);
            f[2] = pack_half2(bf16hi(a0) * u0, bf16hi(a1) * u0);
            f[1] = pack_half2(bf16lo(b0) * u1, bf16lo(b1) * u1);
            f[3] = pack_half2(bf16hi(b0) * u1, bf16hi(b1) * u1);
          } else {
            // E4M3 B fragments hold (+0, +1) and (+2, +3)
            f[0] = pack_half2(bf16lo(a0) * u0, bf16hi(a0) * u0);
            f[2] = pack_half2(bf16lo(a1) * u0, bf16hi(a1) * u0);
            f[1] = pack_half2(bf16lo(b0) * u1, bf16hi(b0) * u1);
            f[3] = pack_half2(bf16lo(b1) * u1, bf16hi(b1) * u1);
          }
        }
      fac0 = base * pow2f(-sg0);
      fac1 = base * pow2f(-sg1);
    }
    if (h0 >= G) fac0 = 0.f;
    if (h1 >= G) fac1 = 0.f;
  }

  // ---------------- online-softmax state
  float m_run0 = -INFINITY, m_run1 = -INFINITY;  // log2-domain running max (uniform in the CTA)
  float l_run0 = 0.f, l_run1 = 0.f;              // this thread's share of sum p
  int e_run = -100;                              // int8: 2^e_run > every V scale seen
  float oacc[8][4];
#pragma unroll
  for (int t = 0; t < 8; ++t) oacc[t][0] = oacc[t][1] = oacc[t][2] = oacc[t][3] = 0.f;

  for (int cs = col0; cs < col1; cs += kIdxCap) {
    const int ce = min(col1, cs + kIdxCap);
    __syncthreads();  // previous chunk's tiles fully consumed
    const int nvalid = stage_indices(a, r, cs, ce, sIdx, sCnt, tid, lane, warp);
    const int ntiles = (nvalid + kTile - 1) / kTile;

#pragma unroll
    for (int st = 0; st < F::kStages - 1; ++st) {
      if (st < ntiles) issue_tile<FMT>(a, h, sIdx, st * kTile, nvalid, smem, st, tid);
      cp_async_commit();
    }

    for (int t = 0; t < ntiles; ++t) {
      cp_async_wait<F::kStages - 2>();
      __syncthreads();
      {
        const int tn = t + F::kStages - 1;
        if (tn < ntiles) issue_tile<FMT>(a, h, sIdx, tn * kTile, nvalid, smem, tn % F::kStages, tid);
        cp_async_commit();
      }
      const int st = t % F::kStages;
      const int tbase = t * kTile;
      const uint8_t* tK = smem + L::kK + size_t(st) * kTile * F::kRowBytes;
      const uint8_t* tV = smem + L::kV + size_t(st) * kTile * F::kRowBytes;

      // ---- q . K^T for this warp's 16 keys
      float sc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        const int row = warp * 16 + nt * 8 + hn;
        const uint32_t rowK = smem_u32(tK + row * F::kRowBytes);
        int delta = 0;
        if (F::kInline) {
          const int key = tbase + row;
          const int64_t slot = key < nvalid ? sIdx[key] : 0;
          delta = static_cast<int>(((slot * H + h) * F::kGlobalRow) & 15);
        }
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          uint32_t kw[8];
          if (F::kBf16) {
            const uint4 x = lds128(rowK + (swz_k<FMT>(8 * blk + 2 * c, row) << 4));
            const uint4 y = lds128(rowK + (swz_k<FMT>(8 * blk + 2 * c + 1, row) << 4));
            kw[0] = x.x; kw[1] = x.y; kw[2] = x.z; kw[3] = x.w;
            kw[4] = y.x; kw[5] = y.y; kw[6] = y.z; kw[7] = y.w;
          } else if (F::kInline) {
            const uint32_t p = rowK + delta + 64 * blk + 16 * c;
            kw[0] = lds32(p); kw[1] = lds32(p + 4); kw[2] = lds32(p + 8); kw[3] = lds32(p + 12);
          } else {
            const uint4 x = lds128(rowK + (swz_k<FMT>(4 * blk + c, row) << 4));
            kw[0] = x.x; kw[1] = x.y; kw[2] = x.z; kw[3] = x.w;
          }
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            uint32_t b0, b1;
            if (F::kBf16) {
              b0 = kw[2 * ks];
              b1 = kw[2 * ks + 1];
              mma_bf16(sc[nt], qf[blk * 4 + ks], b0, b1);
            } else if (F::kInt8) {
              b0 = i8pair_to_f16x2(kw[ks]);       // head dims +0, +2
              b1 = i8pair_to_f16x2(kw[ks] >> 8);  // head dims +1, +3
              mma_f16(sc[nt], qf[blk * 4 + ks], b0, b1);
            } else {
              b0 = e4m3pair_to_f16x2(kw[ks]);        // +0, +1
              b1 = e4m3pair_to_f16x2(kw[ks] >> 16);  // +2, +3
              mma_f16(sc[nt], qf[blk * 4 + ks], b0, b1);
            }
          }
        }
      }

      // ---- logits: hoisted K scale, mask, tile max
      float vsc[2][2];  // int8: V scale of keys (nt, e)
      float mx0 = -INFINITY, mx1 = -INFINITY, vmx = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kt = warp * 16 + nt * 8 + 2 * c + e;
          const bool valid = tbase + kt < nvalid;
          float ks = 1.f, vs = 0.f;
          if (F::kSide) {
            ks = reinterpret_cast<const float*>(smem + L::kKs)[st * kTile + kt];
            vs = reinterpret_cast<const float*>(smem + L::kVs)[st * kTile + kt];
          } else if (F::kInline) {
            const int64_t slot = valid ? sIdx[tbase + kt] : 0;
            const int delta = static_cast<int>(((slot * H + h) * F::kGlobalRow) & 15);
            ks = *reinterpret_cast<const float*>(tK + kt * F::kRowBytes + delta + kHeadDim);
            vs = *reinterpret_cast<const float*>(tV + kt * F::kRowBytes + delta + kHeadDim);
          }
          vs = valid ? vs : 0.f;
          vsc[nt][e] = vs;
          vmx = fmaxf(vmx, vs);
          const float s0 = valid ? sc[nt][e] * fac0 * ks : -INFINITY;
          const float s1 = valid ? sc[nt][2 + e] * fac1 * ks : -INFINITY;
          sc[nt][e] = s0;
          sc[nt][2 + e] = s1;
          mx0 = fmaxf(mx0, s0);
          mx1 = fmaxf(mx1, s1);
        }
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        if (F::kInt8) vmx = fmaxf(vmx, __shfl_xor_sync(0xffffffffu, vmx, off));
      }
      if (c == 0) {
        sRed[warp * 16 + h0] = mx0;
        sRed[warp * 16 + h1] = mx1;
      }
      if (F::kInt8 && lane == 0) sVmax[warp] = vmx;
      __syncthreads();

      float tm0 = sRed[h0], tm1 = sRed[h1];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) {
        tm0 = fmaxf(tm0, sRed[w * 16 + h0]);
        tm1 = fmaxf(tm1, sRed[w * 16 + h1]);
      }
      const float mn0 = fmaxf(m_run0, tm0), mn1 = fmaxf(m_run1, tm1);
      const float al0 = (mn0 == -INFINITY) ? 1.f : fast_exp2(m_run0 - mn0);
      const float al1 = (mn1 == -INFINITY) ? 1.f : fast_exp2(m_run1 - mn1);
      float pm = 1.f, ov = 1.f;
      if (F::kInt8) {
        float vm = sVmax[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) vm = fmaxf(vm, sVmax[w]);
        const int et = vm > 0.f ? max(-100, static_cast<int>(__float_as_uint(vm) >> 23) - 126) : -100;
        const int en = max(e_run, et);
        ov = pow2f(max(e_run - en, -126));
        pm = pow2f(kPShift - en);
        e_run = en;
      } else if (F::kE4m3) {
        pm = pow2f(kPShift);
      }
      m_run0 = mn0;
      m_run1 = mn1;

      // ---- p = exp2(s - m) -> shared memory
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int kt = warp * 16 + nt * 8 + 2 * c;
        float p[4];
        p[0] = (mn0 == -INFINITY) ? 0.f : fast_exp2(sc[nt][0] - mn0);
        p[1] = (mn0 == -INFINITY) ? 0.f : fast_exp2(sc[nt][1] - mn0);
        p[2] = (mn1 == -INFINITY) ? 0.f : fast_exp2(sc[nt][2] - mn1);
        p[3] = (mn1 == -INFINITY) ? 0.f : fast_exp2(sc[nt][3] - mn1);
        ps0 += p[0] + p[1];
        ps1 += p[2] + p[3];
        const uint32_t off0 = h0 * (kTile * 2) + ((((kt >> 3) ^ (h0 & 7))) << 4) + (kt & 7) * 2;
        const uint32_t off1 = h1 * (kTile * 2) + ((((kt >> 3) ^ (h1 & 7))) << 4) + (kt & 7) * 2;
        if (F::kBf16) {
          const __nv_bfloat16 a0 = __float2bfloat16_rn(p[0]), a1 = __float2bfloat16_rn(p[1]);
          const __nv_bfloat16 a2 = __float2bfloat16_rn(p[2]), a3 = __float2bfloat16_rn(p[3]);
          sts32(sP + off0, pack_bf162(__bfloat162float(a0), __bfloat162float(a1)));
          sts32(sP + off1, pack_bf162(__bfloat162float(a2), __bfloat162float(a3)));
          sts32(sPlo + off0, pack_bf162(p[0] - __bfloat162float(a0), p[1] - __bfloat162float(a1)));
          sts32(sPlo + off1, pack_bf162(p[2] - __bfloat162float(a2), p[3] - __bfloat162float(a3)));
        } else {
          const float f0 = F::kInt8 ? vsc[nt][0] * pm : pm, f1 = F::kInt8 ? vsc[nt][1] * pm : pm;
          const float x0 = p[0] * f0, x1 = p[1] * f1, x2 = p[2] * f0, x3 = p[3] * f1;
          const __half2 a = __floats2half2_rn(x0, x1), b = __floats2half2_rn(x2, x3);
          sts32(sP + off0, *reinterpret_cast<const uint32_t*>(&a));
          sts32(sP + off1, *reinterpret_cast<const uint32_t*>(&b));
          sts32(sPlo + off0, pack_half2(x0 - __low2float(a), x1 - __high2float(a)));
          sts32(sPlo + off1, pack_half2(x2 - __low2float(b), x3 - __high2float(b)));
        }
      }
      l_run0 = l_run0 * al0 + ps0;
      l_run1 = l_run1 * al1 + ps1;
      const float ao0 = al0 * ov, ao1 = al1 * ov;
#pragma unroll
      for (int t2 = 0; t2 < 8; ++t2) {
        oacc[t2][0] *= ao0;
        oacc[t2][1] *= ao0;
        oacc[t2][2] *= ao1;
        oacc[t2][3] *= ao1;
      }
      __syncthreads();

      // ---- p . V for head dims [64 warp, 64 warp + 64)
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        uint32_t pa[4], pl[4];
        {
          const int hrow = (lane & 7) + ((lane >> 3) & 1) * 8;
          const int j = 2 * kk + (lane >> 4);
          const uint32_t off = hrow * (kTile * 2) + ((j ^ (hrow & 7)) << 4);
          ldmatrix_x4(sP + off, pa[0], pa[1], pa[2], pa[3]);
          ldmatrix_x4(sPlo + off, pl[0], pl[1], pl[2], pl[3]);
        }
        const int r0 = 16 * kk + 2 * c;
        const int rows[4] = {r0, r0 + 1, r0 + 8, r0 + 9};
        if (F::kBf16) {
          uint4 vv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            vv[i] = lds128(smem_u32(tV + rows[i] * F::kRowBytes) + (swz_v<FMT>(8 * warp + hn, rows[i]) << 4));
          const uint32_t a0[4] = {vv[0].x, vv[0].y, vv[0].z, vv[0].w};
          const uint32_t a1[4] = {vv[1].x, vv[1].y, vv[1].z, vv[1].w};
          const uint32_t a2[4] = {vv[2].x, vv[2].y, vv[2].z, vv[2].w};
          const uint32_t a3[4] = {vv[3].x, vv[3].y, vv[3].z, vv[3].w};
#pragma unroll
          for (int t2 = 0; t2 < 8; ++t2) {
            const uint32_t sel = (t2 & 1) ? 0x7632u : 0x5410u;
            const uint32_t b0 = __byte_perm(a0[t2 >> 1], a1[t2 >> 1], sel);
            const uint32_t b1 = __byte_perm(a2[t2 >> 1], a3[t2 >> 1], sel);
            mma_bf16(oacc[t2], pa, b0, b1);
            mma_bf16(oacc[t2], pl, b0, b1);
          }
        } else {
          uint2 vv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (F::kInline) {
              const int key = tbase + rows[i];
              const int64_t slot = key < nvalid ? sIdx[key] : 0;
              const int delta = static_cast<int>(((slot * H + h) * F::kGlobalRow) & 15);
              const uint32_t p = smem_u32(tV + rows[i] * F::kRowBytes) + delta + 64 * warp + 8 * hn;
              vv[i].x = lds32(p);
              vv[i].y = lds32(p + 4);
            } else {
              vv[i] = lds64(smem_u32(tV + rows[i] * F::kRowBytes) +
                            (swz_v<FMT>(4 * warp + (hn >> 1), rows[i]) << 4) + ((hn & 1) << 3));
            }
          }
          if (F::kInt8) {
#pragma unroll
            for (int t2 = 0; t2 < 8; ++t2) {
              const uint32_t sel = (t2 & 3) | (((t2 & 3) + 4) << 8);
              const uint32_t x0 = (t2 < 4) ? vv[0].x : vv[0].y, x1 = (t2 < 4) ? vv[1].x : vv[1].y;
              const uint32_t x2 = (t2 < 4) ? vv[2].x : vv[2].y, x3 = (t2 < 4) ? vv[3].x : vv[3].y;
              const uint32_t b0 = i8pair_to_f16x2(__byte_perm(x0, x1, sel));
              const uint32_t b1 = i8pair_to_f16x2(__byte_perm(x2, x3, sel));
              mma_f16(oacc[t2], pa, b0, b1);
              mma_f16(oacc[t2], pl, b0, b1);
            }
          } else {
#pragma unroll
            for (int t4 = 0; t4 < 4; ++t4) {
              // [a_t, b_t, a_t+1, b_t+1] for t = 2*(t4&1) within word t4>>1
              const uint32_t sel = (t4 & 1) ? 0x7362u : 0x5140u;
              const uint32_t x0 = (t4 < 2) ? vv[0].x : vv[0].y, x1 = (t4 < 2) ? vv[1].x : vv[1].y;
              const uint32_t x2 = (t4 < 2) ? vv[2].x : vv[2].y, x3 = (t4 < 2) ? vv[3].x : vv[3].y;
              const uint32_t u = __byte_perm(x0, x1, sel), w = __byte_perm(x2, x3, sel);
              const uint32_t b0 = e4m3pair_to_f16x2(u), b1 = e4m3pair_to_f16x2(w);
              const uint32_t c0 = e4m3pair_to_f16x2(u >> 16), c1 = e4m3pair_to_f16x2(w >> 16);
              mma_f16(oacc[2 * t4], pa, b0, b1);
              mma_f16(oacc[2 * t4], pl, b0, b1);
              mma_f16(oacc[2 * t4 + 1], pa, c0, c1);
              mma_f16(oacc[2 * t4 + 1], pl, c0, c1);
            }
          }
        }
      }
    }
  }

  // ---------------- finalize: sum l over the quad and the warps, normalise, store
#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l_run0 += __shfl_xor_sync(0xffffffffu, l_run0, off);
    l_run1 += __shfl_xor_sync(0xffffffffu, l_run1, off);
  }
  __syncthreads();
  if (c == 0) {
    sRed[warp * 16 + h0] = l_run0;
    sRed[warp * 16 + h1] = l_run1;
  }
  __syncthreads();
  float L0 = 0.f, L1 = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    L0 += sRed[w * 16 + h0];
    L1 += sRed[w * 16 + h1];
  }
  float post = 1.f;
  if (F::kInt8) post = pow2f(e_run - kPShift);
  if (F::kE4m3) post = pow2f(-kPShift) * (P == 1 ? a.v_scale_layer : 1.f);

#pragma unroll
  for (int hi = 0; hi < 2; ++hi) {
    const int hh = hi ? h1 : h0;
    if (hh >= G) continue;
    const float Lh = hi ? L1 : L0;
    const float mh = hi ? m_run1 : m_run0;
    const float f = (Lh > 0.f) ? post / Lh : 0.f;
    const int64_t qhead = static_cast<int64_t>(h) * G + hh;
    float* dst = (P == 1) ? a.out + (r * Hq + qhead) * kHeadDim
                          : a.o_part + ((r * P + split) * Hq + qhead) * kHeadDim;
    dst += 64 * warp + 16 * c;
    const int i0 = 2 * hi;
    reinterpret_cast<float4*>(dst)[0] =
        make_float4(oacc[0][i0] * f, oacc[1][i0] * f, oacc[2][i0] * f, oacc[3][i0] * f);
    reinterpret_cast<float4*>(dst)[1] =
        make_float4(oacc[4][i0] * f, oacc[5][i0] * f, oacc[6][i0] * f, oacc[7][i0] * f);
    reinterpret_cast<float4*>(dst)[2] =
        make_float4(oacc[0][i0 + 1] * f, oacc[1][i0 + 1] * f, oacc[2][i0 + 1] * f, oacc[3][i0 + 1] * f);
    reinterpret_cast<float4*>(dst)[3] =
        make_float4(oacc[4][i0 + 1] * f, oacc[5][i0 + 1] * f, oacc[6][i0 + 1] * f, oacc[7][i0 + 1] * f);
    if (warp == 0 && c == 0) {
      const float lse = (Lh > 0.f) ? (mh + log2f(Lh)) * kLn2 : -INFINITY;
      if (P == 1) {
        if (a.lse != nullptr) a.lse[r * Hq + qhead] = lse;
      } else {
        a.lse_part[(r * P + split) * Hq + qhead] = lse;
      }
    }
  }
}

template <int FMT>
cudaError_t launch(const GatherArgs& a, cudaStream_t stream) {
  constexpr size_t smem = Smem<FMT>::kTotal;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(gather_attn_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int64_t grid = a.rows * a.num_kv_heads * a.num_splits;
  gather_attn_kernel<FMT><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace gather
}  // namespace qkv
