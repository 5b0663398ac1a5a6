// Top-k gather decode attention over a quantized slot pool (sm_103a).
//
// Pages: "int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next QSA path" §The finding
// worth upstreaming (each query row gathers its top-k scattered slots; side-tensor vs
// inline 260 B scales); "[Perf][SM70][FP8] Hoist QSA E4M3 KV scales" §Changes (K scale in
// the post-dot softmax factor, V scale once after normalised accumulation or after the
// split-K merge); "[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache" §Implementation
// scope (split-K workspace).
//
// Work decomposition: one CTA (4 warps) per (query row, KV head, K-split) -- and per chunk of
// 16 query heads when the GQA group is larger than 16. The split's index
// columns are cut into tiles of 16 keys, dealt round-robin to the warps; every warp then runs
// on its own -- its own copy ring, online softmax and accumulators -- with no block barrier
// in the main loop. The four partial results are merged once, at the end, through shared
// memory.
//
// Gathering: 16 B cp.async copies, consecutive lanes on consecutive chunks of a row (whole
// lines per request), into a ring per warp: two full K + V stages (E4M3), or three half-stage
// slots that K and V rows rotate through (int8 and 16-bit pools, see kSplitRing). Inline int8
// records, 4 B-aligned only, go by 4 B copies into the same places. The rows' placement keeps every
// fragment read below bank-conflict free: odd K rows sit 64 B (bf16: 16 B) further along the
// bank cycle than even ones, and V row r lands in one of 8 regions whose start rotates with r.
// (Bulk copies on the TMA engine, one 256 B row each, were measured slower on this access
// pattern: 6.4 vs 4.8 TB/s of gathered rows with the math removed.)
//
// Accumulators: each warp's 16 x HD fp32 p.V accumulator lives in tensor memory (TMEM,
// 32 lanes x HD / 2 columns per warp) and streams through registers 128 head dims at a time
// around the MMAs. Registers are what bound this kernel's occupancy; holding the accumulator
// in TMEM leaves room for three CTAs (12 warps) per SM instead of two.
//
// Variants (template parameters): the layout; PAGED (positions through a block table); the
// ring depth and CTAs per SM; QF16 (an IEEE-half query, for the FP16-activation contract of
// the calibrated E4M3 page, and the unquantised fp16 pool); HD (head dim 256 or 128). Run-time
// options: per-row lengths (varlen: columns past a row's length are never read) and the fused
// split-K merge (arrival counters).
//
// Per 16-key tile and warp:
//   q.K^T  mma.sync m16n8k16, M = the GQA group (16 query heads, padded), N = 8 keys, K = 16
//          head dims. Query fragments come from shared memory (ldmatrix; staged once per CTA
//          as fp16 with a per-head power of two, bf16 for the bf16 layout; int8 layouts stage
//          it twice, q_hi and q_lo, for an exact q_hi . c -- see Fmt::kQSplit). Key codes are
//          dequantised straight into B fragments (int8 -> fp16 by an exponent splice, E4M3 ->
//          fp16 by the native cvt, bf16 as stored); the head-dim order inside a fragment
//          follows how a code word unpacks and the staged query uses the same permutation.
//   softmax  logits times the hoisted K scale (per slot for int8; E4M3's per-layer scale is
//          folded into the per-head factor). The running max is only raised when a tile's max
//          exceeds it by more than 2^8 (log2 domain), so the accumulators are rescaled a few
//          times per row rather than every tile; p <= 2^8 is sized for that.
//   p.V    p comes straight from the q.K^T accumulators (the m16n8 C layout of two N-tiles is
//          the m16k16 A layout) as an fp16 hi + lo pair (three bf16 parts for the bf16 layout): with
//          outlier tokens a row can be a near-even mix of two large V rows of opposite sign,
//          and single-fp16 p would lose ~1e-3 of the result to cancellation. int8 p also
//          carries the slot's V scale and a power of two keeping it a normal fp16. HD / 8
//          N-tiles of 8 head dims, two MMAs (hi, lo) each.
// The E4M3 V scale and the power-of-two pre-scale are applied once at the end; split partials
// are written normalised, without the E4M3 V scale.
#pragma once

#include <atomic>
#include "qkv_internal.cuh"

namespace qkv {
namespace gather {

constexpr int kKeys = 16;  // keys per warp tile
constexpr int kHeadsPerCta = 16;  // query heads per CTA: the M = 16 of the MMAs
constexpr int kQkChains = 4;      // q.K^T accumulator chains per N-tile (one per 64 head dims)
constexpr int kQGrain = 7;        // int8 layouts: q_hi is a multiple of 2^7 (see Fmt::kQSplit)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kMaxFinite = 3.4028234663852886e38f;  // largest finite fp32
// p.V operand range. p <= 2^kTau (lazy rescale) and, for int8, a V scale < 2^eu, so the fp16
// operand x = p (v_scale) 2^(kPShift - eu) stays below 2^(kTau + kPShift) = 2^15, finite in
// fp16. The hi + lo pair keeps ~22 bits only while x is well above fp16's normal floor 2^-14;
// below it the pair's absolute error is 2^-25 (x units). So the shift is as large as the
// ceiling allows, and the int8 bound eu sits only 2^2 above the largest scale seen: an
// outlier token's ~16x larger scale costs one rescale instead of 4 bits of every other key.
constexpr float kTau = 8.0f;    // lazy-rescale threshold (log2 units): p <= 2^8
constexpr int kPShift = 7;      // x < 2^15; a key 2^-21 below the running max still has a normal hi
constexpr int kEuHeadroom = 2;  // int8: the V-scale bound 2^eu is raised 2^2 past the largest scale seen

// Per-layout traits. kKShift: extra offset of the odd K rows. Row sizes depend on the head
// dim too: see Geom. kWarps: warps per CTA. kQSplit (the int8 layouts): the query is staged
// twice, q_hi = the pre-scaled query rounded to a multiple of 2^7 and q_lo = the rest, and
// q.K^T runs on both. With integer codes every partial sum of q_hi . c is a multiple of 2^7
// below 2^31, exactly representable in fp32, so that half of the dot product is exact in
// whatever order the MMAs add; q_lo . c is 2^8 times smaller, so its rounding is too. The logit
// is then formed relative to a reference with fused multiply-adds (see the softmax below), which
// keeps the dot product's precision where it matters: a row whose output is a near cancellation
// of two outlier keys with opposite values needs more than a rounded fp32 logit. The second
// staged query leaves no room for two full K + V stages per warp at three CTAs of four warps
// per SM; kSplitRing rotates three half-stage slots instead (see Smem).
// kSide: the scales sit in a per-stage scale area of shared memory; kInline: the pool holds
// (HD + 4)-byte records, codes then the fp32 scale, which the copies realign into exactly the
// side layout's shared memory -- from there on both int8 layouts run the same arithmetic.
template <int FMT>
struct Fmt;
template <>
struct Fmt<QKV_INT8_SIDE> {
  static constexpr int kStages = 2, kMinBlocks = 3, kKShift = 64, kWarps = 4;
  static constexpr bool kInt8 = true, kSide = true, kInline = false, kE4m3 = false, kBf16 = false, kNatural = true;
  static constexpr bool kWide = false, kF16 = false, kQSplit = true, kSplitRing = true;
};
template <>
struct Fmt<QKV_INT8_INLINE> {
  static constexpr int kStages = 2, kMinBlocks = 3, kKShift = 64, kWarps = 4;
  static constexpr bool kInt8 = true, kSide = true, kInline = true, kE4m3 = false, kBf16 = false, kNatural = true;
  static constexpr bool kWide = false, kF16 = false, kQSplit = true, kSplitRing = true;
};
template <>
struct Fmt<QKV_E4M3> {
  static constexpr int kStages = 2, kMinBlocks = 3, kKShift = 64, kWarps = 4;
  static constexpr bool kInt8 = false, kSide = false, kInline = false, kE4m3 = true, kBf16 = false, kNatural = true;
  static constexpr bool kWide = false, kF16 = false, kQSplit = false, kSplitRing = false;
};
template <>
struct Fmt<QKV_BF16> {
  static constexpr int kStages = 2, kMinBlocks = 2, kKShift = 16, kWarps = 4;
  static constexpr bool kInt8 = false, kSide = false, kInline = false, kE4m3 = false, kBf16 = true, kNatural = false;
  static constexpr bool kWide = true, kF16 = false, kQSplit = false, kSplitRing = true;
};
// fp16 pool: the unquantised cache of the FP16-activation contract; moved like bf16 rows,
// multiplied as fp16 (q must be fp16 too)
template <>
struct Fmt<QKV_F16> {
  static constexpr int kStages = 2, kMinBlocks = 2, kKShift = 16, kWarps = 4;
  static constexpr bool kInt8 = false, kSide = false, kInline = false, kE4m3 = false, kBf16 = false, kNatural = false;
  static constexpr bool kWide = true, kF16 = true, kQSplit = false, kSplitRing = true;
};

// Head-dim dependent sizes (HD = 128 or 256).
//   kRowBytes   one K (or V) row in shared memory (an inline record's codes, realigned)
//   kGlobalRow  bytes of one record in the pool
//   kBlocks     64-dim blocks of q.K^T; kSweeps: 128-dim sweeps of p.V and of the final merge
//   kTmemCols   fp32 accumulator columns per TMEM lane (16 heads x HD dims over 32 lanes)
template <int FMT, int HD>
struct Geom {
  static_assert(HD == 128 || HD == 256, "head_dim 128 or 256");
  static constexpr int kRowBytes = Fmt<FMT>::kWide ? 2 * HD : HD;
  static constexpr int kGlobalRow = Fmt<FMT>::kInline ? HD + 4 : (Fmt<FMT>::kWide ? 2 * HD : HD);
  static constexpr int kBlocks = HD / 64, kSweeps = HD / 128, kTmemCols = HD / 2;
  // columns allocated per CTA: warp w uses lanes 32 (w % 4) of columns kTmemCols (w / 4) ..
  static constexpr int kTmemAlloc = kTmemCols * ((Fmt<FMT>::kWarps + 3) / 4);
  static_assert((kTmemAlloc & (kTmemAlloc - 1)) == 0 && kTmemAlloc >= 32, "tensor-memory allocations are powers of two");
};

// V region i (rows i and i + 8) starts 16 B further along the bank cycle than a plain packing
// would put it: by i chunks for 256 B rows, by 0, 0, 1, 1, 4, 4, 5, 5 chunks for 16-bit rows.
template <int FMT>
__host__ __device__ constexpr int v_region_shift(int i) {
  return Fmt<FMT>::kWide ? 16 * ((((i >> 1) & 1)) | (((i >> 2) & 1) << 2)) : 16 * i;
}

// floats per head row of the merge buffer (one 128-dim half), chosen bank-conflict free for the
// layout's fragment-to-head-dim order
template <int FMT>
__host__ __device__ constexpr int merge_row() { return Fmt<FMT>::kNatural ? 136 : 164; }

template <int FMT, int HD = 256, int STAGES = Fmt<FMT>::kStages>
struct Smem {
  using F = Fmt<FMT>;
  using G = Geom<FMT, HD>;
  static constexpr int kWarps = F::kWarps;
  static constexpr size_t kQ = 0;  // [HD / 16 k-steps][16 heads][16] 16-bit, fragment order
  static constexpr size_t kQOne = (HD / 16) * 16 * 16 * 2;
  static constexpr size_t kQ2 = kQ + kQOne;  // the same for q_lo (split layouts)
  static constexpr size_t kQBytes = kQOne * (F::kQSplit ? 2 : 1);
  static constexpr size_t kFac = kQ + kQBytes;  // [16] floats: logit factor per head
  // one stage: K rows, V rows, side scales (K then V), inline record offsets
  static constexpr size_t kKArea = 2 * 8 * size_t(G::kRowBytes) + F::kKShift;
  static constexpr size_t kVRegion = 2 * size_t(G::kRowBytes);
  static constexpr size_t kVArea = 8 * kVRegion + v_region_shift<FMT>(7);
  static constexpr size_t kStageK = 0;
  static constexpr size_t kStageV = kKArea;
  // split ring (kSplitRing): each warp rotates three slots, each holding one tile's K rows or
  // its V rows, so a tile's K and V need not share a stage; the int8 scales of both tensors
  // travel with K. Tile i's K sits in slot 2i mod 3, its V in slot 2i + 1 mod 3; once tile i is
  // done, tile i + 1's V goes into its K slot and tile i + 2's K into its V slot
  static constexpr size_t kSlotRows = kKArea > kVArea ? kKArea : kVArea;
  static constexpr size_t kStageKs = F::kSplitRing ? kSlotRows : kStageV + kVArea;
  // deeper rings keep each stage's valid-key mask here (a two-stage ring keeps it in registers)
  static constexpr size_t kStageMask = (kStageKs + (F::kSide ? 2 * kKeys * 4 : 0) + 3) / 4 * 4;
  static constexpr size_t kStageBytes =
      ((kStageMask + (STAGES > 2 && !F::kSplitRing ? 4 : 0)) + 15) / 16 * 16;  // a stage, or a slot
  static constexpr int kSlots = F::kSplitRing ? 3 : STAGES;
  static constexpr size_t kRing = kFac + 16 * 4;  // [kWarps][kSlots] stages or slots
  static constexpr size_t kWarpRing = size_t(kSlots) * kStageBytes;
  // final merge buffer [kWarps][16][merge_row] floats, reusing the rings (which it may outgrow
  // for small rows)
  static constexpr size_t kMergeBytes = size_t(kWarps) * 16 * merge_row<FMT>() * 4;
  static constexpr size_t kRingArea = kWarps * kWarpRing > kMergeBytes ? kWarps * kWarpRing : kMergeBytes;
  static constexpr size_t kTmem = kRing + kRingArea;  // TMEM base address
  static constexpr size_t kM = kTmem + 16;                         // [kWarps][16] floats
  static constexpr size_t kL = kM + kWarps * 16 * 4;                 // [kWarps][16] floats
  static constexpr size_t kPost = kL + kWarps * 16 * 4;             // [kWarps] floats
  static constexpr size_t kTotal = kPost + kWarps * 4;
  static_assert(kRing % 16 == 0 && kKArea % 16 == 0 && kVArea % 16 == 0, "alignment");
  // the CTAs that fit an SM (228 KB of shared memory, 1 KB reserved each) never ask for more
  // than its 512 TMEM columns, so an allocation never has to wait for another CTA
  static_assert((233472 / (kTotal + 1024)) * G::kTmemAlloc <= 512, "TMEM budget");
};

// Key row (0..15 within a tile) feeding column n of N-tile nt of q.K^T -- and so the key whose
// p a thread holds. The p.V B fragments of the natural layouts come from transposed byte
// matrices: a register holds keys 4c .. 4c + 3 of one head dim, which pair up as (4c, 4c + 2)
// and (4c + 1, 4c + 3) for int8 (exponent splice of bytes 0, 2 / 1, 3) and as (4c, 4c + 1),
// (4c + 2, 4c + 3) for E4M3 (the cvt takes two adjacent bytes). q.K^T produces p in that
// order. The inline layout uses the int8 order too, so it sums exactly like the side layout.
template <int FMT>
__device__ __forceinline__ int key_of(int nt, int n) {
  if (Fmt<FMT>::kInt8) return 2 * n + nt;
  if (Fmt<FMT>::kE4m3) return 4 * (n >> 1) + (n & 1) + 2 * nt;
  return 8 * nt + n;
}

// Byte offsets of tile row r (0..15) inside a stage (K area, V area).
// K: two regions of 8 rows, the second 8 rows + kKShift further on; a row goes to the second
// region when bit b of r is set -- b = 1 for int8 and b = 0 otherwise, so that the two rows a
// quarter-warp reads together (keys 4k + nt and 4k + 2 + nt for int8, 4k + 2nt and
// 4k + 1 + 2nt for E4M3) fall on disjoint banks.
// V: row r in region r mod 8, each region 2 rows plus 16 (r mod 8) B of rotation (bf16: see
// v_region_shift): 8 consecutive rows start on 8 distinct 16 B banks, as the transposed
// matrix loads and the 16 B fragment reads want.
template <int FMT, int HD>
__device__ __forceinline__ uint32_t k_row_off(int r) {
  constexpr int RB = Geom<FMT, HD>::kRowBytes;
  const int b = Fmt<FMT>::kInt8 ? 1 : 0;
  const int region = (r >> b) & 1;
  const int idx = ((r >> (b + 1)) << b) | (r & ((1 << b) - 1));  // r without bit b
  return RB * idx + region * (8 * RB + Fmt<FMT>::kKShift);
}
template <int FMT, int HD>
__device__ __forceinline__ uint32_t v_row_off(int r) {
  constexpr int RB = Geom<FMT, HD>::kRowBytes;
  return Smem<FMT, HD>::kStageV + (r & 7) * (2 * RB) + v_region_shift<FMT>(r & 7) + RB * (r >> 3);
}

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// ks (acc + accl) - R with the product and the subtraction fused: near the reference the
// difference keeps the dot product's full precision (SPLIT: accl is the q_lo part)
template <bool SPLIT>
__device__ __forceinline__ float logit_rel(float ks, float acc, float accl, float R) {
  const float u = fmaf(ks, acc, -R);
  return SPLIT ? fmaf(ks, accl, u) : u;
}

// Byte offset of query element (k-step k, head hd, k-index kappa) in the staged query.
__device__ __forceinline__ uint32_t q_off(int k, int hd, int kappa) {
  return k * 512 + hd * 32 + ((((kappa >> 3) ^ ((hd >> 2) & 1))) << 4) + (kappa & 7) * 2;
}

// PAGED: topk_idx holds logical positions of the row's sequence (a.row_seq), mapped to slots
// through a.block_table; otherwise it holds slot ids.
// STAGES: depth of each warp's copy ring (tiles in flight); MINB: CTAs per SM the register
// budget is sized for. The default (2, the format's) suits full-GPU launches; a deeper ring
// with fewer CTAs per SM suits launches with too few CTAs to fill the GPU.
// QF16: q is IEEE half instead of bf16 (the FP16-activation contract); it only changes how
// the query is staged.
template <int FMT, bool PAGED, int STAGES = Fmt<FMT>::kStages, int MINB = Fmt<FMT>::kMinBlocks,
          bool QF16 = false, int HD = 256>
__global__ void __launch_bounds__(32 * Fmt<FMT>::kWarps, MINB) gather_attn_kernel(const GatherArgs a) {
  using F = Fmt<FMT>;
  using GM = Geom<FMT, HD>;
  using L = Smem<FMT, HD, STAGES>;
  constexpr int kWarps = F::kWarps, kThreads = 32 * kWarps;
  static_assert(STAGES >= 2, "the ring needs a stage in flight while one is computed");
  static_assert(!(F::kBf16 && QF16) && !(F::kF16 && !QF16), "a 16-bit pool takes a query of its own type");
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = lane & 3, hn = lane >> 2;
  const int h0 = hn, h1 = hn + 8;
  const int P = a.num_splits, H = a.num_kv_heads, Hq = a.num_q_heads, G = Hq / H;
  // a GQA group above 16 query heads runs as chunks of 16, one item each (adjacent in launch
  // order, so a chunk's second gather of the same slots mostly hits L2)
  const int QC = (G + kHeadsPerCta - 1) / kHeadsPerCta;
  float* sFac = reinterpret_cast<float*>(smem + L::kFac);
  uint8_t* ring = smem + L::kRing + warp * L::kWarpRing;
  const uint32_t sQ = smem_u32(smem + L::kQ);
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(smem + L::kTmem);
  volatile uint32_t* sItem = reinterpret_cast<volatile uint32_t*>(smem + L::kTmem + 4);
  if (warp == 0) {
    tmem_alloc(smem_u32(sTmem), GM::kTmemAlloc);
    tmem_relinquish_alloc_permit();
  }
  // Work items (row, KV head, head chunk, split), split fastest. One CTA per item, or (a.sched
  // set) a resident grid whose CTAs take item blockIdx.x first and then pull the next free one
  // from the counter a.sched[0] until none is left -- no CTA ever waits for another.
  const int64_t num_items = a.rows * H * QC * P;
  int64_t bid = blockIdx.x;
  for (;;) {
  // (the host keeps the item count below 2^31: 32-bit division, not the 64-bit routine)
  const uint32_t ub = static_cast<uint32_t>(bid);
  const int split = static_cast<int>(ub % static_cast<uint32_t>(P));
  const uint32_t unit32 = ub / static_cast<uint32_t>(P);
  const int64_t unit = unit32;  // (row, KV head, head chunk): the fused merge's counter index
  const int qc = static_cast<int>(unit32 % static_cast<uint32_t>(QC));
  const uint32_t rh = unit32 / static_cast<uint32_t>(QC);
  const int h = static_cast<int>(rh % static_cast<uint32_t>(H));
  const int64_t r = rh / static_cast<uint32_t>(H);
  const int hq0 = h * G + kHeadsPerCta * qc;            // first query head of this item
  const int Gc = min(kHeadsPerCta, G - kHeadsPerCta * qc);  // query heads of this item (1..16)
  // the split partition is over the full width topk; a row with a valid length (varlen) ends
  // there, and its columns past it are never read
  int len = a.topk;
  if (a.topk_len != nullptr) {
    const int l = __ldg(a.topk_len + r);
    if ((l < 0 || l > a.topk) && tid == 0 && split == 0 && qc == 0 && a.dev_status != nullptr)
      atomicOr(a.dev_status, QKV_DEV_BAD_INDEX);
    len = min(max(l, 0), a.topk);
  }
  const int per_split = (a.topk + P - 1) / P;
  const int col0 = min(len, split * per_split);
  const int col1 = min(len, split * per_split + per_split);

  // ---------------- this warp's tiles: split tiles warp, warp + 4, ... (an empty pool has
  // no valid index: every row is empty)
  const int ntiles = (col1 - col0 + kKeys - 1) / kKeys;
  // paged: the row's sequence picks its block-table row; a row outside [0, num_seqs) is empty
  int64_t seq = 0;
  bool seq_ok = true;
  if (PAGED) {
    seq = __ldg(a.row_seq + r);
    seq_ok = seq >= 0 && seq < a.num_seqs;
    if (!seq_ok && tid == 0 && split == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, QKV_DEV_BAD_INDEX);
  }
  const int my = (ntiles > warp && a.num_slots > 0 && seq_ok) ? (ntiles - warp + kWarps - 1) / kWarps : 0;
  const int32_t* idx_row = a.topk_idx + r * a.topk;
  if (a.num_slots == 0 && a.dev_status != nullptr) {  // no tiles run: still flag the bad entries
    for (int col = col0 + tid; col < col1; col += kThreads) {
      const int v = __ldg(idx_row + col);
      if (a.shard ? v < -1 : v != -1) atomicOr(a.dev_status, QKV_DEV_BAD_INDEX);
    }
  }

  // Start the load of tile i's index of key `lane` (-1 past the split's end). The value is
  // only checked where it is used, one tile later, so the load's latency stays hidden.
  auto load_idx = [&](int i) -> int {
    if (i >= my || lane >= kKeys) return -1;
    const int col = col0 + (warp + kWarps * i) * kKeys + lane;
    return col < col1 ? __ldg(idx_row + col) : -1;
  };
  // Entries outside [-1, num_slots) are flagged and become padding.
  // A shard maps a global slot id to its own local id, and skips other shards' slots.
  auto checked = [&](int v) -> int {
    if (a.shard && v >= 0) {
      const int64_t l = static_cast<int64_t>(v) - a.slot_lo;
      return (l >= 0 && l < a.num_slots) ? static_cast<int>(l) : -1;
    }
    if (v < -1 || static_cast<int64_t>(v) >= a.num_slots) {
      if (a.dev_status != nullptr) atomicOr(a.dev_status, QKV_DEV_BAD_INDEX);
      v = -1;
    }
    return v;
  };
  // Paged pools: a position's block-table entry is loaded one tile before its slot is formed
  // (positions themselves two tiles before), so neither dependent load stalls the warp.
  const int32_t* tbl_row = PAGED ? a.block_table + seq * a.max_blocks : nullptr;
  const int bsz = PAGED ? a.block_size : 1;
  const int max_pos = PAGED ? a.max_blocks * a.block_size : 0;  // < 2^31, checked on the host
  const bool bsz_pow2 = (bsz & (bsz - 1)) == 0;
  const int bsz_shift = __ffs(bsz) - 1;
  auto block_of = [&](int pos) -> int { return bsz_pow2 ? pos >> bsz_shift : pos / bsz; };
  auto lookup = [&](int pos) -> int {  // the block id of position pos (-1: none loaded)
    if (!PAGED || pos < 0 || pos >= max_pos) return -1;
    return __ldg(tbl_row + block_of(pos));
  };
  // The slot of position pos in block blk; -1 for padding. Flags positions outside
  // [-1, max_pos), unallocated blocks (id < 0) and slots past the pool.
  auto checked_paged = [&](int pos, int blk) -> int {
    if (pos == -1) return -1;
    const int64_t slot = static_cast<int64_t>(blk) * bsz + (pos - block_of(pos) * bsz);
    if (pos < -1 || pos >= max_pos || blk < 0 || slot >= a.num_slots) {
      if (a.dev_status != nullptr) atomicOr(a.dev_status, QKV_DEV_BAD_INDEX);
      return -1;
    }
    return static_cast<int>(slot);
  };

  // Fixed per-lane parts of the copies of 256 B / 512 B rows. One copy instruction covers
  // four keys, one 128 B line of each (8 consecutive lanes on 8 consecutive 16 B chunks):
  // lane l takes key l / 8 + 4 t (t = 0..3) and chunks l % 8 + 8 u of it, so only the record
  // base changes per key and every chunk of a key is an immediate offset from it. (More
  // keys per instruction split a request over more lines and were measured slower.)
  constexpr int kRowChunks = GM::kRowBytes / 16;
  constexpr int kKpi = 4;                              // keys per copy instruction
  constexpr int kHs = F::kInline ? 1 : kRowChunks / 8;  // lines per key
  const int key_sub = lane >> 3, chunk_sub = lane & 7;
  const uint8_t* kb_l = a.k_cache + 16 * chunk_sub;
  const uint8_t* vb_l = a.v_cache + 16 * chunk_sub;
  const uint32_t dk_l = F::kInline ? 0u : k_row_off<FMT, HD>(key_sub) + 16 * chunk_sub;
  const uint32_t dv_l = F::kInline ? 0u : v_row_off<FMT, HD>(key_sub) - L::kStageV + 16 * chunk_sub;

  // Copies of one 16-key tile. rec_l: record number (slot * H + h; the host keeps it below
  // 2^31) of key `lane`, -1 = padding. K rows go to kdst + k_row_off(r), with the int8 scales
  // of both tensors at kdst + kStageKs; V rows go to vdst + v_row_off(r).
  auto copy_tile = [&](bool do_k, bool do_v, uint32_t kdst, uint32_t vdst, int rec_l) {
    if (!F::kInline) {
#pragma unroll
      for (int t = 0; t < kKeys / kKpi; ++t) {
        int rec = __shfl_sync(0xffffffffu, rec_l, key_sub + kKpi * t);
        // padding copies nothing and zero-fills its row (a zero source size reads no memory):
        // a stale E4M3 or bf16 NaN times p = 0 would still give NaN, and redirecting padding to
        // a real record made every padded row of a batch hammer the same L2 lines (2x slower on
        // causal chunked-prefill rows, whose padding sits at the end)
        const int nb = rec >= 0 ? 16 : 0;
        rec = max(rec, 0);
        const uint64_t off = static_cast<uint64_t>(static_cast<uint32_t>(rec)) * GM::kGlobalRow;
        // offsets of key l / 8 + 4 t relative to key l / 8 (the row layouts are additive)
        const uint32_t tk = k_row_off<FMT, HD>(kKpi * t), tv = v_row_off<FMT, HD>(kKpi * t);
#pragma unroll
        for (int u = 0; u < kHs; ++u) {
          if (do_k) cp_async16(kdst + dk_l + tk + 128 * u, kb_l + off + 128 * u, nb);
          if (do_v) cp_async16(vdst + dv_l + tv + 128 * u, vb_l + off + 128 * u, nb);
        }
      }
    } else {
      // inline records sit on 4 B boundaries only (HD + 4 bytes apart): 4 B copies, lane l taking
      // words l, l + 32, .. of each record's codes, land them 16 B-aligned in the side layout
#pragma unroll
      for (int r = 0; r < kKeys; ++r) {
        const int rec = __shfl_sync(0xffffffffu, rec_l, r);
        const int nb = rec >= 0 ? 4 : 0;
        const uint64_t off = static_cast<uint64_t>(static_cast<uint32_t>(max(rec, 0))) * GM::kGlobalRow + 4 * lane;
#pragma unroll
        for (int u = 0; u < HD / 128; ++u) {
          if (do_k) cp_async4(kdst + k_row_off<FMT, HD>(r) + 4 * lane + 128 * u, a.k_cache + off + 128 * u, nb);
          if (do_v) cp_async4(vdst + v_row_off<FMT, HD>(r) + 4 * lane + 128 * u, a.v_cache + off + 128 * u, nb);
        }
      }
    }
    if (F::kSide && do_k) {
      // lanes 0-15: K scales of the 16 keys; lanes 16-31: V scales (zero for padding), from the
      // side tensors or from the records' last 4 bytes
      const int rec = __shfl_sync(0xffffffffu, rec_l, lane & 15);
      const void* src;
      if (F::kInline) {
        src = ((lane >> 4) ? a.v_cache : a.k_cache) +
              static_cast<uint64_t>(static_cast<uint32_t>(max(rec, 0))) * GM::kGlobalRow + HD;
      } else {
        src = ((lane >> 4) ? a.v_scale_tok : a.k_scale_tok) + max(rec, 0);
      }
      cp_async4(kdst + L::kStageKs + lane * 4, src, rec >= 0 ? 4 : 0);
    }
  };
  auto rec_of = [&](int idxv) -> int { return idxv >= 0 ? idxv * H + h : -1; };
  // Copy one 16-key tile, K and V, into ring stage i % STAGES; returns the tile's valid-key
  // mask (a two-stage ring carries it one tile ahead in a register, a deeper one in the stage).
  auto issue = [&](int i, int idxv) -> uint32_t {  // idxv: this lane's checked slot (or -1)
    const int st = i % STAGES;
    const uint32_t mask = __ballot_sync(0xffffffffu, idxv >= 0) & 0xFFFFu;
    const uint32_t sbase = smem_u32(ring + size_t(st) * L::kStageBytes);
    if (STAGES > 2 && lane == 0) sts32(sbase + L::kStageMask, mask);
    copy_tile(true, true, sbase, sbase, rec_of(idxv));
    return mask;
  };
  // split ring: slot j of this warp (tile i's K in slot 2i mod 3, its V in slot 2i + 1 mod 3)
  const uint32_t ring_u32 = smem_u32(ring);
  auto slot_addr = [&](int j) -> uint32_t { return ring_u32 + static_cast<uint32_t>(j) * L::kStageBytes; };

  // The query's global loads go out first, then the first tiles' index loads and copies: the
  // copies wait for their indices, and the query's latency overlaps both.
  constexpr int kW = HD / 16;  // query: 32-bit words (two head dims each) per thread
  const int qh = tid >> 3, part = tid & 7;  // threads 0 .. 127 stage the query (8 per head)
  const bool live = qh < Gc;
  uint32_t w[kW];
  if (live) {
    const uint4* p = reinterpret_cast<const uint4*>(a.q + (r * Hq + hq0 + qh) * HD + (HD / 8) * part);
#pragma unroll
    for (int i = 0; i < kW / 4; ++i) {
      const uint4 x = __ldg(p + i);
      w[4 * i] = x.x; w[4 * i + 1] = x.y; w[4 * i + 2] = x.z; w[4 * i + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kW; ++i) w[i] = 0u;
  }
  // index pipeline: nidx = tile i + 1's entry (slot id, or position when paged); paged also
  // carries nblk = its block id and ppos = tile i + 2's position
  // The prologue issues tiles 0 .. STAGES - 2 (one commit group each) and loads tile
  // STAGES - 1's entry for the first loop iteration.
  int nidx, nblk = -1, ppos = -1;
  uint32_t mask_cur = 0;  // two-stage ring: valid keys of the tile being computed (bit k = key k)
  // split ring: tile i + 1's mask and records (its V rows go out once tile i is done)
  uint32_t mask_n1 = 0;
  int rec_n1 = -1;
  if (F::kSplitRing) {
    // K of tile 0, V of tile 0, K of tile 1: one commit group each
    const int e0 = load_idx(0), e1 = load_idx(1);
    nidx = load_idx(2);
    int c0, c1;
    if (PAGED) {
      ppos = load_idx(3);
      const int b0 = lookup(e0), b1 = lookup(e1);
      nblk = lookup(nidx);
      c0 = checked_paged(e0, b0);
      c1 = checked_paged(e1, b1);
    } else {
      c0 = checked(e0);
      c1 = checked(e1);
    }
    const int r0 = rec_of(c0);
    rec_n1 = rec_of(c1);
    mask_cur = __ballot_sync(0xffffffffu, c0 >= 0) & 0xFFFFu;
    mask_n1 = __ballot_sync(0xffffffffu, c1 >= 0) & 0xFFFFu;
    if (my > 0) copy_tile(true, false, slot_addr(0), 0u, r0);
    cp_async_commit();
    if (my > 0) copy_tile(false, true, 0u, slot_addr(1) - static_cast<uint32_t>(L::kStageV), r0);
    cp_async_commit();
    if (my > 1) copy_tile(true, false, slot_addr(2), 0u, rec_n1);
    cp_async_commit();
  } else {
    int ent[STAGES - 1];
#pragma unroll
    for (int t = 0; t < STAGES - 1; ++t) ent[t] = load_idx(t);
    nidx = load_idx(STAGES - 1);
    if (PAGED) {
      ppos = load_idx(STAGES);
      int blk[STAGES - 1];
#pragma unroll
      for (int t = 0; t < STAGES - 1; ++t) blk[t] = lookup(ent[t]);
      nblk = lookup(nidx);
#pragma unroll
      for (int t = 0; t < STAGES - 1; ++t) {
        const uint32_t m = (t < my) ? issue(t, checked_paged(ent[t], blk[t])) : 0u;
        if (t == 0) mask_cur = m;
        cp_async_commit();
      }
    } else {
#pragma unroll
      for (int t = 0; t < STAGES - 1; ++t) {
        const uint32_t m = (t < my) ? issue(t, checked(ent[t])) : 0u;
        if (t == 0) mask_cur = m;
        cp_async_commit();
      }
    }
  }

  // ---------------- stage the query once: 8 threads per head, HD / 8 head dims each (its
  // global loads were issued before the first tile's copies, see above)
  {
    int sg = 0;
    if (!F::kBf16) {
      // fp16 operands: a power of two puts the head's largest |q| in [2^14, 2^15)
      // packed |q| maximum over the thread's 32 dims (16-bit float bits order like values
      // when non-negative), then the larger half as fp32 bits
      uint32_t m;
      if (QF16) {
        __half2 mh = __floats2half2_rn(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < kW; ++i) {
          const uint32_t a16 = w[i] & 0x7FFF7FFFu;
          mh = __hmax2(mh, *reinterpret_cast<const __half2*>(&a16));
        }
        m = __float_as_uint(fmaxf(__low2float(mh), __high2float(mh)));
      } else {
        __nv_bfloat162 mh = __floats2bfloat162_rn(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < kW; ++i) {
          const uint32_t a16 = w[i] & 0x7FFF7FFFu;
          mh = __hmax2(mh, *reinterpret_cast<const __nv_bfloat162*>(&a16));
        }
        const uint32_t mw = *reinterpret_cast<const uint32_t*>(&mh);
        m = max((mw & 0xFFFFu) << 16, mw & 0xFFFF0000u);
      }
#pragma unroll
      for (int off = 1; off <= 4; off <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
      sg = m ? max(-64, min(64, 14 - (static_cast<int>(m >> 23) - 127))) : 0;
    }
    const float u = pow2f(sg);
    const uint64_t uu = f2pack(u, u);
    // two head dims per 32-bit store: the pair that shares a B-fragment register of a code
    // word (int8: d, d + 2; E4M3 and bf16: d, d + 1) sits in adjacent k-indices
#pragma unroll
    for (int g4 = 0; g4 < kW / 2; ++g4) {
#pragma unroll
      for (int up = 0; up < 2; ++up) {
        const int i0 = 4 * g4 + (F::kInt8 ? up : 2 * up), i1 = i0 + (F::kInt8 ? 2 : 1);
        const int d = (HD / 8) * part + i0;
        const int blk = d >> 6, cc = (d >> 4) & 3, ks = (d >> 2) & 3;
        const uint32_t b0 = (i0 & 1) ? (w[i0 >> 1] >> 16) : (w[i0 >> 1] & 0xFFFFu);
        const uint32_t b1 = (i1 & 1) ? (w[i1 >> 1] >> 16) : (w[i1 >> 1] & 0xFFFFu);
        uint32_t v32;
        if (F::kBf16) {
          v32 = b0 | (b1 << 16);
        } else {
          float s0, s1, x0, x1;
          if (QF16) {
            x0 = __half2float(__ushort_as_half(static_cast<unsigned short>(b0)));
            x1 = __half2float(__ushort_as_half(static_cast<unsigned short>(b1)));
          } else {
            x0 = __uint_as_float(b0 << 16);
            x1 = __uint_as_float(b1 << 16);
          }
          f2unpack(f2mul(f2pack(x0, x1), uu), s0, s1);
          if (F::kQSplit) {  // q_hi on the 2^7 grid here, the remainder in the second copy
            const float h0v = rintf(s0 * (1.0f / (1 << kQGrain))) * static_cast<float>(1 << kQGrain);
            const float h1v = rintf(s1 * (1.0f / (1 << kQGrain))) * static_cast<float>(1 << kQGrain);
            if (qh < kHeadsPerCta)
              sts32(smem_u32(smem + L::kQ2 + q_off(blk * 4 + ks, qh, up * 8 + 2 * cc)), pack_half2(s0 - h0v, s1 - h1v));
            s0 = h0v;
            s1 = h1v;
          }
          v32 = pack_half2(s0, s1);
        }
        if (qh < kHeadsPerCta) sts32(smem_u32(smem + L::kQ + q_off(blk * 4 + ks, qh, up * 8 + 2 * cc)), v32);
      }
    }
    if (part == 0 && qh < kHeadsPerCta) {
      float base = a.softmax_scale * kLog2e;
      if (F::kE4m3) base *= a.k_scale_layer;
      sFac[qh] = live ? base * pow2f(-sg) : 0.f;
    }
  }
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const float fac0 = sFac[h0], fac1 = sFac[h1];
  const uint64_t fac00 = f2pack(fac0, fac0), fac11 = f2pack(fac1, fac1);
  // this warp's accumulator: its 32 TMEM lanes (quarter warp % 4) of the columns
  // kTmemCols (warp / 4) onwards; column 4 t + j holds the C-fragment value j of N-tile t
  const uint32_t tacc = *sTmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) +
                        static_cast<uint32_t>(GM::kTmemCols * (warp >> 2));
  {
    float z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll
    for (int q = 0; q < GM::kTmemCols / 32; ++q) tmem_st32(tacc + 32 * q, z);
  }

  // ---------------- online-softmax state (per warp)
  // the reference in dot-product units (ks . q . k) the logits are taken against, heads h0, h1;
  // -inf until the head's first valid key; a padded head (no query) keeps 0 with a zero factor
  float R0 = (h0 < Gc) ? -INFINITY : 0.f, R1 = (h1 < Gc) ? -INFINITY : 0.f;
  // this thread's share of sum p for heads h0 (l0) and h1 (l1), each kept as a pair of
  // partial sums (keys e = 0 and e = 1) so that it accumulates with packed adds
  uint64_t l0 = f2pack(0.f, 0.f), l1 = f2pack(0.f, 0.f);
  int eu = -100;                           // int8: 2^eu > every V scale seen
  int ks = 0;  // split ring: the slot of tile i's K rows, 2i mod 3 (its V rows: the next slot)
  for (int i = 0; i < my; ++i) {
    uint32_t mask_next = 0u;
    if (!F::kSplitRing) {
      const int inext = i + STAGES - 1;  // the tile issued now, into the stage freed last iteration
      mask_next = (inext < my) ? issue(inext, PAGED ? checked_paged(nidx, nblk) : checked(nidx)) : 0u;
      cp_async_commit();
      if (PAGED) {
        nidx = ppos;
        nblk = lookup(ppos);
        ppos = load_idx(i + STAGES + 1);
      } else {
        nidx = load_idx(i + STAGES);
      }
      cp_async_wait<STAGES - 1>();
    } else {
      cp_async_wait<2>();  // K of tile i (V of tile i and K of tile i + 1 may be in flight)
    }
    const int st = i % STAGES;
    __syncwarp();

    // where this tile's K rows and scales (kslot) and V rows (vbase + v_row_off) are: one stage,
    // or two slots of the split ring
    const uint32_t sbase = smem_u32(ring + size_t(st) * L::kStageBytes);
    const uint32_t kslot = F::kSplitRing ? slot_addr(ks) : sbase;
    const uint32_t vslot = F::kSplitRing ? slot_addr(ks == 2 ? 0 : ks + 1) : sbase;
    ks = ks == 0 ? 2 : ks - 1;  // (2i + 2) mod 3 for the next tile
    const uint32_t vbase = F::kSplitRing ? vslot - static_cast<uint32_t>(L::kStageV) : sbase;
    const uint32_t mask = (STAGES == 2 || F::kSplitRing) ? mask_cur : lds32(sbase + L::kStageMask);

    // ---- q . K^T for this warp's 16 keys
    // kQkChains independent accumulator chains per N-tile (64-dim blocks dealt round-robin),
    // added at the end: shorter chains of smaller partial sums round less. Outlier keys give
    // logits of ~2^4.5 (log2 units) built from partial sums ~10x larger, so a near-tie of two
    // outlier keys with opposite V values turns the dot product's rounding into output error.
    float accc[kQkChains][2][4];
#pragma unroll
    for (int ch = 0; ch < kQkChains; ++ch)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) accc[ch][nt][0] = accc[ch][nt][1] = accc[ch][nt][2] = accc[ch][nt][3] = 0.f;
    uint32_t rowK[2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) rowK[nt] = kslot + k_row_off<FMT, HD>(key_of<FMT>(nt, hn));
#pragma unroll
    for (int blk = 0; blk < GM::kBlocks; ++blk) {
      uint32_t kw[2][8];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        if (F::kWide) {
          const uint4 x = lds128(rowK[nt] + (8 * blk + 2 * c) * 16);
          const uint4 y = lds128(rowK[nt] + (8 * blk + 2 * c + 1) * 16);
          kw[nt][0] = x.x; kw[nt][1] = x.y; kw[nt][2] = x.z; kw[nt][3] = x.w;
          kw[nt][4] = y.x; kw[nt][5] = y.y; kw[nt][6] = y.z; kw[nt][7] = y.w;
        } else {
          const uint4 x = lds128(rowK[nt] + (4 * blk + c) * 16);
          kw[nt][0] = x.x; kw[nt][1] = x.y; kw[nt][2] = x.z; kw[nt][3] = x.w;
        }
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t qa[4], ql[4];
        {
          const int mtx = lane >> 3, j = lane & 7;
          const int hd = (mtx & 1) * 8 + j;
          const uint32_t qoff = (blk * 4 + ks) * 512 + hd * 32 + ((((mtx >> 1) ^ ((hd >> 2) & 1))) << 4);
          ldmatrix_x4(sQ + qoff, qa[0], qa[1], qa[2], qa[3]);
          if (F::kQSplit) ldmatrix_x4(sQ + L::kQOne + qoff, ql[0], ql[1], ql[2], ql[3]);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          if (F::kQSplit) {  // q_hi chains 0, 1 (even / odd 64-dim blocks), q_lo chains 2, 3
            const uint32_t b0 = i8pair_to_f16x2(kw[nt][ks]), b1 = i8pair_to_f16x2(kw[nt][ks] >> 8);
            mma_f16(accc[blk & 1][nt], qa, b0, b1);
            mma_f16(accc[2 + (blk & 1)][nt], ql, b0, b1);
          } else if (F::kBf16) {
            mma_bf16(accc[blk % kQkChains][nt], qa, kw[nt][2 * ks], kw[nt][2 * ks + 1]);
          } else if (F::kF16) {
            mma_f16(accc[blk % kQkChains][nt], qa, kw[nt][2 * ks], kw[nt][2 * ks + 1]);
          } else if (F::kInt8) {
            mma_f16(accc[blk % kQkChains][nt], qa, i8pair_to_f16x2(kw[nt][ks]), i8pair_to_f16x2(kw[nt][ks] >> 8));
          } else {
            mma_f16(accc[blk % kQkChains][nt], qa, e4m3pair_to_f16x2(kw[nt][ks]), e4m3pair_to_f16x2(kw[nt][ks] >> 16));
          }
        }
      }
    }

    // acc: the dot products (split layouts: the exact q_hi part); accl: the q_lo part
    float acc[2][4], accl[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      if (F::kQSplit) {  // q_hi chains hold multiples of 2^7 below 2^31: their sum is exact
        uint64_t a01 = f2add(f2pack(accc[0][nt][0], accc[0][nt][1]), f2pack(accc[1][nt][0], accc[1][nt][1]));
        uint64_t a23 = f2add(f2pack(accc[0][nt][2], accc[0][nt][3]), f2pack(accc[1][nt][2], accc[1][nt][3]));
        f2unpack(a01, acc[nt][0], acc[nt][1]);
        f2unpack(a23, acc[nt][2], acc[nt][3]);
        a01 = f2add(f2pack(accc[2][nt][0], accc[2][nt][1]), f2pack(accc[3][nt][0], accc[3][nt][1]));
        a23 = f2add(f2pack(accc[2][nt][2], accc[2][nt][3]), f2pack(accc[3][nt][2], accc[3][nt][3]));
        f2unpack(a01, accl[nt][0], accl[nt][1]);
        f2unpack(a23, accl[nt][2], accl[nt][3]);
      } else {
        accl[nt][0] = accl[nt][1] = accl[nt][2] = accl[nt][3] = 0.f;  // (no q_lo part)
        uint64_t a01 = f2pack(accc[0][nt][0], accc[0][nt][1]), a23 = f2pack(accc[0][nt][2], accc[0][nt][3]);
#pragma unroll
        for (int ch = 1; ch < kQkChains; ++ch) {
          a01 = f2add(a01, f2pack(accc[ch][nt][0], accc[ch][nt][1]));
          a23 = f2add(a23, f2pack(accc[ch][nt][2], accc[ch][nt][3]));
        }
        f2unpack(a01, acc[nt][0], acc[nt][1]);
        f2unpack(a23, acc[nt][2], acc[nt][3]);
      }
    }

    // ---- logits with the hoisted K scale; masked keys -> -inf
    float s[2][4];  // [nt][0..1: head h0 keys e=0,1; 2..3: head h1]
    float vsc[2][2];
    float mx0 = -INFINITY, mx1 = -INFINITY;
    float kscs[2][2];
    bool valids[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      float ksc2[2];
      bool valid2[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kt = key_of<FMT>(nt, 2 * c + e);
        const bool valid = (mask >> kt) & 1u;
        valid2[e] = valid;
        float ksc = 1.f, vs = 0.f;
        if (F::kSide) {
          ksc = __uint_as_float(lds32(kslot + L::kStageKs + kt * 4));
          vs = __uint_as_float(lds32(kslot + L::kStageKs + (kKeys + kt) * 4));
        }
        // (padding keys already carry a zero V scale: their scale copies zero-fill)
        vsc[nt][e] = vs;
        ksc2[e] = ksc;
      }
      kscs[nt][0] = ksc2[0];
      kscs[nt][1] = ksc2[1];
      valids[nt][0] = valid2[0];
      valids[nt][1] = valid2[1];
      // logits of keys e = 0, 1 for heads h0 (acc 0, 1) and h1 (acc 2, 3), as fp32 pairs
      // relative to the references (ks . acc - R, one rounding near the maximum), in log2 units
      const float t0 = logit_rel<F::kQSplit>(ksc2[0], acc[nt][0], accl[nt][0], R0) * fac0;
      const float t1 = logit_rel<F::kQSplit>(ksc2[1], acc[nt][1], accl[nt][1], R0) * fac0;
      const float t2 = logit_rel<F::kQSplit>(ksc2[0], acc[nt][2], accl[nt][2], R1) * fac1;
      const float t3 = logit_rel<F::kQSplit>(ksc2[1], acc[nt][3], accl[nt][3], R1) * fac1;
      s[nt][0] = valid2[0] ? t0 : -INFINITY;
      s[nt][1] = valid2[1] ? t1 : -INFINITY;
      s[nt][2] = valid2[0] ? t2 : -INFINITY;
      s[nt][3] = valid2[1] ? t3 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }

    // ---- lazy rescale: raise the max in use only past the threshold
    bool rescale;
    float rf0 = 1.f, rf1 = 1.f;  // accumulator factors for heads h0, h1 when rescaling
    {
      // a logit more than 2^kTau above its reference (any valid key when there is none yet), or
      // an int8 V scale at the bound, moves the reference to the tile's largest ks . (q . k).
      // int8: the largest |V scale| of this thread's four keys, as fp32 bits (non-negative
      // floats order as integers); the threads' keys together are the tile's 16
      uint32_t myv = 0u;
      if (F::kInt8) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) myv = max(myv, __float_as_uint(vsc[nt][e]) & 0x7FFFFFFFu);
      }
      const bool vup = F::kInt8 && myv != 0u && static_cast<int>(myv >> 23) - 126 > eu;
      // (this thread's own logits decide whether any head needs a look; the four threads of a
      // head agree on it inside, from their common maximum)
      rescale = false;
      int ne = eu;
      if (__any_sync(0xffffffffu, mx0 > kTau || mx1 > kTau || vup)) {
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const bool up0 = mx0 > kTau, up1 = mx1 > kTau;
        if (F::kInt8) {  // the new bound from the tile's largest V scale (warp-uniform)
          const uint32_t vmx_bits = __reduce_max_sync(0xffffffffu, myv);
          if (vmx_bits != 0u) {
            const int ev = static_cast<int>(vmx_bits >> 23) - 126;
            if (ev > eu) ne = ev + kEuHeadroom;
          }
        }
        float v0 = -INFINITY, v1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            if (valids[nt][e]) {
              v0 = fmaxf(v0, kscs[nt][e] * (F::kQSplit ? acc[nt][e] + accl[nt][e] : acc[nt][e]));
              v1 = fmaxf(v1, kscs[nt][e] * (F::kQSplit ? acc[nt][2 + e] + accl[nt][2 + e] : acc[nt][2 + e]));
            }
          }
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
          v0 = fmaxf(v0, __shfl_xor_sync(0xffffffffu, v0, off));
          v1 = fmaxf(v1, __shfl_xor_sync(0xffffffffu, v1, off));
        }
        const float nR0 = up0 ? v0 : R0, nR1 = up1 ? v1 : R1;
        const bool live0 = R0 != -INFINITY, live1 = R1 != -INFINITY;
        rescale = __any_sync(0xffffffffu, (live0 && (nR0 != R0 || ne != eu)) || (live1 && (nR1 != R1 || ne != eu)));
        const float ov = F::kInt8 ? pow2f(max(eu - ne, -126)) : 1.f;
        const float al0 = (nR0 == R0) ? 1.f : (live0 ? fast_exp2((R0 - nR0) * fac0) : 0.f);
        const float al1 = (nR1 == R1) ? 1.f : (live1 ? fast_exp2((R1 - nR1) * fac1) : 0.f);
        rf0 = al0 * ov;
        rf1 = al1 * ov;
        l0 = f2mul(l0, f2pack(al0, al0));
        l1 = f2mul(l1, f2pack(al1, al1));
        R0 = nR0;
        R1 = nR1;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float k = kscs[nt][e];
            s[nt][e] = valids[nt][e] ? logit_rel<F::kQSplit>(k, acc[nt][e], accl[nt][e], R0) * fac0 : -INFINITY;
            s[nt][2 + e] =
                valids[nt][e] ? logit_rel<F::kQSplit>(k, acc[nt][2 + e], accl[nt][2 + e], R1) * fac1 : -INFINITY;
          }
      }
      eu = ne;
    }

    // ---- p = exp2(logit relative to the reference): fp32 sums, hi + lo A fragments (bf16: hi,
    //      mid, lo -- three bf16 parts hold the 24 bits two fp16 parts give)
    uint32_t pa[4], pl[4], p3[4];
    {
      const float pm = F::kInt8 ? pow2f(kPShift - eu) : (F::kBf16 ? 1.f : pow2f(kPShift));
      const uint64_t pm2 = f2pack(pm, pm);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float p[4];
        {
          float d0, d1, d2, d3;
          d0 = s[nt][0];  // the logits are already relative to the references
          d1 = s[nt][1];
          d2 = s[nt][2];
          d3 = s[nt][3];
          p[0] = fast_exp2(d0);  // masked: exp2(-inf) = 0
          p[1] = fast_exp2(d1);
          p[2] = fast_exp2(d2);
          p[3] = fast_exp2(d3);
        }
        const uint64_t p01 = f2pack(p[0], p[1]), p23 = f2pack(p[2], p[3]);
        l0 = f2add(l0, p01);
        l1 = f2add(l1, p23);
        // x = p times the key's V scale (int8) and the power-of-two pre-scale
        const uint64_t f01 = F::kInt8 ? f2mul(f2pack(vsc[nt][0], vsc[nt][1]), pm2) : pm2;
        float x0, x1, x2, x3;
        const uint64_t x01 = f2mul(p01, f01), x23 = f2mul(p23, f01);
        f2unpack(x01, x0, x1);
        f2unpack(x23, x2, x3);
        float r0, r1, r2, r3;
        if (F::kBf16) {
          const __nv_bfloat162 a0 = __floats2bfloat162_rn(x0, x1), a1 = __floats2bfloat162_rn(x2, x3);
          pa[2 * nt] = *reinterpret_cast<const uint32_t*>(&a0);
          pa[2 * nt + 1] = *reinterpret_cast<const uint32_t*>(&a1);
          const uint64_t y01 = f2sub(x01, f2pack(__low2float(a0), __high2float(a0)));
          const uint64_t y23 = f2sub(x23, f2pack(__low2float(a1), __high2float(a1)));
          f2unpack(y01, r0, r1);
          f2unpack(y23, r2, r3);
          const __nv_bfloat162 b0 = __floats2bfloat162_rn(r0, r1), b1 = __floats2bfloat162_rn(r2, r3);
          pl[2 * nt] = *reinterpret_cast<const uint32_t*>(&b0);
          pl[2 * nt + 1] = *reinterpret_cast<const uint32_t*>(&b1);
          f2unpack(f2sub(y01, f2pack(__low2float(b0), __high2float(b0))), r0, r1);
          f2unpack(f2sub(y23, f2pack(__low2float(b1), __high2float(b1))), r2, r3);
          p3[2 * nt] = pack_bf162(r0, r1);
          p3[2 * nt + 1] = pack_bf162(r2, r3);
        } else {
          const __half2 a0 = __floats2half2_rn(x0, x1), a1 = __floats2half2_rn(x2, x3);
          pa[2 * nt] = *reinterpret_cast<const uint32_t*>(&a0);
          pa[2 * nt + 1] = *reinterpret_cast<const uint32_t*>(&a1);
          f2unpack(f2sub(x01, f2pack(__low2float(a0), __high2float(a0))), r0, r1);
          f2unpack(f2sub(x23, f2pack(__low2float(a1), __high2float(a1))), r2, r3);
          pl[2 * nt] = pack_half2(r0, r1);
          pl[2 * nt + 1] = pack_half2(r2, r3);
        }
      }
    }

    // ---- p . V: sweep sw covers head dims [128 sw, 128 sw + 128).
    //      Natural layouts: N-tile t holds head dims 8 t .. 8 t + 7; its B fragments come from
    //      transposed 16 x 16 byte matrices (keys x 16 head dims) of the V rows.
    //      Others: lane group n reads the 16 head dims 128 sw + 16 n .. + 16 of the four key
    //      rows whose p it holds; N-tile 16 s + t, column n covers head dim 128 s + 16 n + t.
    {
      const int rows[4] = {key_of<FMT>(0, 2 * c), key_of<FMT>(0, 2 * c + 1), key_of<FMT>(1, 2 * c),
                           key_of<FMT>(1, 2 * c + 1)};
      uint32_t rowV[4];
      if (F::kSplitRing) {  // V of tile i (K of tile i + 1 may be in flight)
        cp_async_wait<1>();
        __syncwarp();
      }
#pragma unroll
      for (int ri = 0; ri < 4; ++ri) rowV[ri] = vbase + v_row_off<FMT, HD>(rows[ri]);
      // natural layouts: lane l addresses key row l % 16 of the 16 B column block l / 16 (+ 2 m)
      const uint32_t vmat = vbase + v_row_off<FMT, HD>(lane & 15) + 16 * (lane >> 4);
#pragma unroll
      for (int sw = 0; sw < GM::kSweeps; ++sw) {
        // accumulator quarters 2 sw (N-tiles 16 sw + 0..7) and 2 sw + 1 (16 sw + 8..15)
        float ob[2][32];
        // the previous sweep's stores have read these registers (and the previous tile's
        // stores of these columns are done)
        tmem_wait_st();
        tmem_ld32(tacc + 64 * sw, ob[0]);
        tmem_ld32(tacc + 64 * sw + 32, ob[1]);
        uint32_t bb[16][2];
        if (F::kNatural) {
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            // 16 B column blocks 8 sw + 2 m and 8 sw + 2 m + 1: N-tiles 4 m .. 4 m + 3 of the sweep
            uint32_t x[4];
            ldmatrix_x2_trans_b8(vmat + 16 * (8 * sw + 2 * m), x[0], x[1], x[2], x[3]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (F::kInt8) {
                bb[4 * m + u][0] = i8pair_to_f16x2(x[u]);       // keys 4c, 4c + 2
                bb[4 * m + u][1] = i8pair_to_f16x2(x[u] >> 8);  // keys 4c + 1, 4c + 3
              } else {
                bb[4 * m + u][0] = e4m3pair_to_f16x2(x[u]);        // keys 4c, 4c + 1
                bb[4 * m + u][1] = e4m3pair_to_f16x2(x[u] >> 16);  // keys 4c + 2, 4c + 3
              }
            }
          }
        } else if (F::kWide) {
          uint32_t vw[4][8];
#pragma unroll
          for (int ri = 0; ri < 4; ++ri) {
            const uint32_t p = rowV[ri] + 2 * (128 * sw + 16 * hn);
            const uint4 x = lds128(p), y = lds128(p + 16);
            vw[ri][0] = x.x; vw[ri][1] = x.y; vw[ri][2] = x.z; vw[ri][3] = x.w;
            vw[ri][4] = y.x; vw[ri][5] = y.y; vw[ri][6] = y.z; vw[ri][7] = y.w;
          }
#pragma unroll
          for (int tt = 0; tt < 16; ++tt) {
            const uint32_t sel = (tt & 1) ? 0x7632u : 0x5410u;
            bb[tt][0] = __byte_perm(vw[0][tt >> 1], vw[1][tt >> 1], sel);
            bb[tt][1] = __byte_perm(vw[2][tt >> 1], vw[3][tt >> 1], sel);
          }
        }
        tmem_wait_ld(ob[0]);
        tmem_wait_ld(ob[1]);
        if (rescale) {
          const uint64_t r00 = f2pack(rf0, rf0), r11 = f2pack(rf1, rf1);
#pragma unroll
          for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              f2scale(&ob[b][4 * t], r00);
              f2scale(&ob[b][4 * t + 2], r11);
            }
        }
#pragma unroll
        for (int tt = 0; tt < 16; ++tt) {
          float* acc4 = &ob[tt >> 3][4 * (tt & 7)];
          if (F::kBf16)
            mma_bf16(acc4, pa, bb[tt][0], bb[tt][1]);
          else
            mma_f16(acc4, pa, bb[tt][0], bb[tt][1]);
        }
#pragma unroll
        for (int tt = 0; tt < 16; ++tt) {
          float* acc4 = &ob[tt >> 3][4 * (tt & 7)];
          if (F::kBf16)
            mma_bf16(acc4, pl, bb[tt][0], bb[tt][1]);
          else
            mma_f16(acc4, pl, bb[tt][0], bb[tt][1]);
        }
        if (F::kBf16) {
#pragma unroll
          for (int tt = 0; tt < 16; ++tt) mma_bf16(&ob[tt >> 3][4 * (tt & 7)], p3, bb[tt][0], bb[tt][1]);
        }
        tmem_st32(tacc + 64 * sw, ob[0]);
        tmem_st32(tacc + 64 * sw + 32, ob[1]);
      }
    }
    if (F::kSplitRing) {
      // every lane is done with this tile's slots: the V rows of tile i + 1 go to its K slot, the
      // K rows of tile i + 2 to its V slot
      __syncwarp();
      if (i + 1 < my) copy_tile(false, true, 0u, kslot - static_cast<uint32_t>(L::kStageV), rec_n1);
      cp_async_commit();
      const int c2 = (i + 2 < my) ? (PAGED ? checked_paged(nidx, nblk) : checked(nidx)) : -1;
      const int r2 = rec_of(c2);
      const uint32_t m2 = __ballot_sync(0xffffffffu, c2 >= 0) & 0xFFFFu;
      if (i + 2 < my) copy_tile(true, false, vslot, 0u, r2);
      cp_async_commit();
      if (PAGED) {
        nidx = ppos;
        nblk = lookup(ppos);
        ppos = load_idx(i + 4);
      } else {
        nidx = load_idx(i + 3);
      }
      mask_cur = mask_n1;
      mask_n1 = m2;
      rec_n1 = r2;
    } else if (STAGES == 2) {
      mask_cur = mask_next;
    }
    if (!F::kSplitRing) __syncwarp();
  }

  // ---------------- merge the warps' partial results, one 128-dim half at a time
  cp_async_wait<0>();
#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l0 = f2add(l0, __shfl_xor_sync(0xffffffffu, l0, off));
    l1 = f2add(l1, __shfl_xor_sync(0xffffffffu, l1, off));
  }
  tmem_wait_st();
  __syncthreads();  // every warp is done with its ring: reuse the rings as the merge buffer
  constexpr int kORow = merge_row<FMT>();
  float* sO = reinterpret_cast<float*>(smem + L::kRing);  // [kWarps][16][kORow]
  float* sM = reinterpret_cast<float*>(smem + L::kM);
  float* sL = reinterpret_cast<float*>(smem + L::kL);
  float* sPost = reinterpret_cast<float*>(smem + L::kPost);
  // the references in log2 units (-inf for a head that saw no valid key)
  const float mu0 = R0 * fac0, mu1 = R1 * fac1;
  if (c == 0) {
    sM[warp * 16 + h0] = mu0;
    sM[warp * 16 + h1] = mu1;
    float a0, b0, a1, b1;
    f2unpack(l0, a0, b0);
    f2unpack(l1, a1, b1);
    sL[warp * 16 + h0] = a0 + b0;
    sL[warp * 16 + h1] = a1 + b1;
  }
  // the accumulators carry p times 2^(kPShift - eu) (int8) or 2^kPShift (E4M3, fp16); that power of
  // two is undone in the combine weights rather than on every accumulator value
  if (lane == 0) sPost[warp] = F::kInt8 ? pow2f(eu - kPShift) : (F::kBf16 ? 1.f : pow2f(-kPShift));
  __syncthreads();
  // combine weights, once per CTA: thread (hh, part) owns head hh and a quarter of each half's
  // head dims; warp w's partial enters with exp2(m_w - M) 2^(its pre-scale) / l
  const int hh = qh;  // = tid >> 3; part = tid & 7 as in the query staging
  float wo[kWarps];
  float lse_h = -INFINITY;
  if (hh < Gc) {
    float mw[kWarps], M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      mw[w] = sM[w * 16 + hh];
      M = fmaxf(M, mw[w]);
    }
    float ww[kWarps], lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      ww[w] = (mw[w] == -INFINITY) ? 0.f : fast_exp2(mw[w] - M);
      lsum += ww[w] * sL[w * 16 + hh];
    }
    float f = (lsum > 0.f) ? 1.f / lsum : 0.f;
    if (F::kE4m3 && P == 1) f *= a.v_scale_layer;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) wo[w] = ww[w] * sPost[w] * f;
    lse_h = (lsum > 0.f) ? (M + log2f(lsum)) * kLn2 : -INFINITY;
  }
#pragma unroll 1
  for (int sw = 0; sw < GM::kSweeps; ++sw) {
    {
      float ob[2][32];
      tmem_ld32(tacc + 64 * sw, ob[0]);
      tmem_ld32(tacc + 64 * sw + 32, ob[1]);
      tmem_wait_ld(ob[0]);
      tmem_wait_ld(ob[1]);
      if (F::kNatural) {
        // N-tile tt of the half holds local head dims 8 tt + 2c, 8 tt + 2c + 1 (heads h0, h1)
        float* o0 = sO + (warp * 16 + h0) * kORow + 2 * c;
        float* o1 = sO + (warp * 16 + h1) * kORow + 2 * c;
#pragma unroll
        for (int tt = 0; tt < 16; ++tt) {
          const float* q = &ob[tt >> 3][4 * (tt & 7)];
          *reinterpret_cast<float2*>(o0 + 8 * tt) = make_float2(q[0], q[1]);
          *reinterpret_cast<float2*>(o1 + 8 * tt) = make_float2(q[2], q[3]);
        }
      }
      // local head dim 32 c + x sits at 40 c + x of a head row: x < 8 and 16 <= x < 24 come
      // from quarter 0 (columns 2c and 2c + 1 of N-tile x mod 8), the others from quarter 1
      float* o0 = sO + (warp * 16 + h0) * kORow + 40 * c;
      float* o1 = sO + (warp * 16 + h1) * kORow + 40 * c;
#pragma unroll
      for (int k = 0; k < (F::kNatural ? 0 : 8); ++k) {
        const int b = (k >> 1) & 1;            // quarter of x = 4k .. 4k + 3
        const int j = (k >> 2);                // column 2c (0) or 2c + 1 (1)
        const int t = 4 * (k & 1);             // first N-tile within the quarter
        const float* q = ob[b];
        reinterpret_cast<float4*>(o0)[k] = make_float4(q[4 * t + j], q[4 * (t + 1) + j], q[4 * (t + 2) + j],
                                                       q[4 * (t + 3) + j]);
        reinterpret_cast<float4*>(o1)[k] = make_float4(q[4 * t + 2 + j], q[4 * (t + 1) + 2 + j],
                                                       q[4 * (t + 2) + 2 + j], q[4 * (t + 3) + 2 + j]);
      }
    }
    __syncthreads();
    {
      // part covers the local head dims d(k) .. d(k) + 3, k = 0..3 (natural layouts:
      // d(k) = 4 part + 32 k, so that 8 consecutive threads read all 32 banks; others:
      // d(k) = 16 part + 4 k, stored at 40 (part / 2) + 16 (part % 2) + 4 k)
      if (hh < Gc) {
        uint64_t res[8];  // 16 floats as packed pairs
#pragma unroll
        for (int i2 = 0; i2 < 8; ++i2) res[i2] = f2pack(0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float* src = sO + (w * 16 + hh) * kORow + (F::kNatural ? 4 * part : 40 * (part >> 1) + 16 * (part & 1));
          const uint64_t ww2 = f2pack(wo[w], wo[w]);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float4 x = *reinterpret_cast<const float4*>(src + (F::kNatural ? 32 * k : 4 * k));
            res[2 * k] = f2fma(f2pack(x.x, x.y), ww2, res[2 * k]);
            res[2 * k + 1] = f2fma(f2pack(x.z, x.w), ww2, res[2 * k + 1]);
          }
        }
        const int64_t qhead = hq0 + hh;
        float* dst = (P == 1) ? a.out + (r * Hq + qhead) * HD : a.o_part + ((r * P + split) * Hq + qhead) * HD;
        dst += 128 * sw + (F::kNatural ? 4 * part : 16 * part);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float4 y;
          f2unpack(res[2 * k], y.x, y.y);
          f2unpack(res[2 * k + 1], y.z, y.w);
          *reinterpret_cast<float4*>(dst + (F::kNatural ? 32 * k : 4 * k)) = y;
        }
        if (sw == 0 && part == 0) {
          const float lse = lse_h;
          if (P == 1) {
            if (a.lse != nullptr) a.lse[r * Hq + qhead] = lse;
          } else {
            a.lse_part[(r * P + split) * Hq + qhead] = lse;
          }
        }
      }
    }
    __syncthreads();  // the merge buffer is rewritten by the next half
  }

  // ---------------- fused split-K merge: the split CTA of this (row, KV head) that finishes
  // last merges all P partials into out / lse. No CTA waits for another: the others just leave.
  if (P > 1 && a.counters != nullptr) {
    uint32_t* sLast = reinterpret_cast<uint32_t*>(smem + L::kPost);  // the weights above are formed
    __threadfence();  // this CTA's partial is visible device-wide before it is announced
    __syncthreads();
    if (tid == 0) sLast[0] = (atomicAdd(a.counters + unit, 1u) == static_cast<uint32_t>(P - 1)) ? 1u : 0u;
    __syncthreads();
    if (sLast[0] != 0u) {
      __threadfence();  // order the reads of the other CTAs' partials after their announcements
      if (hh < Gc) {
        // thread (hh, part) merges head hh's float4 columns part + 8 i: 8 threads of a head
        // read one contiguous 128 B line per load
        int col4[HD / 32];
#pragma unroll
        for (int i = 0; i < HD / 32; ++i) col4[i] = part + 8 * i;
        const int64_t qhead = hq0 + hh;
        merge_head<HD / 32, 2>(a.o_part + (r * P * Hq + qhead) * HD, a.lse_part + r * P * Hq + qhead, Hq, P, HD,
                               F::kE4m3 ? a.v_scale_layer : 1.f, col4, a.out + (r * Hq + qhead) * HD,
                      (a.lse != nullptr && part == 0) ? a.lse + r * Hq + qhead : nullptr);
      }
      if (tid == 0) a.counters[unit] = 0u;  // every split has arrived: ready for the next call
    }
  }
  if (a.sched == nullptr) break;
  // next item: the query, the rings, the merge buffer and the accumulators are rewritten, so
  // every thread is past this one first
  tmem_fence_before_sync();
  __syncthreads();
  if (tid == 0) *sItem = gridDim.x + atomicAdd(a.sched, 1u);
  __syncthreads();
  tmem_fence_after_sync();
  bid = *sItem;
  if (bid >= num_items) break;
  }  // items
  if (a.sched != nullptr && tid == 0) {
    // the CTA that finishes last (every CTA has taken its last item by then) leaves the
    // counters zero for the next launch
    __threadfence();
    if (atomicAdd(a.sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(a.sched, 0u);
      atomicExch(a.sched + 1, 0u);
    }
  }
  // every warp's TMEM accesses are complete (the loads above were waited for): free the columns
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  if (warp == 0) tmem_dealloc(*sTmem, GM::kTmemAlloc);
}

// CTAs of one launch: (row, KV head, 16-head chunk, split).
inline int64_t gather_grid(const GatherArgs& a) {
  const int64_t chunks = (a.num_q_heads / a.num_kv_heads + kHeadsPerCta - 1) / kHeadsPerCta;
  return a.rows * a.num_kv_heads * chunks * a.num_splits;
}

// Opt the kernel into its dynamic shared memory, once per device. Host threads may race here on
// a device's first call: both set the same attributes (idempotent), and the flags are atomic.
template <int FMT, bool PAGED, int STAGES, int MINB, bool QF16 = false, int HD = 256>
cudaError_t prepare_variant() {
  static std::atomic<bool> attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(gather_attn_kernel<FMT, PAGED, STAGES, MINB, QF16, HD>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Smem<FMT, HD, STAGES>::kTotal));
    if (e != cudaSuccess) return e;
    // all of the unified L1 / shared array as shared memory: the copies bypass L1 anyway, and
    // the occupancy query then sees the CTAs per SM that a launch gets
    e = cudaFuncSetAttribute(gather_attn_kernel<FMT, PAGED, STAGES, MINB, QF16, HD>,
                             cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(true, std::memory_order_release);
  }
  return cudaSuccess;
}

// CTAs of a variant that one SM holds at once: the smaller of its shared-memory and register
// limits (registers allocated per warp in units of 256).
template <int FMT, bool PAGED, int STAGES, int MINB, bool QF16, int HD>
cudaError_t variant_ctas_per_sm(int* n) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, gather_attn_kernel<FMT, PAGED, STAGES, MINB, QF16, HD>);
  if (e != cudaSuccess) return e;
  int dev = 0, smem_sm = 0, reserved = 0, regs_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev)) != cudaSuccess) return e;
  const size_t per_cta = Smem<FMT, HD, STAGES>::kTotal + fa.sharedSizeBytes + static_cast<size_t>(reserved);
  const int by_smem = static_cast<int>(static_cast<size_t>(smem_sm) / per_cta);
  const int regs_warp = (fa.numRegs * 32 + 255) / 256 * 256;
  const int by_regs = regs_warp > 0 ? regs_sm / (regs_warp * Fmt<FMT>::kWarps) : by_smem;
  *n = by_smem < by_regs ? by_smem : by_regs;
  return cudaSuccess;
}

// CTAs of the variant that stay resident on the whole device (the persistent grid), once per
// device.
template <int FMT, bool PAGED, int STAGES, int MINB, bool QF16, int HD>
cudaError_t resident_ctas(int64_t* out) {
  static std::atomic<int64_t> cached[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int64_t n = cached[dev].load(std::memory_order_acquire);
  if (n == 0) {
    int per_sm = 0, sms = 0;
    if ((e = variant_ctas_per_sm<FMT, PAGED, STAGES, MINB, QF16, HD>(&per_sm)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    n = static_cast<int64_t>(per_sm > 0 ? per_sm : 1) * sms;
    cached[dev].store(n, std::memory_order_release);
  }
  *out = n;
  return cudaSuccess;
}

template <int FMT, bool PAGED, int STAGES = Fmt<FMT>::kStages, int MINB = Fmt<FMT>::kMinBlocks,
          bool QF16 = false, int HD = 256>
cudaError_t launch_variant(const GatherArgs& a, cudaStream_t stream) {
  cudaError_t e = prepare_variant<FMT, PAGED, STAGES, MINB, QF16, HD>();
  if (e != cudaSuccess) return e;
  int64_t grid = gather_grid(a);
  if (a.sched != nullptr) {
    int64_t resident = 0;
    e = resident_ctas<FMT, PAGED, STAGES, MINB, QF16, HD>(&resident);
    if (e != cudaSuccess) return e;
    grid = grid < resident ? grid : resident;
  }
  gather_attn_kernel<FMT, PAGED, STAGES, MINB, QF16, HD>
      <<<static_cast<unsigned>(grid), 32 * Fmt<FMT>::kWarps, Smem<FMT, HD, STAGES>::kTotal, stream>>>(a);
  return cudaGetLastError();
}

// The default ring and occupancy of the layout, for the launch's head dim (256 or 128).
template <int FMT, bool PAGED, bool QF16>
cudaError_t launch_hd(const GatherArgs& a, cudaStream_t stream) {
  constexpr int S = Fmt<FMT>::kStages, B = Fmt<FMT>::kMinBlocks;
  if (a.head_dim == 128) return launch_variant<FMT, PAGED, S, B, QF16, 128>(a, stream);
  return launch_variant<FMT, PAGED, S, B, QF16, 256>(a, stream);
}

// The query is IEEE half (FP16-activation contract).
template <int FMT>
cudaError_t launch_f16q(const GatherArgs& a, cudaStream_t stream) {
  return launch_hd<FMT, false, true>(a, stream);
}

// CTAs of the default kernel of this layout that one SM holds at once.
template <int FMT>
cudaError_t resident_ctas_per_sm(int* n) {
  constexpr int S = Fmt<FMT>::kStages, B = Fmt<FMT>::kMinBlocks;
  return variant_ctas_per_sm<FMT, false, S, B, false, 256>(n);
}

template <int FMT, bool PAGED = false>
cudaError_t launch(const GatherArgs& a, cudaStream_t stream) {
  return launch_hd<FMT, PAGED, false>(a, stream);
}

}  // namespace gather
}  // namespace qkv
