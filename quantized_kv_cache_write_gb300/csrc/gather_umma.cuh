// Top-k gather decode attention over an int8 pool with side-tensor scales: q.K^T on the
// fifth-generation tensor cores (tcgen05.mma, accumulators in tensor memory), p.V on mma.sync,
// with the warps specialised into two gather producers, an MMA issuer and eight compute warps.
//
// Pages: "int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next QSA path" §The finding
// worth upstreaming (each query row gathers its top-k scattered slots from an int8 pool with
// per-(token, head) scales); "[Perf][SM70][FP8] Hoist QSA E4M3 KV scales" §Changes (the K
// scale multiplies the logit after the dot product; the V scale is applied once per key, in
// p, instead of on every element); "[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache"
// §Implementation scope (split-K partials).
//
// A persistent grid of one CTA per SM walks the work items (row, KV head, K-split) of the launch
// in a fixed stride. An item's index columns are cut into blocks of 128 keys, and the CTA
// streams the blocks of all its items through one pipeline:
//   producers (warps 8, 9)  cp.async 16 B copies of each block's 128 K rows and V rows (256 B
//            each; 64 keys per warp) and scales into two three-stage rings, K and V apart
//            (one warp alone could not issue a block's copies in the time the compute warps
//            spend on it): K is consumed a block earlier than V, so each ring gets its full
//            depth of latency cover. 16 B chunk c of key row j sits at chunk (c + j) mod 16,
//            so that the row-wise K reads and the transposed V reads below are free of bank
//            conflicts.
//   compute (warps 0-7), per block g:
//     front  the two threads that own a key of block g + 1 dequantise its K row into tensor
//            memory, where it is the A operand of S^T[128 keys x 32] = K . Qs^T.
//     softmax  one thread per (key, 8 heads) reads its S^T row of block g and forms the logit
//            relative to the running reference M_h with fused multiply-adds,
//              d = (fma(ks_j, s_hi, -M_h) + ks_j s_lo) . fac_h   (log2 units),
//            so that near the maximum the difference keeps the dot product's full precision.
//            M_h is raised only when a logit exceeds it by 2^8 (a vote of the compute warps);
//            p = 2^d <= 2^8. p times the key's V scale and a power of two is split into fp16
//            hi + lo and stored as two 16 x 128 A operands.
//     p.V    mma.sync m16n8k16: warp w owns head dims 32 w .. 32 w + 31 of all 16 heads; V's B
//            fragments come from transposed byte-matrix loads of the int8 rows, turned into
//            exact fp16 by an exponent splice; two MMAs per fragment (p hi, p lo).
//   MMA (warp 10)  issues the 16 MMAs of each block's S^T once its K is in tensor memory.
//            Qs holds each query head twice: q_hi is the head, pre-scaled by a power of two,
//            rounded to multiples of 2^7; q_lo is the rest. Every partial sum of q_hi . codes is
//            a multiple of 2^7 below 2^31, exactly representable in fp32, so that half of the
//            dot product is exact in whatever order the tensor core adds; the q_lo half is 2^8
//            times smaller, so its rounding is too.
// The warps hand blocks to each other through mbarriers; every wait is bounded, and a wait that
// runs out sets QKV_DEV_TIMEOUT in the status word and stops the CTA (it then waits for its own
// copies and tensor-core work, frees its tensor memory and returns).
#pragma once

#include <atomic>
#include <cstdlib>
#include "qkv_internal.cuh"

namespace qkv {
namespace umma {

constexpr int kComputeWarps = 8;
constexpr int kCompute = 32 * kComputeWarps;  // compute threads (named barrier 1)
constexpr int kProducerWarps = 2;             // warps 8, 9: each gathers 64 keys of every block
constexpr int kProducerWarp0 = 8, kMmaWarp = kProducerWarp0 + kProducerWarps;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr int kKeys = 128;     // keys per block = tensor-memory lanes = M of q.K^T
constexpr int kHeads = 16;     // query heads per CTA (GQA groups up to 16)
constexpr int kN = 2 * kHeads; // q.K^T columns: q hi and q lo of every head
constexpr int kHD = 256;
constexpr int kStages = 3;
constexpr float kTau = 8.0f;      // lazy-rescale threshold (log2 units): p <= 2^8
constexpr int kPShift = 7;        // the fp16 p.V operand p v_scale 2^(7 - eu) stays below 2^15
constexpr int kEuHeadroom = 2;    // the V-scale bound 2^eu is raised 2^2 past the largest scale seen
constexpr int kQGrain = 7;        // q_hi is a multiple of 2^7 (the pre-scaled head maximum is below 2^15)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kWaitLimit = 1u << 22;  // mbarrier polls before a wait is declared lost (about a second)

// ---------------------------------------------------------------- shared memory (bytes)
constexpr uint32_t kRow = kHD;  // one int8 K or V row
// K ring stage: rows only (released once dequantised)
constexpr uint32_t kKStage = kKeys * kRow;
// V ring stage: rows, V scales, K scales, checked slot ids (-1: none) -- everything the softmax
// and p.V of the block read, released together after p.V
constexpr uint32_t kVsOff = kKeys * kRow, kKsOff = kVsOff + 4 * kKeys, kIdxOff = kKsOff + 4 * kKeys;
constexpr uint32_t kVStage = kIdxOff + 4 * kKeys;
constexpr uint32_t kKRing = 0;
constexpr uint32_t kVRing = kKRing + kStages * kKStage;
// Qs: [32 rows n][256 k] fp16, K-major, no swizzle: (n, k) at (n%8)16 + (n/8)SBO + (k%8)2 + (k/8)LBO
constexpr uint32_t kQ = kVRing + kStages * kVStage;
constexpr uint32_t kQLbo = 128, kQSbo = 128 * (kHD / 8);
// Ps: p hi then p lo, each [16 heads][128 k-columns] fp16, rows padded to 272 B (the eight rows
// an ldmatrix phase reads start on distinct 16 B banks)
constexpr uint32_t kP = kQ + kN * kHD * 2;
constexpr uint32_t kPRow = 2 * kKeys + 16;
constexpr uint32_t kPPart = kHeads * kPRow;
constexpr uint32_t kRedM = kP + 2 * kPPart;      // [8 warps][8] block maxima
constexpr uint32_t kRedL = kRedM + 8 * 8 * 4;    // [8 warps][8] row-sum partials
constexpr uint32_t kRedV = kRedL + 8 * 8 * 4;    // [8 warps] V-scale maxima (fp32 bits)
constexpr uint32_t kM = kRedV + 8 * 4;           // [16] references M_h
constexpr uint32_t kAlpha = kM + 16 * 4;         // [16] rescale factors of the last raise
constexpr uint32_t kFac = kAlpha + 16 * 4;       // [2 items][16] logit factor per head
constexpr uint32_t kBar = kFac + 2 * 16 * 4;     // mbarriers (8 B each), see below
constexpr uint32_t kBarKFull = kBar, kBarKEmpty = kBar + 24, kBarVFull = kBar + 48, kBarVEmpty = kBar + 72;
constexpr uint32_t kBarTK = kBar + 96;   // [2] K of block g in tensor memory (compute -> MMA)
constexpr uint32_t kBarS = kBar + 112;   // [2] S^T of block g complete (MMA -> compute)
constexpr uint32_t kTmemSlot = kBar + 128;
constexpr uint32_t kFlag = kTmemSlot + 4;  // a wait ran out: the CTA stops
constexpr uint32_t kEu = kFlag + 4;        // the V-scale bound exponent
constexpr uint32_t kSmemTotal = kEu + 4;
static_assert(kBar % 8 == 0, "mbarrier alignment");
static_assert(kQ % 16 == 0 && kP % 16 == 0 && kKStage % 16 == 0 && kVStage % 16 == 0, "alignment");
static_assert(kSmemTotal <= 232448, "one CTA per SM");

// ---------------------------------------------------------------- tensor memory (columns)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTK = 0;    // K operand, two buffers of 128 columns: lane = key, column c = k-indices 2c, 2c + 1
constexpr uint32_t kTS = 256;  // S^T accumulators, two buffers of 32 columns: lane = key, column n

// Instruction descriptor (kind::f16: fp16 A and B, fp32 D; M = 128, N = 32; A in tensor memory,
// B K-major): bits 4-5 D format (1 = fp32), 17-22 N / 8, 24-28 M / 16.
constexpr uint32_t kIdescS = (1u << 4) | (uint32_t(kN >> 3) << 17) | (uint32_t(kKeys >> 4) << 24);

// Shared-memory matrix descriptor, no swizzle: start address, leading-dimension byte offset
// (between core matrices along K), stride byte offset (along M / N), version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46);
}
__device__ __forceinline__ void mma_a_tmem(uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar)
               : "memory");
}
__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(mbar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(mbar) : "memory");
}
// the arrival happens once every cp.async this thread issued before it has completed
__device__ __forceinline__ void mbar_arrive_cp(uint32_t mbar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(mbar) : "memory");
}
// Wait for the phase with the given parity to complete; false if `limit` polls ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, uint32_t limit) {
  for (uint32_t it = 0; it < limit; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(mbar), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }  // e in [-126, 127]
// named barrier 1: the compute warps only
__device__ __forceinline__ void bar_compute() { asm volatile("bar.sync 1, %0;\n" ::"n"(kCompute) : "memory"); }
__device__ __forceinline__ bool bar_compute_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kCompute)
      : "memory");
  return r != 0u;
}

__device__ __forceinline__ void tmem_st_u32x32(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld_x8(uint32_t taddr, float (&v)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld8(float (&v)[8]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n"
               : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]), "+f"(v[7])::"memory");
}

// Head-dim order inside the fp16 K operand: the int8 -> fp16 splice turns code bytes (0, 2) and
// (1, 3) of a word into one fp16 pair each, so k-index 4i + {0, 1, 2, 3} holds head dim
// 4i + {0, 2, 1, 3}; the staged query follows the same order.
__host__ __device__ __forceinline__ int dim_of(int k) { return (k & ~3) | ((k & 1) << 1) | ((k >> 1) & 1); }
// Column of key kk (0..15 within a 16-key step) in the p.V A operand: the B fragments built from a
// transposed byte matrix hold keys (4c, 4c + 2) in k-indices (2c, 2c + 1) and (4c + 1, 4c + 3) in
// (2c + 8, 2c + 9).
__device__ __forceinline__ int pcol_of(int kk) { return 2 * (kk >> 2) + ((kk >> 1) & 1) + 8 * (kk & 1); }

struct Item {
  int64_t r;
  int h, split, c0, c1, nb;
};

// (row, KV head, split) of work item `it`, its index columns [c0, c1) and its 128-key blocks.
__device__ __forceinline__ Item item_info(const GatherArgs& a, int64_t it) {
  Item t;
  const int P = a.num_splits, H = a.num_kv_heads;
  t.split = static_cast<int>(it % P);
  const int64_t unit = it / P;
  t.h = static_cast<int>(unit % H);
  t.r = unit / H;
  int len = a.topk;
  if (a.topk_len != nullptr) len = min(max(__ldg(a.topk_len + t.r), 0), a.topk);
  const int per = (a.topk + P - 1) / P;
  t.c0 = min(len, t.split * per);
  t.c1 = min(len, t.split * per + per);
  t.nb = (t.c1 - t.c0 + kKeys - 1) / kKeys;
  return t;
}

// A position in the sequence of 128-key blocks of one CTA's items (items without a valid column
// have no blocks and are skipped).
struct Cursor {
  int64_t it;  // >= num_items: past the end
  Item info;
  int bi;
};
__device__ __forceinline__ void cursor_settle(const GatherArgs& a, Cursor& c, int64_t num_items, int64_t stride) {
  while (c.it < num_items && c.bi >= c.info.nb) {
    c.it += stride;
    c.bi = 0;
    if (c.it < num_items) c.info = item_info(a, c.it);
  }
}
__device__ __forceinline__ Cursor cursor_first(const GatherArgs& a, int64_t num_items, int64_t stride) {
  Cursor c;
  c.it = blockIdx.x;
  c.bi = 0;
  if (c.it < num_items) c.info = item_info(a, c.it);
  cursor_settle(a, c, num_items, stride);
  return c;
}
__device__ __forceinline__ void cursor_next(const GatherArgs& a, Cursor& c, int64_t num_items, int64_t stride) {
  ++c.bi;
  cursor_settle(a, c, num_items, stride);
}
__device__ __forceinline__ Cursor cursor_next_item(const GatherArgs& a, Cursor c, int64_t num_items, int64_t stride) {
  c.bi = c.info.nb;
  cursor_settle(a, c, num_items, stride);
  return c;
}

// wait_limit: mbarrier polls before a wait is declared lost (kWaitLimit). drop_tk: the block
// whose K hand-off to the MMA warp the compute warps leave out, -1 for none -- a test of the
// lost-wait path (see launch); with it, the MMA warp's wait for that block and the compute
// warps' wait for its scores both run out, and the CTA winds down with QKV_DEV_TIMEOUT set.
template <int FMT>
__global__ void __launch_bounds__(kThreads, 1)
    umma_gather_kernel(const GatherArgs a, int64_t num_items, uint32_t wait_limit, int64_t drop_tk) {
  static_assert(FMT == QKV_INT8_SIDE, "int8 pool with side-tensor scales");
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t sb = smem_u32(smem);
  const int H = a.num_kv_heads, Hq = a.num_q_heads, G = Hq / H, P = a.num_splits;
  const int64_t stride = gridDim.x;
  volatile uint32_t* sFlag = reinterpret_cast<volatile uint32_t*>(smem + kFlag);
  float* sFac = reinterpret_cast<float*>(smem + kFac);
  float* sM = reinterpret_cast<float*>(smem + kM);
  float* sAlpha = reinterpret_cast<float*>(smem + kAlpha);
  float* sRedM = reinterpret_cast<float*>(smem + kRedM);
  float* sRedL = reinterpret_cast<float*>(smem + kRedL);
  uint32_t* sRedV = reinterpret_cast<uint32_t*>(smem + kRedV);

  if (warp == 0) {
    tmem_alloc(sb + kTmemSlot, kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  if (tid == kThreads - 1) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(sb + kBarKFull + 8 * s, 32 * kProducerWarps);  // copy-completion arrivals
      mbar_init(sb + kBarKEmpty + 8 * s, 1);
      mbar_init(sb + kBarVFull + 8 * s, 64 * kProducerWarps);  // copy-completion and ordinary (slot ids)
      mbar_init(sb + kBarVEmpty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sb + kBarTK + 8 * b, 1);
      mbar_init(sb + kBarS + 8 * b, 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    *sFlag = 0u;
  }
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(smem + kTmemSlot);

  if (warp >= kProducerWarp0 && warp < kMmaWarp) {
    // ================================================================ producers
    // Producer warp p gathers its share of the keys of every block: their K rows as soon as the
    // block's K stage is free, then their V rows, scales and slot ids as soon as the V stage is.
    const int pw = warp - kProducerWarp0;
    constexpr int kPer = kKeys / 32 / kProducerWarps;  // 32-key groups per producer warp
    Cursor pc = cursor_first(a, num_items, stride);
    int idx[kPer], prev_rec[kPer], prev_idx[kPer];  // this lane's keys 32 (kPer pw + i) + lane: the
                                                    // next block's entries; the last block's
                                                    // records and checked slot ids
    Cursor vc = pc;           // the block whose V rows are issued next
    auto load_idx = [&](const Cursor& c) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        idx[i] = -1;
        if (c.it < num_items) {
          const int col = c.info.c0 + c.bi * kKeys + 32 * (kPer * pw + i) + lane;
          if (col < c.info.c1) idx[i] = __ldg(a.topk_idx + c.info.r * a.topk + col);
        }
      }
    };
    // copies of this warp's rows of one ring stage: 16 lanes per 256 B row, two rows per
    // instruction
    auto copy_rows = [&](uint32_t dst_base, const uint8_t* src, const int (&rec)[kPer]) {
      const int c = lane & 15;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
#pragma unroll 4
        for (int pp = 0; pp < 16; ++pp) {
          const int kl = 2 * pp + (lane >> 4);  // key 32 (kPer pw + i) + kl, held by lane kl
          const int key = 32 * (kPer * pw + i) + kl;
          const int rk = __shfl_sync(0xffffffffu, rec[i], kl);
          const uint32_t dst = dst_base + key * kRow + (((c + key) & 15) << 4);
          cp_async16(dst, src + static_cast<uint64_t>(static_cast<uint32_t>(max(rk, 0))) * kRow + 16 * c,
                     rk >= 0 ? 16 : 0);  // padding copies nothing and zero-fills its row
        }
      }
    };
    load_idx(pc);
    int64_t kb = 0, vb = 0;  // blocks whose K / V rows were issued
    bool ok = true;
    while (ok && (pc.it < num_items || vc.it < num_items)) {
      if (pc.it < num_items) {
        const int st = static_cast<int>(kb % kStages);
        const uint32_t stb = sb + kKRing + st * kKStage;
        if (kb >= kStages) {
          int stop = 0;
          if (lane == 0) {
            if (!mbar_wait(sb + kBarKEmpty + 8 * st, static_cast<uint32_t>((kb / kStages - 1) & 1), wait_limit)) *sFlag = 1u;
            stop = *sFlag != 0u;
          }
          if (__shfl_sync(0xffffffffu, stop, 0)) { ok = false; break; }
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          int v = idx[i];
          if (v < -1 || static_cast<int64_t>(v) >= a.num_slots) {  // out of range: flagged, read as padding
            if (a.dev_status != nullptr) atomicOr(a.dev_status, QKV_DEV_BAD_INDEX);
            v = -1;
          }
          prev_idx[i] = v;
          prev_rec[i] = v >= 0 ? v * H + pc.info.h : -1;
        }
        copy_rows(stb, a.k_cache, prev_rec);
        mbar_arrive_cp(sb + kBarKFull + 8 * st);
        ++kb;
        cursor_next(a, pc, num_items, stride);
        load_idx(pc);
      }
      // V rows of the block whose K went out last (one behind the K stream, or the tail)
      if (vb < kb) {
        const int st = static_cast<int>(vb % kStages);
        const uint32_t stb = sb + kVRing + st * kVStage;
        if (vb >= kStages) {
          int stop = 0;
          if (lane == 0) {
            if (!mbar_wait(sb + kBarVEmpty + 8 * st, static_cast<uint32_t>((vb / kStages - 1) & 1), wait_limit)) *sFlag = 1u;
            stop = *sFlag != 0u;
          }
          if (__shfl_sync(0xffffffffu, stop, 0)) { ok = false; break; }
        }
        // vb == kb - 1: its slots are prev_rec; its slot ids and both scales travel with V
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int key = 32 * (kPer * pw + i) + lane, rk = prev_rec[i];
          sts32(stb + kIdxOff + 4 * key, static_cast<uint32_t>(prev_idx[i]));
          cp_async4(stb + kVsOff + 4 * key, a.v_scale_tok + max(rk, 0), rk >= 0 ? 4 : 0);
          cp_async4(stb + kKsOff + 4 * key, a.k_scale_tok + max(rk, 0), rk >= 0 ? 4 : 0);
        }
        copy_rows(stb, a.v_cache, prev_rec);
        mbar_arrive_cp(sb + kBarVFull + 8 * st);
        mbar_arrive(sb + kBarVFull + 8 * st);
        ++vb;
        cursor_next(a, vc, num_items, stride);
      }
    }
  } else if (warp == kMmaWarp) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      Cursor c = cursor_first(a, num_items, stride);
      int64_t gk = 0;
      for (; c.it < num_items; ++gk) {
        const int b = static_cast<int>(gk & 1);
        if (!mbar_wait(sb + kBarTK + 8 * b, static_cast<uint32_t>((gk >> 1) & 1), wait_limit)) {
          *sFlag = 1u;
          break;
        }
        if (*sFlag != 0u) break;
        tmem_fence_after_sync();
        const uint32_t kbuf = kTK + 128 * b, sbuf = kTS + 32 * b;
#pragma unroll
        for (int ks = 0; ks < kHD / 16; ++ks)
          mma_a_tmem(tbase + sbuf, tbase + kbuf + 8 * ks, sdesc(sb + kQ + ks * 2 * kQLbo, kQLbo, kQSbo), kIdescS,
                     ks > 0 ? 1u : 0u);
        mma_commit(sb + kBarS + 8 * b);
        cursor_next(a, c, num_items, stride);
      }
      // after an abort the compute warps may not wait for the last batch: it completes before the
      // tensor memory it writes is freed
      if (gk > 0 && *sFlag != 0u)
        mbar_wait(sb + kBarS + 8 * ((gk - 1) & 1), static_cast<uint32_t>(((gk - 1) >> 1) & 1), wait_limit);
    }
    __syncwarp();
  } else {
    // ================================================================ compute warps
    const int q4 = warp & 3, hf = warp >> 2;
    const int j = 32 * q4 + lane;  // the key of a block this thread dequantises and scores
    const int fg = lane >> 2, fc = lane & 3;  // mma fragment row group / column pair
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;

    // items with no valid column: zero output, lse = -inf
    for (int64_t it = blockIdx.x; it < num_items; it += stride) {
      const Item t = item_info(a, it);
      if (t.nb != 0) continue;
      const int64_t hq0 = static_cast<int64_t>(t.h) * G;
      for (int e = tid; e < G * kHD; e += kCompute) {
        if (P == 1) a.out[(t.r * Hq + hq0) * kHD + e] = 0.f;
        else a.o_part[((t.r * P + t.split) * Hq + hq0) * kHD + e] = 0.f;
      }
      if (tid < G) {
        if (P == 1) {
          if (a.lse != nullptr) a.lse[t.r * Hq + hq0 + tid] = -INFINITY;
        } else {
          a.lse_part[(t.r * P + t.split) * Hq + hq0 + tid] = -INFINITY;
        }
      }
    }

    // thread 0 polls an mbarrier for the compute warps; true when its wait ran out
    auto wait0 = [&](uint32_t mbar, uint32_t parity) -> bool {
      if (tid == 0 && !mbar_wait(mbar, parity, wait_limit)) {
        *sFlag = 1u;
        return true;
      }
      return false;
    };
    // barrier of the compute warps that also agrees on stopping (the flag may be set by another
    // warp at any time, so each thread's reading is OR-ed into one result)
    auto sync_go = [&](bool failed) -> bool { return !bar_compute_or(failed || *sFlag != 0u); };

    // query staging (thread (head qh, part) holds 16 dims, prefetched an item ahead)
    const int qh = tid >> 4, qpart = tid & 15;
    uint4 qn[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    auto q_prefetch = [&](const Cursor& c) {
      if (c.it < num_items && qh < G) {
        const uint4* p =
            reinterpret_cast<const uint4*>(a.q + (c.info.r * Hq + c.info.h * G + qh) * kHD + 16 * qpart);
        qn[0] = __ldg(p);
        qn[1] = __ldg(p + 1);
      }
    };
    // per head a power of two puts max |q| in [2^14, 2^15); q_hi = that rounded to a multiple of
    // 2^7, q_lo = the remainder (both exact in fp16). Writes Qs and the logit factors (buffer fb).
    auto stage_q = [&](int fb) {
      const uint32_t w[8] = {qn[0].x, qn[0].y, qn[0].z, qn[0].w, qn[1].x, qn[1].y, qn[1].z, qn[1].w};
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) m = max(m, max((w[i] & 0x7FFFu) << 16, w[i] & 0x7FFF0000u));
#pragma unroll
      for (int off = 1; off <= 8; off <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
      const int sg = m ? max(-64, min(64, 14 - (static_cast<int>(m >> 23) - 127))) : 0;
      const float u = pow2f(sg);
      uint32_t hi[8], lo[8];
#pragma unroll
      for (int kk = 0; kk < 16; kk += 2) {
        float xh[2], xl[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int d = dim_of(kk + e);  // dim within the thread's 16 (k-indices 16 qpart + kk)
          const uint32_t b = (d & 1) ? (w[d >> 1] & 0xFFFF0000u) : (w[d >> 1] << 16);
          const float x = (qh < G) ? __uint_as_float(b) * u : 0.f;
          const float xhv = rintf(x * (1.0f / (1 << kQGrain))) * static_cast<float>(1 << kQGrain);
          xh[e] = xhv;
          xl[e] = x - xhv;
        }
        hi[kk >> 1] = pack_half2(xh[0], xh[1]);
        lo[kk >> 1] = pack_half2(xl[0], xl[1]);
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int n = half ? kHeads + qh : qh;
        const uint32_t* v = half ? lo : hi;
#pragma unroll
        for (int kg = 0; kg < 2; ++kg)
          sts128(sb + kQ + (n & 7) * 16 + (n >> 3) * kQSbo + (2 * qpart + kg) * kQLbo,
                 make_uint4(v[4 * kg], v[4 * kg + 1], v[4 * kg + 2], v[4 * kg + 3]));
      }
      if (qpart == 0) sFac[16 * fb + qh] = (qh < G) ? a.softmax_scale * kLog2e * pow2f(-sg) : 0.f;
      fence_async_smem();
    };
    // K of block gk (K stage gk % kStages) into tensor-memory buffer gk % 2
    auto dequant_k = [&](int64_t gk) {
      const uint32_t row = sb + kKRing + static_cast<uint32_t>(gk % kStages) * kKStage + j * kRow;
      const uint32_t tk = tbase + lane_off + kTK + 128 * static_cast<uint32_t>(gk & 1) + 64 * hf;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        uint32_t kw[32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int c = 8 * hf + 4 * part + cc;
          const uint4 x = lds128(row + (((c + j) & 15) << 4));
          kw[8 * cc + 0] = i8pair_to_f16x2(x.x);
          kw[8 * cc + 1] = i8pair_to_f16x2(x.x >> 8);
          kw[8 * cc + 2] = i8pair_to_f16x2(x.y);
          kw[8 * cc + 3] = i8pair_to_f16x2(x.y >> 8);
          kw[8 * cc + 4] = i8pair_to_f16x2(x.z);
          kw[8 * cc + 5] = i8pair_to_f16x2(x.z >> 8);
          kw[8 * cc + 6] = i8pair_to_f16x2(x.w);
          kw[8 * cc + 7] = i8pair_to_f16x2(x.w >> 8);
        }
        tmem_st_u32x32(tk + 32 * part, kw);
      }
      tmem_wait_st();
    };

    // ---------------- prologue: the first block's query and K
    Cursor fcur = cursor_first(a, num_items, stride);  // front: next block whose K is dequantised
    Cursor bcur = fcur;                                 // back: next block whose softmax and p.V run
    int f_items = 0, b_items = 0;  // items begun by the front / back (parity = logit-factor buffer)
    bool aborted = false;
    if (fcur.it < num_items && !sync_go(wait0(sb + kBarKFull, 0u))) aborted = true;
    if (fcur.it < num_items && !aborted) {
      q_prefetch(fcur);
      stage_q(0);
      ++f_items;
      q_prefetch(cursor_next_item(a, fcur, num_items, stride));
      dequant_k(0);
      tmem_fence_before_sync();
      bar_compute();
      if (tid == 0) {
        if (drop_tk != 0) mbar_arrive(sb + kBarTK);
        mbar_arrive(sb + kBarKEmpty);  // block 0's K rows are no longer needed
      }
      cursor_next(a, fcur, num_items, stride);
    }

    // softmax state: this thread's row sums (its 8 heads), this warp's p.V accumulators (its 32
    // head dims of heads fg and fg + 8), the V-scale bound; the references live in shared memory
    float l[8];
    float acc[4][4];
    int eu = -100;
    float M0 = 0.f, M1 = 0.f;  // references of heads fg, fg + 8 (for the epilogue's lse)
    for (int64_t g = 0; bcur.it < num_items && !aborted; ++g) {
      const bool item_first = bcur.bi == 0, item_last = bcur.bi == bcur.info.nb - 1;
      const int kst = static_cast<int>(g % kStages);
      const uint32_t vstb = sb + kVRing + kst * kVStage;
      // ---- front: K of block g + 1 into tensor memory (a new item first restages Qs, once the
      //      q.K^T of block g has read the old one)
      const bool front = fcur.it < num_items;
      if (front) {
        const int fst = static_cast<int>((g + 1) % kStages);
        if (fcur.bi == 0) {
          if (!sync_go(wait0(sb + kBarS + 8 * static_cast<uint32_t>(g & 1), static_cast<uint32_t>((g >> 1) & 1)))) {
            aborted = true;
            break;
          }
          stage_q(f_items & 1);
          ++f_items;
          q_prefetch(cursor_next_item(a, fcur, num_items, stride));
        }
        if (!sync_go(wait0(sb + kBarKFull + 8 * fst, static_cast<uint32_t>(((g + 1) / kStages) & 1)))) {
          aborted = true;  // (otherwise block g + 1's K rows are visible)
          break;
        }
        dequant_k(g + 1);
        tmem_fence_before_sync();
        bar_compute();
        if (tid == 0) {
          if (g + 1 != drop_tk) mbar_arrive(sb + kBarTK + 8 * static_cast<uint32_t>((g + 1) & 1));
          mbar_arrive(sb + kBarKEmpty + 8 * fst);  // its K rows are no longer needed
        }
      }
      // ---- softmax of block g (its S^T, its V scales)
      const bool f1 = wait0(sb + kBarS + 8 * static_cast<uint32_t>(g & 1), static_cast<uint32_t>((g >> 1) & 1));
      const bool f2 = !f1 && wait0(sb + kBarVFull + 8 * kst, static_cast<uint32_t>((g / kStages) & 1));
      if (item_first && tid < kHeads) sM[tid] = (tid < G) ? -INFINITY : 0.f;
      if (!sync_go(f1 || f2)) {
        aborted = true;
        break;
      }
      if (item_first) {
#pragma unroll
        for (int e = 0; e < 8; ++e) l[e] = 0.f;
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
        eu = -100;
        ++b_items;
      }
      const float* fac = sFac + 16 * ((b_items - 1) & 1);
      tmem_fence_after_sync();
      const bool valid = static_cast<int32_t>(lds32(vstb + kIdxOff + 4 * j)) >= 0;
      const float ksc = __uint_as_float(lds32(vstb + kKsOff + 4 * j));
      const uint32_t vsc_bits = lds32(vstb + kVsOff + 4 * j);
      const float vsc = __uint_as_float(vsc_bits);
      float shi[8], slo[8];
      {
        const uint32_t ts = tbase + lane_off + kTS + 32 * static_cast<uint32_t>(g & 1);
        tmem_ld_x8(ts + 8 * hf, shi);
        tmem_ld_x8(ts + kHeads + 8 * hf, slo);
        tmem_wait_ld8(shi);
        tmem_wait_ld8(slo);
        tmem_fence_before_sync();  // this buffer is rewritten by a later q.K^T
      }
      float d[8], Mh[8], fh[8];
      bool exceed = valid && eu < 127 && vsc_bits >= static_cast<uint32_t>(max(eu + 127, 0)) << 23;
#pragma unroll
      for (int e = 0; e < 8; ++e) {  // this thread's heads 8 hf + e
        Mh[e] = sM[8 * hf + e];
        fh[e] = fac[8 * hf + e];
        d[e] = valid ? fmaf(ksc, slo[e], fmaf(ksc, shi[e], -Mh[e])) * fh[e] : -INFINITY;
        exceed |= d[e] > kTau;
      }
      if (bar_compute_or(exceed)) {  // rare after an item's first block: raise the references
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float mv = valid ? ksc * (shi[e] + slo[e]) : -INFINITY;
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, off));
          if (lane == 0) sRedM[warp * 8 + e] = mv;
        }
        const uint32_t vm = __reduce_max_sync(0xffffffffu, valid ? (vsc_bits & 0x7FFFFFFFu) : 0u);
        if (lane == 0) sRedV[warp] = vm;
        bar_compute();
        uint32_t vmax = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) vmax = max(vmax, sRedV[w]);
        int ne = eu;
        if (vmax != 0u) {
          const int ev = static_cast<int>(vmax >> 23) - 126;  // 2^ev > the largest V scale
          if (ev > eu) ne = ev + kEuHeadroom;
        }
        if (tid < kHeads) {  // head tid: its new reference and the factor on what it has so far
          const int h = tid;
          float bm = -INFINITY;
#pragma unroll
          for (int w = 0; w < 4; ++w) bm = fmaxf(bm, sRedM[(4 * (h >> 3) + w) * 8 + (h & 7)]);
          const float om = sM[h], fh_ = fac[h];
          float nm = om;
          if (h < G && bm != -INFINITY && (om == -INFINITY || (bm - om) * fh_ > kTau)) nm = bm;
          sAlpha[h] = (nm == om) ? 1.f : (om == -INFINITY ? 0.f : fast_exp2((om - nm) * fh_));
          sM[h] = nm;
        }
        bar_compute();
        const float ov = pow2f(max(eu - ne, -126));
        const float r0 = sAlpha[fg] * ov, r1 = sAlpha[fg + 8] * ov;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          acc[t][0] *= r0;
          acc[t][1] *= r0;
          acc[t][2] *= r1;
          acc[t][3] *= r1;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          Mh[e] = sM[8 * hf + e];
          l[e] *= sAlpha[8 * hf + e];
          d[e] = valid ? fmaf(ksc, slo[e], fmaf(ksc, shi[e], -Mh[e])) * fh[e] : -INFINITY;
        }
        eu = ne;
      }
      // p = 2^d; p v_scale 2^(7 - eu) as fp16 hi and lo into the A operands, column pcol(j)
      {
        const float pm = vsc * pow2f(kPShift - eu);
        const uint32_t col = 2u * static_cast<uint32_t>(16 * (j >> 4) + pcol_of(j & 15));
        const uint32_t ph = sb + kP + col, pl = ph + kPPart;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float p = fast_exp2(d[e]);  // masked: 2^-inf = 0
          l[e] += p;
          const float x = p * pm;
          const __half xh = __float2half_rn(x);
          const __half xl = __float2half_rn(x - __half2float(xh));
          const uint32_t rowoff = static_cast<uint32_t>(8 * hf + e) * kPRow;
          asm volatile("st.shared.b16 [%0], %1;\n" ::"r"(ph + rowoff), "h"(__half_as_ushort(xh)));
          asm volatile("st.shared.b16 [%0], %1;\n" ::"r"(pl + rowoff), "h"(__half_as_ushort(xl)));
        }
      }
      bar_compute();  // the p operands of block g are complete

      // ---- p.V of block g: this warp's head dims 32 warp .. + 31 (four N-tiles of 8)
      {
        const int mrow = lane & 15;               // ldmatrix: key row of the 16-key step
        const int cidx = 2 * warp + (lane >> 4);  // 16-dim chunk of this lane's matrix
        // A fragments: lanes 0-7 rows 0-7, 8-15 rows 8-15 at k 0; 16-23 / 24-31 the same at k 8
        const uint32_t pa = sb + kP + static_cast<uint32_t>(lane & 15) * kPRow + 16u * (lane >> 4);
#pragma unroll 2
        for (int ks = 0; ks < kKeys / 16; ++ks) {
          const int key = 16 * ks + mrow;
          uint32_t v[4];
          ldmatrix_x2_trans_b8(vstb + key * kRow + (((cidx + key) & 15) << 4), v[0], v[1], v[2], v[3]);
          uint32_t ahi[4], alo[4];
          ldmatrix_x4(pa + 32u * ks, ahi[0], ahi[1], ahi[2], ahi[3]);
          ldmatrix_x4(pa + kPPart + 32u * ks, alo[0], alo[1], alo[2], alo[3]);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint32_t b0 = i8pair_to_f16x2(v[t]), b1 = i8pair_to_f16x2(v[t] >> 8);
            mma_f16(acc[t], ahi, b0, b1);
            mma_f16(acc[t], alo, b0, b1);
          }
        }
      }
      if (item_last) {  // the references of this warp's output heads, before they are reset
        M0 = sM[fg];
        M1 = sM[fg + 8];
      }
      bar_compute();  // block g's V stage and the p operands are free
      if (tid == 0) mbar_arrive(sb + kBarVEmpty + 8 * kst);

      // ---- item epilogue: normalise and write this item's output (or split partial)
      if (item_last) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float s = l[e];
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
          if (lane == 0) sRedL[warp * 8 + e] = s;
        }
        bar_compute();
        const Item& ci = bcur.info;
        const int64_t hq0 = static_cast<int64_t>(ci.h) * G;
        float* dst = (P == 1) ? a.out + (ci.r * Hq + hq0) * kHD : a.o_part + ((ci.r * P + ci.split) * Hq + hq0) * kHD;
        const float post = pow2f(eu - kPShift);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int h = fg + 8 * hh;
          float lh = 0.f;
#pragma unroll
          for (int w = 0; w < 4; ++w) lh += sRedL[(4 * hh + w) * 8 + fg];
          const float f = lh > 0.f ? post / lh : 0.f;
          if (h < G) {
#pragma unroll
            for (int t = 0; t < 4; ++t)
              *reinterpret_cast<float2*>(dst + h * kHD + 32 * warp + 8 * t + 2 * fc) =
                  make_float2(acc[t][2 * hh] * f, acc[t][2 * hh + 1] * f);
            if (warp == 0 && fc == 0) {
              const float lse = lh > 0.f ? ((hh ? M1 : M0) * fac[h] + log2f(lh)) * kLn2 : -INFINITY;
              if (P == 1) {
                if (a.lse != nullptr) a.lse[ci.r * Hq + hq0 + h] = lse;
              } else {
                a.lse_part[(ci.r * P + ci.split) * Hq + hq0 + h] = lse;
              }
            }
          }
        }
        bar_compute();  // sRedL and the references are rewritten by the next item
      }
      cursor_next(a, bcur, num_items, stride);
      if (front) cursor_next(a, fcur, num_items, stride);
    }
  }

  // ---------------- every warp: wait for the CTA's outstanding work, free tensor memory
  cp_async_wait<0>();
  tmem_fence_before_sync();
  __syncthreads();
  if (*sFlag != 0u && tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, QKV_DEV_TIMEOUT);
  tmem_fence_after_sync();
  if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

// Opt into the dynamic shared memory once per device; the SM count is cached with it.
template <int FMT>
cudaError_t prepare(int* sms) {
  static std::atomic<int> sm_count[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int n = sm_count[dev].load(std::memory_order_acquire);
  if (n == 0) {
    e = cudaFuncSetAttribute(umma_gather_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemTotal));
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidDevice;
    sm_count[dev].store(n, std::memory_order_release);
  }
  *sms = n;
  return cudaSuccess;
}

template <int FMT>
cudaError_t launch(const GatherArgs& a, cudaStream_t stream) {
  int sms = 0;
  cudaError_t e = prepare<FMT>(&sms);
  if (e != cudaSuccess) return e;
  const int64_t items = a.rows * a.num_kv_heads * a.num_splits;
  const int grid = static_cast<int>(items < sms ? items : sms);
  // Test of the lost-wait path: QKV_TEST_TCGEN05_DROP_HANDOFF=<block> makes the compute warps
  // leave out that block's K hand-off (read at each launch; unset in any other use). The poll
  // limit then drops to 2^14, so that the waits run out in milliseconds, not seconds.
  int64_t drop_tk = -1;
  uint32_t wait_limit = kWaitLimit;
  if (const char* t = std::getenv("QKV_TEST_TCGEN05_DROP_HANDOFF")) {
    char* end = nullptr;
    const long long b = std::strtoll(t, &end, 10);
    if (end != t && b >= 0) {
      drop_tk = b;
      wait_limit = 1u << 14;
    }
  }
  umma_gather_kernel<FMT><<<static_cast<unsigned>(grid), kThreads, kSmemTotal, stream>>>(a, items, wait_limit,
                                                                                           drop_tk);
  return cudaGetLastError();
}

}  // namespace umma
}  // namespace qkv
