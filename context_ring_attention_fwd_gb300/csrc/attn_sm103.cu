// Ring-attention forward on sm_103a tensor cores (tcgen05): bf16 inputs, and
// E4M3 (FP8) inputs with per-(b, h) scales.
//
// What is computed ("上下文並行（Context Parallelism, CP）", compassingai.com,
// section 線上 Softmax, algorithm "Ring Attention + FlashAttention 分塊計算"):
// every virtual rank i holds the query shard Q_i and visits the K/V shards j
// in ascending ring order; for each visited block it forms
// S = Q K^T / sqrt(d) with the causal / document mask, the row max, P =
// exp(S - m), the row sum and P V, and folds them into a running (O, m, l)
// with the online-softmax merge; at the end O / l and the log-sum-exp are
// written.  Shard pairs and tiles with no visible (q, k) are never loaded or
// computed (section 因果掩碼的特殊處理).  The inner tile loop that the page
// leaves out is this kernel's main loop.
//
// GB300 mapping.  One persistent CTA per SM (384 threads, three warpgroups):
//   warps 0-3  softmax + merge + epilogue for query tile 0 (128 rows)
//   warps 4-7  the same for query tile 1 (the next 128 rows)
//   warp  8    TMA producer: Q tiles once per work item, then K/V tiles of
//              each visited shard into a 2-stage shared-memory ring
//              (the ring's send/receive becomes this double-buffered walk)
//   warp  9    issues every tcgen05.mma (the whole warp runs the loop; one
//              lane, picked by elect.sync, issues each instruction)
//   warps 10-11 idle (they complete the third warpgroup, which gives its
//              registers to the softmax warpgroups through setmaxnreg)
// TMEM (512 columns): S_0 | S_1 | O_0 | O_1.  S_t = Q_t K^T lands in TMEM
// (fp32); the softmax warps read it with tcgen05.ld, write P (bf16 pairs)
// back over S_t, and the MMA warp issues O_t += P V with P taken from TMEM
// (bf16: in two halves of 64 keys, the first signalled before the second is
// computed).  While one warpgroup does its exponentials the tensor cores work
// on the other tile, so the two tiles ping-pong.
//
// Running state.  m is kept in base-2 units (scores pre-multiplied by
// log2(e)/sqrt(d)).  The reference point used for the exponentials moves
// only when the row max grows by more than 2^8 (so most tiles need no
// rescale of O); the exact row max is tracked separately and the result is
// converted to the pages' (O, m, l) with m the true row max at the end.
//
// FP8 form (ring_attn_fp8_kernel).  Q and K arrive as E4M3 [B, S, H, d] and
// V as E4M3 [B, H, d, S] (keys contiguous, so V is K-major for the PV MMA),
// each with one fp32 descale per (b, h).  Both MMAs run as kind::f8f6f4 with
// both operands in shared memory: the softmax writes P as E4M3 into one of
// two shared-memory buffers of its query tile and keeps every P <= 2^8,
// inside E4M3's range of 448.  Because P does not overwrite S in TMEM, the
// next key tile's S is computed while the softmax still works on the
// current one.  The descales enter as the score scale (q_descale *
// k_descale) and the output scale (v_descale).  The communication-volume
// note of the first page ties the bytes moved to FP8 transfer; this form
// halves the K/V bytes.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <climits>
#include <cmath>
#include <cstdio>
#include <atomic>
#include <mutex>
#include <type_traits>

#include "attn_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace cpring {
namespace {

constexpr int kBM = kTileRows;  // query rows per tile = TMEM lanes
constexpr int kBN = kTileRows;  // key rows per K/V tile
constexpr int kQTiles = 2;      // query tiles per work item
constexpr int kStages = 2;      // K/V ring depth
constexpr int kThreads = 384;   // three warpgroups
constexpr int kLaunchRegs = 168;  // registers per thread at launch (checked by the build)
constexpr int kSoftmaxRegs = 200; // softmax warpgroups after setmaxnreg.inc
constexpr int kControlRegs = 104; // producer / MMA warpgroup after setmaxnreg.dec
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch's register pool");
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
// Tuning switches (all give the same result up to rounding):
//  CPRING_BALANCE          items are dealt in groups of heads holding at least
//                          this many rounds of the grid (see head_group) ...
//  CPRING_GROUP_MIN_ROUNDS ... when the launch has at least this many rounds;
//                          shorter launches deal every item from one pool.
//  CPRING_GROUP_DOCS       launches with documents group heads too.
//  CPRING_DYNAMIC_ALWAYS   the whole-sequence bf16 launch without documents
//                          claims its items too (otherwise it takes the
//                          fixed snake deal; every other launch claims).
//  CPRING_RANK_DYNAMIC     one rank's launch without documents claims its
//                          items (1) or takes the fixed deal (0).
//  CPRING_FUSED_NOMAX      fused forward only: after the first tile, skip the
//                          row max and redo a tile only if its first 64 keys'
//                          row sum or its last 64 keys' row max shows an
//                          exponential above 2^64 (the reference point never
//                          affects P's relative precision, only its range).
//                          P then goes out in two halves of 64 keys, each
//                          signalled as soon as it is stored.
//  CPRING_PACKED_F32X2     fast pass: scale-and-shift and row sum with the
//                          paired fp32 FMA / ADD (two elements per instruction).
//  CPRING_FP8_FAST         the FP8 kernel uses the same no-max fast pass, with
//                          the guards at 2^8 so that every P it keeps is at
//                          most 2^8, inside E4M3's range (448).
//  CPRING_FP8_EARLY_SFREE  the FP8 softmax releases a tile's S columns as
//                          soon as it has loaded them (the rare redo then
//                          works from the scores kept in registers) instead
//                          of after its exponentials.
//  CPRING_FP8_EXP_F16      FP8 fast pass: P = 2^x from the paired half-precision
//                          exponential (two per instruction) and converted to
//                          E4M3 from half precision; row sums in half pairs
//                          over 32 keys, then added into fp32.
#ifndef CPRING_BALANCE
#define CPRING_BALANCE 1
#endif
#ifndef CPRING_GROUP_MIN_ROUNDS
#define CPRING_GROUP_MIN_ROUNDS 16
#endif
#ifndef CPRING_GROUP_DOCS
#define CPRING_GROUP_DOCS 0
#endif
#ifndef CPRING_DYNAMIC_ALWAYS
#define CPRING_DYNAMIC_ALWAYS 0
#endif
#ifndef CPRING_RANK_DYNAMIC
#define CPRING_RANK_DYNAMIC 0
#endif
#ifndef CPRING_FUSED_NOMAX
#define CPRING_FUSED_NOMAX 1
#endif
#ifndef CPRING_PACKED_F32X2
#define CPRING_PACKED_F32X2 1
#endif
#ifndef CPRING_FP8_FAST
#define CPRING_FP8_FAST 1
#endif
#ifndef CPRING_FP8_EARLY_SFREE
#define CPRING_FP8_EARLY_SFREE 0
#endif
#ifndef CPRING_FP8_EXP_F16
#define CPRING_FP8_EXP_F16 1
#endif
constexpr int kPReadyCount = 128;
constexpr float kOverflowGuard = 18446744073709551616.0f;  // 2^64
constexpr float kOverflowGuardFp8 = 256.0f;                  // 2^8: P <= 2^8 < 448
constexpr float kOverflowGuardLog2 = 64.0f;                  // 2^64 as an exponent
constexpr unsigned long long kTimeoutNs = 4000000000ull;  // per wait

template <int D, int E>  // E = bytes per element (2 bf16, 1 E4M3)
struct Layout {
  static constexpr int kTileBytes = kBM * D * E;    // 128 rows x D elements
  static constexpr int kPanelBytes = kBM * 128;     // 128 rows x 128 bytes (one swizzle panel)
  static constexpr int kPanelCols = 128 / E;        // elements per panel row
  static constexpr int kPanels = D * E / 128;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQTiles * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  static constexpr int kRingOff = kBarOff + 256;  // the item ring
  static constexpr int kBytes = kRingOff + 256;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024 B
};

// mbarrier slots (8 bytes each) after the tiles
enum Bar : int {
  kQFull = 0,
  kQEmpty = 1,
  kKFull = 2,     // + stage
  kVFull = 4,     // + stage
  kKEmpty = 6,    // + stage: K tile consumed by both S MMAs
  kVEmpty = 8,    // + stage: V tile consumed by both PV MMAs
  kSFull = 10,    // + tile
  kPReady = 12,   // + tile: the first 64 keys' P of tile t stored
  kPReadyB = 14,  // + tile: the last 64 keys' P of tile t stored (and O rescaled)
  kOBar = 16,     // + tile: every PV of tile t in the item done (once per item)
  kDrain = 18,
  kNumBars = 19
};
constexpr int kTmemSlot = kNumBars * 8;       // u32: TMEM base address
constexpr int kAbortSlot = kNumBars * 8 + 4;  // u32: CTA abort flag

struct KParams {
  int B, S, H, L, n_shards;
  int q_shard, k_shard;  // -1 = all shards
  int causal;
  const int32_t* doc_offsets;
  const int32_t* doc_info;
  int n_qshards;
  int pairs_per_shard;   // ceil(L / 256)
  int tiles_per_shard;   // ceil(L / 128)
  int n_items;
  float scale_log2;      // log2(e) / sqrt(d)
  __nv_bfloat16* out;
  float* lse;
  float* o_part;
  float* m_part;
  float* l_part;
  int* err;
  unsigned long long timeout_ns;
  int fault_drop_k;  // test hook: CTA 0 never loads its first K tile
  int kv_row0;       // key index of row 0 of the K/V tensors (0 unless a block)
  int head_group;    // (b, h) heads whose items are dealt out together
  const int32_t* slot_perm;  // or null: slots heaviest first by measured cost
  unsigned long long* work_slot;  // this launch's claim counter (see claim_first)
  uint32_t epoch;                 // this launch's tag in that counter
  const float* q_descale;  // FP8 form: [B * H] each
  const float* k_descale;
  const float* v_descale;
};

struct Item {
  int b, h, i;
  int q0[kQTiles];
  int rows[kQTiles];
  int f_lo[kQTiles], f_hi[kQTiles];  // flattened K/V tile range (empty if lo > hi)
  int F_lo, F_hi;
  int klo, khi;                      // key range this launch may use
};

// Work item w: (b, h, query shard, pair of 128-row tiles).  Items are laid
// out head group by head group (p.head_group (b, h) heads at a time), and
// inside a group heaviest first; CTAs claim them in that order, so the CTAs
// running at any moment stream the K/V of few heads and reuse each K/V tile
// from L2, and the lightest items come last.
// A tile's visible keys are [max(doc_start(q_first), klo), min(h(q_last), khi)]
// with h(q) = q (causal) or doc_end(q) - 1: every key of that interval is
// seen by at least one row of the tile, so the K/V tiles it touches are
// exactly the tiles holding a visible (q, k).
__device__ __forceinline__ void decode_item(const KParams& p, int n_docs, int w, Item& it) {
  const int BH = p.B * p.H;
  const int slots = p.n_qshards * p.pairs_per_shard;
  const int HG = p.head_group;
  const int gi = w / (HG * slots);                  // head group
  const int r = w - gi * HG * slots;
  const int hg = min(HG, BH - gi * HG);             // heads in this group
  const int g = p.slot_perm ? __ldg(p.slot_perm + r / hg) : slots - 1 - r / hg;
  const int bh = gi * HG + r % hg;
  it.b = bh / p.H;
  it.h = bh - it.b * p.H;
  const int ii = g / p.pairs_per_shard;
  const int pp = g - ii * p.pairs_per_shard;
  it.i = (p.q_shard < 0) ? ii : p.q_shard;
  it.klo = (p.k_shard < 0) ? 0 : p.k_shard * p.L;
  it.khi = (p.k_shard < 0) ? p.S - 1 : (p.k_shard + 1) * p.L - 1;
  const int shard_end = (it.i + 1) * p.L;
  it.F_lo = INT_MAX;
  it.F_hi = -1;
#pragma unroll
  for (int t = 0; t < kQTiles; ++t) {
    const int q0 = it.i * p.L + pp * (kBM * kQTiles) + t * kBM;
    const int rows = max(0, min(kBM, shard_end - q0));
    it.q0[t] = q0;
    it.rows[t] = rows;
    it.f_lo[t] = 1;
    it.f_hi[t] = 0;
    if (rows > 0) {
      const int qa = q0, qb = q0 + rows - 1;
      const int2 da = doc_span(p, n_docs, qa);
      const int lo = max(da.x, it.klo);
      int hi;
      if (p.causal) {
        hi = qb;
      } else {
        hi = doc_span(p, n_docs, qb).y - 1;
      }
      hi = min(hi, it.khi);
      if (lo <= hi) {
        it.f_lo[t] = flat_tile(p, lo);
        it.f_hi[t] = flat_tile(p, hi);
        it.F_lo = min(it.F_lo, it.f_lo[t]);
        it.F_hi = max(it.F_hi, it.f_hi[t]);
      }
    }
  }
}

// The softmax warps read the item ring; the MMA warp learns each item from
// its Q load instead (see the producer).
constexpr int kSoftmaxRingReaders = 8;

// ---------------------------------------------------------------- softmax pieces
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// This thread's 128 scores of the S tile (one TMEM lane), with columns
// outside [c_lo, c_hi] set to -inf.
__device__ __forceinline__ void load_scores(uint32_t tS, int c_lo, int c_hi,
                                            uint32_t (&sv)[4][32]) {
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) ptx::tmem_ld32(tS + ch * 32, sv[ch]);
  ptx::tmem_wait_ld();
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) ptx::reg_fence(sv[ch]);
  if (c_lo > 0 || c_hi < kBN - 1) {
#pragma unroll
    for (int ch = 0; ch < 4; ++ch)
#pragma unroll
      for (int x = 0; x < 32; ++x) {
        const int cc = ch * 32 + x;
        if (cc < c_lo || cc > c_hi) sv[ch][x] = __float_as_uint(-INFINITY);
      }
  }
}

__device__ __forceinline__ float row_max(const uint32_t (&sv)[4][32]) {
  float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int ch = 0; ch < 4; ++ch)
#pragma unroll
    for (int x = 0; x < 32; x += 2)
      m[ch] = max3(m[ch], __uint_as_float(sv[ch][x]), __uint_as_float(sv[ch][x + 1]));
  return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

// Two exponent arguments s * sc - base at once (paired fp32 FMA).
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float sc,
                                     float nb) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %4};\n\tmov.b64 rc, {%5, %5};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(sc), "f"(nb));
}
// acc (two fp32 lanes) += (p0, p1) with one paired add.
__device__ __forceinline__ void add2(uint64_t& acc, float p0, float p1) {
  asm("{\n\t.reg .b64 rp;\n\tmov.b64 rp, {%1, %2};\n\tadd.rn.f32x2 %0, %0, rp;\n\t}"
      : "+l"(acc)
      : "f"(p0), "f"(p1));
}
__device__ __forceinline__ float sum2(uint64_t acc) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(acc));
  return lo + hi;
}

// P = 2^(s * sc - base), its row sum, and the raw row max of the scores.  P is
// packed as bf16 pairs (P[2c] low, P[2c+1] high) into pk[0..1][32], or for
// the FP8 form as E4M3 quads (P[4c] lowest byte) into pk[0][32].
// kPaired (the step kernel, where every tile takes this path): paired fp32
// FMA / ADD.  The fused kernel reaches it only on the first tile of a row or
// a rare redo and keeps scalar arithmetic there, which measured faster for
// its hot loop.
template <bool kFp8 = false, bool kPaired = false>
__device__ __forceinline__ void exponentials(const uint32_t (&sv)[4][32], float sc, float base,
                                             uint32_t (&pk)[2][32], float& lsum, float& mx) {
  float ls[4] = {0.f, 0.f, 0.f, 0.f};
  float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  if constexpr (kFp8) {
#pragma unroll
    for (int ch = 0; ch < 4; ++ch)
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const float s0 = __uint_as_float(sv[ch][4 * x]);
        const float s1 = __uint_as_float(sv[ch][4 * x + 1]);
        const float s2 = __uint_as_float(sv[ch][4 * x + 2]);
        const float s3 = __uint_as_float(sv[ch][4 * x + 3]);
        m[ch] = max3(m[ch], max3(s0, s1, s2), s3);
        const float p0 = ptx::ex2(fmaf(s0, sc, -base));
        const float p1 = ptx::ex2(fmaf(s1, sc, -base));
        const float p2 = ptx::ex2(fmaf(s2, sc, -base));
        const float p3 = ptx::ex2(fmaf(s3, sc, -base));
        ls[ch] += (p0 + p1) + (p2 + p3);
        pk[0][ch * 8 + x] = ptx::pack_e4m3x4(p0, p1, p2, p3);
      }
  } else if (kPaired) {
    // paired fp32 FMA / ADD, two scores per instruction
    uint64_t acc = 0;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch)
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const float s0 = __uint_as_float(sv[ch][2 * x]);
        const float s1 = __uint_as_float(sv[ch][2 * x + 1]);
        m[ch] = max3(m[ch], s0, s1);
        float e0, e1;
        fma2(e0, e1, s0, s1, sc, -base);
        const float p0 = ptx::ex2(e0);
        const float p1 = ptx::ex2(e1);
        add2(acc, p0, p1);
        pk[ch >> 1][(ch & 1) * 16 + x] = ptx::pack_bf16(p0, p1);
      }
    ls[0] = sum2(acc);
  } else {
#pragma unroll
    for (int ch = 0; ch < 4; ++ch)
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const float s0 = __uint_as_float(sv[ch][2 * x]);
        const float s1 = __uint_as_float(sv[ch][2 * x + 1]);
        m[ch] = max3(m[ch], s0, s1);
        const float p0 = ptx::ex2(fmaf(s0, sc, -base));
        const float p1 = ptx::ex2(fmaf(s1, sc, -base));
        ls[ch] += p0 + p1;
        pk[ch >> 1][(ch & 1) * 16 + x] = ptx::pack_bf16(p0, p1);
      }
  }
  lsum = (ls[0] + ls[1]) + (ls[2] + ls[3]);
  mx = fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

// P for two 32-column chunks of S against `base`, into pk row `half`.
__device__ __forceinline__ void exp_chunks(const uint32_t (&sv)[4][32], int half, float sc,
                                           float base, uint32_t (&pk)[2][32], uint64_t& acc,
                                           float& ls) {
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int ch = 2 * half + cc;
#pragma unroll
    for (int x = 0; x < 16; ++x) {
      const float s0 = __uint_as_float(sv[ch][2 * x]);
      const float s1 = __uint_as_float(sv[ch][2 * x + 1]);
      float e0, e1;
      if (CPRING_PACKED_F32X2) {
        fma2(e0, e1, s0, s1, sc, -base);
      } else {
        e0 = fmaf(s0, sc, -base);
        e1 = fmaf(s1, sc, -base);
      }
      const float p0 = ptx::ex2(e0);
      const float p1 = ptx::ex2(e1);
      if (CPRING_PACKED_F32X2) {
        add2(acc, p0, p1);
      } else {
        ls += p0 + p1;
      }
      pk[half][cc * 16 + x] = ptx::pack_bf16(p0, p1);
    }
  }
}

// The FP8 form of exp_chunks: P as E4M3 quads into pk[0] (P[4c] lowest byte).
__device__ __forceinline__ void exp_chunks_f8(const uint32_t (&sv)[4][32], int half, float sc,
                                              float base, uint32_t (&pk)[2][32], uint64_t& acc) {
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int ch = 2 * half + cc;
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      float e0, e1, e2, e3;
      fma2(e0, e1, __uint_as_float(sv[ch][4 * x]), __uint_as_float(sv[ch][4 * x + 1]), sc, -base);
      fma2(e2, e3, __uint_as_float(sv[ch][4 * x + 2]), __uint_as_float(sv[ch][4 * x + 3]), sc, -base);
      const float p0 = ptx::ex2(e0), p1 = ptx::ex2(e1), p2 = ptx::ex2(e2), p3 = ptx::ex2(e3);
      add2(acc, p0, p1);
      add2(acc, p2, p3);
      pk[0][ch * 8 + x] = ptx::pack_e4m3x4(p0, p1, p2, p3);
    }
  }
}

// exp_chunks_f8 with the exponentials in half precision: 2^x for two keys
// per ex2.approx.f16x2, E4M3 from the half pair, and the row sum of each
// 32-key chunk formed in half pairs (at most 32 * 2^8, exact to 11 bits per
// add) before it enters the fp32 sum.  The argument is rounded to half
// precision (10 bits): 2^x then carries a relative error below 2^-8 for
// x >= -8, far inside E4M3's 2^-4 rounding, and keys further below the
// reference give P under E4M3's smallest step either way.  An argument
// above half precision's range gives +inf, which the caller's 2^8 guard
// sends to the fp32 redo.
__device__ __forceinline__ void exp_chunks_f8h(const uint32_t (&sv)[4][32], int half, float sc,
                                               float base, uint32_t (&pk)[2][32], float& ls) {
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int ch = 2 * half + cc;
    uint32_t hs = 0;  // two half-precision zeros
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      float e0, e1, e2, e3;
      fma2(e0, e1, __uint_as_float(sv[ch][4 * x]), __uint_as_float(sv[ch][4 * x + 1]), sc, -base);
      fma2(e2, e3, __uint_as_float(sv[ch][4 * x + 2]), __uint_as_float(sv[ch][4 * x + 3]), sc, -base);
      uint32_t h01, h23;
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h01) : "f"(e1), "f"(e0));
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h23) : "f"(e3), "f"(e2));
      asm("ex2.approx.f16x2 %0, %0;" : "+r"(h01));
      asm("ex2.approx.f16x2 %0, %0;" : "+r"(h23));
      uint16_t lo, hi;
      asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(lo) : "r"(h01));
      asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(hi) : "r"(h23));
      pk[0][ch * 8 + x] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      asm("add.rn.f16x2 %0, %0, %1;" : "+r"(hs) : "r"(h01));
      asm("add.rn.f16x2 %0, %0, %1;" : "+r"(hs) : "r"(h23));
    }
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %0, hi, %0;\n\t}"
        : "+f"(ls)
        : "r"(hs));
  }
}

// Raw max of the scores of chunks 2*half, 2*half+1 (64 keys).
__device__ __forceinline__ float half_max(const uint32_t (&sv)[4][32], int half) {
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
  for (int x = 0; x < 32; x += 2) {
    m0 = max3(m0, __uint_as_float(sv[2 * half][x]), __uint_as_float(sv[2 * half][x + 1]));
    m1 = max3(m1, __uint_as_float(sv[2 * half + 1][x]), __uint_as_float(sv[2 * half + 1][x + 1]));
  }
  return fmaxf(m0, m1);
}

// bf16 P of 64 keys (half 0: keys 0-63, half 1: keys 64-127) against `base`
// into pk[half], and its row sum.
__device__ __forceinline__ float exp_half(const uint32_t (&sv)[4][32], int half, float sc,
                                          float base, uint32_t (&pk)[2][32]) {
  uint64_t acc = 0;  // two fp32 zeros
  float ls = 0.f;
  exp_chunks(sv, half, sc, base, pk, acc, ls);
  return CPRING_PACKED_F32X2 ? sum2(acc) : ls;
}

// Stores one half of the keys' bf16 P (columns 32*half .. +32 of the lane's
// S row).
__device__ __forceinline__ void store_p_half(uint32_t tS, const uint32_t (&pk)[2][32], int half) {
  ptx::tmem_st32(tS + 32u * half, pk[half]);
}

// ---------------------------------------------------------------- kernel
// The body shared by the bf16 and the FP8 kernels (see the wrappers below).
// kDynamic: CTAs claim items at run time (the producer hands each to the
// softmax warps through the item ring and to the MMA warp with its Q load);
// otherwise every role walks the fixed snake deal by itself.
template <int D, bool kPartial, bool kDynamic>
__device__ __forceinline__ void attn_body(const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                          const CUtensorMap& tmap_v, const KParams& p) {
  using Lay = Layout<D, 2>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t bars = sbase + Lay::kBarOff;
  auto bar = [&](int idx) -> uint32_t { return bars + 8u * static_cast<uint32_t>(idx); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kBarOff + kTmemSlot);
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(smem + Lay::kBarOff + kAbortSlot);
  const ItemRing ring{sbase + Lay::kRingOff,
                      reinterpret_cast<volatile int*>(smem + Lay::kRingOff + 2 * kRing * 8)};
  // the item whose Q the producer is loading (the MMA warp's copy of the work)
  volatile int* q_item = reinterpret_cast<volatile int*>(smem + Lay::kRingOff + 128);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int n_docs = 1;
  if (p.doc_offsets != nullptr) {
    n_docs = __ldg(p.doc_info);
    if (n_docs <= 0) return;  // malformed doc_offsets: the scan already flagged it
  }

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(kQFull), 1);
    ptx::mbar_init(bar(kQEmpty), 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar(kKFull + s), 1);
      ptx::mbar_init(bar(kVFull + s), 1);
      ptx::mbar_init(bar(kKEmpty + s), 1);
      ptx::mbar_init(bar(kVEmpty + s), 1);
    }
    for (int t = 0; t < kQTiles; ++t) {
      ptx::mbar_init(bar(kSFull + t), 1);
      ptx::mbar_init(bar(kPReady + t), kPReadyCount);
      ptx::mbar_init(bar(kPReadyB + t), kPReadyCount);
      ptx::mbar_init(bar(kOBar + t), 1);
    }
    ptx::mbar_init(bar(kDrain), 1);
    if (kDynamic) ring_init(ring, kSoftmaxRingReaders);
    *abort_flag = 0u;
    ptx::fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int G = gridDim.x;
  const int c = blockIdx.x;

  if (warp >= kProducerWarp) {
   // the third warpgroup gives registers away, then splits into its roles
   ptx::setmaxnreg_dec<kControlRegs>();
   if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmap_q);
      ptx::tma_prefetch_desc(&tmap_k);
      ptx::tma_prefetch_desc(&tmap_v);
      uint32_t kv_iter = 0, q_iter = 0;
      unsigned long long ahead = 0;  // the claim of the CTA's next item
      // Loads started into each stage: the n-th one completes phase n - 1.
      uint32_t k_armed0 = 0, k_armed1 = 0, v_armed0 = 0, v_armed1 = 0;
      bool dropped = false;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int w = !kDynamic ? item_of(k, c, G)
                      : (k == 0) ? c : G + claimed_index(ahead, p.epoch, p.err);
        if constexpr (kDynamic) {
          if (!ring_put(ring, static_cast<uint32_t>(k), w, abort_flag, p)) { ok = false; break; }
        }
        if (w >= p.n_items) break;
        if constexpr (kDynamic)  // claim the CTA's next item now; it is read when that item starts
          ahead = (k == 0) ? claim_first(p.work_slot, p.epoch) : claim_next(p.work_slot);
        Item it;
        decode_item(p, n_docs, w, it);
        if (it.F_lo > it.F_hi) continue;
        if (!wait1(bar(kQEmpty), (q_iter & 1u) ^ 1u, abort_flag, p)) { ok = false; break; }
        if constexpr (kDynamic) *q_item = w;  // the MMA warp reads it with this phase of kQFull
        ptx::mbar_arrive_expect_tx(bar(kQFull), kQTiles * Lay::kTileBytes);
#pragma unroll
        for (int t = 0; t < kQTiles; ++t)
#pragma unroll
          for (int pn = 0; pn < Lay::kPanels; ++pn)
            ptx::tma_load_4d(sbase + Lay::kQOff + t * Lay::kTileBytes + pn * Lay::kPanelBytes,
                             &tmap_q, bar(kQFull), pn * Lay::kPanelCols, it.h, it.q0[t], it.b);
        ++q_iter;
        for (int f = it.F_lo; f <= it.F_hi; ++f) {
          const uint32_t st = kv_iter % kStages;
          const uint32_t ph = (kv_iter / kStages) & 1u;
          int ks, ke;
          tile_keys(p, f, ks, ke);
          if (!wait1(bar(kKEmpty + st), ph ^ 1u, abort_flag, p)) { ok = false; break; }
          if (p.fault_drop_k && c == 0 && !dropped) {
            // Test hook: this K tile is never loaded, so the MMA warp's
            // bounded wait for it runs out and the CTA takes its abort path.
            dropped = true;
          } else {
            ptx::mbar_arrive_expect_tx(bar(kKFull + st), Lay::kTileBytes);
            for (int pn = 0; pn < Lay::kPanels; ++pn)
              ptx::tma_load_4d(sbase + Lay::kKOff + st * Lay::kTileBytes + pn * Lay::kPanelBytes,
                               &tmap_k, bar(kKFull + st), pn * Lay::kPanelCols, it.h,
                               ks - p.kv_row0, it.b);
            if (st == 0) ++k_armed0; else ++k_armed1;
          }
          if (!wait1(bar(kVEmpty + st), ph ^ 1u, abort_flag, p)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(bar(kVFull + st), Lay::kTileBytes);
          for (int pn = 0; pn < Lay::kPanels; ++pn)
            ptx::tma_load_4d(sbase + Lay::kVOff + st * Lay::kTileBytes + pn * Lay::kPanelBytes,
                             &tmap_v, bar(kVFull + st), pn * Lay::kPanelCols, it.h,
                             ks - p.kv_row0, it.b);
          if (st == 0) ++v_armed0; else ++v_armed1;
          ++kv_iter;
        }
      }
      // No more items: tell the MMA warp through the next phase of kQFull.
      if (kDynamic && ok && wait1(bar(kQEmpty), (q_iter & 1u) ^ 1u, abort_flag, p)) {
        *q_item = p.n_items;
        ptx::mbar_arrive(bar(kQFull));
        ++q_iter;
      }
      // Let every copy this thread started land before the CTA can exit.
      if (q_iter > 0) wait1(bar(kQFull), (q_iter - 1) & 1u, abort_flag, p, false);
      if (k_armed0 > 0) wait1(bar(kKFull + 0), (k_armed0 - 1) & 1u, abort_flag, p, false);
      if (k_armed1 > 0) wait1(bar(kKFull + 1), (k_armed1 - 1) & 1u, abort_flag, p, false);
      if (v_armed0 > 0) wait1(bar(kVFull + 0), (v_armed0 - 1) & 1u, abort_flag, p, false);
      if (v_armed1 > 0) wait1(bar(kVFull + 1), (v_armed1 - 1) & 1u, abort_flag, p, false);
    }
   } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop with warp-uniform values; each MMA and
    // commit is issued by one lane that elect.sync picks (the warp-collective
    // forms in ptx.cuh), and every wait is the warp-uniform one.
    {
      constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(kBM, kBN, false);
      constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kBM, D, true);
      constexpr int kKStep = 16;  // K elements per MMA (32 bytes)
      uint32_t kv_iter = 0, q_iter = 0;
      uint32_t p_cnt0 = 0, p_cnt1 = 0;
      bool ok = true;
      // Shared-memory descriptors of every operand tile, built once.  A k-step
      // moves the start address (bits 0-13, in 16-byte units) by a constant,
      // so each MMA needs one add: this warp issues 32 MMAs per K/V tile
      // while sharing its scheduler with two softmax warps.
      // (Shared addresses stay below 2^18 bytes, so the 14-bit start field
      // never carries into the offsets above it.)
      const uint64_t d_qk = ptx::smem_desc_sw128(sbase, 16, 1024);
      const uint64_t d_v = ptx::smem_desc_sw128(sbase, Lay::kPanelBytes, 1024);
      // O_t (+)= P_t V: P_t from TMEM (8 columns per K step), V MN-major from
      // the given stage.  Half `part` of the K steps: keys 0-63 (part 0) or
      // 64-127 (part 1), whose P the softmax signals separately.
      auto issue_pv = [&](int t, uint32_t st, bool first, int part) {
        constexpr int kHalfSteps = kBN / kKStep / 2;
        const uint64_t dv = d_v + ((Lay::kVOff + st * Lay::kTileBytes) >> 4);
#pragma unroll
        for (int s = part * kHalfSteps; s < (part + 1) * kHalfSteps; ++s) {
          ptx::mma_ts_w(tmem_base + 256 + t * D, tmem_base + t * 128 + s * 8,
                        dv + static_cast<uint64_t>((s * 16 * 128) >> 4), kIdescPV,
                        (first && s == 0) ? 0u : 1u);
        }
      };
      // S_t = Q_t K^T (both K-major, 128-byte swizzled panels; a K step is
      // 32 bytes, four steps per panel).
      auto issue_s = [&](int t, uint32_t st) {
        const uint64_t dq = d_qk + ((Lay::kQOff + t * Lay::kTileBytes) >> 4);
        const uint64_t dk = d_qk + ((Lay::kKOff + st * Lay::kTileBytes) >> 4);
#pragma unroll
        for (int s = 0; s < D / kKStep; ++s) {
          const uint64_t step = static_cast<uint64_t>(((s >> 2) * Lay::kPanelBytes + (s & 3) * 32) >> 4);
          ptx::mma_ss_w(tmem_base + t * 128, dq + step, dk + step, kIdescQK, s > 0 ? 1u : 0u);
        }
        ptx::mma_commit_w(bar(kSFull + t));
      };
      for (int k = 0;; ++k) {
        // Claimed items: the producer publishes each item that has work with
        // its Q load (and the end of the work with a plain arrival), so this
        // warp needs no wait beyond the one for Q.  The fixed deal: this
        // warp walks it and skips items with nothing to compute.
        Item it;
        if constexpr (kDynamic) {
          if (!wait_warp(bar(kQFull), q_iter & 1u, abort_flag, p)) { ok = false; break; }
          ++q_iter;
          const int w = *q_item;
          if (w >= p.n_items) break;
          decode_item(p, n_docs, w, it);
        } else {
          const int w = item_of(k, c, G);
          if (w >= p.n_items) break;
          decode_item(p, n_docs, w, it);
          if (it.F_lo > it.F_hi) continue;
          if (!wait_warp(bar(kQFull), q_iter & 1u, abort_flag, p)) { ok = false; break; }
          ++q_iter;
        }
        ptx::tc_fence_after();
        bool pend0 = false, pend1 = false;    // an S issued whose PV is still owed
        bool first0 = true, first1 = true;    // next PV overwrites O
        uint32_t prev_st = 0, prev_ph = 0;
        bool have_prev = false, prev_v_ready = false;
        // Owed PV of tile t on the previous K/V stage: wait for V and P, issue.
        // After the item's last PV of tile t, O_t is final: commit kOBar + t
        // (the epilogue waits on it; nothing else does).
        auto flush = [&](int t, uint32_t& pc, bool& first, bool last) -> bool {
          if (!prev_v_ready) {
            if (!wait_warp(bar(kVFull + prev_st), prev_ph, abort_flag, p)) return false;
            prev_v_ready = true;
          }
          if (!wait_warp(bar(kPReady + t), pc & 1u, abort_flag, p)) return false;
          ptx::tc_fence_after();
          issue_pv(t, prev_st, first, 0);
          if (!wait_warp(bar(kPReadyB + t), pc & 1u, abort_flag, p)) return false;
          ++pc;
          ptx::tc_fence_after();
          issue_pv(t, prev_st, false, 1);
          if (last) ptx::mma_commit_w(bar(kOBar + t));
          first = false;
          return true;
        };
        for (int f = it.F_lo; f <= it.F_hi; ++f) {
          const uint32_t st = kv_iter % kStages;
          const uint32_t ph = (kv_iter / kStages) & 1u;
          if (pend0) {
            if (!flush(0, p_cnt0, first0, f - 1 == it.f_hi[0])) { ok = false; break; }
            pend0 = false;
          }
          if (!wait_warp(bar(kKFull + st), ph, abort_flag, p)) { ok = false; break; }
          ptx::tc_fence_after();
          if (f >= it.f_lo[0] && f <= it.f_hi[0]) {
            issue_s(0, st);
            pend0 = true;
          }
          if (pend1) {
            if (!flush(1, p_cnt1, first1, f - 1 == it.f_hi[1])) { ok = false; break; }
            pend1 = false;
          }
          if (f >= it.f_lo[1] && f <= it.f_hi[1]) {
            issue_s(1, st);
            pend1 = true;
          }
          ptx::mma_commit_w(bar(kKEmpty + st));                      // K(f) read by every S
          if (have_prev) ptx::mma_commit_w(bar(kVEmpty + prev_st));  // V(f-1) read by every PV
          prev_st = st;
          prev_ph = ph;
          have_prev = true;
          prev_v_ready = false;
          ++kv_iter;
        }
        if (!ok) break;
        ptx::mma_commit_w(bar(kQEmpty));  // every S of this item has been issued
        if (pend0) {
          if (!flush(0, p_cnt0, first0, true)) { ok = false; break; }
        }
        if (pend1) {
          if (!flush(1, p_cnt1, first1, true)) { ok = false; break; }
        }
        if (have_prev) ptx::mma_commit_w(bar(kVEmpty + prev_st));
      }
      // Wait until every MMA this warp issued has finished.
      ptx::mma_commit_w(bar(kDrain));
      wait_warp(bar(kDrain), 0u, abort_flag, p, false);
    }
   }
  } else {
    ptx::setmaxnreg_inc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;  // query tile of this warpgroup
    const int wq = warp & 3;  // TMEM lane quarter
    const int row_in_tile = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem_base + lane_off + static_cast<uint32_t>(t * 128);
    const uint32_t tO = tmem_base + lane_off + 256u + static_cast<uint32_t>(t * D);
    const float sc = p.scale_log2;
    uint32_t s_cnt = 0, o_cnt = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int w;
      if constexpr (kDynamic) {
        w = ring_get(ring, static_cast<uint32_t>(k), abort_flag, p);
        if (w < 0) { ok = false; break; }
      } else {
        w = item_of(k, c, G);
      }
      if (w >= p.n_items) break;
      Item it;
      decode_item(p, n_docs, w, it);
      // this warpgroup's tile (selects keep the item in registers)
      const int rows = t ? it.rows[1] : it.rows[0];
      const int f_lo = t ? it.f_lo[1] : it.f_lo[0];
      const int f_hi = t ? it.f_hi[1] : it.f_hi[0];
      if (rows == 0) continue;
      const bool row_valid = row_in_tile < rows;
      const int r = (t ? it.q0[1] : it.q0[0]) + row_in_tile;
      int klo_r = 0, khi_r = -1;
      if (row_valid) {
        const int2 ds = doc_span(p, n_docs, r);
        klo_r = max(ds.x, it.klo);
        khi_r = min(p.causal ? r : ds.y - 1, it.khi);
      }
      const int rloc = r - it.i * p.L;
      const size_t mrow = (static_cast<size_t>(it.b) * p.H + it.h) * p.L + rloc;
      if (f_lo > f_hi) {
        // No visible key for the whole tile (a skipped step): empty partial.
        if (kPartial && row_valid) {
          float4* o4 = reinterpret_cast<float4*>(
              p.o_part + ((static_cast<size_t>(it.b) * p.L + rloc) * p.H + it.h) * D);
#pragma unroll
          for (int x = 0; x < D / 4; ++x) o4[x] = make_float4(0.f, 0.f, 0.f, 0.f);
          p.m_part[mrow] = -INFINITY;
          p.l_part[mrow] = 0.f;
        }
        continue;
      }
      float m_used = -INFINITY, m_true = -INFINITY, l_run = 0.f;
      for (int f = f_lo; f <= f_hi; ++f) {
        if (!wait_warp(bar(kSFull + t), s_cnt & 1u, abort_flag, p)) { ok = false; break; }
        ++s_cnt;
        ptx::tc_fence_after();
        int ks, ke;
        tile_keys(p, f, ks, ke);
        const int c_lo = klo_r - ks;
        const int c_hi = min(khi_r, ke - 1) - ks;
        uint32_t sv[4][32];
        uint32_t pk[2][32];
        float lsum, mx;
        float alpha = 1.f;
        bool rescale_o = false;
        const bool fast = CPRING_FUSED_NOMAX && !kPartial &&
                          !__any_sync(0xffffffffu, m_used == -INFINITY);
        if (fast) {
          // P in two halves of 64 keys: the first half is stored and
          // signalled (kPReady + t) before the second half's exponentials
          // run, so the MMA warp starts that half of P V meanwhile.  Both
          // halves use the current reference; before anything is stored the
          // first half's row sum and the second half's row max are checked
          // against the guard (2^64, as a sum and as an exponent).
          load_scores(tS, c_lo, c_hi, sv);
          const float lsum1 = exp_half(sv, 0, sc, m_used, pk);
          const float mx2 = half_max(sv, 1);
          const bool in_range =
              (lsum1 <= kOverflowGuard) & (mx2 * sc <= m_used + kOverflowGuardLog2);
          if (__all_sync(0xffffffffu, in_range)) {
            store_p_half(tS, pk, 0);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(kPReady + t));
            const float lsum2 = exp_half(sv, 1, sc, m_used, pk);
            l_run += lsum1 + lsum2;
            store_p_half(tS, pk, 1);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(kPReadyB + t));
            continue;
          }
          // Rare: a row ran past the guard, so this tile's max is above the
          // reference (64 entries of at most 1 sum to 64 or less).  Nothing
          // is stored yet and sv still holds the scores: move the reference
          // of those rows to this tile's max and let every lane recompute
          // (lanes that keep theirs get the same P).
          {
            const float m_tile = row_max(sv) * sc;
            if (!in_range && m_tile > m_used) {
              rescale_o = true;
              alpha = ptx::ex2(m_used - m_tile);
              l_run *= alpha;
              m_used = m_tile;
            }
            exponentials<false, kPartial>(sv, sc, m_used, pk, lsum, mx);
          }
        } else {
        load_scores(tS, c_lo, c_hi, sv);
        if (__any_sync(0xffffffffu, m_used == -INFINITY)) {
          // Some row of this warp has no reference yet: row max first.
          mx = row_max(sv);
          const float m_tile = mx * sc;
          m_true = fmaxf(m_true, m_tile);
          if (m_tile > m_used + kRescaleLog2) {
            rescale_o = (m_used != -INFINITY);
            alpha = rescale_o ? ptx::ex2(m_used - m_tile) : 0.f;
            l_run *= alpha;
            m_used = m_tile;
          }
          exponentials<false, kPartial>(sv, sc, (m_used == -INFINITY) ? 0.f : m_used, pk, lsum, mx);
        } else if constexpr (kPartial) {
          // Step kernel: the exact row max first (its epilogue exports it),
          // then P in two halves of 64 keys, each signalled once stored, as
          // in the fused pass.  When a row's reference has to move, O is
          // rescaled before any of this tile's P V, so P goes out whole.
          mx = row_max(sv);
          const float m_tile = mx * sc;
          m_true = fmaxf(m_true, m_tile);
          if (m_tile > m_used + kRescaleLog2) {
            rescale_o = true;
            alpha = ptx::ex2(m_used - m_tile);
            l_run *= alpha;
            m_used = m_tile;
          }
          if (!__any_sync(0xffffffffu, rescale_o)) {
            const float lsum1 = exp_half(sv, 0, sc, m_used, pk);
            store_p_half(tS, pk, 0);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(kPReady + t));
            const float lsum2 = exp_half(sv, 1, sc, m_used, pk);
            l_run += lsum1 + lsum2;
            store_p_half(tS, pk, 1);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(kPReadyB + t));
            continue;
          }
          exponentials<false, kPartial>(sv, sc, m_used, pk, lsum, mx);
        } else {
          // Exponentials against the current reference; the row max is
          // taken in the same pass and only forces a redo (rare) when it
          // moved more than 2^8 above the reference.
          {
            exponentials<false, kPartial>(sv, sc, m_used, pk, lsum, mx);
            const float m_tile = mx * sc;
            m_true = fmaxf(m_true, m_tile);
            const bool redo = m_tile > m_used + kRescaleLog2;
            if (__any_sync(0xffffffffu, redo)) {
              if (redo) {
                rescale_o = true;
                alpha = ptx::ex2(m_used - m_tile);
                l_run *= alpha;
                m_used = m_tile;
              }
              load_scores(tS, c_lo, c_hi, sv);  // S is still in TMEM: P not yet written
              exponentials<false, kPartial>(sv, sc, m_used, pk, lsum, mx);
            }
          }
        }
        }
        l_run += lsum;
        ptx::tmem_st32(tS, pk[0]);
        ptx::tmem_st32(tS + 32, pk[1]);
        if (__any_sync(0xffffffffu, rescale_o)) {
          // O_t already holds the sum up to the previous tile: the MMA warp
          // issued that PV before this tile's S, and the commit this warp
          // waited on for S tracks every MMA issued before it.
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t ov[32];
            ptx::tmem_ld32(tO + ch * 32, ov);
            ptx::tmem_wait_ld();
            ptx::reg_fence(ov);
#pragma unroll
            for (int x = 0; x < 32; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * alpha);
            ptx::tmem_st32(tO + ch * 32, ov);
          }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(kPReady + t));
        ptx::mbar_arrive(bar(kPReadyB + t));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!wait_warp(bar(kOBar + t), o_cnt & 1u, abort_flag, p)) { ok = false; break; }
      ++o_cnt;
      ptx::tc_fence_after();
      if (!kPartial) {
        const float inv_l = 1.f / l_run;
        uint4* dst = reinterpret_cast<uint4*>(
            p.out + ((static_cast<size_t>(it.b) * p.S + r) * p.H + it.h) * D);
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t ov[32];
          ptx::tmem_ld32(tO + ch * 32, ov);
          ptx::tmem_wait_ld();
          ptx::reg_fence(ov);
          if (row_valid) {
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              uint4 v4;
              v4.x = ptx::pack_bf16(__uint_as_float(ov[8 * x + 0]) * inv_l,
                                    __uint_as_float(ov[8 * x + 1]) * inv_l);
              v4.y = ptx::pack_bf16(__uint_as_float(ov[8 * x + 2]) * inv_l,
                                    __uint_as_float(ov[8 * x + 3]) * inv_l);
              v4.z = ptx::pack_bf16(__uint_as_float(ov[8 * x + 4]) * inv_l,
                                    __uint_as_float(ov[8 * x + 5]) * inv_l);
              v4.w = ptx::pack_bf16(__uint_as_float(ov[8 * x + 6]) * inv_l,
                                    __uint_as_float(ov[8 * x + 7]) * inv_l);
              dst[ch * 4 + x] = v4;
            }
          }
        }
        if (row_valid) {
          p.lse[(static_cast<size_t>(it.b) * p.H + it.h) * p.S + r] =
              (m_used + log2f(l_run)) * 0.69314718055994531f;
        }
      } else {
        const bool empty = (m_true == -INFINITY);
        const float fac = empty ? 0.f : ptx::ex2(m_used - m_true);
        float4* dst = reinterpret_cast<float4*>(
            p.o_part + ((static_cast<size_t>(it.b) * p.L + rloc) * p.H + it.h) * D);
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t ov[32];
          ptx::tmem_ld32(tO + ch * 32, ov);
          ptx::tmem_wait_ld();
          ptx::reg_fence(ov);
          if (row_valid) {
#pragma unroll
            for (int x = 0; x < 8; ++x)
              dst[ch * 8 + x] = make_float4(__uint_as_float(ov[4 * x + 0]) * fac,
                                            __uint_as_float(ov[4 * x + 1]) * fac,
                                            __uint_as_float(ov[4 * x + 2]) * fac,
                                            __uint_as_float(ov[4 * x + 3]) * fac);
          }
        }
        if (row_valid) {
          p.m_part[mrow] = empty ? -INFINITY : m_true * 0.69314718055994531f;
          p.l_part[mrow] = empty ? 0.f : l_run * fac;
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- FP8 kernel
// The FP8 form hands P to the PV product through shared memory instead of
// TMEM.  P in E4M3 is 16 KB per 128 x 128 tile, so two buffers per query tile
// fit beside the FP8 Q/K/V tiles.  With P out of TMEM, the S columns of a
// query tile are free as soon as its softmax has loaded them, so the MMA warp
// issues S = Q K^T of the next key tile right then, while the softmax is
// still exponentiating the current one: a softmax warpgroup never waits for
// its own PV and next S in turn, which is what bound the FP8 form (its
// products run at twice the bf16 rate; the exponentials do not).
constexpr int kStages8 = 3;  // K/V ring depth of the FP8 kernel

struct Fp8Layout {
  static constexpr int kTileBytes = kBM * 128;  // 128 rows x 128 E4M3 = one swizzle panel
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQTiles * kTileBytes;
  static constexpr int kVOff = kKOff + kStages8 * kTileBytes;
  static constexpr int kPOff = kVOff + kStages8 * kTileBytes;   // [tile][buffer] P tiles
  static constexpr int kBarOff = kPOff + kQTiles * 2 * kTileBytes;
  static constexpr int kRingOff = kBarOff + 256;  // the item ring
  static constexpr int kBytes = kRingOff + 256;
  static constexpr int kAlloc = kBytes + 1024;
};

enum Bar8 : int {
  k8QFull = 0,
  k8QEmpty = 1,
  k8KFull = 2,    // + stage
  k8VFull = 5,    // + stage
  k8KEmpty = 8,   // + stage: K tile read by both S products
  k8VEmpty = 11,  // + stage: V tile read by both PV products
  k8SFull = 14,   // + tile: S of the tile's next key tile in TMEM
  k8SFree = 16,   // + tile: the softmax has loaded that S (its columns may be reused)
  k8PReady = 18,  // + 2 * tile + buffer: P stored in that shared-memory buffer
  k8PFree = 22,   // + 2 * tile + buffer: the PV that read that buffer is done
  k8OBar = 26,    // + tile: every PV of tile t in the item done (once per item)
  k8Drain = 28,
  k8NumBars = 29
};
static_assert(k8NumBars * 8 + 8 <= 256, "FP8 barrier block");
constexpr int kTmemSlot8 = k8NumBars * 8;
constexpr int kAbortSlot8 = k8NumBars * 8 + 4;

template <int D>
__device__ __forceinline__ void attn_body_fp8(const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                              const CUtensorMap& tmap_v, const KParams& p) {
  static_assert(D == 128, "the FP8 form takes d = 128");
  using Lay = Fp8Layout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t bars = sbase + Lay::kBarOff;
  auto bar = [&](int idx) -> uint32_t { return bars + 8u * static_cast<uint32_t>(idx); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kBarOff + kTmemSlot8);
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(smem + Lay::kBarOff + kAbortSlot8);
  const ItemRing ring{sbase + Lay::kRingOff,
                      reinterpret_cast<volatile int*>(smem + Lay::kRingOff + 2 * kRing * 8)};
  // the item whose Q the producer is loading (the MMA warp's copy of the work)
  volatile int* q_item = reinterpret_cast<volatile int*>(smem + Lay::kRingOff + 128);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int n_docs = 1;
  if (p.doc_offsets != nullptr) {
    n_docs = __ldg(p.doc_info);
    if (n_docs <= 0) return;  // malformed doc_offsets: the scan already flagged it
  }

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(k8QFull), 1);
    ptx::mbar_init(bar(k8QEmpty), 1);
    for (int s = 0; s < kStages8; ++s) {
      ptx::mbar_init(bar(k8KFull + s), 1);
      ptx::mbar_init(bar(k8VFull + s), 1);
      ptx::mbar_init(bar(k8KEmpty + s), 1);
      ptx::mbar_init(bar(k8VEmpty + s), 1);
    }
    for (int t = 0; t < kQTiles; ++t) {
      ptx::mbar_init(bar(k8SFull + t), 1);
      ptx::mbar_init(bar(k8SFree + t), kPReadyCount);
      ptx::mbar_init(bar(k8OBar + t), 1);
      for (int b = 0; b < 2; ++b) {
        ptx::mbar_init(bar(k8PReady + 2 * t + b), kPReadyCount);
        ptx::mbar_init(bar(k8PFree + 2 * t + b), 1);
      }
    }
    ptx::mbar_init(bar(k8Drain), 1);
    ring_init(ring, kSoftmaxRingReaders);
    *abort_flag = 0u;
    ptx::fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int G = gridDim.x;
  const int c = blockIdx.x;

  if (warp >= kProducerWarp) {
   ptx::setmaxnreg_dec<kControlRegs>();
   if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmap_q);
      ptx::tma_prefetch_desc(&tmap_k);
      ptx::tma_prefetch_desc(&tmap_v);
      uint32_t kv_iter = 0, q_iter = 0;
      unsigned long long ahead = 0;  // the claim of the CTA's next item
      // Loads started into each stage (the n-th completes phase n - 1), held
      // in registers: a runtime index into a local array would live in memory.
      uint32_t k_armed0 = 0, k_armed1 = 0, k_armed2 = 0;
      uint32_t v_armed0 = 0, v_armed1 = 0, v_armed2 = 0;
      auto bump = [](uint32_t st, uint32_t& a0, uint32_t& a1, uint32_t& a2) {
        if (st == 0) ++a0; else if (st == 1) ++a1; else ++a2;
      };
      bool dropped = false;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int w = (k == 0) ? c : G + claimed_index(ahead, p.epoch, p.err);
        if (!ring_put(ring, static_cast<uint32_t>(k), w, abort_flag, p)) { ok = false; break; }
        if (w >= p.n_items) break;
        // claim the CTA's next item now; it is read when that item starts
        ahead = (k == 0) ? claim_first(p.work_slot, p.epoch) : claim_next(p.work_slot);
        Item it;
        decode_item(p, n_docs, w, it);
        if (it.F_lo > it.F_hi) continue;
        if (!wait1(bar(k8QEmpty), (q_iter & 1u) ^ 1u, abort_flag, p)) { ok = false; break; }
        *q_item = w;  // the MMA warp reads it once this phase of k8QFull completes
        ptx::mbar_arrive_expect_tx(bar(k8QFull), kQTiles * Lay::kTileBytes);
#pragma unroll
        for (int t = 0; t < kQTiles; ++t)
          ptx::tma_load_4d(sbase + Lay::kQOff + t * Lay::kTileBytes, &tmap_q, bar(k8QFull), 0,
                           it.h, it.q0[t], it.b);
        ++q_iter;
        for (int f = it.F_lo; f <= it.F_hi; ++f) {
          const uint32_t st = kv_iter % kStages8;
          const uint32_t ph = (kv_iter / kStages8) & 1u;
          int ks, ke;
          tile_keys(p, f, ks, ke);
          if (!wait1(bar(k8KEmpty + st), ph ^ 1u, abort_flag, p)) { ok = false; break; }
          if (p.fault_drop_k && c == 0 && !dropped) {
            // Test hook: this K tile is never loaded, so the MMA warp's
            // bounded wait for it runs out and the CTA takes its abort path.
            dropped = true;
          } else {
            ptx::mbar_arrive_expect_tx(bar(k8KFull + st), Lay::kTileBytes);
            ptx::tma_load_4d(sbase + Lay::kKOff + st * Lay::kTileBytes, &tmap_k, bar(k8KFull + st),
                             0, it.h, ks - p.kv_row0, it.b);
            bump(st, k_armed0, k_armed1, k_armed2);
          }
          if (!wait1(bar(k8VEmpty + st), ph ^ 1u, abort_flag, p)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(bar(k8VFull + st), Lay::kTileBytes);
          // V^T [B, H, d, S]: one box of 128 keys x D rows (keys contiguous)
          ptx::tma_load_4d(sbase + Lay::kVOff + st * Lay::kTileBytes, &tmap_v, bar(k8VFull + st),
                           ks - p.kv_row0, 0, it.h, it.b);
          bump(st, v_armed0, v_armed1, v_armed2);
          ++kv_iter;
        }
      }
      // No more items: tell the MMA warp through the next phase of k8QFull.
      if (ok && wait1(bar(k8QEmpty), (q_iter & 1u) ^ 1u, abort_flag, p)) {
        *q_item = p.n_items;
        ptx::mbar_arrive(bar(k8QFull));
        ++q_iter;
      }
      // Let every copy this thread started land before the CTA can exit.
      if (q_iter > 0) wait1(bar(k8QFull), (q_iter - 1) & 1u, abort_flag, p, false);
      const uint32_t k_armed[kStages8] = {k_armed0, k_armed1, k_armed2};
      const uint32_t v_armed[kStages8] = {v_armed0, v_armed1, v_armed2};
#pragma unroll
      for (int s = 0; s < kStages8; ++s) {
        if (k_armed[s] > 0) wait1(bar(k8KFull + s), (k_armed[s] - 1) & 1u, abort_flag, p, false);
        if (v_armed[s] > 0) wait1(bar(k8VFull + s), (v_armed[s] - 1) & 1u, abort_flag, p, false);
      }
    }
   } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // Per key tile f: S(f) of both query tiles as soon as each softmax has
    // loaded its previous S, then PV(f - 1) of both tiles as each P lands in
    // shared memory.  The whole warp runs the loop; elect.sync picks the lane
    // that issues each MMA and commit.
    {
      constexpr uint32_t kIdesc = ptx::idesc_e4m3_f32(kBM, kBN);  // S and PV: 128 x 128
      static_assert(kBN == D, "one instruction descriptor for both products");
      // Per-tile state in scalars (a runtime index into a local array would
      // put it in memory).
      uint32_t kv_iter = 0, q_iter = 0;
      uint32_t s_issued0 = 0, s_issued1 = 0;   // S products issued, per query tile
      uint32_t pv_issued0 = 0, pv_issued1 = 0; // PV products issued, per query tile
      bool ok = true;
      const uint64_t d_sw = ptx::smem_desc_sw128(sbase, 16, 1024);
      // O_t (+)= P_t V: P from its shared-memory buffer, V^T K-major; a K step
      // is 32 E4M3 (32 bytes) along the 128-byte swizzled rows of both.
      auto issue_pv = [&](int t, uint32_t& n_pv, uint32_t st, bool& first, bool last) -> bool {
        const uint32_t n = n_pv;
        const int b = static_cast<int>(n & 1u);
        if (!wait_warp(bar(k8PReady + 2 * t + b), (n >> 1) & 1u, abort_flag, p)) return false;
        ptx::tc_fence_after();
        const uint64_t dp = d_sw + ((Lay::kPOff + (2 * t + b) * Lay::kTileBytes) >> 4);
        const uint64_t dv = d_sw + ((Lay::kVOff + st * Lay::kTileBytes) >> 4);
#pragma unroll
        for (int s = 0; s < kBN / 32; ++s)
          ptx::mma_ss_f8_w(tmem_base + 256 + t * D, dp + static_cast<uint64_t>(2 * s),
                           dv + static_cast<uint64_t>(2 * s), kIdesc, (first && s == 0) ? 0u : 1u);
        ptx::mma_commit_w(bar(k8PFree + 2 * t + b));
        if (last) ptx::mma_commit_w(bar(k8OBar + t));
        first = false;
        n_pv = n + 1;
        return true;
      };
      // S_t = Q_t K^T (both K-major, one 128-byte swizzled panel each), once
      // the softmax has loaded the tile's previous S.
      auto issue_s = [&](int t, uint32_t& n_s, uint32_t st) -> bool {
        if (n_s > 0) {
          if (!wait_warp(bar(k8SFree + t), (n_s - 1) & 1u, abort_flag, p)) return false;
          ptx::tc_fence_after();
        }
        const uint64_t dq = d_sw + ((Lay::kQOff + t * Lay::kTileBytes) >> 4);
        const uint64_t dk = d_sw + ((Lay::kKOff + st * Lay::kTileBytes) >> 4);
#pragma unroll
        for (int s = 0; s < D / 32; ++s)
          ptx::mma_ss_f8_w(tmem_base + t * 128, dq + static_cast<uint64_t>(2 * s),
                           dk + static_cast<uint64_t>(2 * s), kIdesc, s > 0 ? 1u : 0u);
        ptx::mma_commit_w(bar(k8SFull + t));
        ++n_s;
        return true;
      };
      for (;;) {
        // The producer publishes each item that has work with its Q load
        // (and the end of the work with a plain arrival), so this warp needs
        // no wait beyond the one for Q.
        if (!wait_warp(bar(k8QFull), q_iter & 1u, abort_flag, p)) { ok = false; break; }
        ++q_iter;
        const int w = *q_item;
        if (w >= p.n_items) break;
        Item it;
        decode_item(p, n_docs, w, it);
        ptx::tc_fence_after();
        bool pend0 = false, pend1 = false;    // S issued whose PV is still owed
        bool first0 = true, first1 = true;    // next PV overwrites O
        uint32_t prev_st = 0, prev_ph = 0;
        bool have_prev = false;
        // Owed PVs on the previous K/V stage (V(f_prev)); then release it.
        auto flush = [&](int f_prev) -> bool {
          if (pend0 || pend1) {
            if (!wait_warp(bar(k8VFull + prev_st), prev_ph, abort_flag, p)) return false;
          }
          if (pend0 && !issue_pv(0, pv_issued0, prev_st, first0, f_prev == it.f_hi[0]))
            return false;
          if (pend1 && !issue_pv(1, pv_issued1, prev_st, first1, f_prev == it.f_hi[1]))
            return false;
          pend0 = pend1 = false;
          ptx::mma_commit_w(bar(k8VEmpty + prev_st));
          return true;
        };
        for (int f = it.F_lo; f <= it.F_hi; ++f) {
          const uint32_t st = kv_iter % kStages8;
          const uint32_t ph = (kv_iter / kStages8) & 1u;
          if (!wait_warp(bar(k8KFull + st), ph, abort_flag, p)) { ok = false; break; }
          ptx::tc_fence_after();
          const bool now0 = (f >= it.f_lo[0] && f <= it.f_hi[0]);
          const bool now1 = (f >= it.f_lo[1] && f <= it.f_hi[1]);
          if (now0 && !issue_s(0, s_issued0, st)) { ok = false; break; }
          if (now1 && !issue_s(1, s_issued1, st)) { ok = false; break; }
          ptx::mma_commit_w(bar(k8KEmpty + st));  // K(f) read by every S
          if (have_prev && !flush(f - 1)) { ok = false; break; }
          pend0 = now0;
          pend1 = now1;
          prev_st = st;
          prev_ph = ph;
          have_prev = true;
          ++kv_iter;
        }
        if (!ok) break;
        ptx::mma_commit_w(bar(k8QEmpty));  // every S of this item has been issued
        if (have_prev && !flush(it.F_hi)) { ok = false; break; }
      }
      // Wait until every MMA this warp issued has finished.
      ptx::mma_commit_w(bar(k8Drain));
      wait_warp(bar(k8Drain), 0u, abort_flag, p, false);
    }
   }
  } else {
    ptx::setmaxnreg_inc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;  // query tile of this warpgroup
    const int wq = warp & 3;  // TMEM lane quarter
    const int row_in_tile = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem_base + lane_off + static_cast<uint32_t>(t * 128);
    const uint32_t tO = tmem_base + lane_off + 256u + static_cast<uint32_t>(t * D);
    // this thread's row of a P buffer: 128 bytes, 16-byte chunk c stored at
    // chunk c ^ (row % 8) of its row (the 128-byte swizzle the MMA reads)
    const uint32_t p_row = sbase + Lay::kPOff + static_cast<uint32_t>(2 * t * Lay::kTileBytes) +
                           static_cast<uint32_t>((row_in_tile >> 3) * 1024 + (row_in_tile & 7) * 128);
    const uint32_t r8 = static_cast<uint32_t>(row_in_tile & 7);
    uint32_t s_cnt = 0, p_cnt = 0, o_cnt = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int w = ring_get(ring, static_cast<uint32_t>(k), abort_flag, p);
      if (w < 0) { ok = false; break; }
      if (w >= p.n_items) break;
      Item it;
      decode_item(p, n_docs, w, it);
      const int rows = t ? it.rows[1] : it.rows[0];
      const int f_lo = t ? it.f_lo[1] : it.f_lo[0];
      const int f_hi = t ? it.f_hi[1] : it.f_hi[0];
      if (rows == 0 || f_lo > f_hi) continue;
      const int bh = it.b * p.H + it.h;
      const float sc = p.scale_log2 * __ldg(p.q_descale + bh) * __ldg(p.k_descale + bh);
      const bool row_valid = row_in_tile < rows;
      const int r = (t ? it.q0[1] : it.q0[0]) + row_in_tile;
      int klo_r = 0, khi_r = -1;
      if (row_valid) {
        const int2 ds = doc_span(p, n_docs, r);
        klo_r = max(ds.x, it.klo);
        khi_r = min(p.causal ? r : ds.y - 1, it.khi);
      }
      float m_used = -INFINITY, l_run = 0.f;
      for (int f = f_lo; f <= f_hi; ++f) {
        if (!wait_warp(bar(k8SFull + t), s_cnt & 1u, abort_flag, p)) { ok = false; break; }
        ++s_cnt;
        ptx::tc_fence_after();
        int ks, ke;
        tile_keys(p, f, ks, ke);
        const int c_lo = klo_r - ks;
        const int c_hi = min(khi_r, ke - 1) - ks;
        uint32_t sv[4][32];
        uint32_t pk[2][32];
        load_scores(tS, c_lo, c_hi, sv);
        if (CPRING_FP8_EARLY_SFREE) {
          // S is in registers: its TMEM columns may take the next key tile's S.
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(k8SFree + t));
        }
        float lsum = 0.f, mx;
        float alpha = 1.f;
        bool rescale_o = false;
        if (CPRING_FP8_FAST && !__any_sync(0xffffffffu, m_used == -INFINITY)) {
          // One pass over the 128 keys against the current reference; a row
          // sum above 2^8 sends the tile to the redo below, which keeps every
          // P inside E4M3's range (448).
          if (CPRING_FP8_EXP_F16) {
            exp_chunks_f8h(sv, 0, sc, m_used, pk, lsum);
            exp_chunks_f8h(sv, 1, sc, m_used, pk, lsum);
          } else {
            uint64_t acc = 0;  // two fp32 zeros
            exp_chunks_f8(sv, 0, sc, m_used, pk, acc);
            exp_chunks_f8(sv, 1, sc, m_used, pk, acc);
            lsum = sum2(acc);
          }
          const bool redo = !(lsum <= kOverflowGuardFp8);
          if (__any_sync(0xffffffffu, redo)) {
            // Rare: a sum above the guard means this tile's max is above the
            // reference (128 entries of at most 1 sum to 128 or less).  Move
            // the reference of those rows to this tile's max and recompute
            // (from the registers, or from S still held in TMEM).
            if (!CPRING_FP8_EARLY_SFREE) load_scores(tS, c_lo, c_hi, sv);
            const float m_tile = row_max(sv) * sc;
            if (redo && m_tile > m_used) {
              rescale_o = true;
              alpha = ptx::ex2(m_used - m_tile);
              l_run *= alpha;
              m_used = m_tile;
            }
            exponentials<true>(sv, sc, m_used, pk, lsum, mx);
          }
        } else {
          // Some row of this warp has no reference yet: row max first.
          mx = row_max(sv);
          const float m_tile = mx * sc;
          if (m_tile > m_used + kRescaleLog2) {
            rescale_o = (m_used != -INFINITY);
            alpha = rescale_o ? ptx::ex2(m_used - m_tile) : 0.f;
            l_run *= alpha;
            m_used = m_tile;
          }
          exponentials<true>(sv, sc, (m_used == -INFINITY) ? 0.f : m_used, pk, lsum, mx);
        }
        if (!CPRING_FP8_EARLY_SFREE) {
          // This tile's S is no longer needed: its TMEM columns may take the
          // next key tile's S while P goes out and PV runs.
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(k8SFree + t));
        }
        l_run += lsum;
        const uint32_t n = p_cnt++;
        const uint32_t b = n & 1u;
        bool rescaled = false;
        if (__any_sync(0xffffffffu, rescale_o)) {
          // O_t must hold every earlier PV of this tile before it is scaled:
          // wait for the PV of the previous key tile (the one before it was
          // already waited for by the P-buffer reuse below).
          if (n >= 1 && !wait_warp(bar(k8PFree + 2 * t + ((n - 1) & 1u)), ((n - 1) >> 1) & 1u,
                                   abort_flag, p)) { ok = false; break; }
          ptx::tc_fence_after();
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t ov[32];
            ptx::tmem_ld32(tO + ch * 32, ov);
            ptx::tmem_wait_ld();
            ptx::reg_fence(ov);
#pragma unroll
            for (int x = 0; x < 32; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * alpha);
            ptx::tmem_st32(tO + ch * 32, ov);
          }
          rescaled = true;
        }
        // The buffer's previous P (two key tiles back) must have been read.
        if (n >= 2 && !wait_warp(bar(k8PFree + 2 * t + b), ((n >> 1) - 1) & 1u, abort_flag, p)) {
          ok = false;
          break;
        }
        const uint32_t dst = p_row + b * static_cast<uint32_t>(Lay::kTileBytes);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          ptx::st_shared_v4(dst + ((static_cast<uint32_t>(ch) ^ r8) << 4), pk[0][4 * ch],
                            pk[0][4 * ch + 1], pk[0][4 * ch + 2], pk[0][4 * ch + 3]);
        ptx::fence_proxy_async_shared();
        if (rescaled) ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(k8PReady + 2 * t + b));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!wait_warp(bar(k8OBar + t), o_cnt & 1u, abort_flag, p)) { ok = false; break; }
      ++o_cnt;
      ptx::tc_fence_after();
      const float inv_l = __ldg(p.v_descale + bh) / l_run;
      uint4* dst = reinterpret_cast<uint4*>(
          p.out + ((static_cast<size_t>(it.b) * p.S + r) * p.H + it.h) * D);
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t ov[32];
        ptx::tmem_ld32(tO + ch * 32, ov);
        ptx::tmem_wait_ld();
        ptx::reg_fence(ov);
        if (row_valid) {
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            uint4 v4;
            v4.x = ptx::pack_bf16(__uint_as_float(ov[8 * x + 0]) * inv_l,
                                  __uint_as_float(ov[8 * x + 1]) * inv_l);
            v4.y = ptx::pack_bf16(__uint_as_float(ov[8 * x + 2]) * inv_l,
                                  __uint_as_float(ov[8 * x + 3]) * inv_l);
            v4.z = ptx::pack_bf16(__uint_as_float(ov[8 * x + 4]) * inv_l,
                                  __uint_as_float(ov[8 * x + 5]) * inv_l);
            v4.w = ptx::pack_bf16(__uint_as_float(ov[8 * x + 6]) * inv_l,
                                  __uint_as_float(ov[8 * x + 7]) * inv_l);
            dst[ch * 4 + x] = v4;
          }
        }
      }
      if (row_valid) {
        p.lse[(static_cast<size_t>(it.b) * p.H + it.h) * p.S + r] =
            (m_used + log2f(l_run)) * 0.69314718055994531f;
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int D, bool kPartial, bool kDynamic>
__global__ void __launch_bounds__(kThreads, 1)
    ring_attn_bf16_kernel(const __grid_constant__ CUtensorMap tmap_q,
                          const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, const KParams p) {
  attn_body<D, kPartial, kDynamic>(tmap_q, tmap_k, tmap_v, p);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    ring_attn_fp8_kernel(const __grid_constant__ CUtensorMap tmap_q,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const KParams p) {
  attn_body_fp8<D>(tmap_q, tmap_k, tmap_v, p);
}

// ---------------------------------------------------------------- host side
// V^T [B, H, D, S] of bytes viewed as (S, D, H, B); box = 128 keys x D rows.
// Needs S % 16 == 0 (row stride a multiple of 16 bytes).
bool make_map_vt8(CUtensorMap* m, const void* base, int B, int S, int H, int D) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(D),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(D) * S,
                           static_cast<cuuint64_t>(H) * D * S};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(kBN), static_cast<cuuint32_t>(D), 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Test hook state (see cp_test_set_wait_fault).
std::atomic<int> g_fault_drop_k{0};
std::atomic<unsigned long long> g_wait_limit_ns{kTimeoutNs};

// With documents the work of a slot (query shard, pair of query tiles) is
// its number of visible key tiles, which depends on the layout, not on the
// position: rank the slots by that cost, heaviest first (ties: later slot
// first, the order used without documents), so the CTAs claim the heavy
// items first and the tail holds only light ones.  Every (b, h) shares the layout, so one block ranks the slots of
// (b, h) = (0, 0); O(slots^2) compares, used up to kMaxRankedSlots.

__global__ void __launch_bounds__(1024) slot_order_kernel(KParams p, int32_t* __restrict__ perm) {
  __shared__ int cost[kMaxRankedSlots];
  const int slots = p.n_qshards * p.pairs_per_shard;
  int n_docs = 1;
  if (p.doc_offsets != nullptr) {
    n_docs = __ldg(p.doc_info);
    if (n_docs <= 0) return;
  }
  p.B = 1;
  p.H = 1;
  p.head_group = 1;
  p.slot_perm = nullptr;
  for (int s = threadIdx.x; s < slots; s += blockDim.x) {
    Item it;
    decode_item(p, n_docs, slots - 1 - s, it);   // item w = slots - 1 - s is slot s
    int c = 0;
#pragma unroll
    for (int t = 0; t < kQTiles; ++t)
      if (it.f_lo[t] <= it.f_hi[t]) c += it.f_hi[t] - it.f_lo[t] + 1;
    cost[s] = c;
  }
  __syncthreads();
  for (int s = threadIdx.x; s < slots; s += blockDim.x) {
    const int cs = cost[s];
    int rank = 0;
    for (int u = 0; u < slots; ++u) {
      const int cu = cost[u];
      rank += (cu > cs) || (cu == cs && u > s);
    }
    perm[rank] = s;
  }
}

template <int D, bool kPartial, bool kFp8 = false, bool kDynamic = true>
cudaError_t launch_t(const AttnArgs& a, cudaStream_t stream) {
  using Lay = std::conditional_t<kFp8, Fp8Layout, Layout<D, 2>>;
  static_assert(Lay::kAlloc <= 232448, "shared memory budget");
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, KParams);
  if constexpr (kFp8)
    kern = ring_attn_fp8_kernel<D>;
  else
    kern = ring_attn_bf16_kernel<D, kPartial, kDynamic>;
  const cudaError_t attr_err = ensure_smem_limit(reinterpret_cast<const void*>(kern), Lay::kAlloc);
  if (attr_err != cudaSuccess) return attr_err;

  CUtensorMap mq, mk, mv;
  const int kv_rows = a.kv_rows > 0 ? a.kv_rows : a.S;
  if constexpr (kFp8) {
    if (a.kv_rows > 0) return cudaErrorInvalidValue;  // the FP8 form reads whole tensors
    if (!make_map(&mq, a.q, a.B, a.S, a.H, D, 1) || !make_map(&mk, a.k, a.B, a.S, a.H, D, 1) ||
        !make_map_vt8(&mv, a.v, a.B, a.S, a.H, D))
      return cudaErrorInvalidValue;
  } else {
    if (!make_map(&mq, a.q, a.B, a.S, a.H, D) || !make_map(&mk, a.k, a.B, kv_rows, a.H, D) ||
        !make_map(&mv, a.v, a.B, kv_rows, a.H, D))
      return cudaErrorInvalidValue;
  }

  KParams p{};
  p.B = a.B;
  p.S = a.S;
  p.H = a.H;
  p.n_shards = a.n_shards;
  p.L = a.S / a.n_shards;
  p.q_shard = a.q_shard;
  p.k_shard = a.k_shard;
  p.kv_row0 = a.kv_rows > 0 ? a.kv_row0 : 0;
  p.causal = a.causal;
  p.doc_offsets = a.doc_offsets;
  p.doc_info = a.doc_info;
  p.n_qshards = (a.q_shard < 0) ? a.n_shards : 1;
  p.pairs_per_shard = (p.L + kBM * kQTiles - 1) / (kBM * kQTiles);
  p.tiles_per_shard = (p.L + kBN - 1) / kBN;
  const long long items = static_cast<long long>(a.B) * a.H * p.n_qshards * p.pairs_per_shard;
  if (items > INT_MAX) return cudaErrorInvalidValue;
  p.n_items = static_cast<int>(items);
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.o_part = a.o_part;
  p.m_part = a.m_part;
  p.l_part = a.l_part;
  p.q_descale = a.q_descale;
  p.k_descale = a.k_descale;
  p.v_descale = a.v_descale;
  p.err = device_error_word();
  if (!p.err) return cudaErrorInvalidValue;
  p.timeout_ns = g_wait_limit_ns.load();
  p.fault_drop_k = g_fault_drop_k.load();
  unsigned long long* slots = work_slots_address();
  if (!slots) return cudaErrorInvalidValue;
  const uint32_t epoch = next_epoch(slots);
  if (epoch == 0) return cudaErrorInvalidValue;
  p.epoch = epoch;
  p.work_slot = slots + epoch % kWorkSlots;
  const int grid = static_cast<int>(std::min<long long>(items, sm_count()));
  // Head groups: fewer heads in flight reuse each K/V tile from L2.  A long
  // launch (many rounds of the grid) takes the smallest group whose items
  // fill CPRING_BALANCE rounds; a short one keeps a single pool, so that its
  // lightest items come last.  With documents the item count says little
  // about the work (the layout decides it), so CPRING_GROUP_DOCS decides.
  {
    const int BH = a.B * a.H;
    const long long slots = static_cast<long long>(p.n_qshards) * p.pairs_per_shard;
    long long hg = BH;
    if ((a.doc_offsets == nullptr || CPRING_GROUP_DOCS) &&
        items >= static_cast<long long>(CPRING_GROUP_MIN_ROUNDS) * grid) {
      hg = (static_cast<long long>(CPRING_BALANCE) * grid + slots - 1) / slots;
      hg = std::max<long long>(1, std::min<long long>(hg, BH));
    }
    p.head_group = static_cast<int>(hg);
  }
  p.slot_perm = nullptr;
  if (a.doc_offsets != nullptr && a.slot_perm != nullptr &&
      p.n_qshards * p.pairs_per_shard <= kMaxRankedSlots) {
    slot_order_kernel<<<1, 1024, 0, stream>>>(p, a.slot_perm);
    count_launch(2);
    p.slot_perm = a.slot_perm;
  }
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, kThreads, Lay::kAlloc, stream>>>(mq, mk, mv, p);
  count_launch(0);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bf16(const AttnArgs& a, cudaStream_t stream) {
  const bool partial = (a.k_shard >= 0);
  // Claimed items pay where the items' costs are uneven or few: documents
  // and one step's launch.  A launch without documents over whole key ranges
  // (all ranks, or one rank's query shard) takes the fixed snake deal, which
  // measured faster there (81.4 against 85.7 ms for all ranks at 128K, and
  // 87.2 against 89.5 ms for the four rank launches of the same shape).
  const bool dynamic = CPRING_DYNAMIC_ALWAYS || a.doc_offsets != nullptr ||
                       (CPRING_RANK_DYNAMIC && a.q_shard >= 0) || partial;
  if (a.d == 128) {
    if (partial) return launch_t<128, true, false, true>(a, stream);
    return dynamic ? launch_t<128, false, false, true>(a, stream)
                   : launch_t<128, false, false, false>(a, stream);
  }
  if (a.d == 64) {
    if (partial) return launch_t<64, true, false, true>(a, stream);
    return dynamic ? launch_t<64, false, false, true>(a, stream)
                   : launch_t<64, false, false, false>(a, stream);
  }
  return cudaErrorInvalidValue;
}

// The tile ranges the fused kernel walks, from its own decode_item: for
// every 128-row query tile (flat order) the first and last flat key tile.
__global__ void schedule_probe_kernel(const KParams p, int32_t* __restrict__ ranges) {
  const int w = blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= p.n_items) return;
  int n_docs = 1;
  if (p.doc_offsets != nullptr) {
    n_docs = __ldg(p.doc_info);
    if (n_docs <= 0) return;
  }
  Item it;
  decode_item(p, n_docs, w, it);
#pragma unroll
  for (int t = 0; t < kQTiles; ++t) {
    if (it.rows[t] == 0) continue;
    const int qt = it.i * p.tiles_per_shard + (it.q0[t] - it.i * p.L) / kBM;
    ranges[2 * qt] = it.f_lo[t];
    ranges[2 * qt + 1] = it.f_hi[t];
  }
}

cudaError_t launch_schedule_probe(const AttnArgs& a, int32_t* ranges, cudaStream_t stream) {
  KParams p{};
  p.B = 1;
  p.S = a.S;
  p.H = 1;
  p.n_shards = a.n_shards;
  p.L = a.S / a.n_shards;
  p.q_shard = -1;
  p.k_shard = -1;
  p.causal = a.causal;
  p.doc_offsets = a.doc_offsets;
  p.doc_info = a.doc_info;
  p.n_qshards = a.n_shards;
  p.pairs_per_shard = (p.L + kBM * kQTiles - 1) / (kBM * kQTiles);
  p.tiles_per_shard = (p.L + kBN - 1) / kBN;
  p.n_items = p.n_qshards * p.pairs_per_shard;
  p.head_group = 1;
  const int grid = (p.n_items + 127) / 128;
  schedule_probe_kernel<<<grid, 128, 0, stream>>>(p, ranges);
  count_launch(2);
  return cudaGetLastError();
}

cudaError_t launch_attn_fp8(const AttnArgs& a, cudaStream_t stream) {
  if (a.d != 128 || a.k_shard >= 0 || a.q_shard >= 0 || !a.q_descale || !a.k_descale ||
      !a.v_descale)
    return cudaErrorInvalidValue;
  return launch_t<128, false, true>(a, stream);
}

int test_fault_drop() { return g_fault_drop_k.load(); }
unsigned long long test_wait_limit_ns() { return g_wait_limit_ns.load(); }

}  // namespace cpring

extern "C" void cp_test_set_wait_fault(int drop_first_k_tile, long long wait_limit_ns) {
  cpring::g_fault_drop_k.store(drop_first_k_tile ? 1 : 0);
  cpring::g_wait_limit_ns.store(wait_limit_ns > 0 ? static_cast<unsigned long long>(wait_limit_ns)
                                                  : cpring::kTimeoutNs);
}
