// Ring-attention backward for bf16 inputs on sm_103a tensor cores (tcgen05).
//
// What is computed.  "上下文並行（Context Parallelism, CP）" (compassingai.com),
// section 反向傳播: the backward walks the ring's K/V blocks again;
// "大语言模型并行策略（五）：上下文并行" (wangyu.me): the gradients of K and V
// travel with their blocks.  For L = sum(out * dout), per (b, h), with P the
// forward's softmax recomputed from its saved log-sum-exp:
//   D = rowsum(dO * O);  dP = dO V^T;  dS = P * (dP - D);
//   dV = P^T dO;  dK = dS^T Q / sqrt(d);  dQ = dS K / sqrt(d),
// summed over the visible shard pairs and tiles of the forward (tiles are
// laid from each shard's first row; pairs with no visible (q, k) are never
// loaded).
//
// Two kernels share one body:
//   kDKDV  a CTA owns a 128-key tile of one (b, h) - the dK_j / dV_j
//          accumulators that travel with K_j, V_j around the ring - and walks
//          the query tiles that see it: S^T = K Q^T and dP^T = V dO^T on the
//          tensor cores with both operands in shared memory, P^T and dS^T in
//          the softmax warps, then dV += P^T dO and dK += dS^T Q with the A
//          operand taken from TMEM.
//   kDQ    a CTA owns a 128-query tile and walks the key tiles it sees:
//          S = Q K^T, dP = dO V^T, dS, then dQ += dS K.
// Every CTA finishes its own output tile, so no atomics are needed; the price
// is that S and dP are formed by both kernels (7 tile products where the
// gradient needs 5).
//
// CTA (384 threads): warps 0-3 and 4-7 split the 128 columns of each S / dP
// tile (64 each) over the same 128 rows, one thread per TMEM lane; warp 8
// is the TMA producer (the two fixed tiles once per item, the streamed tiles
// of every step into their slot rings); warp 9 issues every tcgen05.mma
// (one lane, picked by elect.sync, per instruction); warps 10-11 only
// complete the third warpgroup, which hands its registers to the softmax
// warpgroups through setmaxnreg.
// TMEM (512 columns).  kDQ: S | dP | dQ | two buffers of packed dS.  kDKDV
// runs each 128-query tile as two 64-query halves in two buffers
// (S^T 64 | dP^T 64) x 2 | dV | dK, so the products of the next half overlap
// the softmax of the current one.  A warpgroup writes its packed bf16 P / dS
// into the first columns of the range it read itself, so nothing is
// overwritten before its owner has read it; the TS products gather their A
// operand from the warpgroups' pieces.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <mutex>

#include "attn_common.cuh"
#include "internal.h"
#include "ptx.cuh"

// Head-group size of the backward's deal: the smallest group of heads whose
// items fill this many rounds of the grid (see launch_bwd_t).
#ifndef CPRING_BWD_BALANCE
#define CPRING_BWD_BALANCE 1
#endif

namespace cpring {
namespace {

constexpr int kT = kTileRows;       // rows of every tile
constexpr int kThreads = 384;        // three warpgroups (warps 10, 11 idle)
constexpr int kLaunchRegs = 168;     // registers per thread at launch (checked by the build)
constexpr int kSoftmaxRegs = 200;    // softmax warpgroups after setmaxnreg.inc
constexpr int kControlRegs = 104;    // producer / MMA warpgroup after setmaxnreg.dec
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch's register pool");
constexpr int kSoftmaxThreads = 256;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

// Streamed tiles run in two rings of single-tile slots: X0 (K for kDQ, Q for
// kDKDV) and X1 (V or dO).  kDQ holds K until dQ += dS K is done but V only
// until dP, and issues the next step's products early, so its K ring is one
// slot deeper.
template <int D, bool kDKDV>
struct BLayout {
  static constexpr int kTileBytes = kT * D * 2;
  static constexpr int kPanelBytes = kT * 128;   // 128 rows x 64 bf16 columns
  static constexpr int kPanels = D / 64;
  static constexpr int kX0Slots = kDKDV ? 2 : 3;
  static constexpr int kX1Slots = 2;
  static constexpr int kF0 = 0;                  // fixed tiles
  static constexpr int kF1 = kTileBytes;
  static constexpr int kX0 = 2 * kTileBytes;
  static constexpr int kX1 = kX0 + kX0Slots * kTileBytes;
  static constexpr int kVec = kX1 + kX1Slots * kTileBytes;    // kDKDV: [2][-lse2, -D][128] fp32
  static constexpr int kBar = kVec + (kDKDV ? 2 * 2 * kT * 4 : 0);
  static constexpr int kRingOff = kBar + 256;  // the item ring
  static constexpr int kBytes = kRingOff + 256;
  static constexpr int kAlloc = kBytes + 1024;
  __host__ __device__ static constexpr int x0(int slot) { return kX0 + slot * kTileBytes; }
  __host__ __device__ static constexpr int x1(int slot) { return kX1 + slot * kTileBytes; }
};

enum BBar : int {
  kFixFull = 0,
  kFixEmpty = 1,
  kX0Full = 2,     // + slot (3)
  kX1Full = 5,     // + slot (2)
  kX0Empty = 7,    // + slot (3)
  kX1Empty = 10,   // + slot (2)
  kSFull = 12,     // + TMEM buffer (kDKDV; kDQ uses +0): S and dP of a step are in TMEM
  kPReady = 14,    // + step parity: P / dS written by all softmax threads
  kSConsumed = 16, // kDQ: every softmax thread has read S and dP of the step
  kAccFull = 17,   // the item's accumulators are final
  kVecFull = 18,   // + buffer: per-column lse / delta of a query tile written (kDKDV)
  kVecFree = 20,   // + buffer: every softmax thread is done reading it
  kPReadyS = 22,   // + TMEM buffer (kDKDV): dS^T written (kPReady + buffer: P^T written)
  kDrain = 24,
  kNumBars = 25
};
// kDQ keeps packed dS in its own double buffer of TMEM columns (acc0 ends at
// 256 + D <= 384), so S and dP of the next step can be issued while the
// softmax still works on the current one.
constexpr uint32_t kDsBuf = 384;
constexpr int kTmemSlot = kNumBars * 8;
constexpr int kAbortSlot = kNumBars * 8 + 4;

struct BParams {
  int B, S, H, L, n_shards, causal;
  const int32_t* doc_offsets;
  const int32_t* doc_info;
  int tiles_per_shard, n_tiles, n_items;
  int head_group;       // (b, h) heads whose items are dealt out together
  float scale_log2;     // log2(e) / sqrt(d)
  float scale;          // 1 / sqrt(d)
  const float* lse;     // [B, H, S], natural log
  const float* delta;   // [B, H, S]
  __nv_bfloat16* g0;    // dQ (kDQ) or dV (kDKDV)
  __nv_bfloat16* g1;    // dK (kDKDV)
  int* err;
  unsigned long long timeout_ns;
  int fault_drop;       // test hook: CTA 0 never loads its first streamed X0 tile
  unsigned long long* work_slot;  // this launch's claim counter (see claim_first)
  uint32_t epoch;                 // this launch's tag in that counter
};

struct BItem {
  int b, h;
  int r0, r1;        // fixed rows [r0, r1)
  int x_lo, x_hi;    // flattened streamed tile range
};

// Item w: items are laid out head group by head group (head_group (b, h)
// heads at a time, so the CTAs in flight stream the tiles of few heads and
// re-read them from L2), and inside a group heaviest slot first (under
// causality the last query tiles see the most keys and the first key tiles
// are seen by the most queries); CTAs claim them in that order.
template <bool kDKDV>
__device__ __forceinline__ void decode_bitem(const BParams& p, int n_docs, int w, BItem& it) {
  const int BH = p.B * p.H;
  const int HG = p.head_group;
  const int gi = w / (HG * p.n_tiles);
  const int rr = w - gi * HG * p.n_tiles;
  const int hg = min(HG, BH - gi * HG);
  const int slot = rr / hg;
  const int bh = gi * HG + rr % hg;
  it.b = bh / p.H;
  it.h = bh - it.b * p.H;
  const int g = kDKDV ? slot : p.n_tiles - 1 - slot;
  tile_keys(p, g, it.r0, it.r1);
  int lo, hi;
  if (kDKDV) {  // queries that see a key of [r0, r1)
    lo = p.causal ? it.r0 : doc_span(p, n_docs, it.r0).x;
    hi = doc_span(p, n_docs, it.r1 - 1).y - 1;
  } else {      // keys seen by a query of [r0, r1)
    lo = doc_span(p, n_docs, it.r0).x;
    hi = p.causal ? it.r1 - 1 : doc_span(p, n_docs, it.r1 - 1).y - 1;
  }
  it.x_lo = flat_tile(p, lo);
  it.x_hi = flat_tile(p, hi);
}

template <int D, bool kDKDV>
__global__ void __launch_bounds__(kThreads, 1)
    ring_attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_f0,
                         const __grid_constant__ CUtensorMap tm_f1,
                         const __grid_constant__ CUtensorMap tm_x0,
                         const __grid_constant__ CUtensorMap tm_x1, const BParams p) {
  using Lay = BLayout<D, kDKDV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t bars = sbase + Lay::kBar;
  auto bar = [&](int idx) -> uint32_t { return bars + 8u * static_cast<uint32_t>(idx); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kBar + kTmemSlot);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + Lay::kBar + kAbortSlot);
  float* vec = reinterpret_cast<float*>(smem + Lay::kVec);
  const ItemRing ring{sbase + Lay::kRingOff,
                      reinterpret_cast<volatile int*>(smem + Lay::kRingOff + 2 * kRing * 8)};
  // the item whose fixed tiles the producer is loading (the MMA warp's copy)
  volatile int* fix_item = reinterpret_cast<volatile int*>(smem + Lay::kRingOff + 128);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int n_docs = 1;
  if (p.doc_offsets != nullptr) {
    n_docs = __ldg(p.doc_info);
    if (n_docs <= 0) return;  // malformed doc_offsets: the scan already flagged it
  }

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(kFixFull), 1);
    ptx::mbar_init(bar(kFixEmpty), 1);
    for (int s = 0; s < Lay::kX0Slots; ++s) {
      ptx::mbar_init(bar(kX0Full + s), 1);
      ptx::mbar_init(bar(kX0Empty + s), 1);
    }
    for (int s = 0; s < Lay::kX1Slots; ++s) {
      ptx::mbar_init(bar(kX1Full + s), 1);
      ptx::mbar_init(bar(kX1Empty + s), 1);
    }
    ptx::mbar_init(bar(kSFull), 1);
    ptx::mbar_init(bar(kSFull + 1), 1);
    ptx::mbar_init(bar(kPReady), kSoftmaxThreads);
    ptx::mbar_init(bar(kPReady + 1), kSoftmaxThreads);
    ptx::mbar_init(bar(kSConsumed), kSoftmaxThreads);
    ptx::mbar_init(bar(kAccFull), 1);
    for (int b2 = 0; b2 < 2; ++b2) {
      ptx::mbar_init(bar(kVecFull + b2), kT);
      ptx::mbar_init(bar(kVecFree + b2), kSoftmaxThreads);
    }
    ptx::mbar_init(bar(kPReadyS), kSoftmaxThreads);
    ptx::mbar_init(bar(kPReadyS + 1), kSoftmaxThreads);
    ptx::mbar_init(bar(kDrain), 1);
    ring_init(ring, kSoftmaxThreads / 32);  // the softmax warps read the ring
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
      ptx::tma_prefetch_desc(&tm_f0);
      ptx::tma_prefetch_desc(&tm_f1);
      ptx::tma_prefetch_desc(&tm_x0);
      ptx::tma_prefetch_desc(&tm_x1);
      uint32_t x_iter = 0, fix_iter = 0;
      uint32_t armed0[3] = {0u, 0u, 0u}, armed1[2] = {0u, 0u};  // loads started per slot
      unsigned long long ahead = 0;  // the claim of the CTA's next item
      bool dropped = false;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int w = !CPRING_DYNAMIC ? item_of(k, c, G)
                      : (k == 0) ? c : G + claimed_index(ahead, p.epoch, p.err);
        if (!ring_put(ring, static_cast<uint32_t>(k), w, abort_flag, p)) { ok = false; break; }
        if (w >= p.n_items) break;
        if (CPRING_DYNAMIC)  // claim the CTA's next item now; it is read when that item starts
          ahead = (k == 0) ? claim_first(p.work_slot, p.epoch) : claim_next(p.work_slot);
        BItem it;
        decode_bitem<kDKDV>(p, n_docs, w, it);
        if (!wait1(bar(kFixEmpty), (fix_iter & 1u) ^ 1u, abort_flag, p)) { ok = false; break; }
        *fix_item = w;  // the MMA warp reads it once this phase of kFixFull completes
        ptx::mbar_arrive_expect_tx(bar(kFixFull), 2 * Lay::kTileBytes);
        for (int pn = 0; pn < Lay::kPanels; ++pn) {
          ptx::tma_load_4d(sbase + Lay::kF0 + pn * Lay::kPanelBytes, &tm_f0, bar(kFixFull),
                           pn * 64, it.h, it.r0, it.b);
          ptx::tma_load_4d(sbase + Lay::kF1 + pn * Lay::kPanelBytes, &tm_f1, bar(kFixFull),
                           pn * 64, it.h, it.r0, it.b);
        }
        ++fix_iter;
        for (int f = it.x_lo; f <= it.x_hi; ++f) {
          const uint32_t s0 = x_iter % Lay::kX0Slots, ph0 = (x_iter / Lay::kX0Slots) & 1u;
          const uint32_t s1 = x_iter % Lay::kX1Slots, ph1 = (x_iter / Lay::kX1Slots) & 1u;
          int xs, xe;
          tile_keys(p, f, xs, xe);
          if (!wait1(bar(kX0Empty + s0), ph0 ^ 1u, abort_flag, p)) { ok = false; break; }
          if (p.fault_drop && c == 0 && !dropped) {
            // Test hook: this tile is never loaded, so the MMA warp's
            // bounded wait for it runs out and the CTA takes its abort path.
            dropped = true;
          } else {
            ptx::mbar_arrive_expect_tx(bar(kX0Full + s0), Lay::kTileBytes);
            for (int pn = 0; pn < Lay::kPanels; ++pn)
              ptx::tma_load_4d(sbase + Lay::x0(s0) + pn * Lay::kPanelBytes, &tm_x0,
                               bar(kX0Full + s0), pn * 64, it.h, xs, it.b);
            ++armed0[s0];
          }
          if (!wait1(bar(kX1Empty + s1), ph1 ^ 1u, abort_flag, p)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(bar(kX1Full + s1), Lay::kTileBytes);
          for (int pn = 0; pn < Lay::kPanels; ++pn)
            ptx::tma_load_4d(sbase + Lay::x1(s1) + pn * Lay::kPanelBytes, &tm_x1,
                             bar(kX1Full + s1), pn * 64, it.h, xs, it.b);
          ++armed1[s1];
          ++x_iter;
        }
      }
      // No more items: tell the MMA warp through the next phase of kFixFull.
      if (ok && wait1(bar(kFixEmpty), (fix_iter & 1u) ^ 1u, abort_flag, p)) {
        *fix_item = p.n_items;
        ptx::mbar_arrive(bar(kFixFull));
        ++fix_iter;
      }
      // Let every copy this thread started land before the CTA can exit.
      if (fix_iter > 0) wait1(bar(kFixFull), (fix_iter - 1) & 1u, abort_flag, p, false);
      for (int s = 0; s < Lay::kX0Slots; ++s)
        if (armed0[s] > 0) wait1(bar(kX0Full + s), (armed0[s] - 1) & 1u, abort_flag, p, false);
      for (int s = 0; s < Lay::kX1Slots; ++s)
        if (armed1[s] > 0) wait1(bar(kX1Full + s), (armed1[s] - 1) & 1u, abort_flag, p, false);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop with warp-uniform values; one lane picked
    // by elect.sync issues each MMA and commit (the warp-collective forms in
    // ptx.cuh), and every wait is the warp-uniform one.
    {
      constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(kT, kT, false);   // N = streamed rows
      constexpr uint32_t kIdescG = ptx::idesc_bf16_f32(kT, D, true);     // N = d, B MN-major
      const uint64_t d_k = ptx::smem_desc_sw128(sbase, 16, 1024);                // K-major
      const uint64_t d_mn = ptx::smem_desc_sw128(sbase, Lay::kPanelBytes, 1024);  // MN-major
      const uint32_t tS = tmem_base, tdP = tmem_base + 128;
      const uint32_t tA0 = tmem_base + 256, tA1 = tmem_base + 256 + D;
      uint32_t x_iter = 0, fix_iter = 0;
      bool ok = true;
      // D_t = A B^T over the head dimension, both tiles K-major.
      auto issue_ss = [&](uint32_t d_tmem, int a_off, int b_off) {
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint64_t step =
              static_cast<uint64_t>(((s >> 2) * Lay::kPanelBytes + (s & 3) * 32) >> 4);
          ptx::mma_ss_w(d_tmem, d_k + (a_off >> 4) + step, d_k + (b_off >> 4) + step, kIdescS,
                      s > 0 ? 1u : 0u);
        }
      };
      // acc (+)= A B: A = packed bf16 columns at a_tmem, in two halves
      // `half` columns apart (64: the halves of S / dP; 32: contiguous),
      // B = the streamed tile at b_off read MN-major (rows = K).
      auto issue_ts = [&](uint32_t acc, uint32_t a_tmem, int b_off, bool first, int half) {
#pragma unroll
        for (int s = 0; s < kT / 16; ++s) {
          const uint32_t a_col = static_cast<uint32_t>((s >> 2) * half + (s & 3) * 8);
          ptx::mma_ts_w(acc, a_tmem + a_col, d_mn + (b_off >> 4) + static_cast<uint64_t>(s * 128),
                      kIdescG, (first && s == 0) ? 0u : 1u);
        }
      };
      uint32_t n = 0;       // kDQ: steps issued so far (all items)
      uint32_t m_half = 0;  // kDKDV: halves issued so far (all items)
      constexpr uint32_t kIdescS64 = ptx::idesc_bf16_f32(kT, 64, false);
      // D = A B^T over the head dimension with B 64 rows (a half tile).
      auto issue_ss64 = [&](uint32_t d_tmem, int a_off, int b_off) {
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint64_t step =
              static_cast<uint64_t>(((s >> 2) * Lay::kPanelBytes + (s & 3) * 32) >> 4);
          ptx::mma_ss_w(d_tmem, d_k + (a_off >> 4) + step, d_k + (b_off >> 4) + step, kIdescS64,
                      s > 0 ? 1u : 0u);
        }
      };
      // acc (+)= A B over 64 queries: A = the two warpgroups' packed pieces
      // (32 columns apart), B = the half tile at b_off read MN-major.
      auto issue_ts64 = [&](uint32_t acc, uint32_t a_tmem, int b_off, bool first) {
#pragma unroll
        for (int s = 0; s < 64 / 16; ++s) {
          const uint32_t a_col = static_cast<uint32_t>((s >> 1) * 32 + (s & 1) * 8);
          ptx::mma_ts_w(acc, a_tmem + a_col, d_mn + (b_off >> 4) + static_cast<uint64_t>(s * 128),
                      kIdescG, (first && s == 0) ? 0u : 1u);
        }
      };
      for (;;) {
        // The producer publishes each item with its fixed tiles' load (and
        // the end of the work with a plain arrival), so this warp needs no
        // wait beyond the one for those tiles.
        if (!wait_warp(bar(kFixFull), fix_iter & 1u, abort_flag, p)) { ok = false; break; }
        ++fix_iter;
        const int w = *fix_item;
        if (w >= p.n_items) break;
        BItem it;
        decode_bitem<kDKDV>(p, n_docs, w, it);
        ptx::tc_fence_after();
        if constexpr (!kDKDV) {
          // S, dP of step n + 1 go out once the softmax has read those of
          // step n; dQ += dS K of step n once its dS is in buffer n % 2.
          bool have = false;  // S, dP of the current step already issued
          // S, dP of streamed step x: K from X0 slot x % 3, V from X1 slot
          // x % 2; V's slot is free once dP is done.
          auto issue_step = [&](uint32_t x) -> bool {
            const uint32_t s0 = x % Lay::kX0Slots, s1 = x % Lay::kX1Slots;
            if (!wait_warp(bar(kX0Full + s0), (x / Lay::kX0Slots) & 1u, abort_flag, p)) return false;
            if (!wait_warp(bar(kX1Full + s1), (x / Lay::kX1Slots) & 1u, abort_flag, p)) return false;
            ptx::tc_fence_after();
            issue_ss(tS, Lay::kF0, Lay::x0(s0));
            issue_ss(tdP, Lay::kF1, Lay::x1(s1));
            ptx::mma_commit_w(bar(kSFull));
            ptx::mma_commit_w(bar(kX1Empty + s1));
            return true;
          };
          for (int f = it.x_lo; f <= it.x_hi; ++f) {
            if (!have) {
              if (n > 0 && !wait_warp(bar(kSConsumed), (n - 1u) & 1u, abort_flag, p)) { ok = false; break; }
              if (!issue_step(x_iter)) { ok = false; break; }
            }
            have = false;
            if (f < it.x_hi) {
              if (!wait_warp(bar(kSConsumed), n & 1u, abort_flag, p)) { ok = false; break; }
              if (!issue_step(x_iter + 1)) { ok = false; break; }
              have = true;
            }
            if (!wait_warp(bar(kPReady + (n & 1u)), (n >> 1) & 1u, abort_flag, p)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t s0 = x_iter % Lay::kX0Slots;
            issue_ts(tA0, tmem_base + kDsBuf + (n & 1u) * 64u, Lay::x0(s0), f == it.x_lo, 32);
            ptx::mma_commit_w(bar(kX0Empty + s0));
            ++n;
            ++x_iter;
          }
          if (!ok) break;
          ptx::mma_commit_w(bar(kFixEmpty));
          ptx::mma_commit_w(bar(kAccFull));
          continue;
        }
        // kDKDV: half hh of the item is query rows 64 (hh % 2) .. of its
        // streamed tile x_iter + hh / 2; m counts halves over all items and
        // half m uses TMEM buffer m % 2.  S^T, dP^T of half m + 1 are issued
        // before dV, dK of half m, so they run during the softmax of half m.
        const int nh = 2 * (it.x_hi - it.x_lo + 1);
        auto issue_half = [&](uint32_t mm, int hh2) -> bool {
          const uint32_t xi = x_iter + static_cast<uint32_t>(hh2 >> 1);
          const uint32_t st = xi % Lay::kX0Slots, ph = (xi / Lay::kX0Slots) & 1u;
          if (!wait_warp(bar(kX0Full + st), ph, abort_flag, p)) return false;
          if (!wait_warp(bar(kX1Full + st), ph, abort_flag, p)) return false;
          ptx::tc_fence_after();
          const uint32_t b = mm & 1u;
          const int rows = (hh2 & 1) * 64 * 128;   // byte offset of query row 64 in a panel
          issue_ss64(tmem_base + 128u * b, Lay::kF0, Lay::x0(st) + rows);         // S^T = K Q_h^T
          issue_ss64(tmem_base + 128u * b + 64u, Lay::kF1, Lay::x1(st) + rows);   // dP^T = V dO_h^T
          ptx::mma_commit_w(bar(kSFull + b));
          return true;
        };
        if (!issue_half(m_half, 0)) { ok = false; break; }
        for (int hh = 0; hh < nh; ++hh) {
          const uint32_t b = m_half & 1u;
          if (hh + 1 < nh && !issue_half(m_half + 1, hh + 1)) { ok = false; break; }
          // dV += P^T dO_h as soon as P^T is in TMEM, dK += dS^T Q_h once dS^T is
          if (!wait_warp(bar(kPReady + b), (m_half >> 1) & 1u, abort_flag, p)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t st = (x_iter + static_cast<uint32_t>(hh >> 1)) % Lay::kX0Slots;
          const int rows = (hh & 1) * 64 * 128;
          issue_ts64(tA0, tmem_base + 128u * b, Lay::x1(st) + rows, hh == 0);
          if (!wait_warp(bar(kPReadyS + b), (m_half >> 1) & 1u, abort_flag, p)) { ok = false; break; }
          ptx::tc_fence_after();
          issue_ts64(tA1, tmem_base + 128u * b + 64u, Lay::x0(st) + rows, hh == 0);
          if (hh & 1) {
            ptx::mma_commit_w(bar(kX0Empty + st));
            ptx::mma_commit_w(bar(kX1Empty + st));
          }
          ++m_half;
        }
        if (!ok) break;
        x_iter += static_cast<uint32_t>(nh >> 1);
        if (!ok) break;
        ptx::mma_commit_w(bar(kFixEmpty));
        ptx::mma_commit_w(bar(kAccFull));
      }
      // Wait until every MMA this warp issued has finished.
      ptx::mma_commit_w(bar(kDrain));
      wait_warp(bar(kDrain), 0u, abort_flag, p, false);
    }
   }
  } else {
    ptx::setmaxnreg_inc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax
    const int wg = warp >> 2;        // column half of this warpgroup
    const int wq = warp & 3;         // TMEM lane quarter
    const int row_in_tile = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem_base + lane_off;
    const uint32_t tdP = tS + 128;
    const uint32_t tA0 = tS + 256, tA1 = tS + 256 + D;
    const int col0 = wg * 64;
    const float sc = p.scale_log2;
    uint32_t s_cnt = 0, item_cnt = 0, h_cnt = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int w = ring_get(ring, static_cast<uint32_t>(k), abort_flag, p);
      if (w < 0) { ok = false; break; }
      if (w >= p.n_items) break;
      BItem it;
      decode_bitem<kDKDV>(p, n_docs, w, it);
      const int r = it.r0 + row_in_tile;
      const bool row_valid = r < it.r1;
      const size_t bh_off = (static_cast<size_t>(it.b) * p.H + it.h) * p.S;
      int lo_r = 0, hi_r = -1;           // streamed indices this row sees
      float lse2_r = 0.f, d_r = 0.f;     // kDQ: per-row constants
      if (row_valid) {
        const int2 ds = doc_span(p, n_docs, r);
        if (kDKDV) {
          lo_r = p.causal ? r : ds.x;
          hi_r = ds.y - 1;
        } else {
          lo_r = ds.x;
          hi_r = p.causal ? r : ds.y - 1;
          lse2_r = __ldg(p.lse + bh_off + r) * kLog2e;
          d_r = __ldg(p.delta + bh_off + r);
        }
      }
      for (int f = it.x_lo; f <= it.x_hi; ++f) {
        int xs, xe;
        tile_keys(p, f, xs, xe);
        const int buf = static_cast<int>(s_cnt & 1u);
        const uint32_t use = s_cnt >> 1;  // uses of this buffer before this one
        if (kDKDV) {
          // Per-column constants of the streamed query tile, shared by all
          // rows: warps 0-3 write them once the previous user of the buffer
          // is done, every softmax warp waits for them (all waits bounded).
          if (threadIdx.x < kT) {
            if (use > 0 &&
                !wait_warp(bar(kVecFree + buf), (use - 1u) & 1u, abort_flag, p)) { ok = false; break; }
            const int q = xs + threadIdx.x;
            vec[(buf * 2 + 0) * kT + threadIdx.x] = q < xe ? -__ldg(p.lse + bh_off + q) * kLog2e : 0.f;
            vec[(buf * 2 + 1) * kT + threadIdx.x] = q < xe ? -__ldg(p.delta + bh_off + q) : 0.f;
            ptx::mbar_arrive(bar(kVecFull + buf));
          }
          if (!wait_warp(bar(kVecFull + buf), use & 1u, abort_flag, p)) { ok = false; break; }
        }
        const int c_lo = lo_r - xs;
        const int c_hi = min(hi_r, xe - 1) - xs;
        if constexpr (!kDKDV) {
          const uint32_t n = s_cnt;
          if (!wait_warp(bar(kSFull), s_cnt & 1u, abort_flag, p)) { ok = false; break; }
          ++s_cnt;
          ptx::tc_fence_after();
          // Read all of this half of S and dP, release them for the next
          // step's products, then form dS into buffer n % 2.
          uint32_t sv[2][32], dv[2][32];
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            ptx::tmem_ld32(tS + col0 + ch * 32, sv[ch]);
            ptx::tmem_ld32(tdP + col0 + ch * 32, dv[ch]);
          }
          ptx::tmem_wait_ld();
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            ptx::reg_fence(sv[ch]);
            ptx::reg_fence(dv[ch]);
          }
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(kSConsumed));
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            const int c0 = col0 + ch * 32;
            uint32_t pk_s[16];
            if (__all_sync(0xffffffffu, c_lo <= c0 && c_hi >= c0 + 31)) {
              // every column visible to every row of the warp: paired fp32
#pragma unroll
              for (int x = 0; x < 16; ++x) {
                float e0, e1, g0, g1;
                ptx::fma_f32x2(e0, e1, __uint_as_float(sv[ch][2 * x]), __uint_as_float(sv[ch][2 * x + 1]),
                               sc, sc, -lse2_r, -lse2_r);
                const float p0 = ptx::ex2(e0), p1 = ptx::ex2(e1);
                ptx::fma_f32x2(g0, g1, __uint_as_float(dv[ch][2 * x]), __uint_as_float(dv[ch][2 * x + 1]),
                               1.f, 1.f, -d_r, -d_r);
                ptx::fma_f32x2(g0, g1, p0, p1, g0, g1, 0.f, 0.f);
                pk_s[x] = ptx::pack_bf16(g0, g1);
              }
            } else {
#pragma unroll
              for (int x = 0; x < 16; ++x) {
                float dsr[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const int cc = c0 + 2 * x + e;
                  const bool vis = cc >= c_lo && cc <= c_hi;
                  const float pv =
                      vis ? ptx::ex2(fmaf(__uint_as_float(sv[ch][2 * x + e]), sc, -lse2_r)) : 0.f;
                  dsr[e] = pv * (__uint_as_float(dv[ch][2 * x + e]) - d_r);
                }
                pk_s[x] = ptx::pack_bf16(dsr[0], dsr[1]);
              }
            }
            ptx::tmem_st16(tmem_base + lane_off + kDsBuf + (n & 1u) * 64u + c0 / 2, pk_s);
          }
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(kPReady + (n & 1u)));
          continue;
        }
        ++s_cnt;  // query tiles seen: selects the per-column buffer
        // The two 64-query halves of this tile; half m uses TMEM buffer m % 2.
        for (int h = 0; h < 2; ++h) {
          const uint32_t b = h_cnt & 1u;
          if (!wait_warp(bar(kSFull + b), (h_cnt >> 1) & 1u, abort_flag, p)) { ok = false; break; }
          ptx::tc_fence_after();
          // this warpgroup's 32 columns of S^T and dP^T in buffer b
          const uint32_t tb = tmem_base + lane_off + 128u * b + 32u * static_cast<uint32_t>(wg);
          uint32_t sv[32], dv[32];
          ptx::tmem_ld32(tb, sv);
          ptx::tmem_ld32(tb + 64, dv);
          ptx::tmem_wait_ld();
          ptx::reg_fence(sv);
          ptx::reg_fence(dv);
          const int c0 = 64 * h + 32 * wg;   // first tile column of this piece
          uint32_t pk_p[16], pk_s[16];
          float pf[32];  // this chunk's P in fp32, for dS
          // per-column -lse2 and -D of this chunk, four columns per load
          const float4* nl4 = reinterpret_cast<const float4*>(vec + (buf * 2 + 0) * kT + c0);
          const float4* nd4 = reinterpret_cast<const float4*>(vec + (buf * 2 + 1) * kT + c0);
          // P^T first: it is stored and announced (kPReady) before dS^T is
          // formed, so the MMA warp starts dV += P^T dO meanwhile.
          const bool all_visible = __all_sync(0xffffffffu, c_lo <= c0 && c_hi >= c0 + 31);
          if (all_visible) {
            // every column visible to every row of the warp: paired fp32
#pragma unroll
            for (int x4 = 0; x4 < 8; ++x4) {
              const float4 nl = nl4[x4];
              const float nla[4] = {nl.x, nl.y, nl.z, nl.w};
#pragma unroll
              for (int hx = 0; hx < 2; ++hx) {
                const int x = 2 * x4 + hx;
                float e0, e1;
                ptx::fma_f32x2(e0, e1, __uint_as_float(sv[2 * x]), __uint_as_float(sv[2 * x + 1]), sc,
                               sc, nla[2 * hx], nla[2 * hx + 1]);
                pf[2 * x] = ptx::ex2(e0);
                pf[2 * x + 1] = ptx::ex2(e1);
                pk_p[x] = ptx::pack_bf16(pf[2 * x], pf[2 * x + 1]);
              }
            }
          } else {
#pragma unroll
            for (int x = 0; x < 16; ++x) {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int cc = c0 + 2 * x + e;
                const bool vis = cc >= c_lo && cc <= c_hi;
                pf[2 * x + e] =
                    vis ? ptx::ex2(fmaf(__uint_as_float(sv[2 * x + e]), sc, vec[(buf * 2 + 0) * kT + cc]))
                        : 0.f;
              }
              pk_p[x] = ptx::pack_bf16(pf[2 * x], pf[2 * x + 1]);
            }
          }
          ptx::tmem_st16(tb, pk_p);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(kPReady + b));
          // dS^T = P^T (dP^T - D)
          if (all_visible) {
#pragma unroll
            for (int x4 = 0; x4 < 8; ++x4) {
              const float4 nd = nd4[x4];
              const float nda[4] = {nd.x, nd.y, nd.z, nd.w};
#pragma unroll
              for (int hx = 0; hx < 2; ++hx) {
                const int x = 2 * x4 + hx;
                float g0, g1;
                ptx::fma_f32x2(g0, g1, __uint_as_float(dv[2 * x]), __uint_as_float(dv[2 * x + 1]), 1.f,
                               1.f, nda[2 * hx], nda[2 * hx + 1]);
                ptx::fma_f32x2(g0, g1, pf[2 * x], pf[2 * x + 1], g0, g1, 0.f, 0.f);
                pk_s[x] = ptx::pack_bf16(g0, g1);
              }
            }
          } else {
#pragma unroll
            for (int x = 0; x < 16; ++x) {
              float dsr[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int cc = c0 + 2 * x + e;
                dsr[e] = pf[2 * x + e] * (__uint_as_float(dv[2 * x + e]) + vec[(buf * 2 + 1) * kT + cc]);
              }
              pk_s[x] = ptx::pack_bf16(dsr[0], dsr[1]);
            }
          }
          ptx::tmem_st16(tb + 64, pk_s);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(kPReadyS + b));
          ++h_cnt;
        }
        if (!ok) break;
        ptx::mbar_arrive(bar(kVecFree + buf));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!wait_warp(bar(kAccFull), item_cnt & 1u, abort_flag, p)) { ok = false; break; }
      ++item_cnt;
      ptx::tc_fence_after();
#pragma unroll
      for (int a = 0; a < (kDKDV ? 2 : 1); ++a) {
        const uint32_t tacc = a == 0 ? tA0 : tA1;
        __nv_bfloat16* g = a == 0 ? p.g0 : p.g1;
        const float fac = (kDKDV && a == 0) ? 1.f : p.scale;  // dV unscaled; dK, dQ / sqrt(d)
        uint4* dst = reinterpret_cast<uint4*>(g + ((static_cast<size_t>(it.b) * p.S + r) * p.H + it.h) * D);
#pragma unroll
        for (int ch = 0; ch < D / 64; ++ch) {
          const int c0 = wg * (D / 2) + ch * 32;
          uint32_t ov[32];
          ptx::tmem_ld32(tacc + c0, ov);
          ptx::tmem_wait_ld();
          ptx::reg_fence(ov);
          if (row_valid) {
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              uint4 v4;
              v4.x = ptx::pack_bf16(__uint_as_float(ov[8 * x + 0]) * fac, __uint_as_float(ov[8 * x + 1]) * fac);
              v4.y = ptx::pack_bf16(__uint_as_float(ov[8 * x + 2]) * fac, __uint_as_float(ov[8 * x + 3]) * fac);
              v4.z = ptx::pack_bf16(__uint_as_float(ov[8 * x + 4]) * fac, __uint_as_float(ov[8 * x + 5]) * fac);
              v4.w = ptx::pack_bf16(__uint_as_float(ov[8 * x + 6]) * fac, __uint_as_float(ov[8 * x + 7]) * fac);
              dst[c0 / 8 + x] = v4;
            }
          }
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

// D[b, h, s] = sum_c dO[b, s, h, c] * O[b, s, h, c] (fp32), one warp per row.
__global__ void __launch_bounds__(256)
    bwd_delta_kernel(const __nv_bfloat162* __restrict__ out, const __nv_bfloat162* __restrict__ dout,
                     float* __restrict__ delta, int B, int S, int H, int D) {
  const long long rows = static_cast<long long>(B) * S * H;
  const int lane = threadIdx.x & 31;
  const int pairs = D / 2;
  for (long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       row < rows; row += (static_cast<long long>(gridDim.x) * blockDim.x) >> 5) {
    float acc = 0.f;
    for (int i = lane; i < pairs; i += 32) {
      const float2 o = __bfloat1622float2(out[row * pairs + i]);
      const float2 g = __bfloat1622float2(dout[row * pairs + i]);
      acc = fmaf(o.x, g.x, fmaf(o.y, g.y, acc));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      const int h = static_cast<int>(row % H);
      const long long bs = row / H;
      const int s = static_cast<int>(bs % S);
      const int b = static_cast<int>(bs / S);
      delta[(static_cast<long long>(b) * H + h) * S + s] = acc;
    }
  }
}

template <int D, bool kDKDV>
cudaError_t launch_bwd_t(const BwdArgs& a, cudaStream_t stream) {
  using Lay = BLayout<D, kDKDV>;
  static_assert(Lay::kAlloc <= 232448, "shared memory budget");
  static_assert(Lay::kX0Slots <= 3 && Lay::kX1Slots == 2, "barrier slots");
  auto kern = ring_attn_bwd_kernel<D, kDKDV>;
  const cudaError_t attr_err = ensure_smem_limit(reinterpret_cast<const void*>(kern), Lay::kAlloc);
  if (attr_err != cudaSuccess) return attr_err;
  // kDQ: fixed (Q, dO), streamed (K, V); kDKDV: fixed (K, V), streamed (Q, dO)
  const void* f0 = kDKDV ? a.k : a.q;
  const void* f1 = kDKDV ? a.v : a.dout;
  const void* x0 = kDKDV ? a.q : a.k;
  const void* x1 = kDKDV ? a.dout : a.v;
  CUtensorMap m0, m1, m2, m3;
  if (!make_map(&m0, f0, a.B, a.S, a.H, D) || !make_map(&m1, f1, a.B, a.S, a.H, D) ||
      !make_map(&m2, x0, a.B, a.S, a.H, D) || !make_map(&m3, x1, a.B, a.S, a.H, D))
    return cudaErrorInvalidValue;
  BParams p{};
  p.B = a.B;
  p.S = a.S;
  p.H = a.H;
  p.n_shards = a.n_shards;
  p.L = a.S / a.n_shards;
  p.causal = a.causal;
  p.doc_offsets = a.doc_offsets;
  p.doc_info = a.doc_info;
  p.tiles_per_shard = (p.L + kT - 1) / kT;
  p.n_tiles = a.n_shards * p.tiles_per_shard;
  const long long items = static_cast<long long>(a.B) * a.H * p.n_tiles;
  if (items > INT_MAX) return cudaErrorInvalidValue;
  p.n_items = static_cast<int>(items);
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
  p.lse = a.lse;
  p.delta = a.delta;
  p.g0 = static_cast<__nv_bfloat16*>(kDKDV ? a.dv : a.dq);
  p.g1 = static_cast<__nv_bfloat16*>(kDKDV ? a.dk : nullptr);
  p.err = device_error_word();
  if (!p.err) return cudaErrorInvalidValue;
  p.timeout_ns = test_wait_limit_ns();
  p.fault_drop = test_fault_drop();
  unsigned long long* slots = work_slots_address();
  if (!slots) return cudaErrorInvalidValue;
  const uint32_t epoch = next_epoch(slots);
  if (epoch == 0) return cudaErrorInvalidValue;
  p.epoch = epoch;
  p.work_slot = slots + epoch % kWorkSlots;
  const int grid = static_cast<int>(std::min<long long>(items, sm_count()));
  // Head groups as in the forward: a launch with at least 16 rounds of the
  // grid and no document layout takes the smallest group whose items fill
  // CPRING_BWD_BALANCE rounds; otherwise one pool, so that the lightest
  // items come last.
  {
    const int BH = a.B * a.H;
    long long hg = BH;
    if (a.doc_offsets == nullptr && items >= 16LL * grid) {
      hg = (static_cast<long long>(CPRING_BWD_BALANCE) * grid + p.n_tiles - 1) / p.n_tiles;
      hg = std::max<long long>(1, std::min<long long>(hg, BH));
    }
    p.head_group = static_cast<int>(hg);
  }
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, kThreads, Lay::kAlloc, stream>>>(m0, m1, m2, m3, p);
  count_launch(0);
  return cudaGetLastError();
}

// The dQ launch reads nothing that the dK/dV launch writes, so it can run on
// a second stream of the library's (one per device, created on first use
// and kept for the process's life): its CTAs then take the SMs that the
// dK/dV launch's last items leave idle instead of waiting for all of them.
// The caller's stream waits for it before anything enqueued later.
#ifndef CPRING_BWD_OVERLAP
#define CPRING_BWD_OVERLAP 1
#endif
struct BwdSideStream {
  std::mutex mu;
  cudaStream_t s = nullptr;
};
constexpr int kMaxBwdDevices = 64;
BwdSideStream g_bwd_side[kMaxBwdDevices];

cudaStream_t bwd_side_stream() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxBwdDevices) return nullptr;
  BwdSideStream& b = g_bwd_side[dev];
  std::lock_guard<std::mutex> lock(b.mu);
  if (!b.s && cudaStreamCreateWithFlags(&b.s, cudaStreamNonBlocking) != cudaSuccess) b.s = nullptr;
  return b.s;
}

// dK/dV on `stream`, dQ beside it; both after everything already on `stream`.
template <int D>
cudaError_t launch_bwd_pair(const BwdArgs& a, cudaStream_t stream) {
  cudaStream_t side = CPRING_BWD_OVERLAP ? bwd_side_stream() : nullptr;
  if (!side) {
    cudaError_t e = launch_bwd_t<D, true>(a, stream);
    return e == cudaSuccess ? launch_bwd_t<D, false>(a, stream) : e;
  }
  cudaEvent_t ready = nullptr, dq_done = nullptr;
  if (cudaEventCreateWithFlags(&ready, cudaEventDisableTiming) != cudaSuccess) return cudaErrorUnknown;
  if (cudaEventCreateWithFlags(&dq_done, cudaEventDisableTiming) != cudaSuccess) {
    cudaEventDestroy(ready);
    return cudaErrorUnknown;
  }
  cudaError_t e = cudaEventRecord(ready, stream);
  if (e == cudaSuccess) e = launch_bwd_t<D, true>(a, stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(side, ready, 0);
  if (e == cudaSuccess) e = launch_bwd_t<D, false>(a, side);
  if (e == cudaSuccess) e = cudaEventRecord(dq_done, side);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, dq_done, 0);
  // (destroying a recorded event releases it once the work it marks is done)
  cudaEventDestroy(ready);
  cudaEventDestroy(dq_done);
  return e;
}

}  // namespace

cudaError_t launch_attn_bwd(const BwdArgs& a, cudaStream_t stream) {
  {
    const long long rows = static_cast<long long>(a.B) * a.S * a.H;
    const long long want = (rows * 32 + 255) / 256;
    const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(want, 8LL * sm_count())));
    bwd_delta_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat162*>(a.out),
                                               static_cast<const __nv_bfloat162*>(a.dout),
                                               a.delta, a.B, a.S, a.H, a.d);
    count_launch(2);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.d == 128) return launch_bwd_pair<128>(a, stream);
  if (a.d == 64) return launch_bwd_pair<64>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace cpring
