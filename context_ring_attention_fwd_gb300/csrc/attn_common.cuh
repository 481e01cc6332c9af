// Device helpers shared by the tcgen05 attention kernels (forward and
// backward): the shard-aligned tiling of the sequence, the document of a
// token, the claiming of work items by persistent CTAs (and the fixed snake
// deal it replaced), and the bounded mbarrier waits.  Templates over the
// kernel's parameter struct, which must provide S, L (shard length),
// tiles_per_shard, doc_offsets, timeout_ns and err.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <atomic>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace cpring {
namespace {

constexpr int kTileRows = 128;  // rows of every Q / K / V / dO tile = TMEM lanes

// Document [start, end) containing token r.
template <class P>
__device__ __forceinline__ int2 doc_span(const P& p, int n_docs, int r) {
  if (p.doc_offsets == nullptr) return make_int2(0, p.S);
  int lo = 0, hi = n_docs;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (__ldg(p.doc_offsets + mid) <= r) lo = mid; else hi = mid;
  }
  return make_int2(__ldg(p.doc_offsets + lo), __ldg(p.doc_offsets + lo + 1));
}

// Tiles are laid from each shard's first row and never cross a shard
// boundary; tile f of the flattened order is tile f % tiles_per_shard of
// shard f / tiles_per_shard.
template <class P>
__device__ __forceinline__ int flat_tile(const P& p, int key) {
  int j = key / p.L;
  return j * p.tiles_per_shard + (key - j * p.L) / kTileRows;
}

template <class P>
__device__ __forceinline__ void tile_keys(const P& p, int f, int& ks, int& ke) {
  int j = f / p.tiles_per_shard;
  int kt = f - j * p.tiles_per_shard;
  ks = j * p.L + kt * kTileRows;
  ke = min(ks + kTileRows, (j + 1) * p.L);
}

// k-th item of CTA c in a grid of G: rows of G items, dealt in a snake.
__device__ __forceinline__ int item_of(int k, int c, int G) {
  return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// Single-thread bounded wait.  Returns false on abort or timeout.
template <class P>
__device__ __forceinline__ bool wait1(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                      const P& p, bool honour_abort = true) {
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (honour_abort && *abort_flag) return false;
    if ((it & 255u) == 0) {
      const uint64_t now = ptx::globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > p.timeout_ns) {
        *abort_flag = 1u;
        atomicOr(p.err, kErrTimeout);
        return false;
      }
    }
  }
}

// Warp-uniform bounded wait (every lane calls it; all lanes get one answer).
// It returns once every lane has itself seen the phase complete, so whichever
// lane then issues an MMA or a tcgen05 access has acquired the barrier.
// With honour_abort false it ignores the CTA's abort flag and ends only on the
// phase or its own time limit (the final drain of a CTA that is giving up).
template <class P>
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity,
                                          volatile uint32_t* abort_flag, const P& p,
                                          bool honour_abort = true) {
  uint64_t t0 = 0;
  const int lane = threadIdx.x & 31;
  for (uint32_t it = 1;; ++it) {
    const bool ok = ptx::mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if (honour_abort && __any_sync(0xffffffffu, *abort_flag != 0u)) return false;
    if ((it & 255u) == 0) {
      int tout = 0;
      if (lane == 0) {
        const uint64_t now = ptx::globaltimer();
        if (t0 == 0) {
          t0 = now;
        } else if (now - t0 > p.timeout_ns) {
          *abort_flag = 1u;
          atomicOr(p.err, kErrTimeout);
          tout = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, tout, 0)) return false;
    }
  }
}

// ---------------------------------------------------------------- work queue
// Work items of the persistent tcgen05 kernels are claimed at run time.  CTA
// c starts with item c; every later item comes from a counter the launch's
// CTAs share, in the order the kernel lays its items out (heaviest first),
// so a CTA that finishes early takes more work and the tail stays short
// whatever the items cost.  The counter is one of kWorkSlots 64-bit
// slots of a device array that launches use in turn; a slot holds
// (launch epoch << 32 | next index), and epochs only grow, so no launch
// clears it and none allocates it.  At most kWorkSlots launches can run at
// once on a device before one would reuse the slot of another still running.
constexpr int kWorkSlots = 256;
__device__ unsigned long long g_work_slots[kWorkSlots];
// Tuning switch of the backward kernels: CTAs claim items from the launch's
// counter (1) or take them in the fixed snake order of item_of (0).  (The
// forward chooses per launch.)
#ifndef CPRING_DYNAMIC
#define CPRING_DYNAMIC 1
#endif

// A CTA's first claim of a launch: raise the slot to (epoch << 32 | 0) if it
// still holds an older launch's tag (an atomic max leaves this launch's
// running count alone), then take the next index with one atomic add.  Both
// are single atomics to one address, so 152 CTAs claiming at once cost no
// retries.  The result is read only when the item starts.
__device__ __forceinline__ unsigned long long claim_first(unsigned long long* slot, uint32_t epoch) {
  atomicMax(slot, static_cast<unsigned long long>(epoch) << 32);
  return atomicAdd(slot, 1ull);
}

// A CTA's later claims: the slot carries this launch's tag already.  The
// producer issues each one item ahead, so the atomic's latency hides behind
// the current item's loads.
__device__ __forceinline__ unsigned long long claim_next(unsigned long long* slot) {
  return atomicAdd(slot, 1ull);
}

// The item index of a claim, or past every item (with the error word set)
// if the slot did not carry this launch's tag, which only another launch
// using the same slot at the same time could cause.
__device__ __forceinline__ int claimed_index(unsigned long long v, uint32_t epoch, int* err) {
  if (static_cast<uint32_t>(v >> 32) != epoch) {
    atomicOr(err, kErrTimeout);
    return INT_MAX / 2;
  }
  return static_cast<int>(v & 0xffffffffull);
}

// The CTA's ring of claimed item indices: the producer publishes each item
// it claims (its k-th item in slot k % kRing); the reading warps (by default
// the MMA warp and the eight softmax warps) read them in the same order, so
// every role walks the same items.  Full barriers take the producer's
// arrival, empty ones one arrival per reading warp.
constexpr int kRing = 4;
constexpr int kRingReaders = 9;  // the MMA warp and the eight softmax warps
constexpr int kRingBytes = 2 * kRing * 8 + kRing * 4;
static_assert(kRingBytes <= 256, "the item ring's shared-memory block");

struct ItemRing {
  uint32_t bars;      // shared address: kRing full barriers, then kRing empty barriers
  volatile int* idx;  // kRing item indices
  __device__ uint32_t full(int s) const { return bars + 8u * static_cast<uint32_t>(s); }
  __device__ uint32_t empty(int s) const { return bars + 8u * static_cast<uint32_t>(kRing + s); }
};

__device__ __forceinline__ void ring_init(const ItemRing& r, int readers = kRingReaders) {
  for (int s = 0; s < kRing; ++s) {
    ptx::mbar_init(r.full(s), 1);
    ptx::mbar_init(r.empty(s), readers);
  }
}

// Producer (one thread): publish w as the CTA's k-th item.
template <class P>
__device__ __forceinline__ bool ring_put(const ItemRing& r, uint32_t k, int w,
                                         volatile uint32_t* abort_flag, const P& p) {
  const int s = static_cast<int>(k % kRing);
  const uint32_t use = k / kRing;
  if (use > 0 && !wait1(r.empty(s), (use - 1) & 1u, abort_flag, p)) return false;
  r.idx[s] = w;
  ptx::mbar_arrive(r.full(s));
  return true;
}

// A reading warp (every lane): the CTA's k-th item, or -1 if the wait gave up.
template <class P>
__device__ __forceinline__ int ring_get(const ItemRing& r, uint32_t k,
                                        volatile uint32_t* abort_flag, const P& p) {
  const int s = static_cast<int>(k % kRing);
  if (!wait_warp(r.full(s), (k / kRing) & 1u, abort_flag, p)) return -1;
  const int w = r.idx[s];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(r.empty(s));
  return w;
}

// ---------------------------------------------------------------- host side
// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// [B, S, H, D] viewed as a 4-D tensor (D, H, S, B) of E-byte elements;
// box = one 128-byte panel x 1 x 128 rows x 1.
bool make_map(CUtensorMap* m, const void* base, int B, int S, int H, int D, int E = 2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t e = static_cast<cuuint64_t>(E);
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * e, static_cast<cuuint64_t>(H) * D * e,
                           static_cast<cuuint64_t>(S) * H * D * e};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / E), 1, static_cast<cuuint32_t>(kTileRows), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, E == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
                  const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Device address of the claim counters (g_work_slots) for the current
// device, looked up once per device with that device current.
unsigned long long* work_slots_address() {
  static std::mutex mu;
  static unsigned long long* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_work_slots) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned long long*>(ptr);
  }
  return addr[dev];
}

// Launch epochs, per device: every launch that claims items gets the next one
// and the counter slot epoch % kWorkSlots.  Epoch 0 is the counters'
// initial tag and is never handed out; when the count wraps (after 2^32 - 1
// launches) the device is synchronised and its counters cleared, because a
// claim can only raise a slot's tag.
std::atomic<uint32_t> g_epoch[64];

// The next epoch of the current device, or 0 if clearing the counters failed.
uint32_t next_epoch(unsigned long long* slots) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  uint32_t e = ++g_epoch[dev];
  if (e == 0) {
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemset(slots, 0, sizeof(unsigned long long) * kWorkSlots) != cudaSuccess)
      return 0;
    e = ++g_epoch[dev];
  }
  return e;
}

}  // namespace
}  // namespace cpring
