// Device helpers shared by the tcgen05 attention kernels (forward and
// backward): the shard-aligned tiling of the sequence, the document of a
// token, the snake deal of work items to persistent CTAs, and the bounded
// mbarrier waits.  Templates over the kernel's parameter struct, which must
// provide S, L (shard length), tiles_per_shard, doc_offsets, timeout_ns and
// err.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

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

}  // namespace
}  // namespace cpring
