// FP8 (E4M3) storage of Q, K and V for the FP8 form of the forward.
//
// "上下文並行（Context Parallelism, CP）" (compassingai.com), section 通訊量分析:
// the bytes a CP scheme moves depend on whether K/V travel in FP8.  The format
// is OCP E4M3 (largest finite 448) with one fp32 scale per (b, h):
//   amax    = max |x| over (S, d) of head (b, h)
//   inv     = 448 / amax                (fp32, rounded to nearest)
//   x8      = E4M3(x * inv)             (fp32 product rounded to nearest, then
//                                        to the nearest E4M3, ties to even,
//                                        saturated at +-448)
//   descale = amax / 448                (fp32), so x ~ x8 * descale
// and an all-zero head gets inv = descale = 1.  Every step is an exactly
// rounded fp32 operation, so the codes are reproducible bit for bit.
//
// Kernels (all HBM-bound; x is bf16 [B, S, H, d], d in {64, 128}):
//   fp8_amax_kernel     one pass over x, per-(b, h) max |x| with an unsigned
//                       atomic max on the fp32 bit pattern (non-negative
//                       floats order like their bits), one atomic per head
//                       per column sweep of a block
//   fp8_quant_kernel    x8 in the same [B, S, H, d] layout (Q and K)
//   fp8_quant_t_kernel  x8 as [B, H, d, S] (V^T, keys contiguous), through a
//                       shared-memory tile of 128 tokens
//   fp8_descale_kernel  amax -> descale in place
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace cpring {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerBlock = 64;

__device__ __forceinline__ float abs_max8(const uint4& v) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
  }
  return m;
}

__device__ __forceinline__ float inv_scale(float amax) {
  return amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
}

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight bf16 values times inv, as eight E4M3 bytes (element 0 lowest).
__device__ __forceinline__ uint2 quant8(const uint4& v, float inv) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    w[i] = e4m3x2(__fmul_rn(f.x, inv), __fmul_rn(f.y, inv));
  }
  return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// Block (x, y) covers tokens [x * kRowsPerBlock, ...) of batch row b = y.  A
// thread owns columns vi = c0 + threadIdx.x (16-byte vectors of one token
// row, H * d / 8 per row); the g = d / 8 lanes of a column group share one
// head, so a shuffle reduction leaves one atomic per head and sweep.
__global__ void __launch_bounds__(kThreads)
    fp8_amax_kernel(const uint4* __restrict__ x, unsigned* __restrict__ amax, int S, int H,
                    int d) {
  const int b = blockIdx.y;
  const int row0 = blockIdx.x * kRowsPerBlock;
  const int nr = min(kRowsPerBlock, S - row0);
  const int vpr = H * d / 8;
  const int g = d / 8;
  for (int c0 = 0; c0 < vpr; c0 += kThreads) {
    const int vi = c0 + threadIdx.x;
    float m = 0.f;
    if (vi < vpr) {
      const uint4* col = x + (static_cast<long long>(b) * S + row0) * vpr + vi;
#pragma unroll 4
      for (int r = 0; r < nr; ++r) m = fmaxf(m, abs_max8(col[static_cast<long long>(r) * vpr]));
    }
    for (int off = g / 2; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (vi < vpr && vi % g == 0) atomicMax(amax + b * H + vi / g, __float_as_uint(m));
  }
}

__global__ void __launch_bounds__(kThreads)
    fp8_quant_kernel(const uint4* __restrict__ x, uint2* __restrict__ y,
                     const float* __restrict__ amax, int S, int H, int d) {
  const int b = blockIdx.y;
  const int row0 = blockIdx.x * kRowsPerBlock;
  const int nr = min(kRowsPerBlock, S - row0);
  const int vpr = H * d / 8;
  const int g = d / 8;
  for (int vi = threadIdx.x; vi < vpr; vi += kThreads) {
    const float inv = inv_scale(amax[b * H + vi / g]);
    const long long base = (static_cast<long long>(b) * S + row0) * vpr + vi;
#pragma unroll 4
    for (int r = 0; r < nr; ++r) {
      const long long at = base + static_cast<long long>(r) * vpr;
      y[at] = quant8(x[at], inv);
    }
  }
}

constexpr int kTTokens = 128;  // tokens per transposed tile (one 128-byte output segment)

// Block (x, h, b) covers tokens [s0, s0 + 128) of head h, s0 = 128 x.
// Phase 1: the block reads the 128 token rows of d bf16 (coalesced 16-byte
// loads, all of a thread's loads issued before the first is used, so that
// enough bytes are in flight to cover the memory latency), quantizes them
// and stores the codes row-major in shared memory,
// 128 bytes per token row, word w of token r at word w ^ (4 (r / 16)) of its
// row.  Phase 2: thread (d4, g) gathers words d4 (four consecutive channels)
// of tokens 16 g .. 16 g + 15, transposes the 4 x 16 bytes in registers and
// writes four 16-byte segments, channel rows 4 d4 .. 4 d4 + 3 of
// y[b, h, :, s0 + 16 g ..].  With g the fastest thread index, 8 lanes write
// one full 128-byte segment of a row; the swizzle makes both phases' shared
// accesses conflict-free.  S % 16 == 0, so a 16-token segment is either
// wholly inside [0, S) or wholly past it.
template <int D>
__global__ void __launch_bounds__(kThreads)
    fp8_quant_t_kernel(const uint4* __restrict__ x, uint8_t* __restrict__ y,
                       const float* __restrict__ amax, int S, int H) {
  __shared__ __align__(16) uint32_t tile[kTTokens * 32];  // 128 rows x 128 bytes
  constexpr int g8 = D / 8;                         // 16-byte input vectors per token row
  constexpr int kVecs = kTTokens * g8 / kThreads;   // of them per thread: 8 (d = 128), 4 (64)
  static_assert(kVecs * kThreads == kTTokens * g8, "whole vectors per thread");
  const int h = blockIdx.y, b = blockIdx.z;
  const int s0 = blockIdx.x * kTTokens;
  uint4 v[kVecs];
#pragma unroll
  for (int i = 0; i < kVecs; ++i) {
    const int idx = threadIdx.x + i * kThreads;
    const int r = idx / g8, cv = idx % g8;
    v[i] = make_uint4(0u, 0u, 0u, 0u);
    if (s0 + r < S) v[i] = x[((static_cast<long long>(b) * S + s0 + r) * H + h) * g8 + cv];
  }
  const float inv = inv_scale(amax[b * H + h]);
#pragma unroll
  for (int i = 0; i < kVecs; ++i) {
    const int idx = threadIdx.x + i * kThreads;
    const int r = idx / g8, cv = idx % g8;
    const uint2 q = (s0 + r < S) ? quant8(v[i], inv) : make_uint2(0u, 0u);
    const int w = (2 * cv) ^ (4 * (r >> 4));  // words 2 cv, 2 cv + 1 stay adjacent
    *reinterpret_cast<uint2*>(tile + r * 32 + w) = q;
  }
  __syncthreads();
  constexpr int n_d4 = D / 4;
  for (int idx = threadIdx.x; idx < n_d4 * 8; idx += kThreads) {
    const int g = idx & 7, d4 = idx >> 3;
    const int s = s0 + 16 * g;
    if (s >= S) continue;
    uint32_t wv[16];  // word d4 (channels 4 d4 .. +3) of tokens 16 g + j
#pragma unroll
    for (int j = 0; j < 16; ++j) wv[j] = tile[(16 * g + j) * 32 + (d4 ^ (4 * g))];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      // channel 4 d4 + c of the 16 tokens: byte c of each word, token j at byte j
      uint32_t o[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint32_t lo = __byte_perm(wv[4 * q4 + 0], wv[4 * q4 + 1], 0x0040 | (c << 4) | c) & 0xffffu;
        const uint32_t hi = __byte_perm(wv[4 * q4 + 2], wv[4 * q4 + 3], 0x0040 | (c << 4) | c) & 0xffffu;
        o[q4] = lo | (hi << 16);
      }
      *reinterpret_cast<uint4*>(y + ((static_cast<long long>(b) * H + h) * D + 4 * d4 + c) * S + s) =
          make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

__global__ void fp8_descale_kernel(float* v, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    const float a = v[i];
    v[i] = a > 0.f ? __fdiv_rn(a, 448.f) : 1.f;
  }
}

}  // namespace
}  // namespace cpring

extern "C" cp_status cp_fp8_quantize(const void* x, void* x8, float* descale, int B, int S, int H,
                                     int d, int transpose, cudaStream_t stream) {
  cpring::TraceRange trace_("cp_fp8_quantize");
  using namespace cpring;
  if (!x || !x8 || !descale) return CP_ERR_NULL;
  if (B < 1 || S < 1 || H < 1 || B > 65535 || H > 65535) return CP_ERR_SHAPE;
  if (transpose != 0 && transpose != 1) return CP_ERR_SHAPE;
  if (d != 64 && d != 128) return CP_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * S * H * d > (1LL << 40)) return CP_ERR_SHAPE;
  if (transpose && S % 16 != 0) return CP_ERR_SHAPE;
  auto aligned = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; };
  if (!aligned(x, 16) || !aligned(x8, 16) || !aligned(descale, 4)) return CP_ERR_ALIGN;
  if (device_cc() != 103) return CP_ERR_DEVICE;

  const int n = B * H;
  cudaError_t e = cudaMemsetAsync(descale, 0, static_cast<size_t>(n) * sizeof(float), stream);
  if (e != cudaSuccess) return CP_ERR_CUDA;
  const dim3 grid_rows((S + kRowsPerBlock - 1) / kRowsPerBlock, B);
  fp8_amax_kernel<<<grid_rows, kThreads, 0, stream>>>(static_cast<const uint4*>(x),
                                                      reinterpret_cast<unsigned*>(descale), S, H, d);
  if (transpose) {
    const dim3 grid_t((S + kTTokens - 1) / kTTokens, H, B);
    if (d == 128)
      fp8_quant_t_kernel<128><<<grid_t, kThreads, 0, stream>>>(
          static_cast<const uint4*>(x), static_cast<uint8_t*>(x8), descale, S, H);
    else
      fp8_quant_t_kernel<64><<<grid_t, kThreads, 0, stream>>>(
          static_cast<const uint4*>(x), static_cast<uint8_t*>(x8), descale, S, H);
  } else {
    fp8_quant_kernel<<<grid_rows, kThreads, 0, stream>>>(static_cast<const uint4*>(x),
                                                         static_cast<uint2*>(x8), descale, S, H, d);
  }
  fp8_descale_kernel<<<(n + 255) / 256, 256, 0, stream>>>(descale, n);
  for (int i = 0; i < 3; ++i) count_launch(2);
  return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}
