// Standalone online-softmax merge and final normalisation, the doc_offsets
// scan, and the library's per-device error word.
//
// Merge ("上下文並行（Context Parallelism, CP）", compassingai.com, section
// 線上 Softmax, the 線上合併 lines of the algorithm):
//   m_new = max(m, m'); O = O e^{m - m_new} + O' e^{m' - m_new};
//   l = l e^{m - m_new} + l' e^{m' - m_new}; m = m_new.
// Finalisation (last line of the same algorithm): O / l, plus the
// log-sum-exp m + log l.
//
// Both are elementwise over [B, rows, H, d] fp32 state and bound by HBM
// bandwidth.  A warp takes 32 consecutive rows of one (b, h): the per-row
// scalars (m, l, lse) are read and written coalesced along [B, H, rows], and
// the rows' d-vectors stream with 16-byte accesses, several rows in flight
// per lane.  The grid is a multiple of the SM count and strides over the
// work.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <atomic>
#include <cmath>
#include <mutex>
#include <vector>

#include "internal.h"

namespace cpring {

// Sticky error word: one per device that loads this library.
__device__ int g_cp_error_word;

namespace {

constexpr int kMergeThreads = 256;

__device__ __forceinline__ void merge_factors(float m, float mp, float& a, float& c, float& mn) {
  mn = fmaxf(m, mp);
  if (mn == -INFINITY) {  // both empty
    a = 0.f;
    c = 0.f;
    return;
  }
  a = (m == -INFINITY) ? 0.f : expf(m - mn);
  c = (mp == -INFINITY) ? 0.f : expf(mp - mn);
}

// Work unit of both kernels: 32 consecutive rows of one (b, h).  Lane i
// handles the scalars (m, l, lse) of row r0 + i, so those accesses are
// coalesced along the [B, H, rows] layout; then the warp streams the rows'
// d-vectors of O ([B, rows, H, d]: one row is d contiguous floats), with the
// row's factors broadcast by shuffles and kRowsInFlight rows loaded before any
// is written, so several loads per lane are in flight.
constexpr int kRowsInFlight = 4;

__global__ void __launch_bounds__(kMergeThreads)
    lse_merge_kernel(float* __restrict__ o_acc, float* __restrict__ m_acc,
                     float* __restrict__ l_acc, const float* __restrict__ o_part,
                     const float* __restrict__ m_part, const float* __restrict__ l_part, int B,
                     int rows, int H, int d, bool vec4) {
  const int lane = threadIdx.x & 31;
  const int chunks = (rows + 31) / 32;
  const long long n_units = static_cast<long long>(B) * H * chunks;
  const long long wstride = static_cast<long long>(gridDim.x) * (kMergeThreads / 32);
  for (long long u = static_cast<long long>(blockIdx.x) * (kMergeThreads / 32) + (threadIdx.x >> 5);
       u < n_units; u += wstride) {
    const int chunk = static_cast<int>(u % chunks);
    const long long bh = u / chunks;
    const int h = static_cast<int>(bh % H);
    const int b = static_cast<int>(bh / H);
    const int r0 = chunk * 32;
    const int n_rows = min(32, rows - r0);
    // this lane's row: merge factors and the new (m, l)
    float a = 0.f, cf = 0.f;
    if (lane < n_rows) {
      const size_t mi = static_cast<size_t>(bh) * rows + r0 + lane;
      const float m = m_acc[mi], mp = m_part[mi];
      float mn;
      merge_factors(m, mp, a, cf, mn);
      l_acc[mi] = l_acc[mi] * a + l_part[mi] * cf;
      m_acc[mi] = mn;
    }
    const size_t row_stride = static_cast<size_t>(H) * d;  // floats between consecutive rows
    float* o = o_acc + (static_cast<size_t>(b) * rows + r0) * row_stride + static_cast<size_t>(h) * d;
    const float* op = o_part + (static_cast<size_t>(b) * rows + r0) * row_stride +
                      static_cast<size_t>(h) * d;
    if (vec4) {
      const int nv = d / 4;
      for (int j0 = 0; j0 < n_rows; j0 += kRowsInFlight) {
        float4 u4[kRowsInFlight], q4[kRowsInFlight];
#pragma unroll
        for (int j = 0; j < kRowsInFlight; ++j) {
          if (j0 + j < n_rows && lane < nv) {
            u4[j] = reinterpret_cast<const float4*>(o + (j0 + j) * row_stride)[lane];
            q4[j] = reinterpret_cast<const float4*>(op + (j0 + j) * row_stride)[lane];
          }
        }
#pragma unroll
        for (int j = 0; j < kRowsInFlight; ++j) {
          const float aj = __shfl_sync(0xffffffffu, a, (j0 + j) & 31);
          const float cj = __shfl_sync(0xffffffffu, cf, (j0 + j) & 31);
          if (j0 + j < n_rows && lane < nv) {
            float4 v = u4[j];
            v.x = v.x * aj + q4[j].x * cj;
            v.y = v.y * aj + q4[j].y * cj;
            v.z = v.z * aj + q4[j].z * cj;
            v.w = v.w * aj + q4[j].w * cj;
            reinterpret_cast<float4*>(o + (j0 + j) * row_stride)[lane] = v;
          }
        }
      }
    } else {
      for (int j = 0; j < n_rows; ++j) {
        const float aj = __shfl_sync(0xffffffffu, a, j);
        const float cj = __shfl_sync(0xffffffffu, cf, j);
        for (int x = lane; x < d; x += 32)
          o[j * row_stride + x] = o[j * row_stride + x] * aj + op[j * row_stride + x] * cj;
      }
    }
  }
}

template <bool kBf16>
__global__ void __launch_bounds__(kMergeThreads)
    lse_finalize_kernel(const float* __restrict__ o_acc, const float* __restrict__ m_acc,
                        const float* __restrict__ l_acc, void* __restrict__ out,
                        float* __restrict__ lse, int B, int rows, int H, int d, bool vec4,
                        long long out_bstride, long long lse_bstride, long long lse_hstride) {
  const int lane = threadIdx.x & 31;
  const int chunks = (rows + 31) / 32;
  const long long n_units = static_cast<long long>(B) * H * chunks;
  const long long wstride = static_cast<long long>(gridDim.x) * (kMergeThreads / 32);
  for (long long u = static_cast<long long>(blockIdx.x) * (kMergeThreads / 32) + (threadIdx.x >> 5);
       u < n_units; u += wstride) {
    const int chunk = static_cast<int>(u % chunks);
    const long long bh = u / chunks;
    const int h = static_cast<int>(bh % H);
    const int b = static_cast<int>(bh / H);
    const int r0 = chunk * 32;
    const int n_rows = min(32, rows - r0);
    float inv = 0.f;
    if (lane < n_rows) {
      const size_t mi = static_cast<size_t>(bh) * rows + r0 + lane;
      const float l = l_acc[mi];
      inv = (l > 0.f) ? 1.f / l : 0.f;
      lse[static_cast<size_t>(b) * lse_bstride + static_cast<size_t>(h) * lse_hstride + r0 + lane] =
          (l > 0.f) ? m_acc[mi] + logf(l) : -INFINITY;
    }
    const size_t row_stride = static_cast<size_t>(H) * d;
    const float* o = o_acc + (static_cast<size_t>(b) * rows + r0) * row_stride +
                     static_cast<size_t>(h) * d;
    const size_t orow0 = static_cast<size_t>(b) * out_bstride +
                         (static_cast<size_t>(r0) * H + h) * d;
    if (vec4) {
      const int nv = d / 4;
      for (int j0 = 0; j0 < n_rows; j0 += kRowsInFlight) {
        float4 u4[kRowsInFlight];
#pragma unroll
        for (int j = 0; j < kRowsInFlight; ++j)
          if (j0 + j < n_rows && lane < nv)
            u4[j] = reinterpret_cast<const float4*>(o + (j0 + j) * row_stride)[lane];
#pragma unroll
        for (int j = 0; j < kRowsInFlight; ++j) {
          const float ij = __shfl_sync(0xffffffffu, inv, (j0 + j) & 31);
          if (j0 + j < n_rows && lane < nv) {
            const size_t orow = orow0 + (j0 + j) * row_stride;
            if (kBf16) {
              __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(out) + orow;
              __nv_bfloat162 lo = __floats2bfloat162_rn(u4[j].x * ij, u4[j].y * ij);
              __nv_bfloat162 hi = __floats2bfloat162_rn(u4[j].z * ij, u4[j].w * ij);
              uint2 pk;
              pk.x = *reinterpret_cast<uint32_t*>(&lo);
              pk.y = *reinterpret_cast<uint32_t*>(&hi);
              reinterpret_cast<uint2*>(dst)[lane] = pk;
            } else {
              float* dst = static_cast<float*>(out) + orow;
              reinterpret_cast<float4*>(dst)[lane] =
                  make_float4(u4[j].x * ij, u4[j].y * ij, u4[j].z * ij, u4[j].w * ij);
            }
          }
        }
      }
    } else {
      for (int j = 0; j < n_rows; ++j) {
        const float ij = __shfl_sync(0xffffffffu, inv, j);
        const size_t orow = orow0 + j * row_stride;
        for (int x = lane; x < d; x += 32) {
          const float val = o[j * row_stride + x] * ij;
          if (kBf16)
            static_cast<__nv_bfloat16*>(out)[orow + x] = __float2bfloat16_rn(val);
          else
            static_cast<float*>(out)[orow + x] = val;
        }
      }
    }
  }
}

// Scan a device doc_offsets array that ends at the first entry equal to S.
// Writes the number of documents to info[0], or -1 (and raises the error
// word) when the array is not 0 = o_0 < o_1 < ... < o_n = S.  The scan reads
// one entry at a time and never past the terminator or past S + 1 entries.
__global__ void doc_scan_kernel(const int32_t* __restrict__ offs, int S, int32_t* info,
                                int* err) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  int32_t prev = offs[0];
  bool ok = (prev == 0) && (S > 0);
  int n = 0;
  if (ok) {
    for (int idx = 1; idx <= S; ++idx) {
      const int32_t x = offs[idx];
      if (x <= prev || x > S) {
        ok = false;
        break;
      }
      prev = x;
      if (x == S) {
        n = idx;
        break;
      }
    }
    if (n == 0) ok = false;
  }
  info[0] = ok ? n : -1;
  if (!ok) atomicOr(err, kErrDocOffsets);
}

int grid_for(long long warps) {
  const long long blocks = (warps + (kMergeThreads / 32) - 1) / (kMergeThreads / 32);
  const long long cap = 8LL * sm_count();
  return static_cast<int>(std::max<long long>(1, std::min(blocks, cap)));
}

std::atomic<long long> g_launches[4];

}  // namespace

void count_launch(int which) { g_launches[which].fetch_add(1, std::memory_order_relaxed); }

int* device_error_word() {
  // One address per device; cudaGetSymbolAddress is called with the device
  // current and the result cached for that device.
  static std::mutex mu;
  static int* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_cp_error_word) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<int*>(p);
  }
  return addr[dev];
}

cudaError_t ensure_smem_limit(const void* kern, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  struct Done {
    const void* kern;
    int dev;
    cudaError_t err;
  };
  static std::mutex mu;
  static std::vector<Done> done;
  std::lock_guard<std::mutex> lock(mu);
  for (const Done& d : done)
    if (d.kern == kern && d.dev == dev) return d.err;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  done.push_back(Done{kern, dev, e});
  return e;
}

// The two device attributes below are cached per device in atomics: host
// threads calling at once may both query the device, and store the same
// value.
int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    v = n > 0 ? n : 1;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

int device_cc() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int ma = 0, mi = 0;
    cudaDeviceGetAttribute(&ma, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev);
    v = ma * 10 + mi;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

cudaError_t launch_doc_scan(const int32_t* doc_offsets, int S, int32_t* doc_info,
                            cudaStream_t stream) {
  int* err = device_error_word();
  if (!err) return cudaErrorInvalidValue;
  doc_scan_kernel<<<1, 32, 0, stream>>>(doc_offsets, S, doc_info, err);
  count_launch(3);
  return cudaGetLastError();
}

cudaError_t launch_merge(float* o_acc, float* m_acc, float* l_acc, const float* o_part,
                         const float* m_part, const float* l_part, int B, int rows, int H, int d,
                         cudaStream_t stream) {
  const long long n = static_cast<long long>(B) * H * ((rows + 31) / 32);  // warp units
  const bool vec4 = (d % 4 == 0) && ((reinterpret_cast<uintptr_t>(o_acc) |
                                       reinterpret_cast<uintptr_t>(o_part)) % 16 == 0);
  lse_merge_kernel<<<grid_for(n), kMergeThreads, 0, stream>>>(o_acc, m_acc, l_acc, o_part, m_part,
                                                              l_part, B, rows, H, d, vec4);
  count_launch(2);
  return cudaGetLastError();
}

cudaError_t launch_finalize_strided(const float* o_acc, const float* m_acc, const float* l_acc,
                                    void* out, float* lse, int B, int rows, int H, int d,
                                    int out_is_bf16, long long out_bstride, long long lse_bstride,
                                    long long lse_hstride, cudaStream_t stream) {
  const long long n = static_cast<long long>(B) * H * ((rows + 31) / 32);  // warp units
  const size_t esz = out_is_bf16 ? 2 : 4;
  const bool vec4 = (d % 4 == 0) &&
                    ((reinterpret_cast<uintptr_t>(o_acc) | reinterpret_cast<uintptr_t>(out)) % 16 == 0) &&
                    ((static_cast<size_t>(out_bstride) * esz) % 16 == 0) &&
                    ((static_cast<size_t>(d) * esz) % (out_is_bf16 ? 8 : 16) == 0);
  if (out_is_bf16)
    lse_finalize_kernel<true><<<grid_for(n), kMergeThreads, 0, stream>>>(
        o_acc, m_acc, l_acc, out, lse, B, rows, H, d, vec4 && d % 8 == 0, out_bstride, lse_bstride,
        lse_hstride);
  else
    lse_finalize_kernel<false><<<grid_for(n), kMergeThreads, 0, stream>>>(
        o_acc, m_acc, l_acc, out, lse, B, rows, H, d, vec4, out_bstride, lse_bstride, lse_hstride);
  count_launch(2);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const float* o_acc, const float* m_acc, const float* l_acc, void* out,
                            float* lse, int B, int rows, int H, int d, int out_is_bf16,
                            cudaStream_t stream) {
  return launch_finalize_strided(o_acc, m_acc, l_acc, out, lse, B, rows, H, d, out_is_bf16,
                                 static_cast<long long>(rows) * H * d,
                                 static_cast<long long>(H) * rows, rows, stream);
}

}  // namespace cpring

extern "C" void cp_launch_counts(int64_t* counts4) {
  if (!counts4) return;
  for (int i = 0; i < 4; ++i)
    counts4[i] = cpring::g_launches[i].load(std::memory_order_relaxed);
}
