// Ring-attention forward and single ring step in true fp32 on CUDA cores.
//
// Same method as the tensor-core path ("上下文並行（Context Parallelism, CP）",
// compassingai.com, section 線上 Softmax): each virtual rank i visits the K/V
// shards j = 0..N-1 in ascending order, skipping shards with no visible key,
// and folds 32-key blocks into a running (O, m, l) with the online-softmax
// merge.  Scores use fp32 FFMA (no TF32), exponentials use expf, so the
// result stays within 1e-4 of an fp64 evaluation.
//
// One warp owns one query row of one (b, h): every lane scores one key of the
// current 32-key block, the block max and sum are warp reductions, and each
// lane accumulates d/32 output columns.
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"

namespace cpring {
namespace {

constexpr int kWarpsPerBlock = 4;
constexpr int kMaxD = 128;

struct F32Params {
  const float* q;
  const float* k;
  const float* v;
  int B, S, H, d, L, n_shards;
  int q_shard, k_shard;
  int causal;
  const int32_t* doc_offsets;
  const int32_t* doc_info;
  float scale;  // 1/sqrt(d)
  long long n_rows;  // B * H * rows processed
  float* out;
  float* lse;
  float* o_part;
  float* m_part;
  float* l_part;
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <bool kPartial>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    ring_attn_f32_kernel(const F32Params p) {
  __shared__ float qs[kWarpsPerBlock][kMaxD];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int n_docs = 1;
  if (p.doc_offsets != nullptr) {
    n_docs = __ldg(p.doc_info);
    if (n_docs <= 0) return;
  }
  const int rows_per_bh = (p.q_shard < 0) ? p.S : p.L;
  for (long long gw = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + warp; gw < p.n_rows;
       gw += static_cast<long long>(gridDim.x) * kWarpsPerBlock) {
    const int rr = static_cast<int>(gw % rows_per_bh);
    const long long bh = gw / rows_per_bh;
    const int h = static_cast<int>(bh % p.H);
    const int b = static_cast<int>(bh / p.H);
    const int r = (p.q_shard < 0) ? rr : p.q_shard * p.L + rr;  // global query row
    // visible keys of row r: [doc_start, causal ? r : doc_end - 1]
    int ds = 0, de = p.S;
    if (p.doc_offsets != nullptr) {
      int lo = 0, hi = n_docs;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(p.doc_offsets + mid) <= r) lo = mid; else hi = mid;
      }
      ds = __ldg(p.doc_offsets + lo);
      de = __ldg(p.doc_offsets + lo + 1);
    }
    const int vis_lo = ds;
    const int vis_hi = p.causal ? r : de - 1;

    const float* qrow = p.q + ((static_cast<size_t>(b) * p.S + r) * p.H + h) * p.d;
    __syncwarp();
    for (int x = lane; x < p.d; x += 32) qs[warp][x] = qrow[x];
    __syncwarp();

    float m = -INFINITY, l = 0.f;
    float acc[kMaxD / 32];
#pragma unroll
    for (int x = 0; x < kMaxD / 32; ++x) acc[x] = 0.f;

    const int j_first = (p.k_shard < 0) ? 0 : p.k_shard;
    const int j_last = (p.k_shard < 0) ? p.n_shards - 1 : p.k_shard;
    for (int j = j_first; j <= j_last; ++j) {
      const int a = max(vis_lo, j * p.L);
      const int e = min(vis_hi, (j + 1) * p.L - 1);
      if (a > e) continue;  // shard pair with no visible key: skipped
      for (int k0 = a; k0 <= e; k0 += 32) {
        const int key = k0 + lane;
        const bool valid = key <= e;
        float s = -INFINITY;
        if (valid) {
          const float* krow = p.k + ((static_cast<size_t>(b) * p.S + key) * p.H + h) * p.d;
          float dot = 0.f;
          for (int x = 0; x < p.d; ++x) dot = fmaf(qs[warp][x], __ldg(krow + x), dot);
          s = dot * p.scale;
        }
        const float m_new = fmaxf(m, warp_max(s));
        const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
        const float pr = valid ? expf(s - m_new) : 0.f;
        l = l * alpha + warp_sum(pr);
#pragma unroll
        for (int x = 0; x < kMaxD / 32; ++x) acc[x] *= alpha;
        const int nk = min(32, e - k0 + 1);
        for (int t = 0; t < nk; ++t) {
          const float pt = __shfl_sync(0xffffffffu, pr, t);
          const float* vrow = p.v + ((static_cast<size_t>(b) * p.S + k0 + t) * p.H + h) * p.d;
#pragma unroll
          for (int x = 0; x < kMaxD / 32; ++x) {
            const int col = x * 32 + lane;
            if (col < p.d) acc[x] = fmaf(pt, __ldg(vrow + col), acc[x]);
          }
        }
        m = m_new;
      }
    }
    if (!kPartial) {
      float* orow = p.out + ((static_cast<size_t>(b) * p.S + r) * p.H + h) * p.d;
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
      for (int x = 0; x < kMaxD / 32; ++x) {
        const int col = x * 32 + lane;
        if (col < p.d) orow[col] = acc[x] * inv;
      }
      if (lane == 0)
        p.lse[(static_cast<size_t>(b) * p.H + h) * p.S + r] = (l > 0.f) ? m + logf(l) : -INFINITY;
    } else {
      float* orow = p.o_part + ((static_cast<size_t>(b) * p.L + rr) * p.H + h) * p.d;
#pragma unroll
      for (int x = 0; x < kMaxD / 32; ++x) {
        const int col = x * 32 + lane;
        if (col < p.d) orow[col] = acc[x];
      }
      if (lane == 0) {
        const size_t mi = (static_cast<size_t>(b) * p.H + h) * p.L + rr;
        p.m_part[mi] = m;
        p.l_part[mi] = l;
      }
    }
  }
}

}  // namespace

cudaError_t launch_attn_f32(const AttnArgs& a, cudaStream_t stream) {
  F32Params p{};
  p.q = static_cast<const float*>(a.q);
  p.k = static_cast<const float*>(a.k);
  p.v = static_cast<const float*>(a.v);
  p.B = a.B;
  p.S = a.S;
  p.H = a.H;
  p.d = a.d;
  p.n_shards = a.n_shards;
  p.L = a.S / a.n_shards;
  p.q_shard = a.q_shard;
  p.k_shard = a.k_shard;
  p.causal = a.causal;
  p.doc_offsets = a.doc_offsets;
  p.doc_info = a.doc_info;
  p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(a.d)));
  const long long rows = (a.q_shard < 0) ? a.S : a.S / a.n_shards;
  p.n_rows = static_cast<long long>(a.B) * a.H * rows;
  p.out = static_cast<float*>(a.out);
  p.lse = a.lse;
  p.o_part = a.o_part;
  p.m_part = a.m_part;
  p.l_part = a.l_part;
  const long long want = (p.n_rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int grid = static_cast<int>(std::min<long long>(want, 8LL * sm_count()));
  if (grid <= 0) return cudaSuccess;
  if (a.k_shard >= 0)
    ring_attn_f32_kernel<true><<<grid, kWarpsPerBlock * 32, 0, stream>>>(p);
  else
    ring_attn_f32_kernel<false><<<grid, kWarpsPerBlock * 32, 0, stream>>>(p);
  count_launch(1);
  return cudaGetLastError();
}

}  // namespace cpring
