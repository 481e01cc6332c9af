// The all-to-all form of context parallelism on one GPU.
//
// "上下文並行（Context Parallelism, CP）" (compassingai.com), section 方案二:
// All-to-All (DeepSpeed Ulysses): step 1, an all-to-all turns every GPU's
// Q/K/V from "split by sequence" into "split by attention head"; step 2, each
// GPU computes full-sequence attention for its heads; step 3, an all-to-all
// turns the result back into "split by sequence".  The communication-volume
// table of the same page counts two all-to-alls against the ring's single
// pass of K/V.
//
// With N virtual ranks on one GPU both all-to-alls are layout permutations:
// rank g's head group is the contiguous run of H/N heads g*H/N .. (g+1)*H/N-1
// of every token, so [B, S, H, d] becomes N tensors [B, S, H/N, d] (one per
// rank, stored back to back) and back.  The permutation kernel moves 16-byte
// vectors with no per-element division; it is bound by HBM bandwidth.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <optional>

#include "internal.h"

namespace cpring {
namespace {

constexpr int kPermThreads = 256;
constexpr int kPermUnroll = 4;            // 16-byte vectors in flight per thread
constexpr int kPermBlockVecs = 4096;      // about 64 KB moved per block

// Chunk (row, g) of cv 16-byte vectors: in[row][g][c] <-> out[g][row][c].
// to_heads: src = [rows][N][cv] (sequence layout), dst = [N][rows][cv] (head
// groups); otherwise the inverse.  Block (x, y) moves rows
// [x * rows_per_block, ...) of head group g = y.  Each thread splits its first
// vector index into (row, c) once and then steps by the block size with a
// carry, so the loop does no division.
__global__ void __launch_bounds__(kPermThreads)
    a2a_permute_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, long long rows,
                       int n_groups, int cv, int rows_per_block, bool to_heads) {
  const int g = blockIdx.y;
  const long long row0 = static_cast<long long>(blockIdx.x) * rows_per_block;
  const int nr = static_cast<int>(min(static_cast<long long>(rows_per_block), rows - row0));
  const int dr = kPermThreads / cv, dc = kPermThreads % cv;
  int r = threadIdx.x / cv, c = threadIdx.x % cv;
  const long long src_row_stride = to_heads ? static_cast<long long>(n_groups) * cv : cv;
  const long long dst_row_stride = to_heads ? cv : static_cast<long long>(n_groups) * cv;
  const long long src_base = to_heads ? (row0 * n_groups + g) * cv : (g * rows + row0) * cv;
  const long long dst_base = to_heads ? (g * rows + row0) * cv : (row0 * n_groups + g) * cv;
  while (r < nr) {
    uint4 val[kPermUnroll];
    long long di[kPermUnroll];
    int n = 0;
#pragma unroll
    for (int u = 0; u < kPermUnroll; ++u) {
      if (r < nr) {
        val[u] = src[src_base + r * src_row_stride + c];
        di[u] = dst_base + r * dst_row_stride + c;
        n = u + 1;
        c += dc;
        r += dr;
        if (c >= cv) {
          c -= cv;
          ++r;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kPermUnroll; ++u)
      if (u < n) dst[di[u]] = val[u];
  }
}

cudaError_t permute(const void* src, void* dst, long long rows, int n_groups, int chunk_bytes,
                    bool to_heads, cudaStream_t stream) {
  const int cv = chunk_bytes / 16;
  const int rows_per_block = std::max(1, kPermBlockVecs / cv);
  const long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  if (blocks > 0x7fffffffLL || n_groups > 65535) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(n_groups));
  a2a_permute_kernel<<<grid, kPermThreads, 0, stream>>>(static_cast<const uint4*>(src),
                                                        static_cast<uint4*>(dst), rows, n_groups,
                                                        cv, rows_per_block, to_heads);
  count_launch(2);
  return cudaGetLastError();
}

}  // namespace
}  // namespace cpring

extern "C" int64_t cp_ulysses_workspace_bytes(int B, int S, int H, int d, int n_shards) {
  if (B < 1 || S < 1 || H < 1 || d < 1 || n_shards < 1 || H % n_shards != 0) return -1;
  const int64_t t = static_cast<int64_t>(B) * S * H * d * 2;  // one bf16 tensor
  const int64_t lse = static_cast<int64_t>(B) * H * S * 4;
  return 4 * ((t + 255) / 256 * 256) + (lse + 255) / 256 * 256;
}

extern "C" cp_status cp_ulysses_attn_fwd(const void* q, const void* k, const void* v, void* out,
                                         float* lse, int B, int S, int H, int d, int n_shards,
                                         int causal, const int32_t* doc_offsets, void* workspace,
                                         int64_t workspace_bytes, cudaStream_t stream,
                                         int64_t* a2a_bytes) {
  cpring::TraceRange trace_("cp_ulysses_attn_fwd");
  using namespace cpring;
  if (!q || !k || !v || !out || !lse || !workspace) return CP_ERR_NULL;
  if (B < 1 || S < 1 || H < 1 || n_shards < 1 || n_shards > S || S % n_shards != 0)
    return CP_ERR_SHAPE;
  if (H % n_shards != 0) return CP_ERR_SHAPE;  // heads are dealt out evenly
  if (causal != 0 && causal != 1) return CP_ERR_SHAPE;
  if (d != 64 && d != 128) return CP_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * S * H * d > (1LL << 40)) return CP_ERR_SHAPE;
  auto aligned = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; };
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(workspace, 256) || !aligned(doc_offsets, 4))
    return CP_ERR_ALIGN;
  const int64_t need = cp_ulysses_workspace_bytes(B, S, H, d, n_shards);
  if (workspace_bytes < need) return CP_ERR_BUFFER;
  if (device_cc() != 103) return CP_ERR_DEVICE;

  const int N = n_shards;
  const int Hg = H / N;
  const int64_t t_bytes = (static_cast<int64_t>(B) * S * H * d * 2 + 255) / 256 * 256;
  char* ws = static_cast<char*>(workspace);
  char* qh = ws;
  char* kh = ws + t_bytes;
  char* vh = ws + 2 * t_bytes;
  char* oh = ws + 3 * t_bytes;
  float* lh = reinterpret_cast<float*>(ws + 4 * t_bytes);
  const long long rows = static_cast<long long>(B) * S;
  const int chunk = Hg * d * 2;  // bytes of one head group of one token

  int32_t* info = nullptr;
  cudaError_t e = cudaSuccess;
  // with documents: the doc-scan word and the attention launch's slot order,
  // in the library's cached scratch for the rest of this call
  std::optional<ScratchLease> lease;
  if (doc_offsets) {
    lease.emplace(doc_scratch_bytes(S, 1, -1, true), stream);
    if (!lease->ok()) return CP_ERR_CUDA;
  }
  auto chk = [&](cudaError_t x) {
    if (e == cudaSuccess && x != cudaSuccess) e = x;
  };
  // step 1: sequence-split -> head-split (all-to-all of Q, K, V)
  chk(permute(q, qh, rows, N, chunk, true, stream));
  chk(permute(k, kh, rows, N, chunk, true, stream));
  chk(permute(v, vh, rows, N, chunk, true, stream));
  if (doc_offsets) {
    info = static_cast<int32_t*>(lease->get());
    chk(launch_doc_scan(doc_offsets, S, info, stream));
  }
  // step 2: rank g attends over the whole sequence for its H/N heads.  The
  // N head-group tensors [B, S, H/N, d] lie back to back, which is one
  // problem of batch N * B with H/N heads: a single launch covers every rank
  // (lse comes out as [N, B, H/N, S]).
  if (e == cudaSuccess) {
    AttnArgs a{};
    a.q = qh;
    a.k = kh;
    a.v = vh;
    a.B = N * B; a.S = S; a.H = Hg; a.d = d; a.n_shards = 1;
    a.q_shard = -1; a.k_shard = -1;
    a.causal = causal;
    a.doc_offsets = doc_offsets;
    a.doc_info = info;
    a.slot_perm = info ? info + 4 : nullptr;
    a.out = oh;
    a.lse = lh;
    chk(launch_attn_bf16(a, stream));
  }
  // step 3: head-split -> sequence-split (all-to-all of the output)
  chk(permute(oh, out, rows, N, chunk, false, stream));
  // lse: rank g's [B, H/N, S] block lands in heads g*H/N .. of [B, H, S]
  for (int g = 0; g < N && e == cudaSuccess; ++g)
    chk(cudaMemcpy2DAsync(lse + static_cast<int64_t>(g) * Hg * S, static_cast<size_t>(H) * S * 4,
                          lh + static_cast<int64_t>(g) * B * Hg * S,
                          static_cast<size_t>(Hg) * S * 4, static_cast<size_t>(Hg) * S * 4, B,
                          cudaMemcpyDeviceToDevice, stream));
  if (a2a_bytes) {
    // every rank keeps 1/N of its shard and exchanges the rest, both ways:
    // Q, K, V before the attention and O after it, per rank sent + received
    const int64_t shard = static_cast<int64_t>(B) * (S / N) * H * d * 2;
    *a2a_bytes = 4 * 2 * shard * (N - 1) / N * N;  // summed over the N ranks
  }
  return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}
