// C ABI of the ring-attention library: argument checks, dispatch to the
// kernels, the host-side skip schedule and traffic counts, and status
// reporting.  Every argument is checked before anything is launched.
#include <cuda_runtime_api.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <vector>

#include "internal.h"

namespace {

using cpring::AttnArgs;
using cpring::aligned;
using cpring::check_shape;

cp_status check_device() {
  if (cpring::device_cc() != 103) return CP_ERR_DEVICE;
  return CP_OK;
}

// kind: 0 fp32 CUDA-core kernel, 1 bf16 tcgen05 kernel, 2 FP8 tcgen05 kernel.
// With documents the launch reads the doc-scan word and (tensor-core paths)
// the cost-ranked slot order from the library's cached per-device scratch.
cp_status run_attn(AttnArgs a, int kind, cudaStream_t stream) {
  cp_status st = check_device();
  if (st != CP_OK) return st;
  if (!a.doc_offsets) {
    const cudaError_t e = kind == 2   ? cpring::launch_attn_fp8(a, stream)
                          : kind == 1 ? cpring::launch_attn_bf16(a, stream)
                                      : cpring::launch_attn_f32(a, stream);
    return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
  }
  cpring::ScratchLease lease(cpring::doc_scratch_bytes(a.S, a.n_shards, a.q_shard, kind != 0),
                             stream);
  if (!lease.ok()) return CP_ERR_CUDA;
  int32_t* info = static_cast<int32_t*>(lease.get());
  if (cpring::launch_doc_scan(a.doc_offsets, a.S, info, stream) != cudaSuccess) return CP_ERR_CUDA;
  a.doc_info = info;
  if (kind != 0) a.slot_perm = info + 4;
  const cudaError_t e = kind == 2   ? cpring::launch_attn_fp8(a, stream)
                        : kind == 1 ? cpring::launch_attn_bf16(a, stream)
                                    : cpring::launch_attn_f32(a, stream);
  return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

// Document [start, end) of every token from host offsets; false if malformed.
bool host_docs(const int32_t* offs, int S, std::vector<int>& start, std::vector<int>& end) {
  start.assign(S, 0);
  end.assign(S, S);
  if (!offs) return true;
  if (offs[0] != 0) return false;
  int prev = 0;
  for (int idx = 1; idx <= S; ++idx) {
    const int x = offs[idx];
    if (x <= prev || x > S) return false;
    for (int t = prev; t < x; ++t) {
      start[t] = prev;
      end[t] = x;
    }
    prev = x;
    if (x == S) return true;
  }
  return false;
}

}  // namespace

extern "C" {

cp_status cp_ring_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                           int B, int S, int H, int d, int n_shards, int causal,
                           const int32_t* doc_offsets, cudaStream_t stream) {
  cpring::TraceRange trace_("cp_ring_attn_fwd");
  if (!q || !k || !v || !out || !lse) return CP_ERR_NULL;
  cp_status st = check_shape(B, S, H, d, n_shards);
  if (st != CP_OK) return st;
  if (d != 64 && d != 128) return CP_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return CP_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(doc_offsets, 4))
    return CP_ERR_ALIGN;
  AttnArgs a{};
  a.q = q; a.k = k; a.v = v;
  a.B = B; a.S = S; a.H = H; a.d = d; a.n_shards = n_shards;
  a.q_shard = -1; a.k_shard = -1;
  a.causal = causal;
  a.doc_offsets = doc_offsets;
  a.out = out; a.lse = lse;
  return run_attn(a, true, stream);
}

cp_status cp_ring_attn_fwd_rank(const void* q, const void* k, const void* v, void* out, float* lse,
                                int B, int S, int H, int d, int n_shards, int rank, int causal,
                                const int32_t* doc_offsets, cudaStream_t stream) {
  cpring::TraceRange trace_("cp_ring_attn_fwd_rank");
  if (!q || !k || !v || !out || !lse) return CP_ERR_NULL;
  cp_status st = check_shape(B, S, H, d, n_shards);
  if (st != CP_OK) return st;
  if (rank < 0 || rank >= n_shards) return CP_ERR_SHAPE;
  if (d != 64 && d != 128) return CP_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return CP_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(doc_offsets, 4))
    return CP_ERR_ALIGN;
  AttnArgs a{};
  a.q = q; a.k = k; a.v = v;
  a.B = B; a.S = S; a.H = H; a.d = d; a.n_shards = n_shards;
  a.q_shard = rank; a.k_shard = -1;
  a.causal = causal;
  a.doc_offsets = doc_offsets;
  a.out = out; a.lse = lse;
  return run_attn(a, 1, stream);
}

cp_status cp_ring_attn_fwd_fp8(const void* q8, const void* k8, const void* v8t,
                               const float* q_descale, const float* k_descale,
                               const float* v_descale, void* out, float* lse, int B, int S, int H,
                               int d, int n_shards, int causal, const int32_t* doc_offsets,
                               cudaStream_t stream) {
  cpring::TraceRange trace_("cp_ring_attn_fwd_fp8");
  if (!q8 || !k8 || !v8t || !q_descale || !k_descale || !v_descale || !out || !lse)
    return CP_ERR_NULL;
  cp_status st = check_shape(B, S, H, d, n_shards);
  if (st != CP_OK) return st;
  if (d != 128) return CP_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return CP_ERR_SHAPE;
  if ((S / n_shards) % 16 != 0) return CP_ERR_SHAPE;
  if (!aligned(q8, 16) || !aligned(k8, 16) || !aligned(v8t, 16) || !aligned(out, 16) ||
      !aligned(q_descale, 4) || !aligned(k_descale, 4) || !aligned(v_descale, 4) ||
      !aligned(lse, 4) || !aligned(doc_offsets, 4))
    return CP_ERR_ALIGN;
  AttnArgs a{};
  a.q = q8; a.k = k8; a.v = v8t;
  a.q_descale = q_descale; a.k_descale = k_descale; a.v_descale = v_descale;
  a.B = B; a.S = S; a.H = H; a.d = d; a.n_shards = n_shards;
  a.q_shard = -1; a.k_shard = -1;
  a.causal = causal;
  a.doc_offsets = doc_offsets;
  a.out = out; a.lse = lse;
  return run_attn(a, 2, stream);
}

int64_t cp_ring_attn_bwd_workspace_bytes(int B, int S, int H, int d, int n_shards) {
  if (check_shape(B, S, H, d, n_shards) != CP_OK) return -1;
  const int64_t delta = static_cast<int64_t>(B) * H * S * 4;
  return (delta + 255) / 256 * 256 + 256;  // D, then the doc-scan word
}

cp_status cp_ring_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                           const float* lse, const void* dout, void* dq, void* dk, void* dv,
                           int B, int S, int H, int d, int n_shards, int causal,
                           const int32_t* doc_offsets, void* workspace, int64_t workspace_bytes,
                           cudaStream_t stream) {
  cpring::TraceRange trace_("cp_ring_attn_bwd");
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv || !workspace)
    return CP_ERR_NULL;
  cp_status st = check_shape(B, S, H, d, n_shards);
  if (st != CP_OK) return st;
  if (d != 64 && d != 128) return CP_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return CP_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4) || !aligned(doc_offsets, 4) || !aligned(workspace, 256))
    return CP_ERR_ALIGN;
  const int64_t need = cp_ring_attn_bwd_workspace_bytes(B, S, H, d, n_shards);
  if (workspace_bytes < need) return CP_ERR_BUFFER;
  st = check_device();
  if (st != CP_OK) return st;
  cpring::BwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.out = out; a.lse = lse; a.dout = dout;
  a.dq = dq; a.dk = dk; a.dv = dv;
  a.delta = static_cast<float*>(workspace);
  a.B = B; a.S = S; a.H = H; a.d = d; a.n_shards = n_shards;
  a.causal = causal;
  a.doc_offsets = doc_offsets;
  if (doc_offsets) {
    int32_t* info = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + need - 256);
    if (cpring::launch_doc_scan(doc_offsets, S, info, stream) != cudaSuccess) return CP_ERR_CUDA;
    a.doc_info = info;
  }
  return cpring::launch_attn_bwd(a, stream) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

cp_status cp_ring_attn_fwd_f32(const float* q, const float* k, const float* v, float* out,
                               float* lse, int B, int S, int H, int d, int n_shards, int causal,
                               const int32_t* doc_offsets, cudaStream_t stream) {
  cpring::TraceRange trace_("cp_ring_attn_fwd_f32");
  if (!q || !k || !v || !out || !lse) return CP_ERR_NULL;
  cp_status st = check_shape(B, S, H, d, n_shards);
  if (st != CP_OK) return st;
  if (d > 128) return CP_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return CP_ERR_SHAPE;
  if (!aligned(q, 4) || !aligned(k, 4) || !aligned(v, 4) || !aligned(out, 4) ||
      !aligned(lse, 4) || !aligned(doc_offsets, 4))
    return CP_ERR_ALIGN;
  AttnArgs a{};
  a.q = q; a.k = k; a.v = v;
  a.B = B; a.S = S; a.H = H; a.d = d; a.n_shards = n_shards;
  a.q_shard = -1; a.k_shard = -1;
  a.causal = causal;
  a.doc_offsets = doc_offsets;
  a.out = out; a.lse = lse;
  return run_attn(a, false, stream);
}

static cp_status ring_step_common(const void* q, const void* k, const void* v, float* o_part,
                                  float* m_part, float* l_part, int B, int S, int H, int d,
                                  int n_shards, int i, int j, int causal,
                                  const int32_t* doc_offsets, cudaStream_t stream, bool bf16) {
  if (!q || !k || !v || !o_part || !m_part || !l_part) return CP_ERR_NULL;
  cp_status st = check_shape(B, S, H, d, n_shards);
  if (st != CP_OK) return st;
  if (i < 0 || j < 0 || i >= n_shards || j >= n_shards) return CP_ERR_SHAPE;
  if (causal != 0 && causal != 1) return CP_ERR_SHAPE;
  if (bf16) {
    if (d != 64 && d != 128) return CP_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o_part, 16))
      return CP_ERR_ALIGN;
  } else {
    if (d > 128) return CP_ERR_UNSUPPORTED;
    if (!aligned(q, 4) || !aligned(k, 4) || !aligned(v, 4) || !aligned(o_part, 4))
      return CP_ERR_ALIGN;
  }
  if (!aligned(m_part, 4) || !aligned(l_part, 4) || !aligned(doc_offsets, 4)) return CP_ERR_ALIGN;
  AttnArgs a{};
  a.q = q; a.k = k; a.v = v;
  a.B = B; a.S = S; a.H = H; a.d = d; a.n_shards = n_shards;
  a.q_shard = i; a.k_shard = j;
  a.causal = causal;
  a.doc_offsets = doc_offsets;
  a.o_part = o_part; a.m_part = m_part; a.l_part = l_part;
  return run_attn(a, bf16, stream);
}

cp_status cp_ring_step(const void* q, const void* k, const void* v, float* o_part,
                       float* m_part, float* l_part, int B, int S, int H, int d, int n_shards,
                       int i, int j, int causal, const int32_t* doc_offsets,
                       cudaStream_t stream) {
  cpring::TraceRange trace_("cp_ring_step");
  return ring_step_common(q, k, v, o_part, m_part, l_part, B, S, H, d, n_shards, i, j, causal,
                          doc_offsets, stream, true);
}

cp_status cp_ring_step_f32(const float* q, const float* k, const float* v, float* o_part,
                           float* m_part, float* l_part, int B, int S, int H, int d,
                           int n_shards, int i, int j, int causal,
                           const int32_t* doc_offsets, cudaStream_t stream) {
  cpring::TraceRange trace_("cp_ring_step_f32");
  return ring_step_common(q, k, v, o_part, m_part, l_part, B, S, H, d, n_shards, i, j, causal,
                          doc_offsets, stream, false);
}

cp_status cp_lse_merge(float* o_acc, float* m_acc, float* l_acc, const float* o_part,
                       const float* m_part, const float* l_part, int B, int rows, int H, int d,
                       cudaStream_t stream) {
  cpring::TraceRange trace_("cp_lse_merge");
  if (!o_acc || !m_acc || !l_acc || !o_part || !m_part || !l_part) return CP_ERR_NULL;
  if (B < 1 || rows < 1 || H < 1 || d < 1) return CP_ERR_SHAPE;
  if (d > 128) return CP_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * rows * H * d > (1LL << 40)) return CP_ERR_SHAPE;
  if (o_acc == o_part) return CP_ERR_SHAPE;
  if (!aligned(o_acc, 4) || !aligned(m_acc, 4) || !aligned(l_acc, 4) || !aligned(o_part, 4) ||
      !aligned(m_part, 4) || !aligned(l_part, 4))
    return CP_ERR_ALIGN;
  cp_status st = check_device();
  if (st != CP_OK) return st;
  return cpring::launch_merge(o_acc, m_acc, l_acc, o_part, m_part, l_part, B, rows, H, d,
                              stream) == cudaSuccess
             ? CP_OK
             : CP_ERR_CUDA;
}

cp_status cp_lse_finalize(const float* o_acc, const float* m_acc, const float* l_acc, void* out,
                          float* lse, int B, int rows, int H, int d, int out_is_bf16,
                          cudaStream_t stream) {
  cpring::TraceRange trace_("cp_lse_finalize");
  if (!o_acc || !m_acc || !l_acc || !out || !lse) return CP_ERR_NULL;
  if (B < 1 || rows < 1 || H < 1 || d < 1) return CP_ERR_SHAPE;
  if (d > 128) return CP_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * rows * H * d > (1LL << 40)) return CP_ERR_SHAPE;
  if (out_is_bf16 != 0 && out_is_bf16 != 1) return CP_ERR_SHAPE;
  if (!aligned(o_acc, 4) || !aligned(m_acc, 4) || !aligned(l_acc, 4) || !aligned(lse, 4) ||
      !aligned(out, out_is_bf16 ? 2 : 4))
    return CP_ERR_ALIGN;
  cp_status st = check_device();
  if (st != CP_OK) return st;
  return cpring::launch_finalize(o_acc, m_acc, l_acc, out, lse, B, rows, H, d, out_is_bf16,
                                 stream) == cudaSuccess
             ? CP_OK
             : CP_ERR_CUDA;
}

cp_status cp_ring_schedule(int S, int n_shards, int tile_q, int tile_k, int causal,
                           const int32_t* doc_offsets_host, int32_t* pairs_out, int64_t max_pairs,
                           int64_t* n_pairs) {
  if (!n_pairs) return CP_ERR_NULL;
  *n_pairs = 0;
  if (S < 1 || n_shards < 1 || n_shards > S || S % n_shards != 0 || tile_q < 1 || tile_k < 1 ||
      max_pairs < 0)
    return CP_ERR_SHAPE;
  if (causal != 0 && causal != 1) return CP_ERR_SHAPE;
  std::vector<int> ds, de;
  if (!host_docs(doc_offsets_host, S, ds, de)) return CP_ERR_DOC_OFFSETS;
  const int L = S / n_shards;
  const int tq = (L + tile_q - 1) / tile_q;
  const int tk = (L + tile_k - 1) / tile_k;
  int64_t count = 0;
  for (int i = 0; i < n_shards; ++i) {
    for (int a = 0; a < tq; ++a) {
      const int q0 = i * L + a * tile_q;
      const int q1 = std::min(q0 + tile_q, (i + 1) * L) - 1;
      // visible keys of the tile: [doc_start(q0), causal ? q1 : doc_end(q1) - 1]
      const int lo = ds[q0];
      const int hi = causal ? q1 : de[q1] - 1;
      for (int j = 0; j < n_shards; ++j) {
        for (int c = 0; c < tk; ++c) {
          const int k0 = j * L + c * tile_k;
          const int k1 = std::min(k0 + tile_k, (j + 1) * L) - 1;
          if (k0 > hi || k1 < lo) continue;
          if (pairs_out && count < max_pairs) {
            pairs_out[2 * count] = i * tq + a;
            pairs_out[2 * count + 1] = j * tk + c;
          }
          ++count;
        }
      }
    }
  }
  *n_pairs = count;
  if (pairs_out && count > max_pairs) return CP_ERR_BUFFER;
  return CP_OK;
}

cp_status cp_ring_schedule_device(int S, int n_shards, int causal, const int32_t* doc_offsets,
                                  int32_t* ranges, cudaStream_t stream) {
  cpring::TraceRange trace_("cp_ring_schedule_device");
  if (!ranges) return CP_ERR_NULL;
  if (S < 1 || n_shards < 1 || n_shards > S || S % n_shards != 0) return CP_ERR_SHAPE;
  if (causal != 0 && causal != 1) return CP_ERR_SHAPE;
  if (!aligned(ranges, 4) || !aligned(doc_offsets, 4)) return CP_ERR_ALIGN;
  cp_status st = check_device();
  if (st != CP_OK) return st;
  AttnArgs a{};
  a.S = S;
  a.n_shards = n_shards;
  a.causal = causal;
  a.doc_offsets = doc_offsets;
  if (!doc_offsets)
    return cpring::launch_schedule_probe(a, ranges, stream) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
  cpring::ScratchLease lease(cpring::doc_scratch_bytes(S, n_shards, -1, false), stream);
  if (!lease.ok()) return CP_ERR_CUDA;
  int32_t* info = static_cast<int32_t*>(lease.get());
  if (cpring::launch_doc_scan(doc_offsets, S, info, stream) != cudaSuccess) return CP_ERR_CUDA;
  a.doc_info = info;
  return cpring::launch_schedule_probe(a, ranges, stream) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

cp_status cp_ring_traffic(int64_t B, int64_t S, int64_t H, int64_t d, int dtype_bytes,
                          int n_shards, int causal, int64_t* per_rank_bytes) {
  if (!per_rank_bytes) return CP_ERR_NULL;
  if (B < 1 || S < 1 || H < 1 || d < 1 || dtype_bytes < 1 || n_shards < 1 || n_shards > S ||
      S % n_shards != 0)
    return CP_ERR_SHAPE;
  if (causal != 0 && causal != 1) return CP_ERR_SHAPE;
  const int64_t G = 2 * B * S * H * d * dtype_bytes;  // K and V of the whole sequence
  const int64_t blk = G / n_shards;
  for (int r = 0; r < n_shards; ++r) {
    if (!causal) {
      per_rank_bytes[r] = 2 * blk * (n_shards - 1);
    } else {
      const int64_t recv = static_cast<int64_t>(r) * blk;
      const int64_t sent = (r < n_shards - 1) ? static_cast<int64_t>(r + 1) * blk : 0;
      per_rank_bytes[r] = recv + sent;
    }
  }
  return CP_OK;
}

cp_status cp_get_last_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return CP_ERR_CUDA;
  int* word = cpring::device_error_word();
  if (!word) return CP_ERR_CUDA;
  int bits = 0;
  if (cudaMemcpy(&bits, word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return CP_ERR_CUDA;
  if (bits != 0) {
    const int zero = 0;
    if (cudaMemcpy(word, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return CP_ERR_CUDA;
  }
  if (bits & cpring::kErrScratch) return CP_ERR_SCRATCH;
  if (bits & cpring::kErrTimeout) return CP_ERR_TIMEOUT;
  if (bits & cpring::kErrDocOffsets) return CP_ERR_DOC_OFFSETS;
  return CP_OK;
}

const char* cp_status_string(cp_status s) {
  switch (s) {
    case CP_OK: return "ok";
    case CP_ERR_NULL: return "null pointer";
    case CP_ERR_SHAPE: return "bad shape or index";
    case CP_ERR_UNSUPPORTED: return "unsupported head dimension";
    case CP_ERR_ALIGN: return "misaligned pointer";
    case CP_ERR_CUDA: return "CUDA error";
    case CP_ERR_BUFFER: return "output buffer too small";
    case CP_ERR_DOC_OFFSETS: return "malformed doc_offsets";
    case CP_ERR_TIMEOUT: return "device wait timed out";
    case CP_ERR_DEVICE: return "device is not sm_103";
    case CP_ERR_SCRATCH: return "more documents than the fixed scratch of cp_ring_attn_fwd_noalloc holds";
    default: return "unknown status";
  }
}

}  // extern "C"
