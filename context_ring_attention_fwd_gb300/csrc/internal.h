// Host-side declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include <cstdint>
#include <cuda_runtime_api.h>
#include <nvtx3/nvToolsExt.h>

#include "../../include/cpring.h"

namespace cpring {

// What one launch computes: every query shard (q_shard < 0) or one shard
// (q_shard = i), against every key shard (k_shard < 0) or one (k_shard = j).
struct AttnArgs {
  const void* q;
  const void* k;
  const void* v;
  int B, S, H, d, n_shards;
  int q_shard, k_shard;
  int causal;
  const int32_t* doc_offsets;  // device or null
  const int32_t* doc_info;     // device scratch written by the doc scan, or null
  // K/V layout: by default k and v are the whole sequence [B, S, H, d].  With
  // kv_rows > 0 they are one block [B, kv_rows, H, d] whose row 0 is the key
  // kv_row0 of the sequence (a rank's receive buffer in the ring emulation).
  int kv_rows;
  int kv_row0;
  // fused outputs
  void* out;
  float* lse;
  // partial (one step) outputs
  float* o_part;
  float* m_part;
  float* l_part;
  // FP8 form: per-(b, h) descales [B * H] (q, k, v = E4M3 Q, K and V^T)
  const float* q_descale;
  const float* k_descale;
  const float* v_descale;
  // With doc_offsets: device scratch of slot_count() int32 for the
  // cost-ranked work order, or null to deal by position.
  int32_t* slot_perm;
};

// Work slots (query shard, pair of 128-row query tiles) of one (b, h) of a
// tensor-core forward launch: n_qshards * ceil((S / n_shards) / 256).
inline int slot_count(int S, int n_shards, int q_shard) {
  const int L = S / n_shards;
  return (q_shard < 0 ? n_shards : 1) * ((L + 255) / 256);
}

// Launches with documents rank their slots by cost (slot_order_kernel) when
// they hold at most this many; larger ones deal by position.
constexpr int kMaxRankedSlots = 8192;

// Bytes of scratch a forward launch with documents uses: the doc-scan word
// (16 bytes), then the cost-ranked slot order (tensor-core paths only).
inline size_t doc_scratch_bytes(int S, int n_shards, int q_shard, bool ranked) {
  return 16 + (ranked ? 4 * static_cast<size_t>(slot_count(S, n_shards, q_shard)) : 0);
}

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// The shape checks every forward entry point shares: sizes >= 1, an equal
// split into n_shards, at most 2^40 elements and B * H small enough for the
// kernels' int work counters.
inline cp_status check_shape(int B, int S, int H, int d, int n_shards) {
  if (B < 1 || S < 1 || H < 1 || d < 1 || n_shards < 1 || n_shards > S) return CP_ERR_SHAPE;
  if (S % n_shards != 0) return CP_ERR_SHAPE;
  const long long elems = static_cast<long long>(B) * S * H * d;
  if (elems > (1LL << 40)) return CP_ERR_SHAPE;
  if (static_cast<long long>(B) * H > 0x7fffffff / 4) return CP_ERR_SHAPE;
  return CP_OK;
}

// The library's cached per-device scratch (the doc-scan word and the
// cost-ranked slot order of launches with documents).  One buffer per device
// grows on demand with stream-ordered allocation (cudaMallocAsync /
// cudaFreeAsync on the caller's stream) and is kept for the process's life.
// A lease holds the device's lock from construction to destruction, so host
// threads take turns; its constructor orders `stream` after the work of the
// previous lease when that ran on another stream, and its destructor records
// the point after which the next lease may reuse the buffer.  Every launch
// that reads the buffer must be enqueued on `stream` while the lease lives.
class ScratchLease {
 public:
  ScratchLease(size_t bytes, cudaStream_t stream);
  ~ScratchLease();
  ScratchLease(const ScratchLease&) = delete;
  ScratchLease& operator=(const ScratchLease&) = delete;
  void* get() const { return ptr_; }
  bool ok() const { return ok_; }

 private:
  int dev_ = -1;
  void* ptr_ = nullptr;
  bool ok_ = false;
  cudaStream_t stream_ = nullptr;
};

// The backward: gradients of sum(out * dout) for the forward's out and lse.
struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* out;
  const float* lse;
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  float* delta;                // device scratch [B, H, S]
  int B, S, H, d, n_shards;
  int causal;
  const int32_t* doc_offsets;  // device or null
  const int32_t* doc_info;     // written by the doc scan, or null
};

// An NVTX range named after the C-ABI call it covers (tracing for profilers;
// a no-op unless a profiler is attached, and never a device allocation).
struct TraceRange {
  explicit TraceRange(const char* name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};

// Sticky device error word (bits of kErr*), owned by merge.cu.
constexpr int kErrDocOffsets = 1;
constexpr int kErrTimeout = 2;
constexpr int kErrScratch = 4;  // raised only by cp_ring_attn_fwd_noalloc
int* device_error_word();   // device address for the current device, or null

// Launchers: return cudaSuccess or the launch error.
cudaError_t launch_attn_bf16(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_attn_f32(const AttnArgs& a, cudaStream_t stream);
// FP8 form: q, k E4M3 [B, S, H, 128], v E4M3 [B, H, 128, S]; the fused
// forward only (q_shard = k_shard = -1).
cudaError_t launch_attn_fp8(const AttnArgs& a, cudaStream_t stream);
// The fused kernel's per-query-tile key-tile ranges (first, last flat tile),
// computed on the device by the kernel's own work decoding (B = H = 1).
cudaError_t launch_schedule_probe(const AttnArgs& a, int32_t* ranges, cudaStream_t stream);
// Backward: the row sums D, then the dK/dV kernel and the dQ kernel (bf16,
// d in {64, 128}).
cudaError_t launch_attn_bwd(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_doc_scan(const int32_t* doc_offsets, int S, int32_t* doc_info,
                            cudaStream_t stream);
cudaError_t launch_merge(float* o_acc, float* m_acc, float* l_acc, const float* o_part,
                         const float* m_part, const float* l_part, int B, int rows, int H, int d,
                         cudaStream_t stream);
cudaError_t launch_finalize(const float* o_acc, const float* m_acc, const float* l_acc, void* out,
                            float* lse, int B, int rows, int H, int d, int out_is_bf16,
                            cudaStream_t stream);
// Finalize into strided outputs: out row (b, r, h) at b*out_bstride +
// (r*H + h)*d elements; lse (b, h, r) at b*lse_bstride + h*lse_hstride + r.
cudaError_t launch_finalize_strided(const float* o_acc, const float* m_acc, const float* l_acc,
                                    void* out, float* lse, int B, int rows, int H, int d,
                                    int out_is_bf16, long long out_bstride, long long lse_bstride,
                                    long long lse_hstride, cudaStream_t stream);

// Test hook state set by cp_test_set_wait_fault: whether CTA 0 of the next
// tensor-core launches skips one tile load, and the wait limit in ns.
int test_fault_drop();
unsigned long long test_wait_limit_ns();

// Host launch counters (index: 0 tcgen05 attention, 1 fp32 attention,
// 2 merge/finalize, 3 doc scan).
void count_launch(int which);

// Multiprocessor count of the current device (cached per device).
int sm_count();
// Raises `kern`'s dynamic shared-memory limit to `bytes` on the current
// device: once per (kernel, device) for the process's life, under a lock,
// with the first call's result returned to every later one.
cudaError_t ensure_smem_limit(const void* kern, int bytes);
// Compute capability major*10+minor of the current device (cached).
int device_cc();

}  // namespace cpring
