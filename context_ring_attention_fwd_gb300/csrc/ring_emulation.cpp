// The ring with explicit per-rank buffers, on one GPU.
//
// "上下文並行（Context Parallelism, CP）" (compassingai.com), section 線上 Softmax:
// at every step each GPU computes a partial attention of its query shard
// against the K/V block it currently holds, merges it into its running
// (O, m, l), and passes the block to the next GPU while receiving one from
// the previous GPU; "大语言模型并行策略（五）：上下文并行" (wangyu.me), section
// 通信模式: the transfer of the next block is double-buffered so it overlaps
// the computation of the current one.  Section 因果掩碼的特殊處理 of the first
// page: under causality GPU i needs only the blocks of GPUs 0..i, so a block
// travels only to the ranks that need it.
//
// Here every virtual rank owns a two-slot K/V receive buffer in one
// workspace.  At step t rank i holds the block of rank (i - t) mod N in slot
// t % 2.  The compute stream runs cp_ring_step on that slot and the online
// merge; the copy stream moves, for step t + 1, the block each rank holds
// into its successor's other slot (the "send"), ordered by events so that
// a slot is overwritten only after the step that read it has finished and
// read only after its copy has landed.  Without a copy stream the copies run
// in order on the compute stream (no overlap), which measures what the
// overlap hides.  With documents every step applies the document mask, so
// packed sequences keep their boundaries across the ranks' blocks.
#include <cuda_runtime_api.h>

#include <cstdint>
#include <optional>
#include <vector>

#include "internal.h"

namespace {

struct Plan {
  int64_t blk_elems;   // B * L * H * d
  int64_t kv_bytes;    // one K or V block, bf16
  int64_t state_elems; // B * H * L
  // workspace offsets (bytes)
  int64_t off_kv;      // N ranks x 2 slots x (K, V)
  int64_t off_acc;     // N ranks x (O fp32, m, l)
  int64_t off_part;    // one (O, m, l) partial, shared by the serialised steps
  int64_t total;
};

int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }

Plan make_plan(int B, int S, int H, int d, int N) {
  Plan p{};
  const int64_t L = S / N;
  p.blk_elems = static_cast<int64_t>(B) * L * H * d;
  p.kv_bytes = align256(p.blk_elems * 2);
  p.state_elems = static_cast<int64_t>(B) * H * L;
  const int64_t acc = align256(p.blk_elems * 4) + 2 * align256(p.state_elems * 4);
  p.off_kv = 0;
  p.off_acc = p.off_kv + static_cast<int64_t>(N) * 2 * 2 * p.kv_bytes;
  p.off_part = p.off_acc + static_cast<int64_t>(N) * acc;
  p.total = p.off_part + acc;
  return p;
}

}  // namespace

extern "C" int64_t cp_ring_emulated_workspace_bytes(int B, int S, int H, int d, int n_shards) {
  if (B < 1 || S < 1 || H < 1 || d < 1 || n_shards < 1 || n_shards > S || S % n_shards != 0)
    return -1;
  return make_plan(B, S, H, d, n_shards).total;
}

extern "C" cp_status cp_ring_attn_fwd_emulated(const void* q, const void* k, const void* v,
                                               void* out, float* lse, int B, int S, int H, int d,
                                               int n_shards, int causal,
                                               const int32_t* doc_offsets, void* workspace,
                                               int64_t workspace_bytes, cudaStream_t stream,
                                               cudaStream_t copy_stream,
                                               int64_t* recv_bytes_per_rank) {
  cpring::TraceRange trace_("cp_ring_attn_fwd_emulated");
  using cpring::aligned;
  if (!q || !k || !v || !out || !lse || !workspace) return CP_ERR_NULL;
  const cp_status shape = cpring::check_shape(B, S, H, d, n_shards);
  if (shape != CP_OK) return shape;
  if (causal != 0 && causal != 1) return CP_ERR_SHAPE;
  if (d != 64 && d != 128) return CP_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(workspace, 256) || !aligned(doc_offsets, 4))
    return CP_ERR_ALIGN;
  const int N = n_shards;
  const Plan pl = make_plan(B, S, H, d, N);
  if (workspace_bytes < pl.total) return CP_ERR_BUFFER;
  if (cpring::device_cc() != 103) return CP_ERR_DEVICE;

  const int L = S / N;
  char* ws = static_cast<char*>(workspace);
  auto kv_slot = [&](int rank, int slot, int which) -> void* {  // which: 0 = K, 1 = V
    return ws + pl.off_kv + ((static_cast<int64_t>(rank) * 2 + slot) * 2 + which) * pl.kv_bytes;
  };
  const int64_t acc_stride = align256(pl.blk_elems * 4) + 2 * align256(pl.state_elems * 4);
  auto acc = [&](int rank, int part) -> float* {  // part: 0 = O, 1 = m, 2 = l
    char* base = ws + pl.off_acc + static_cast<int64_t>(rank) * acc_stride;
    if (part == 0) return reinterpret_cast<float*>(base);
    base += align256(pl.blk_elems * 4);
    if (part == 2) base += align256(pl.state_elems * 4);
    return reinterpret_cast<float*>(base);
  };
  auto part = [&](int which) -> float* {
    char* base = ws + pl.off_part;
    if (which == 0) return reinterpret_cast<float*>(base);
    base += align256(pl.blk_elems * 4);
    if (which == 2) base += align256(pl.state_elems * 4);
    return reinterpret_cast<float*>(base);
  };
  const bool overlap = copy_stream != nullptr;
  cudaStream_t cs = overlap ? copy_stream : stream;
  // Copy one K or V block of the sequence (rows [j L, (j+1) L) of every batch
  // row) into / between rank buffers: B strided pieces.
  const size_t row_bytes = static_cast<size_t>(H) * d * 2;
  auto copy_in = [&](void* dst, const void* src_seq, int j, cudaStream_t st) -> cudaError_t {
    return cudaMemcpy2DAsync(dst, static_cast<size_t>(L) * row_bytes,
                             static_cast<const char*>(src_seq) + static_cast<size_t>(j) * L * row_bytes,
                             static_cast<size_t>(S) * row_bytes, static_cast<size_t>(L) * row_bytes,
                             B, cudaMemcpyDeviceToDevice, st);
  };
  std::vector<int64_t> recv(N, 0);
  cudaEvent_t ev_copied = nullptr, ev_computed = nullptr;
  if (cudaEventCreateWithFlags(&ev_copied, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&ev_computed, cudaEventDisableTiming) != cudaSuccess)
    return CP_ERR_CUDA;
  cudaError_t err = cudaSuccess;
  auto chk = [&](cudaError_t e) {
    if (err == cudaSuccess && e != cudaSuccess) err = e;
  };
  // Documents ("Context Parallel", section 常见失败模式: packed samples keep
  // their boundaries across shards): every step masks by document as the
  // fused kernel does; the doc-scan word and the step launches' slot order
  // live in the library's cached scratch for the rest of the call.
  std::optional<cpring::ScratchLease> lease;
  int32_t* info = nullptr;
  if (doc_offsets) {
    lease.emplace(cpring::doc_scratch_bytes(S, N, 0, true), stream);
    if (!lease->ok()) {
      cudaEventDestroy(ev_copied);
      cudaEventDestroy(ev_computed);
      return CP_ERR_CUDA;
    }
    info = static_cast<int32_t*>(lease->get());
    chk(cpring::launch_doc_scan(doc_offsets, S, info, stream));
  }
  // Step 0: every rank holds its own block (local placement, not ring traffic).
  for (int i = 0; i < N; ++i) {
    chk(copy_in(kv_slot(i, 0, 0), k, i, stream));
    chk(copy_in(kv_slot(i, 0, 1), v, i, stream));
  }
  chk(cudaEventRecord(ev_computed, stream));  // the first sends read these slots
  std::vector<bool> started(N, false);
  for (int t = 0; t < N && err == cudaSuccess; ++t) {
    const int slot = t & 1;
    // "send": for step t + 1, rank i receives from rank i - 1 the block that
    // rank i - 1 holds at step t, into its other slot.  The other slot was
    // read by step t - 1, which ev_computed marks.
    if (t + 1 < N) {
      if (overlap) chk(cudaStreamWaitEvent(cs, ev_computed, 0));
      for (int i = 0; i < N; ++i) {
        const int src = (i - 1 + N) % N;
        const int j_next = ((i - (t + 1)) % N + N) % N;
        if (causal && j_next > i) continue;  // rank i never needs that block
        chk(cudaMemcpyAsync(kv_slot(i, slot ^ 1, 0), kv_slot(src, slot, 0), pl.blk_elems * 2,
                            cudaMemcpyDeviceToDevice, cs));
        chk(cudaMemcpyAsync(kv_slot(i, slot ^ 1, 1), kv_slot(src, slot, 1), pl.blk_elems * 2,
                            cudaMemcpyDeviceToDevice, cs));
        recv[i] += 2 * pl.blk_elems * 2;
      }
    }
    // compute of step t on slot t % 2
    for (int i = 0; i < N; ++i) {
      const int j = ((i - t) % N + N) % N;
      if (causal && j > i) continue;  // causally dead step: skipped
      cpring::AttnArgs a{};
      a.q = q;
      a.k = kv_slot(i, slot, 0);
      a.v = kv_slot(i, slot, 1);
      a.B = B; a.S = S; a.H = H; a.d = d; a.n_shards = N;
      a.q_shard = i; a.k_shard = j;
      a.causal = causal;
      a.doc_offsets = doc_offsets;
      a.doc_info = info;
      a.slot_perm = info ? info + 4 : nullptr;
      a.kv_rows = L;
      a.kv_row0 = j * L;
      if (!started[i]) {
        a.o_part = acc(i, 0); a.m_part = acc(i, 1); a.l_part = acc(i, 2);
        chk(cpring::launch_attn_bf16(a, stream));
        started[i] = true;
      } else {
        a.o_part = part(0); a.m_part = part(1); a.l_part = part(2);
        chk(cpring::launch_attn_bf16(a, stream));
        chk(cpring::launch_merge(acc(i, 0), acc(i, 1), acc(i, 2), part(0), part(1), part(2), B, L,
                                 H, d, stream));
      }
    }
    chk(cudaEventRecord(ev_computed, stream));
    if (t + 1 < N && overlap) {
      chk(cudaEventRecord(ev_copied, cs));
      chk(cudaStreamWaitEvent(stream, ev_copied, 0));
    }
  }
  // O_i / l_i and the log-sum-exp, into rank i's rows of out and lse.
  for (int i = 0; i < N && err == cudaSuccess; ++i) {
    chk(cpring::launch_finalize_strided(
        acc(i, 0), acc(i, 1), acc(i, 2),
        static_cast<char*>(out) + static_cast<size_t>(i) * L * row_bytes, lse + static_cast<size_t>(i) * L,
        B, L, H, d, 1, static_cast<long long>(S) * H * d, static_cast<long long>(H) * S, S, stream));
  }
  // The copy stream must not outlive the call with work on buffers that the
  // caller may reuse: the compute stream waits for it.
  if (overlap && err == cudaSuccess) {
    chk(cudaEventRecord(ev_copied, cs));
    chk(cudaStreamWaitEvent(stream, ev_copied, 0));
  }
  cudaEventDestroy(ev_copied);
  cudaEventDestroy(ev_computed);
  if (recv_bytes_per_rank)
    for (int i = 0; i < N; ++i) recv_bytes_per_rank[i] = recv[i];
  return err == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}
