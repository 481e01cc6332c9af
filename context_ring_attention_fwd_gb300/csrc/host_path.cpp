// cp_ring_attn_fwd_host: the fused forward end to end from host buffers.
//
// "上下文並行（Context Parallelism, CP）" (compassingai.com), section 線上
// Softmax: each GPU i computes with the K/V block it holds while the next
// block is sent and received, the two running asynchronously side by side;
// section 因果掩碼的特殊處理: under causality GPU i needs only the blocks of
// GPUs 0..i.  On one GPU the host link takes the ring's place: shard i's Q, K
// and V go to the device on a copy stream, rank i starts as soon as every
// shard it reads has landed (shards 0..i under causality, all of them
// otherwise), and its rows of the output go back on a second copy stream
// while later ranks compute.  The result is bitwise that of one
// cp_ring_attn_fwd call on the same inputs, because every rank's launch
// computes its work items exactly as the whole-sequence launch does.
//
// The two copy streams and the events that order them belong to the library
// (one set per device, created on first use and kept for the process's
// life); a per-device lock is held while a call enqueues its work, so host
// threads take turns.  The caller's stream ends up waiting for every copy,
// so synchronising it means the host outputs are complete.
#include <cuda_runtime_api.h>

#include <mutex>
#include <optional>
#include <vector>

#include "internal.h"

namespace cpring {
namespace {

struct HostPathDevice {
  std::mutex mu;
  cudaStream_t h2d = nullptr;
  cudaStream_t d2h = nullptr;
  std::vector<cudaEvent_t> events;
};

constexpr int kMaxDevices = 64;
HostPathDevice g_host_path[kMaxDevices];

int64_t round256(int64_t x) { return (x + 255) / 256 * 256; }

// Workspace layout: q | k | v | out (each B*S*H*d elements) | lse (B*H*S fp32).
struct HostLayout {
  int64_t tensor;  // bytes of one [B, S, H, d] tensor, rounded to 256
  int64_t total;
};

HostLayout host_layout(int B, int S, int H, int d, int elem_bytes) {
  HostLayout l{};
  l.tensor = round256(static_cast<int64_t>(B) * S * H * d * elem_bytes);
  l.total = 4 * l.tensor + round256(static_cast<int64_t>(B) * H * S * 4);
  return l;
}

// The copy streams and events of the current device.
HostPathDevice* host_path_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  return &g_host_path[dev];
}

// Creates the two copy streams and at least n_events events on first use.
bool ensure_resources(HostPathDevice& h, int n_events) {
  if (!h.h2d && cudaStreamCreateWithFlags(&h.h2d, cudaStreamNonBlocking) != cudaSuccess) {
    h.h2d = nullptr;
    return false;
  }
  if (!h.d2h && cudaStreamCreateWithFlags(&h.d2h, cudaStreamNonBlocking) != cudaSuccess) {
    h.d2h = nullptr;
    return false;
  }
  while (static_cast<int>(h.events.size()) < n_events) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
    h.events.push_back(e);
  }
  return true;
}

cp_status host_forward(const void* q_host, const void* k_host, const void* v_host, void* out_host,
                       float* lse_host, int B, int S, int H, int d, int n_shards, int causal,
                       const int32_t* doc_offsets, void* workspace, int64_t workspace_bytes,
                       cudaStream_t stream, bool f32) {
  if (!q_host || !k_host || !v_host || !out_host || !lse_host || !workspace) return CP_ERR_NULL;
  cp_status st = check_shape(B, S, H, d, n_shards);
  if (st != CP_OK) return st;
  if (f32 ? (d > 128) : (d != 64 && d != 128)) return CP_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return CP_ERR_SHAPE;
  if (!aligned(workspace, 256) || !aligned(doc_offsets, 4)) return CP_ERR_ALIGN;
  const int esz = f32 ? 4 : 2;
  const HostLayout lay = host_layout(B, S, H, d, esz);
  if (workspace_bytes < lay.total) return CP_ERR_BUFFER;
  if (device_cc() != 103) return CP_ERR_DEVICE;

  const int N = n_shards;
  HostPathDevice* hp = host_path_device();
  if (!hp) return CP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(hp->mu);
  if (!ensure_resources(*hp, 2 * N + 2)) return CP_ERR_CUDA;
  cudaEvent_t ev_start = hp->events[0];
  cudaEvent_t ev_end = hp->events[1];
  cudaEvent_t* landed = hp->events.data() + 2;
  cudaEvent_t* done = hp->events.data() + 2 + N;

  char* ws = static_cast<char*>(workspace);
  char* qd = ws;
  char* kd = ws + lay.tensor;
  char* vd = ws + 2 * lay.tensor;
  char* od = ws + 3 * lay.tensor;
  float* ld = reinterpret_cast<float*>(ws + 4 * lay.tensor);
  const int L = S / N;
  const size_t row_bytes = static_cast<size_t>(H) * d * esz;    // one token, all heads
  const size_t shard_bytes = static_cast<size_t>(L) * row_bytes;  // one shard of one batch row
  const size_t seq_bytes = static_cast<size_t>(S) * row_bytes;
  auto at = [&](const void* base, int b, int i) {
    return static_cast<const char*>(base) + static_cast<size_t>(b) * seq_bytes +
           static_cast<size_t>(i) * shard_bytes;
  };

  cudaError_t err = cudaSuccess;
  auto chk = [&](cudaError_t e) {
    if (err == cudaSuccess && e != cudaSuccess) err = e;
  };
  // Everything the caller enqueued before (including an earlier call's
  // kernels on these device buffers) comes first.
  chk(cudaEventRecord(ev_start, stream));
  chk(cudaStreamWaitEvent(hp->h2d, ev_start, 0));

  // Documents: the doc-scan word and each rank's slot order live in the
  // library's cached scratch for the rest of the call.
  std::optional<ScratchLease> lease;
  int32_t* info = nullptr;
  if (doc_offsets) {
    lease.emplace(doc_scratch_bytes(S, N, 0, !f32), stream);
    if (!lease->ok()) return CP_ERR_CUDA;
    info = static_cast<int32_t*>(lease->get());
    chk(launch_doc_scan(doc_offsets, S, info, stream));
  }

  // shard i of Q, K, V to the device, in rank order
  for (int i = 0; i < N && err == cudaSuccess; ++i) {
    for (int b = 0; b < B; ++b) {
      const size_t off = static_cast<size_t>(b) * seq_bytes + static_cast<size_t>(i) * shard_bytes;
      chk(cudaMemcpyAsync(qd + off, at(q_host, b, i), shard_bytes, cudaMemcpyHostToDevice, hp->h2d));
      chk(cudaMemcpyAsync(kd + off, at(k_host, b, i), shard_bytes, cudaMemcpyHostToDevice, hp->h2d));
      chk(cudaMemcpyAsync(vd + off, at(v_host, b, i), shard_bytes, cudaMemcpyHostToDevice, hp->h2d));
    }
    chk(cudaEventRecord(landed[i], hp->h2d));
  }
  // rank i once the shards it reads have landed; its rows go back at once
  for (int i = 0; i < N && err == cudaSuccess; ++i) {
    chk(cudaStreamWaitEvent(stream, landed[causal ? i : N - 1], 0));
    AttnArgs a{};
    a.q = qd; a.k = kd; a.v = vd;
    a.B = B; a.S = S; a.H = H; a.d = d; a.n_shards = N;
    a.q_shard = i; a.k_shard = -1;
    a.causal = causal;
    a.doc_offsets = doc_offsets;
    a.doc_info = info;
    a.slot_perm = (info && !f32) ? info + 4 : nullptr;
    a.out = od; a.lse = ld;
    chk(f32 ? launch_attn_f32(a, stream) : launch_attn_bf16(a, stream));
    chk(cudaEventRecord(done[i], stream));
    chk(cudaStreamWaitEvent(hp->d2h, done[i], 0));
    for (int b = 0; b < B; ++b) {
      const size_t off = static_cast<size_t>(b) * seq_bytes + static_cast<size_t>(i) * shard_bytes;
      chk(cudaMemcpyAsync(static_cast<char*>(out_host) + off, od + off, shard_bytes,
                          cudaMemcpyDeviceToHost, hp->d2h));
    }
    // lse [B, H, S]: rank i's L entries of each of the B*H rows
    chk(cudaMemcpy2DAsync(lse_host + static_cast<size_t>(i) * L, static_cast<size_t>(S) * 4,
                          ld + static_cast<size_t>(i) * L, static_cast<size_t>(S) * 4,
                          static_cast<size_t>(L) * 4, static_cast<size_t>(B) * H,
                          cudaMemcpyDeviceToHost, hp->d2h));
  }
  // the caller's stream waits for the last copy back
  chk(cudaEventRecord(ev_end, hp->d2h));
  chk(cudaStreamWaitEvent(stream, ev_end, 0));
  return err == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

}  // namespace
}  // namespace cpring

extern "C" int64_t cp_ring_attn_fwd_host_workspace_bytes(int B, int S, int H, int d, int n_shards,
                                                         int elem_bytes) {
  if (cpring::check_shape(B, S, H, d, n_shards) != CP_OK) return -1;
  if (elem_bytes != 2 && elem_bytes != 4) return -1;
  return cpring::host_layout(B, S, H, d, elem_bytes).total;
}

extern "C" cp_status cp_ring_attn_fwd_host(const void* q_host, const void* k_host,
                                           const void* v_host, void* out_host, float* lse_host,
                                           int B, int S, int H, int d, int n_shards, int causal,
                                           const int32_t* doc_offsets, void* workspace,
                                           int64_t workspace_bytes, cudaStream_t stream) {
  cpring::TraceRange trace_("cp_ring_attn_fwd_host");
  return cpring::host_forward(q_host, k_host, v_host, out_host, lse_host, B, S, H, d, n_shards,
                              causal, doc_offsets, workspace, workspace_bytes, stream, false);
}

extern "C" cp_status cp_ring_attn_fwd_host_f32(const float* q_host, const float* k_host,
                                               const float* v_host, float* out_host,
                                               float* lse_host, int B, int S, int H, int d,
                                               int n_shards, int causal,
                                               const int32_t* doc_offsets, void* workspace,
                                               int64_t workspace_bytes, cudaStream_t stream) {
  cpring::TraceRange trace_("cp_ring_attn_fwd_host_f32");
  return cpring::host_forward(q_host, k_host, v_host, out_host, lse_host, B, S, H, d, n_shards,
                              causal, doc_offsets, workspace, workspace_bytes, stream, true);
}
