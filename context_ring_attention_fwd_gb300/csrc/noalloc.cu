// cp_ring_attn_fwd_noalloc: the fused bf16 forward without any device
// allocation by the library.
//
// Why it exists.  cp_ring_attn_fwd keeps a small cached scratch per device
// for calls that pass doc_offsets, and allocates it (cudaMallocAsync) the
// first time and whenever a call needs more than it holds.  Some callers
// cannot let a library allocate at all: serving processes that hand almost
// all of the GPU's memory to their own pool at start-up and forbid any later
// cudaMalloc/cudaMallocAsync (an allocation there can fail, or fragment or
// shrink the pool under load), and latency-critical loops that must never
// enter the driver's allocator.  This entry point serves them: it computes
// the same result as cp_ring_attn_fwd, but its scratch lives in a fixed
// device array compiled into the library.
//
// The scratch.  g_noalloc_scratch below is a file-scope device array of
// kScratchInts int32 (295,168 bytes).  Every GPU that loads the library holds
// it until the process exits.  It stores the document count (header word 0),
// a validated copy of the document boundaries (from word kHeaderInts on),
// which the attention kernel then reads, and the cost-ranked order of the
// launch's work slots (the last kMaxRankedSlots words), the same order
// cp_ring_attn_fwd deals by.  The copy holds at most kMaxDocs + 1
// boundaries, so at most kMaxDocs = 65,535 documents per call.
//
// Host code must never hand the array's name to a kernel: on the host that
// name is only a stand-in, not a device address.  The device address comes
// from cudaGetSymbolAddress, called once per device with that device
// current, the first time this entry point runs on it.  Make that first call
// on each device before any stream capture.  The address is cached for the
// life of the process, so the library must not be used across
// cudaDeviceReset.
//
// Sharing.  All calls on a device share the one array, and it keeps what the
// last call wrote.  Each call rewrites the header, the boundary copy and the
// slot order before its attention kernel reads them (stream order), so
// nothing from an earlier call is ever read and nothing needs clearing to
// zero.  Calls whose work overlaps on the GPU (different streams, no ordering
// between them) race on the array and must not be issued.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace cpring {
namespace {

constexpr int kHeaderInts = 64;      // word 0: document count, or -1
constexpr int kMaxDocs = 65535;      // boundaries copied: at most kMaxDocs + 1
constexpr int kPermOff = kHeaderInts + kMaxDocs + 1;  // the slot order
constexpr int kScratchInts = kPermOff + kMaxRankedSlots;

static __device__ __align__(256) int32_t g_noalloc_scratch[kScratchInts];
static_assert(sizeof(g_noalloc_scratch) == 295168, "the documented size of the fixed scratch");

// Validate doc_offsets (0 = o_0 < o_1 < ... < o_n = S, read up to the first
// entry equal to S and never past it) and copy it into the scratch.  Writes
// the document count to the header, or -1 with an error bit: kErrDocOffsets
// for a malformed array, kErrScratch when it holds more than kMaxDocs
// documents.
__global__ void doc_scan_copy_kernel(const int32_t* __restrict__ offs, int S, int32_t* scratch,
                                     int* err) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  int32_t* copy = scratch + kHeaderInts;
  int32_t prev = offs[0];
  int code = (prev == 0 && S > 0) ? 0 : kErrDocOffsets;
  int n = 0;
  if (code == 0) {
    copy[0] = 0;
    for (int idx = 1; idx <= S; ++idx) {
      const int32_t x = offs[idx];
      if (x <= prev || x > S) {
        code = kErrDocOffsets;
        break;
      }
      if (idx > kMaxDocs) {
        code = kErrScratch;
        break;
      }
      copy[idx] = x;
      prev = x;
      if (x == S) {
        n = idx;
        break;
      }
    }
    if (code == 0 && n == 0) code = kErrDocOffsets;
  }
  scratch[0] = (code == 0) ? n : -1;
  if (code != 0) atomicOr(err, code);
}

// Device address of g_noalloc_scratch for the current device, looked up once
// per device with that device current.  Null if the lookup failed.
int32_t* scratch_address() {
  static std::mutex mu;
  static int32_t* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    int32_t* ptr = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_scratch) != cudaSuccess)
      return nullptr;
    addr[dev] = ptr;
  }
  return addr[dev];
}

}  // namespace
}  // namespace cpring

extern "C" cp_status cp_ring_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                                              void* out, float* lse, int B, int S, int H, int d,
                                              int n_shards, int causal,
                                              const int32_t* doc_offsets, cudaStream_t stream) {
  cpring::TraceRange trace_("cp_ring_attn_fwd_noalloc");
  using namespace cpring;
  if (!q || !k || !v || !out || !lse) return CP_ERR_NULL;
  const cp_status st = check_shape(B, S, H, d, n_shards);
  if (st != CP_OK) return st;
  if (d != 64 && d != 128) return CP_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return CP_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(doc_offsets, 4))
    return CP_ERR_ALIGN;
  if (device_cc() != 103) return CP_ERR_DEVICE;

  AttnArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.B = B;
  a.S = S;
  a.H = H;
  a.d = d;
  a.n_shards = n_shards;
  a.q_shard = -1;
  a.k_shard = -1;
  a.causal = causal;
  a.out = out;
  a.lse = lse;
  if (doc_offsets) {
    int32_t* scratch = scratch_address();
    int* err = device_error_word();
    if (!scratch || !err) return CP_ERR_CUDA;
    doc_scan_copy_kernel<<<1, 32, 0, stream>>>(doc_offsets, S, scratch, err);
    count_launch(3);
    if (cudaGetLastError() != cudaSuccess) return CP_ERR_CUDA;
    a.doc_offsets = scratch + kHeaderInts;  // the validated copy
    a.doc_info = scratch;
    a.slot_perm = scratch + kPermOff;        // written by the launch's slot ranking
  }
  return launch_attn_bf16(a, stream) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}
