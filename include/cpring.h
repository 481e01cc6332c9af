/*
 * cpring — context-parallel ring-attention forward on one GB300 (sm_103a).
 *
 * The method: the sequence is cut into N contiguous equal shards; every
 * query shard Q_i visits the K/V shards j in ring order, computes a partial
 * attention against each and folds it into a running (O_i, m_i, l_i) with the
 * online-softmax merge; causally dead steps (j > i) are skipped; the output is
 * O_i / l_i and the log-sum-exp.  Sources: the "上下文並行（Context
 * Parallelism, CP）" page (compassingai.com), sections 數學基礎, 線上 Softmax
 * (algorithm "Ring Attention + FlashAttention 分塊計算") and 因果掩碼的特殊處理;
 * the "大语言模型并行策略（五）：上下文并行" page (wangyu.me), sections
 * Attention 的流式计算, Ring Attention and 通信模式; the "Context Parallel"
 * page (process-cxr.github.io), sections 基本机制 and 常见失败模式 (document
 * boundaries of packed samples).
 *
 * All N virtual ranks run on one GPU: the ring's send/receive becomes a
 * double-buffered walk over K/V tiles that TMA streams from HBM.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  Layout      q, k, v, out: [B, S, H, d], row-major, d fastest (contiguous).
 *              lse: [B, H, S] fp32, natural log.  Per-step state: O as
 *              [B, S/N, H, d] fp32, m and l as [B, H, S/N] fp32 (natural-log
 *              units: m is the row max of q.k/sqrt(d)).
 *  Shards      shard i = tokens [i*S/N, (i+1)*S/N); S % N must be 0.
 *  Masks       causal: key k visible to query q iff k <= q.  doc_offsets:
 *              NULL = one document per batch row; otherwise a DEVICE int32
 *              array 0 = o_0 < o_1 < ... < o_n = S, read up to and including
 *              the first entry equal to S (cu_seqlens style); the same
 *              boundaries apply to every batch row; key k is visible to q
 *              only if both lie in the same document.
 *  Ownership   the caller owns every buffer and the stream.  Calls are
 *              asynchronous on `stream`; only cp_get_last_status
 *              synchronises.  When doc_offsets is given the call reads its
 *              doc-scan word and work order from a small scratch that the
 *              library caches per device: it is allocated in stream order
 *              (cudaMallocAsync on `stream`) on first use and whenever a
 *              call needs more than it holds (4 bytes per 256 query rows of
 *              the launch, plus 16), and kept until the process exits.  A
 *              call on another stream than the previous user's first waits
 *              for that user's work.  cp_ring_attn_fwd_noalloc allocates
 *              nothing.  State cached per device (this scratch, the error
 *              word's address, the host path's copy streams) does not
 *              survive cudaDeviceReset: do not use the library across one.
 *  Errors      arguments are checked on the host before any launch; a
 *              violation returns a negative cp_status and launches nothing.
 *              Faults found on the device (malformed doc_offsets, a wait
 *              that ran out) set a sticky device error word; the call that
 *              found them writes none of its outputs, and the error is
 *              reported by cp_get_last_status.
 *  Pointers    q/k/v/out/o_part: 16-byte aligned; lse/m/l: 4-byte aligned.
 */
#ifndef CPRING_H
#define CPRING_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int cp_status;

enum {
  CP_OK = 0,
  CP_ERR_NULL = -1,         /* a required pointer is NULL                       */
  CP_ERR_SHAPE = -2,        /* sizes out of range, S % N != 0, i/j out of range */
  CP_ERR_UNSUPPORTED = -3,  /* head dim not supported by this entry point       */
  CP_ERR_ALIGN = -4,        /* a pointer is not aligned as required             */
  CP_ERR_CUDA = -5,         /* a CUDA runtime call or launch failed             */
  CP_ERR_BUFFER = -6,       /* an output buffer is too small                    */
  CP_ERR_DOC_OFFSETS = -7,  /* doc_offsets not 0 < ... < S terminated by S      */
  CP_ERR_TIMEOUT = -8,      /* a bounded device wait ran out; outputs invalid   */
  CP_ERR_DEVICE = -9,       /* current device is not an sm_103 GPU              */
  CP_ERR_SCRATCH = -10      /* problem too large for the fixed scratch of       */
                            /* cp_ring_attn_fwd_noalloc (more than 65,535 docs) */
};

/*
 * Fused ring-attention forward, bf16 inputs and output, fp32 accumulation.
 * ("Context Parallelism", 線上 Softmax algorithm, run for every rank i with
 * the causal skip of 因果掩碼的特殊處理; log-sum-exp in natural log.)
 *
 *  q, k, v   device, bf16 [B,S,H,d], read only.
 *  out       device, bf16 [B,S,H,d], written: softmax(q k^T/sqrt(d)) v.
 *  lse       device, fp32 [B,H,S], written: log sum_k exp(q.k/sqrt(d)).
 *  B,S,H     >= 1; S < 2^31; n_shards in [1, S], S % n_shards == 0.
 *  d         64 or 128.
 *  causal    0 or 1.
 *  doc_offsets  NULL or device int32 (see Masks).
 *  stream    CUDA stream (0 = legacy default stream).
 * Runs on tcgen05 tensor cores; K/V tiles of each shard are streamed by TMA
 * into a double-buffered shared-memory ring.  The result does not depend on
 * n_shards beyond floating-point rounding.
 */
cp_status cp_ring_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                           int B, int S, int H, int d, int n_shards, int causal,
                           const int32_t* doc_offsets, cudaStream_t stream);

/*
 * One virtual rank's part of cp_ring_attn_fwd: rank i's whole ring ("上下文並行
 * （Context Parallelism, CP）", section 線上 Softmax: GPU i runs the loop over
 * the K/V shards for its own Q_i).  Writes out rows and lse entries of query
 * shard `rank` only ([rank*S/N, (rank+1)*S/N) of every batch row and head);
 * reads Q of that shard and K/V of the shards it needs (under causality,
 * shards 0..rank).  Pointers, layouts, masks and errors as cp_ring_attn_fwd;
 * rank outside [0, n_shards) returns CP_ERR_SHAPE.  The N calls for
 * rank = 0..N-1 give bitwise the result of one cp_ring_attn_fwd call, so a
 * caller can move shard i's inputs in and its output out while other ranks
 * compute.
 */
cp_status cp_ring_attn_fwd_rank(const void* q, const void* k, const void* v, void* out, float* lse,
                                int B, int S, int H, int d, int n_shards, int rank, int causal,
                                const int32_t* doc_offsets, cudaStream_t stream);

/*
 * cp_ring_attn_fwd for callers that cannot let a library allocate device
 * memory.  The pages have no counterpart: this is a deployment variant of the
 * fused forward above, with the same arguments, layouts and result.
 *
 * cp_ring_attn_fwd allocates its small per-device scratch (stream-ordered
 * cudaMallocAsync) the first time a call passes doc_offsets and whenever a call
 * needs more than it holds.  Processes that give nearly all GPU memory to their
 * own pool at start-up and forbid later cudaMalloc/cudaMallocAsync, and loops
 * that must never enter the driver's allocator, call this entry point instead:
 * it allocates nothing and keeps its scratch in a fixed device array built into
 * the library (295,168 bytes per GPU that loads the library, held until the
 * process exits).  It deals the work in the same cost-ranked order.
 *
 * Limit: doc_offsets may describe at most 65,535 documents.  A larger array
 * is rejected on the device: nothing is written, and cp_get_last_status
 * reports CP_ERR_SCRATCH.  A malformed one is rejected the same way with
 * CP_ERR_DOC_OFFSETS.  Host-side checks are those of cp_ring_attn_fwd.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  The address is cached for the process's life:
 * do not use the library across cudaDeviceReset.  All calls share the array
 * and it keeps the last call's contents; every call rewrites what it reads,
 * so nothing needs clearing.  Calls whose GPU work can overlap (unordered
 * streams) race on the array and must not be issued.
 */
cp_status cp_ring_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out,
                                   float* lse, int B, int S, int H, int d, int n_shards,
                                   int causal, const int32_t* doc_offsets, cudaStream_t stream);

/*
 * cp_ring_attn_fwd end to end from HOST buffers ("上下文並行（Context
 * Parallelism, CP）", section 線上 Softmax: a GPU computes on the block it holds
 * while the next one is sent and received, asynchronously and side by side;
 * section 因果掩碼的特殊處理: under causality rank i needs only shards 0..i).
 * Shard i's Q, K, V are copied to the device on a copy stream of the
 * library's, rank i starts once the shards it reads have landed (0..i when
 * causal, all of them otherwise), and its rows of out and lse are copied back
 * on a second copy stream while later ranks compute.  The result equals
 * cp_ring_attn_fwd's bit for bit.
 *
 *  q_host, k_host, v_host  host, bf16 [B,S,H,d], read.
 *  out_host   host, bf16 [B,S,H,d], written.
 *  lse_host   host, fp32 [B,H,S], written.
 *             Host buffers should be page-locked (cudaHostAlloc /
 *             cudaHostRegister) for the copies to overlap the kernels;
 *             pageable memory gives the same result with serialised copies.
 *  doc_offsets  NULL or DEVICE int32, as for cp_ring_attn_fwd.
 *  workspace  device, >= cp_ring_attn_fwd_host_workspace_bytes(B, S, H, d,
 *             n_shards, 2) bytes, 256-byte aligned, owned by the caller: the
 *             device copies of q, k, v, out and lse (its layout is private;
 *             contents undefined after the call).
 *  stream     the caller's stream.  The call is asynchronous: it returns
 *             once everything is enqueued, and `stream` then waits for the
 *             last copy back, so after synchronising `stream` the host
 *             outputs are complete.  The host inputs must stay unchanged and
 *             the host outputs unread until then.
 *  Shapes, masks, d and errors as cp_ring_attn_fwd; workspace too small:
 *  CP_ERR_BUFFER.  With doc_offsets the call uses the cached scratch that
 *  cp_ring_attn_fwd uses.  The copy streams and their events are created on
 *  the first call on each device and kept; a per-device lock is held while a
 *  call enqueues, so concurrent host threads take turns.
 */
int64_t cp_ring_attn_fwd_host_workspace_bytes(int B, int S, int H, int d, int n_shards,
                                              int elem_bytes /* 2 bf16, 4 fp32 */);
cp_status cp_ring_attn_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                                void* out_host, float* lse_host, int B, int S, int H, int d,
                                int n_shards, int causal, const int32_t* doc_offsets,
                                void* workspace, int64_t workspace_bytes, cudaStream_t stream);
/* The same with fp32 host buffers and the fp32 path (d in [1, 128];
 * workspace from cp_ring_attn_fwd_host_workspace_bytes(..., 4)). */
cp_status cp_ring_attn_fwd_host_f32(const float* q_host, const float* k_host,
                                    const float* v_host, float* out_host, float* lse_host, int B,
                                    int S, int H, int d, int n_shards, int causal,
                                    const int32_t* doc_offsets, void* workspace,
                                    int64_t workspace_bytes, cudaStream_t stream);

/* Same operation in true fp32 (CUDA-core FFMA, no TF32): q, k, v, out are
 * float [B,S,H,d]; d in [1, 128]; 4-byte alignment suffices. */
cp_status cp_ring_attn_fwd_f32(const float* q, const float* k, const float* v, float* out,
                               float* lse, int B, int S, int H, int d, int n_shards, int causal,
                               const int32_t* doc_offsets, cudaStream_t stream);

/*
 * One partial-attention step for the shard pair (i, j) ("Context
 * Parallelism", 線上 Softmax algorithm, the body of the j loop before the
 * merge): S_ij = Q_i K_j^T / sqrt(d) with the causal/document mask,
 * m_ij = rowmax(S_ij), P_ij = exp(S_ij - m_ij), l_ij = rowsum(P_ij),
 * O_ij = P_ij V_j (unnormalised).
 *
 *  q, k, v   device bf16 [B,S,H,d] (the whole sequence; the call reads
 *            Q rows of shard i and K/V rows of shard j only).
 *  o_part    device fp32 [B,S/N,H,d], written.
 *  m_part    device fp32 [B,H,S/N], written (natural-log units).
 *  l_part    device fp32 [B,H,S/N], written.
 *  i, j      0 <= i, j < n_shards.
 * Rows of Q_i that see no key of shard j get m = -inf, l = 0, O = 0.
 */
cp_status cp_ring_step(const void* q, const void* k, const void* v, float* o_part,
                       float* m_part, float* l_part, int B, int S, int H, int d, int n_shards,
                       int i, int j, int causal, const int32_t* doc_offsets,
                       cudaStream_t stream);

/* cp_ring_step with fp32 q, k, v (CUDA-core FFMA); d in [1, 128]. */
cp_status cp_ring_step_f32(const float* q, const float* k, const float* v, float* o_part,
                           float* m_part, float* l_part, int B, int S, int H, int d,
                           int n_shards, int i, int j, int causal,
                           const int32_t* doc_offsets, cudaStream_t stream);

/*
 * Online-softmax merge of a partial into a running state, in place
 * ("Context Parallelism", 線上 Softmax algorithm, 線上合併 lines):
 *   m_new = max(m_acc, m_part)
 *   o_acc = o_acc * exp(m_acc - m_new) + o_part * exp(m_part - m_new)
 *   l_acc = l_acc * exp(m_acc - m_new) + l_part * exp(m_part - m_new)
 *   m_acc = m_new
 * A state with m = -inf is empty and contributes nothing (no (-inf)-(-inf)).
 *  o_acc, o_part  device fp32 [B,rows,H,d]; m_*, l_* device fp32 [B,H,rows].
 *  rows >= 1, d in [1, 128].  o_acc must not alias o_part.
 */
cp_status cp_lse_merge(float* o_acc, float* m_acc, float* l_acc, const float* o_part,
                       const float* m_part, const float* l_part, int B, int rows, int H, int d,
                       cudaStream_t stream);

/*
 * Final normalisation ("Context Parallelism", 線上 Softmax algorithm, last
 * line O_i = O_i / l_i) and the log-sum-exp m + log(l).
 *  out   device [B,rows,H,d]: bf16 if out_is_bf16, else fp32.
 *  lse   device fp32 [B,H,rows].
 * Rows with l = 0 (no visible key) get out = 0 and lse = -inf.
 */
cp_status cp_lse_finalize(const float* o_acc, const float* m_acc, const float* l_acc, void* out,
                          float* lse, int B, int rows, int H, int d, int out_is_bf16,
                          cudaStream_t stream);

/*
 * Host-only, integer: the skip schedule ("Context Parallelism",
 * 因果掩碼的特殊處理: steps with no causal dependency are skipped).
 * Each shard is cut into tiles from its first row (tile_q rows for queries,
 * tile_k for keys; a tile never crosses a shard boundary); tiles are numbered
 * in order across shards.  A (q tile, kv tile) pair is listed iff at least
 * one of its (q, k) is visible.  Pairs are ordered by q tile, then by kv tile
 * ascending (the ascending ring order).  With tile_q = tile_k = S/N the list
 * is the shard-pair schedule, N(N+1)/2 pairs when causal without documents.
 *  doc_offsets_host  NULL or HOST int32 (same format as on the device).
 *  pairs_out  host int32 [2*max_pairs] or NULL (count only).
 *  n_pairs    host, written: the number of pairs.
 * Returns CP_ERR_BUFFER (after writing max_pairs pairs and *n_pairs) when
 * the list does not fit.
 */
cp_status cp_ring_schedule(int S, int n_shards, int tile_q, int tile_k, int causal,
                           const int32_t* doc_offsets_host, int32_t* pairs_out, int64_t max_pairs,
                           int64_t* n_pairs);

/*
 * Diagnostic: the tile schedule the fused bf16 / FP8 kernels actually walk,
 * computed on the device by the kernels' own work decoding.  For every
 * 128-row query tile in flat order (tile a of shard i is i * ceil(L/128) + a,
 * L = S / n_shards) it writes the first and the last flat 128-row key tile of
 * its contiguous key-tile range, which must equal the range of the pairs
 * cp_ring_schedule(S, n_shards, 128, 128, causal, ...) lists for that tile.
 * No counterpart on the pages beyond section 因果掩碼的特殊處理 (which pairs
 * are needed); it exists so tests can check the device schedule.
 *  doc_offsets  NULL or device int32 (as cp_ring_attn_fwd).
 *  ranges       device int32 [n_shards * ceil(L/128) * 2], written.
 * With doc_offsets it uses the library's cached per-device scratch.
 */
cp_status cp_ring_schedule_device(int S, int n_shards, int causal, const int32_t* doc_offsets,
                                  int32_t* ranges, cudaStream_t stream);

/*
 * Host-only, integer: bytes each virtual rank would send plus receive if the
 * K/V blocks travelled a real ring ("大语言模型并行策略（五）：上下文并行",
 * 通信模式: 2 x (G/N) x (N-1), G = K and V bytes of the whole sequence,
 * G = 2*B*S*H*d*dtype_bytes).  With causal != 0, a block of shard s is only
 * forwarded to ranks r > s, so rank i receives i blocks and sends i+1
 * (none for the last rank).
 *  per_rank_bytes  host int64 [n_shards], written.
 */
cp_status cp_ring_traffic(int64_t B, int64_t S, int64_t H, int64_t d, int dtype_bytes,
                          int n_shards, int causal, int64_t* per_rank_bytes);

/*
 * Synchronise `stream`, then read and clear the sticky device error word of
 * the current device: CP_OK, CP_ERR_DOC_OFFSETS, CP_ERR_TIMEOUT or
 * CP_ERR_SCRATCH (the lowest code wins when several were raised);
 * CP_ERR_CUDA if the synchronisation itself failed.
 */
cp_status cp_get_last_status(cudaStream_t stream);

/* A static, human-readable name for a status code. */
const char* cp_status_string(cp_status status);

/*
 * The ring with explicit per-rank buffers ("上下文並行（Context Parallelism,
 * CP）", 線上 Softmax: compute against the held K/V block, then pass it to the
 * next GPU; "大语言模型并行策略（五）：上下文并行", 通信模式: double-buffered so
 * the transfer overlaps the computation; 因果掩碼的特殊處理: under causality a
 * block goes only to the ranks that need it).  Every virtual rank owns a
 * two-slot K/V receive buffer in `workspace`; at step t rank i holds the block
 * of rank (i - t) mod N, runs cp_ring_step on it and merges the partial, while
 * the copy engine moves each held block into the next rank's other slot for
 * step t + 1.  Same arguments and result as cp_ring_attn_fwd (bf16, d 64 or
 * 128; doc_offsets NULL or device int32, every step masking by document, the
 * doc-scan word in the library's cached scratch), plus:
 *  workspace        device, >= cp_ring_emulated_workspace_bytes(...) bytes,
 *                   256-byte aligned; owned by the caller; contents undefined
 *                   after the call.
 *  stream           compute stream.
 *  copy_stream      stream for the block transfers; NULL runs them in order
 *                   on `stream` (no overlap).  The call leaves `stream`
 *                   waiting for every transfer it issued.
 *  recv_bytes_per_rank  host int64 [n_shards] or NULL: bytes each rank
 *                   received from its predecessor (K and V).
 */
int64_t cp_ring_emulated_workspace_bytes(int B, int S, int H, int d, int n_shards);
cp_status cp_ring_attn_fwd_emulated(const void* q, const void* k, const void* v, void* out,
                                    float* lse, int B, int S, int H, int d, int n_shards,
                                    int causal, const int32_t* doc_offsets, void* workspace,
                                    int64_t workspace_bytes,
                                    cudaStream_t stream, cudaStream_t copy_stream,
                                    int64_t* recv_bytes_per_rank);

/*
 * The all-to-all form of context parallelism ("上下文並行（Context
 * Parallelism, CP）", 方案二 All-to-All (DeepSpeed Ulysses)): an all-to-all
 * turns the sequence-split Q/K/V into head-split ones, every rank attends
 * over the whole sequence for its H/N heads, and an all-to-all turns the
 * output back.  On one GPU both all-to-alls are layout permutations run by a
 * bandwidth-bound kernel; the attention is the fused kernel.  Same arguments
 * and result as cp_ring_attn_fwd (bf16, d 64 or 128, doc_offsets allowed),
 * with H % n_shards == 0, plus:
 *  workspace  device, >= cp_ulysses_workspace_bytes(...) bytes, 256-byte
 *             aligned, owned by the caller, contents undefined afterwards.
 *  a2a_bytes  host int64 or NULL: bytes the two all-to-alls would move,
 *             sent plus received, summed over the ranks (8 * shard bytes *
 *             (N - 1) with shard = B*(S/N)*H*d*2).
 */
int64_t cp_ulysses_workspace_bytes(int B, int S, int H, int d, int n_shards);
cp_status cp_ulysses_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                              int B, int S, int H, int d, int n_shards, int causal,
                              const int32_t* doc_offsets, void* workspace,
                              int64_t workspace_bytes, cudaStream_t stream, int64_t* a2a_bytes);

/*
 * TEST HOOK (failure detection without a GPU fault).  With drop_first_k_tile
 * != 0, the next tensor-core launches have CTA 0 skip loading its first K
 * tile, so one of its bounded device waits runs out: the CTA drains its own
 * copies and MMAs, frees TMEM, leaves its outputs unwritten and raises
 * CP_ERR_TIMEOUT in the device error word.  wait_limit_ns sets the per-wait
 * limit of later launches (<= 0 restores the default of 4 s).  Call with
 * (0, 0) to return to normal operation.  Not thread-safe; for tests only.
 */
void cp_test_set_wait_fault(int drop_first_k_tile, long long wait_limit_ns);

/* Number of tcgen05 kernel launches, fp32 kernel launches, auxiliary
 * launches (merge, finalize, all-to-all permutation, FP8 quantisation) and
 * doc-scan launches made by this process so far (host-side counters, for
 * launch accounting in benchmarks). */
void cp_launch_counts(int64_t* counts4);

/*
 * Ring-attention backward: the gradients of L = sum(out * dout) with respect
 * to q, k and v, for the forward of cp_ring_attn_fwd (same masks, sharding
 * and tiling).  "上下文並行（Context Parallelism, CP）" (compassingai.com),
 * section 反向傳播: the backward walks the ring's K/V blocks again; the
 * gradients of K_j, V_j travel with them ("大语言模型并行策略（五）：上下文并行").
 * Per (b, h), with P recomputed from the saved lse:
 *   D = rowsum(dout * out);  dP = dout v^T;  dS = P * (dP - D);
 *   dv = P^T dout;  dk = dS^T q / sqrt(d);  dq = dS k / sqrt(d).
 *  q, k, v, out, dout   device, bf16 [B,S,H,d], read only (out, lse from the
 *                       forward on the same inputs).
 *  lse        device, fp32 [B,H,S], read only.
 *  dq, dk, dv device, bf16 [B,S,H,d], written.
 *  workspace  device, >= cp_ring_attn_bwd_workspace_bytes(...) bytes,
 *             256-byte aligned, caller-owned scratch (D and the doc-scan
 *             word); nothing is allocated.
 *  Shapes, masks, d, alignment and errors as cp_ring_attn_fwd; a workspace
 *  too small returns CP_ERR_BUFFER.
 * Three launches (with doc_offsets, four: the doc scan first): D and the
 * dK/dV kernel (one CTA per 128-key tile) on `stream`, and the dQ kernel (one
 * CTA per 128-query tile), which reads nothing the dK/dV kernel writes, on a
 * second stream owned by the library (one per device, kept for the
 * process's life) after D; `stream` then waits for it, so work enqueued
 * later on `stream` sees every gradient.  Both kernels run on tcgen05 with
 * fp32 accumulation and bf16 P / dS operands.
 */
int64_t cp_ring_attn_bwd_workspace_bytes(int B, int S, int H, int d, int n_shards);
cp_status cp_ring_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                           const float* lse, const void* dout, void* dq, void* dk, void* dv,
                           int B, int S, int H, int d, int n_shards, int causal,
                           const int32_t* doc_offsets, void* workspace, int64_t workspace_bytes,
                           cudaStream_t stream);

/*
 * FP8 (E4M3) quantisation of one bf16 tensor, per (b, h).
 * "上下文並行（Context Parallelism, CP）" (compassingai.com), section
 * 通訊量分析: the bytes moved depend on whether K/V travel in FP8.  Format:
 * OCP E4M3 (largest finite 448), one fp32 scale per (b, h):
 *   amax = max |x| over (S, d);  inv = 448 / amax;  x8 = E4M3(x * inv)
 *   (each an fp32 operation rounded to nearest, then rounded to the nearest
 *   E4M3 value, ties to even, saturated at +-448);  descale = amax / 448;
 *   an all-zero head gets inv = descale = 1.
 *  x          device, bf16 [B,S,H,d], read only (finite values).
 *  x8         device, bytes: [B,S,H,d] if transpose == 0 (Q, K), or
 *             [B,H,d,S] if transpose == 1 (V^T for cp_ring_attn_fwd_fp8).
 *  descale    device, fp32 [B,H], written (used as scratch during the call).
 *  B, H       1 .. 65535; S >= 1 (transpose: S % 16 == 0); d 64 or 128.
 *  Alignment  x, x8 16 bytes; descale 4 bytes.
 * Four launches on `stream` (a memset and three kernels); no allocation.
 */
cp_status cp_fp8_quantize(const void* x, void* x8, float* descale, int B, int S, int H, int d,
                          int transpose, cudaStream_t stream);

/*
 * Fused ring-attention forward over FP8 inputs.  Same computation, masks,
 * sharding and outputs as cp_ring_attn_fwd, applied to the dequantized
 * inputs q8 * q_descale, k8 * k_descale, v8 * v_descale ("上下文並行", section
 * 線上 Softmax; FP8 transfer per section 通訊量分析).
 *  q8, k8     device, E4M3 [B,S,H,d] (cp_fp8_quantize, transpose 0).
 *  v8t        device, E4M3 [B,H,d,S] (cp_fp8_quantize, transpose 1).
 *  q_descale, k_descale, v_descale   device, fp32 [B,H].
 *  out        device, bf16 [B,S,H,d];  lse  device, fp32 [B,H,S].
 *  d          128 only (others: CP_ERR_UNSUPPORTED).
 *  Shapes     as cp_ring_attn_fwd, and (S / n_shards) % 16 == 0 so that every
 *             K/V tile starts on a 16-byte boundary of v8t (else CP_ERR_SHAPE).
 *  Alignment  q8, k8, v8t, out 16 bytes; descales, lse, doc_offsets 4 bytes.
 * Both products run on tcgen05 as kind::f8f6f4 with fp32 accumulation; P is
 * rounded to E4M3 before the PV product (relative error <= 2^-4 per entry),
 * so the result differs from the exact attention of the dequantized inputs
 * by up to about 2^-4 max|v| (peaked rows come closest).
 */
cp_status cp_ring_attn_fwd_fp8(const void* q8, const void* k8, const void* v8t,
                               const float* q_descale, const float* k_descale,
                               const float* v_descale, void* out, float* lse, int B, int S, int H,
                               int d, int n_shards, int causal, const int32_t* doc_offsets,
                               cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CPRING_H */
