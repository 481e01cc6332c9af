"""GB300-native context-parallel ring-attention forward.

The sequence is cut into N contiguous shards; each query shard visits the
K/V shards in ring order, computes a partial attention against each and
folds it into a running (O, m, l) with the online-softmax merge, skipping
causally dead steps; the output is O / l with its log-sum-exp ("上下文並行
（Context Parallelism, CP）", compassingai.com, section 線上 Softmax).  All N
virtual ranks run on one GPU.

Every step runs in libcpring.so (hand-written sm_103a CUDA behind a C ABI);
this package only marshals arguments.  The library is loaded lazily and its
absence raises - there is no fallback path.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from ._binding import (  # noqa: F401
    CP_OK, STATUS_CODES, STATUS_NAMES, CpError, LIB_PATH, cp_fp8_quantize, cp_get_last_status,
    cp_ring_attn_fwd_rank, cp_ring_attn_fwd_host, cp_ring_attn_fwd_host_workspace_bytes,
    cp_ring_attn_fwd_noalloc,
    cp_lse_finalize, cp_lse_merge, cp_ring_attn_bwd, cp_ring_attn_bwd_workspace_bytes,
    cp_ring_attn_fwd, cp_ring_attn_fwd_emulated,
    cp_ring_attn_fwd_f32, cp_ring_attn_fwd_fp8,
    cp_ring_emulated_workspace_bytes, cp_ring_schedule, cp_ring_schedule_device, cp_ring_step,
    cp_ulysses_attn_fwd,
    cp_ulysses_workspace_bytes,
    cp_ring_traffic, cp_status_string, doc_offsets_tensor, launch_counts, lib,
    test_set_wait_fault)

__all__ = [
    "cp_ring_attn_fwd", "cp_ring_attn_fwd_f32", "cp_ring_step", "cp_lse_merge",
    "cp_lse_finalize", "cp_ring_schedule", "cp_ring_traffic", "cp_get_last_status",
    "cp_status_string", "ring_attn_fwd", "ring_attn_fwd_host", "ring_attn_composed",
    "cp_ring_attn_fwd_host", "cp_ring_attn_fwd_noalloc",
    "cp_fp8_quantize", "cp_ring_attn_fwd_fp8", "fp8_quantize_qkv", "ring_attn_fwd_fp8",
    "cp_ring_attn_bwd", "ring_attn_bwd",
    "CpError", "lib",
]


def ring_attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, n_shards: int = 1,
                  causal: bool = True, doc_offsets=None, stream=None):
    """Allocate out [B,S,H,d] (q's dtype) and lse [B,H,S] fp32 on q's device
    and run the fused forward (bf16 on tensor cores, fp32 on CUDA cores)."""
    B, S, H, d = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    docs = doc_offsets_tensor(doc_offsets, q.device)
    if q.dtype == torch.bfloat16:
        cp_ring_attn_fwd(q, k, v, out, lse, n_shards, causal, docs, stream)
    elif q.dtype == torch.float32:
        cp_ring_attn_fwd_f32(q, k, v, out, lse, n_shards, causal, docs, stream)
    else:
        raise TypeError("q must be bf16 or fp32")
    return out, lse


def ring_attn_fwd_host(q_host: torch.Tensor, k_host: torch.Tensor, v_host: torch.Tensor,
                       n_shards: int = 1, causal: bool = True, doc_offsets=None,
                       device: str = "cuda", buffers=None, stream=None):
    """End-to-end call from host tensors through cp_ring_attn_fwd_host (the
    library copies Q/K/V in shard by shard, runs rank by rank and copies out
    and lse back while later ranks compute).  `buffers` may hold a reusable
    (workspace, out_host, lse_host); otherwise they are allocated here (the
    host ones page-locked).  Waits for the stream and returns the host
    (out, lse)."""
    B, S, H, d = q_host.shape
    esz = 2 if q_host.dtype == torch.bfloat16 else 4
    dev = torch.device(device)
    if buffers is None:
        need = cp_ring_attn_fwd_host_workspace_bytes(B, S, H, d, int(n_shards), esz)
        if need < 0:
            raise CpError("cp_ring_attn_fwd_host_workspace_bytes", STATUS_CODES["CP_ERR_SHAPE"])
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        hout = torch.empty(q_host.shape, dtype=q_host.dtype, pin_memory=True)
        hlse = torch.empty((B, H, S), dtype=torch.float32, pin_memory=True)
    else:
        ws, hout, hlse = buffers
    docs = doc_offsets_tensor(doc_offsets, ws.device)
    st = stream if stream is not None else torch.cuda.current_stream(ws.device)
    cp_ring_attn_fwd_host(q_host, k_host, v_host, hout, hlse, n_shards, causal, docs, ws, st)
    st.synchronize()
    return hout, hlse


def ring_attn_composed(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, n_shards: int,
                       causal: bool = True, doc_offsets=None,
                       order: str | Sequence[int] | None = "ascending", skip_masked: bool = True,
                       stream=None):
    """The ring walk spelled out as separate launches, one virtual rank at a
    time: for rank i, for each shard j in the visiting order, cp_ring_step(i, j)
    then cp_lse_merge into rank i's running state; finally cp_lse_finalize.
    `order` is "ascending" (j = 0..N-1), "ring" (j = (i - t) mod N at step t)
    or an explicit permutation.  With skip_masked the causally dead pairs
    (j > i, no documents) are not launched.  Returns out (q's dtype) and lse."""
    B, S, H, d = q.shape
    N = int(n_shards)
    L = S // N
    dev = q.device
    docs = doc_offsets_tensor(doc_offsets, dev)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    o_acc = torch.empty((B, L, H, d), dtype=torch.float32, device=dev)
    m_acc = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    l_acc = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    o_p = torch.empty_like(o_acc)
    m_p = torch.empty_like(m_acc)
    l_p = torch.empty_like(l_acc)
    o_fin = torch.empty((B, L, H, d), dtype=q.dtype, device=dev)
    lse_fin = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    for i in range(N):
        if order == "ascending" or order is None:
            js = list(range(N))
        elif order == "ring":
            js = [(i - t) % N for t in range(N)]
        else:
            js = [int(x) for x in order]
        first = True
        for j in js:
            if skip_masked and causal and doc_offsets is None and j > i:
                continue
            if first:  # the first visited step initialises the running state
                cp_ring_step(q, k, v, o_acc, m_acc, l_acc, N, i, j, causal, docs, stream)
                first = False
                continue
            cp_ring_step(q, k, v, o_p, m_p, l_p, N, i, j, causal, docs, stream)
            cp_lse_merge(o_acc, m_acc, l_acc, o_p, m_p, l_p, stream)
        cp_lse_finalize(o_acc, m_acc, l_acc, o_fin, lse_fin, stream)
        out[:, i * L:(i + 1) * L].copy_(o_fin)
        lse[:, :, i * L:(i + 1) * L].copy_(lse_fin)
    return out, lse


def fp8_quantize_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, stream=None):
    """E4M3 storage of bf16 Q, K, V [B,S,H,d]: returns (q8, k8, v8t, q_descale,
    k_descale, v_descale) with q8, k8 [B,S,H,d], v8t [B,H,d,S] (uint8) and the
    descales [B,H] fp32."""
    B, S, H, d = q.shape
    dev = q.device
    q8 = torch.empty((B, S, H, d), dtype=torch.uint8, device=dev)
    k8 = torch.empty_like(q8)
    v8t = torch.empty((B, H, d, S), dtype=torch.uint8, device=dev)
    desc = [torch.empty((B, H), dtype=torch.float32, device=dev) for _ in range(3)]
    cp_fp8_quantize(q, q8, desc[0], False, stream)
    cp_fp8_quantize(k, k8, desc[1], False, stream)
    cp_fp8_quantize(v, v8t, desc[2], True, stream)
    return q8, k8, v8t, desc[0], desc[1], desc[2]


def ring_attn_fwd_fp8(fp8_inputs, n_shards: int = 1, causal: bool = True, doc_offsets=None,
                      stream=None):
    """The FP8 fused forward on the output of fp8_quantize_qkv; allocates and
    returns (out [B,S,H,d] bf16, lse [B,H,S] fp32)."""
    q8, k8, v8t, qd, kd, vd = fp8_inputs
    B, S, H, d = q8.shape
    out = torch.empty((B, S, H, d), dtype=torch.bfloat16, device=q8.device)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q8.device)
    docs = doc_offsets_tensor(doc_offsets, q8.device)
    cp_ring_attn_fwd_fp8(q8, k8, v8t, qd, kd, vd, out, lse, n_shards, causal, docs, stream)
    return out, lse


def ring_attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
                  lse: torch.Tensor, dout: torch.Tensor, n_shards: int = 1, causal: bool = True,
                  doc_offsets=None, stream=None):
    """The bf16 backward for the forward's (out, lse): allocates and returns
    (dq, dk, dv) [B,S,H,d] bf16."""
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    docs = doc_offsets_tensor(doc_offsets, q.device)
    cp_ring_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, n_shards, causal, docs, None, stream)
    return dq, dk, dv
