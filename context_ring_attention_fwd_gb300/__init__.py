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
    cp_ring_attn_fwd_rank,
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


_COPY_STREAMS = {}


def _copy_streams(device):
    """Two streams per device for host <-> device copies (one per direction)."""
    key = torch.device(device).index if torch.device(device).index is not None else \
        torch.cuda.current_device()
    if key not in _COPY_STREAMS:
        _COPY_STREAMS[key] = (torch.cuda.Stream(device=key), torch.cuda.Stream(device=key))
    return _COPY_STREAMS[key]


def ring_attn_fwd_host(q_host: torch.Tensor, k_host: torch.Tensor, v_host: torch.Tensor,
                       n_shards: int = 1, causal: bool = True, doc_offsets=None,
                       device: str = "cuda", buffers=None, stream=None):
    """End-to-end call from host tensors: copy Q/K/V to the device, run the
    fused forward, copy out and lse back.  `buffers` may hold reusable
    (q, k, v, out, lse, out_host, lse_host) tensors.  Returns the host
    (out, lse).

    bf16 runs rank by rank (cp_ring_attn_fwd_rank): shard i's Q/K/V go in on a
    copy stream, rank i starts once the shards it reads have landed (0..i
    under causality, all shards otherwise), and its rows of out come back on
    a second copy stream while later ranks compute.  The result is bitwise
    that of one cp_ring_attn_fwd call."""
    B, S, H, d = q_host.shape
    if buffers is None:
        dq = torch.empty(q_host.shape, dtype=q_host.dtype, device=device)
        dk = torch.empty_like(dq)
        dv = torch.empty_like(dq)
        dout = torch.empty_like(dq)
        dlse = torch.empty((B, H, S), dtype=torch.float32, device=device)
        hout = torch.empty(q_host.shape, dtype=q_host.dtype, pin_memory=True)
        hlse = torch.empty((B, H, S), dtype=torch.float32, pin_memory=True)
    else:
        dq, dk, dv, dout, dlse, hout, hlse = buffers
    docs = doc_offsets_tensor(doc_offsets, dq.device)
    compute = stream if stream is not None else torch.cuda.current_stream(dq.device)
    if dq.dtype != torch.bfloat16:
        with torch.cuda.stream(compute):
            dq.copy_(q_host, non_blocking=True)
            dk.copy_(k_host, non_blocking=True)
            dv.copy_(v_host, non_blocking=True)
            cp_ring_attn_fwd_f32(dq, dk, dv, dout, dlse, n_shards, causal, docs, compute)
            hout.copy_(dout, non_blocking=True)
            hlse.copy_(dlse, non_blocking=True)
        compute.synchronize()
        return hout, hlse
    N = int(n_shards)
    L = S // N
    h2d, d2h = _copy_streams(dq.device)
    landed = []
    h2d.wait_stream(compute)          # the device buffers are free to overwrite
    with torch.cuda.stream(h2d):
        for i in range(N):
            for b in range(B):
                rows = slice(i * L, (i + 1) * L)
                dq[b, rows].copy_(q_host[b, rows], non_blocking=True)
                dk[b, rows].copy_(k_host[b, rows], non_blocking=True)
                dv[b, rows].copy_(v_host[b, rows], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(h2d)
            landed.append(ev)
    d2h.wait_stream(compute)          # the host output buffers are free
    for i in range(N):
        compute.wait_event(landed[i if causal else N - 1])
        cp_ring_attn_fwd_rank(dq, dk, dv, dout, dlse, N, i, causal, docs, compute)
        done = torch.cuda.Event()
        done.record(compute)
        d2h.wait_event(done)
        with torch.cuda.stream(d2h):
            for b in range(B):
                rows = slice(i * L, (i + 1) * L)
                hout[b, rows].copy_(dout[b, rows], non_blocking=True)
    with torch.cuda.stream(d2h):
        hlse.copy_(dlse, non_blocking=True)
    d2h.synchronize()
    compute.wait_stream(d2h)
    compute.synchronize()
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
