"""ctypes binding of libcpring.so: argument marshalling only.

Every computation runs in the library's CUDA kernels; torch supplies device
memory and streams.  If the library is missing the calls raise instead of
falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libcpring.so")

CP_OK = 0
STATUS_NAMES = {
    0: "CP_OK", -1: "CP_ERR_NULL", -2: "CP_ERR_SHAPE", -3: "CP_ERR_UNSUPPORTED",
    -4: "CP_ERR_ALIGN", -5: "CP_ERR_CUDA", -6: "CP_ERR_BUFFER", -7: "CP_ERR_DOC_OFFSETS",
    -8: "CP_ERR_TIMEOUT", -9: "CP_ERR_DEVICE", -10: "CP_ERR_SCRATCH",
}
STATUS_CODES = {v: k for k, v in STATUS_NAMES.items()}

_lib = None
_lock = threading.Lock()

_vp, _i, _i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
_SIGS = {
    "cp_ring_attn_fwd": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp],
    "cp_ring_attn_fwd_noalloc": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp],
    "cp_ring_attn_fwd_rank": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp],
    "cp_ring_attn_fwd_f32": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp],
    "cp_ring_step": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _vp, _vp],
    "cp_ring_step_f32": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _vp, _vp],
    "cp_lse_merge": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp],
    "cp_lse_finalize": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp],
    "cp_ring_schedule": [_i, _i, _i, _i, _i, _vp, _vp, _i64, ctypes.POINTER(_i64)],
    "cp_ring_traffic": [_i64, _i64, _i64, _i64, _i, _i, _i, ctypes.POINTER(_i64)],
    "cp_get_last_status": [_vp],
    "cp_status_string": [_i],
    "cp_launch_counts": [ctypes.POINTER(_i64)],
    "cp_test_set_wait_fault": [_i, _i64],
    "cp_ring_emulated_workspace_bytes": [_i, _i, _i, _i, _i],
    "cp_ulysses_workspace_bytes": [_i, _i, _i, _i, _i],
    "cp_ulysses_attn_fwd": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _i64, _vp,
                            ctypes.POINTER(_i64)],
    "cp_ring_attn_fwd_emulated": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp,
                                  _i64, _vp, _vp, ctypes.POINTER(_i64)],
    "cp_fp8_quantize": [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp],
    "cp_ring_attn_bwd_workspace_bytes": [_i, _i, _i, _i, _i],
    "cp_ring_schedule_device": [_i, _i, _i, _vp, _vp, _vp],
    "cp_ring_attn_bwd": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp,
                         _vp, _i64, _vp],
    "cp_ring_attn_fwd_fp8": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp,
                             _vp],
    "cp_ring_attn_fwd_host_workspace_bytes": [_i, _i, _i, _i, _i, _i],
    "cp_ring_attn_fwd_host": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _i64,
                              _vp],
    "cp_ring_attn_fwd_host_f32": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp,
                                  _i64, _vp],
}


class CpError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{fn} failed: {self.name} ({status})")


def lib() -> ctypes.CDLL:
    """The loaded library (loaded once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            handle = ctypes.CDLL(LIB_PATH)
            for name, argtypes in _SIGS.items():
                fn = getattr(handle, name)
                fn.argtypes = argtypes
                if name == "cp_status_string":
                    fn.restype = ctypes.c_char_p
                elif name in ("cp_launch_counts", "cp_test_set_wait_fault"):
                    fn.restype = None
                elif name in ("cp_ring_emulated_workspace_bytes", "cp_ulysses_workspace_bytes",
                              "cp_ring_attn_bwd_workspace_bytes",
                              "cp_ring_attn_fwd_host_workspace_bytes"):
                    fn.restype = _i64
                else:
                    fn.restype = _i
            _lib = handle
    return _lib


def _check(fn: str, st: int) -> None:
    if st != CP_OK:
        raise CpError(fn, st)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def doc_offsets_tensor(doc_offsets, device) -> Optional[torch.Tensor]:
    """doc_offsets (list, numpy array or tensor) as a device int32 tensor."""
    if doc_offsets is None:
        return None
    if isinstance(doc_offsets, torch.Tensor):
        t = doc_offsets.to(device=device, dtype=torch.int32)
    else:
        t = torch.tensor([int(x) for x in doc_offsets], dtype=torch.int32, device=device)
    return t.contiguous()


# --------------------------------------------------------------------- C ABI
def cp_ring_attn_fwd(q, k, v, out, lse, n_shards: int, causal: bool = True,
                     doc_offsets: Optional[torch.Tensor] = None, stream=None) -> None:
    """bf16 fused forward; q, k, v, out [B,S,H,d] bf16, lse [B,H,S] fp32."""
    B, S, H, d = q.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _need(t, n, torch.bfloat16, (B, S, H, d))
    _need(lse, "lse", torch.float32, (B, H, S))
    if doc_offsets is not None:
        _need(doc_offsets, "doc_offsets", torch.int32)
    _check("cp_ring_attn_fwd", lib().cp_ring_attn_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, S, H, d, int(n_shards),
        int(bool(causal)), _ptr(doc_offsets), _stream(stream)))


def cp_fp8_quantize(x, x8, descale, transpose: bool = False, stream=None) -> None:
    """Per-(b, h) E4M3 quantisation of x [B,S,H,d] bf16 into x8 (uint8,
    [B,S,H,d], or [B,H,d,S] with transpose) and descale [B,H] fp32."""
    B, S, H, d = x.shape
    _need(x, "x", torch.bfloat16)
    _need(x8, "x8", torch.uint8, (B, H, d, S) if transpose else (B, S, H, d))
    _need(descale, "descale", torch.float32, (B, H))
    _check("cp_fp8_quantize", lib().cp_fp8_quantize(
        _ptr(x), _ptr(x8), _ptr(descale), B, S, H, d, int(bool(transpose)), _stream(stream)))


def cp_ring_attn_fwd_fp8(q8, k8, v8t, q_descale, k_descale, v_descale, out, lse, n_shards: int,
                         causal: bool = True, doc_offsets: Optional[torch.Tensor] = None,
                         stream=None) -> None:
    """FP8 fused forward: q8, k8 uint8 E4M3 [B,S,H,d], v8t uint8 E4M3
    [B,H,d,S], descales fp32 [B,H]; out [B,S,H,d] bf16, lse [B,H,S] fp32."""
    B, S, H, d = q8.shape
    _need(q8, "q8", torch.uint8, (B, S, H, d))
    _need(k8, "k8", torch.uint8, (B, S, H, d))
    _need(v8t, "v8t", torch.uint8, (B, H, d, S))
    for t, n in ((q_descale, "q_descale"), (k_descale, "k_descale"), (v_descale, "v_descale")):
        _need(t, n, torch.float32, (B, H))
    _need(out, "out", torch.bfloat16, (B, S, H, d))
    _need(lse, "lse", torch.float32, (B, H, S))
    if doc_offsets is not None:
        _need(doc_offsets, "doc_offsets", torch.int32)
    _check("cp_ring_attn_fwd_fp8", lib().cp_ring_attn_fwd_fp8(
        _ptr(q8), _ptr(k8), _ptr(v8t), _ptr(q_descale), _ptr(k_descale), _ptr(v_descale),
        _ptr(out), _ptr(lse), B, S, H, d, int(n_shards), int(bool(causal)), _ptr(doc_offsets),
        _stream(stream)))


def cp_ring_attn_bwd_workspace_bytes(B: int, S: int, H: int, d: int, n_shards: int) -> int:
    return int(lib().cp_ring_attn_bwd_workspace_bytes(B, S, H, d, n_shards))


def cp_ring_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, n_shards: int, causal: bool = True,
                     doc_offsets: Optional[torch.Tensor] = None, workspace=None,
                     stream=None) -> None:
    """bf16 backward: q, k, v, out, dout, dq, dk, dv [B,S,H,d] bf16, lse
    [B,H,S] fp32; workspace a uint8 device tensor of at least
    cp_ring_attn_bwd_workspace_bytes bytes (allocated here if None)."""
    B, S, H, d = q.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"), (dq, "dq"),
                 (dk, "dk"), (dv, "dv")):
        _need(t, n, torch.bfloat16, (B, S, H, d))
    _need(lse, "lse", torch.float32, (B, H, S))
    if doc_offsets is not None:
        _need(doc_offsets, "doc_offsets", torch.int32)
    need = cp_ring_attn_bwd_workspace_bytes(B, S, H, d, int(n_shards))
    if need < 0:
        raise CpError("cp_ring_attn_bwd_workspace_bytes", STATUS_CODES["CP_ERR_SHAPE"])
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check("cp_ring_attn_bwd", lib().cp_ring_attn_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
        _ptr(dv), B, S, H, d, int(n_shards), int(bool(causal)), _ptr(doc_offsets),
        _ptr(workspace), int(workspace.numel()), _stream(stream)))


def cp_ring_attn_fwd_rank(q, k, v, out, lse, n_shards: int, rank: int, causal: bool = True,
                          doc_offsets: Optional[torch.Tensor] = None, stream=None) -> None:
    """Rank `rank`'s part of the bf16 fused forward (its query shard's rows of
    out and lse); the tensors are the whole-sequence ones."""
    B, S, H, d = q.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _need(t, n, torch.bfloat16, (B, S, H, d))
    _need(lse, "lse", torch.float32, (B, H, S))
    if doc_offsets is not None:
        _need(doc_offsets, "doc_offsets", torch.int32)
    _check("cp_ring_attn_fwd_rank", lib().cp_ring_attn_fwd_rank(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, S, H, d, int(n_shards), int(rank),
        int(bool(causal)), _ptr(doc_offsets), _stream(stream)))


def cp_ring_attn_fwd_host_workspace_bytes(B: int, S: int, H: int, d: int, n_shards: int,
                                          elem_bytes: int = 2) -> int:
    return int(lib().cp_ring_attn_fwd_host_workspace_bytes(B, S, H, d, n_shards, elem_bytes))


def _need_host(t: torch.Tensor, name: str, dtype: torch.dtype, shape) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.is_cuda:
        raise ValueError(f"{name} must live in host memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def cp_ring_attn_fwd_host(q_host, k_host, v_host, out_host, lse_host, n_shards: int,
                          causal: bool = True, doc_offsets: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """The fused forward from host tensors (bf16 or fp32 [B,S,H,d], lse fp32
    [B,H,S]; page-locked for overlap): asynchronous on `stream`, whose
    synchronisation completes out_host and lse_host.  workspace: a uint8
    device tensor of cp_ring_attn_fwd_host_workspace_bytes bytes."""
    B, S, H, d = q_host.shape
    dt = q_host.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise TypeError("q_host must be bf16 or fp32")
    for t, n in ((q_host, "q_host"), (k_host, "k_host"), (v_host, "v_host"),
                 (out_host, "out_host")):
        _need_host(t, n, dt, (B, S, H, d))
    _need_host(lse_host, "lse_host", torch.float32, (B, H, S))
    if doc_offsets is not None:
        _need(doc_offsets, "doc_offsets", torch.int32)
    if workspace is None:
        raise ValueError("workspace is required")
    _need(workspace, "workspace", torch.uint8)
    name = "cp_ring_attn_fwd_host" if dt == torch.bfloat16 else "cp_ring_attn_fwd_host_f32"
    _check(name, getattr(lib(), name)(
        _ptr(q_host), _ptr(k_host), _ptr(v_host), _ptr(out_host), _ptr(lse_host), B, S, H, d,
        int(n_shards), int(bool(causal)), _ptr(doc_offsets), _ptr(workspace),
        int(workspace.numel()), _stream(stream)))


def cp_ring_attn_fwd_noalloc(q, k, v, out, lse, n_shards: int, causal: bool = True,
                             doc_offsets: Optional[torch.Tensor] = None, stream=None) -> None:
    """cp_ring_attn_fwd without any device allocation by the library, for
    callers whose memory pool forbids it; at most 65,535 documents (more is
    reported as CP_ERR_SCRATCH by cp_get_last_status)."""
    B, S, H, d = q.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _need(t, n, torch.bfloat16, (B, S, H, d))
    _need(lse, "lse", torch.float32, (B, H, S))
    if doc_offsets is not None:
        _need(doc_offsets, "doc_offsets", torch.int32)
    _check("cp_ring_attn_fwd_noalloc", lib().cp_ring_attn_fwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, S, H, d, int(n_shards),
        int(bool(causal)), _ptr(doc_offsets), _stream(stream)))


def cp_ring_attn_fwd_emulated(q, k, v, out, lse, n_shards: int, causal: bool = True,
                              workspace: Optional[torch.Tensor] = None, stream=None,
                              copy_stream=None, doc_offsets: Optional[torch.Tensor] = None):
    """The ring with explicit per-rank K/V buffers and copy-engine transfers
    (overlapped on copy_stream, or in order when copy_stream is None).
    Returns the bytes each rank received.  workspace: a uint8 device tensor
    of at least cp_ring_emulated_workspace_bytes(...) bytes (allocated here
    if None)."""
    B, S, H, d = q.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _need(t, n, torch.bfloat16, (B, S, H, d))
    _need(lse, "lse", torch.float32, (B, H, S))
    if doc_offsets is not None:
        _need(doc_offsets, "doc_offsets", torch.int32)
    need = int(lib().cp_ring_emulated_workspace_bytes(B, S, H, d, int(n_shards)))
    if need < 0:
        raise CpError("cp_ring_emulated_workspace_bytes", STATUS_CODES["CP_ERR_SHAPE"])
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    recv = (ctypes.c_int64 * int(n_shards))()
    cs = None if copy_stream is None else _stream(copy_stream)
    _check("cp_ring_attn_fwd_emulated", lib().cp_ring_attn_fwd_emulated(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, S, H, d, int(n_shards),
        int(bool(causal)), _ptr(doc_offsets), _ptr(workspace), int(workspace.numel()),
        _stream(stream), cs, recv))
    return list(recv)


def cp_ulysses_attn_fwd(q, k, v, out, lse, n_shards: int, causal: bool = True,
                        doc_offsets: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, stream=None) -> int:
    """All-to-all (Ulysses) form: head-split attention between two layout
    permutations.  Returns the bytes the two all-to-alls would move."""
    B, S, H, d = q.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _need(t, n, torch.bfloat16, (B, S, H, d))
    _need(lse, "lse", torch.float32, (B, H, S))
    if doc_offsets is not None:
        _need(doc_offsets, "doc_offsets", torch.int32)
    need = int(lib().cp_ulysses_workspace_bytes(B, S, H, d, int(n_shards)))
    if need < 0:
        raise CpError("cp_ulysses_workspace_bytes", STATUS_CODES["CP_ERR_SHAPE"])
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    moved = ctypes.c_int64(0)
    _check("cp_ulysses_attn_fwd", lib().cp_ulysses_attn_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, S, H, d, int(n_shards),
        int(bool(causal)), _ptr(doc_offsets), _ptr(workspace), int(workspace.numel()),
        _stream(stream), ctypes.byref(moved)))
    return int(moved.value)


def cp_ulysses_workspace_bytes(B: int, S: int, H: int, d: int, n_shards: int) -> int:
    return int(lib().cp_ulysses_workspace_bytes(B, S, H, d, n_shards))


def cp_ring_emulated_workspace_bytes(B: int, S: int, H: int, d: int, n_shards: int) -> int:
    return int(lib().cp_ring_emulated_workspace_bytes(B, S, H, d, n_shards))


def cp_ring_attn_fwd_f32(q, k, v, out, lse, n_shards: int, causal: bool = True,
                         doc_offsets: Optional[torch.Tensor] = None, stream=None) -> None:
    """fp32 fused forward; q, k, v, out [B,S,H,d] fp32, lse [B,H,S] fp32."""
    B, S, H, d = q.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _need(t, n, torch.float32, (B, S, H, d))
    _need(lse, "lse", torch.float32, (B, H, S))
    if doc_offsets is not None:
        _need(doc_offsets, "doc_offsets", torch.int32)
    _check("cp_ring_attn_fwd_f32", lib().cp_ring_attn_fwd_f32(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, S, H, d, int(n_shards),
        int(bool(causal)), _ptr(doc_offsets), _stream(stream)))


def cp_ring_step(q, k, v, o_part, m_part, l_part, n_shards: int, i: int, j: int,
                 causal: bool = True, doc_offsets: Optional[torch.Tensor] = None,
                 stream=None) -> None:
    """One partial step (i, j).  bf16 or fp32 q/k/v (dispatched on dtype);
    o_part [B,S/N,H,d] fp32, m_part and l_part [B,H,S/N] fp32."""
    B, S, H, d = q.shape
    L = S // int(n_shards) if n_shards else 0
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise TypeError("q must be bf16 or fp32")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, dt, (B, S, H, d))
    _need(o_part, "o_part", torch.float32, (B, L, H, d))
    _need(m_part, "m_part", torch.float32, (B, H, L))
    _need(l_part, "l_part", torch.float32, (B, H, L))
    if doc_offsets is not None:
        _need(doc_offsets, "doc_offsets", torch.int32)
    name = "cp_ring_step" if dt == torch.bfloat16 else "cp_ring_step_f32"
    _check(name, getattr(lib(), name)(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o_part), _ptr(m_part), _ptr(l_part), B, S, H, d,
        int(n_shards), int(i), int(j), int(bool(causal)), _ptr(doc_offsets), _stream(stream)))


def cp_lse_merge(o_acc, m_acc, l_acc, o_part, m_part, l_part, stream=None) -> None:
    """In-place online merge of (o_part, m_part, l_part) into (o_acc, m_acc, l_acc)."""
    B, rows, H, d = o_acc.shape
    _need(o_acc, "o_acc", torch.float32)
    _need(o_part, "o_part", torch.float32, (B, rows, H, d))
    for t, n in ((m_acc, "m_acc"), (l_acc, "l_acc"), (m_part, "m_part"), (l_part, "l_part")):
        _need(t, n, torch.float32, (B, H, rows))
    _check("cp_lse_merge", lib().cp_lse_merge(
        _ptr(o_acc), _ptr(m_acc), _ptr(l_acc), _ptr(o_part), _ptr(m_part), _ptr(l_part),
        B, rows, H, d, _stream(stream)))


def cp_lse_finalize(o_acc, m_acc, l_acc, out, lse, stream=None) -> None:
    """out = o_acc / l_acc (bf16 or fp32 by out's dtype), lse = m + log(l)."""
    B, rows, H, d = o_acc.shape
    _need(o_acc, "o_acc", torch.float32)
    for t, n in ((m_acc, "m_acc"), (l_acc, "l_acc"), (lse, "lse")):
        _need(t, n, torch.float32, (B, H, rows))
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out must be bf16 or fp32")
    _need(out, "out", out.dtype, (B, rows, H, d))
    _check("cp_lse_finalize", lib().cp_lse_finalize(
        _ptr(o_acc), _ptr(m_acc), _ptr(l_acc), _ptr(out), _ptr(lse), B, rows, H, d,
        int(out.dtype == torch.bfloat16), _stream(stream)))


def cp_ring_schedule(S: int, n_shards: int, tile_q: int, tile_k: int, causal: bool = True,
                     doc_offsets: Optional[Sequence[int]] = None):
    """Host-side skip schedule: list of (q tile, kv tile) pairs."""
    L = lib()
    n = ctypes.c_int64(0)
    docs = None
    if doc_offsets is not None:
        arr = (ctypes.c_int32 * len(doc_offsets))(*[int(x) for x in doc_offsets])
        docs = ctypes.cast(arr, ctypes.c_void_p)
    _check("cp_ring_schedule", L.cp_ring_schedule(S, n_shards, tile_q, tile_k, int(bool(causal)),
                                                  docs, None, 0, ctypes.byref(n)))
    cnt = n.value
    buf = (ctypes.c_int32 * max(1, 2 * cnt))()
    _check("cp_ring_schedule", L.cp_ring_schedule(S, n_shards, tile_q, tile_k, int(bool(causal)),
                                                  docs, ctypes.cast(buf, ctypes.c_void_p), cnt,
                                                  ctypes.byref(n)))
    return [(buf[2 * x], buf[2 * x + 1]) for x in range(cnt)]


def cp_ring_schedule_device(S: int, n_shards: int, causal: bool = True,
                            doc_offsets: Optional[torch.Tensor] = None, device="cuda",
                            stream=None) -> torch.Tensor:
    """The fused kernel's key-tile range per 128-row query tile, computed on the
    device: int32 [n_tiles, 2] (first, last flat key tile)."""
    L = S // n_shards
    n_tiles = n_shards * ((L + 127) // 128)
    out = torch.full((n_tiles, 2), -7, dtype=torch.int32, device=device)
    if doc_offsets is not None:
        _need(doc_offsets, "doc_offsets", torch.int32)
    _check("cp_ring_schedule_device", lib().cp_ring_schedule_device(
        S, n_shards, int(bool(causal)), _ptr(doc_offsets), _ptr(out), _stream(stream)))
    return out


def cp_ring_traffic(B: int, S: int, H: int, d: int, dtype_bytes: int, n_shards: int,
                    causal: bool = False):
    """Per-rank send + receive bytes of the virtual ring."""
    out = (ctypes.c_int64 * n_shards)()
    _check("cp_ring_traffic", lib().cp_ring_traffic(B, S, H, d, dtype_bytes, n_shards,
                                                    int(bool(causal)), out))
    return list(out)


def cp_get_last_status(stream=None) -> int:
    """Synchronise the stream, read and clear the device error word."""
    return int(lib().cp_get_last_status(_stream(stream)))


def cp_status_string(status: int) -> str:
    return lib().cp_status_string(int(status)).decode()


def test_set_wait_fault(drop_first_k_tile: bool, wait_limit_ns: int = 0) -> None:
    """Test hook: make CTA 0 of later tensor-core launches skip its first K
    tile so that a bounded device wait runs out (see include/cpring.h)."""
    lib().cp_test_set_wait_fault(int(bool(drop_first_k_tile)), int(wait_limit_ns))


def launch_counts():
    """(tcgen05 attention, fp32 attention, merge/finalize, doc scan) launches so far."""
    buf = (ctypes.c_int64 * 4)()
    lib().cp_launch_counts(buf)
    return tuple(buf)
