"""cp_ring_attn_fwd_noalloc: the fused forward for callers that cannot let a
library allocate device memory (processes whose memory pool owns the GPU and
forbids later cudaMalloc/cudaMallocAsync, or loops that must stay out of the
driver's allocator).  It keeps its scratch in a fixed array built into the
library instead.

The GPU tests call it through the C ABI and require it to equal
cp_ring_attn_fwd bit for bit (the same kernel computes the same work items;
only where the scratch lives differs), on calls in a row with different
document layouts and shard counts (a later call must not see anything left
by an earlier one), and once against the oracle.  Malformed and oversized
document arrays are rejected on the device and leave the outputs untouched.
This file is collected last so that a run stopping at its first failure has
run everything else.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import context_ring_attention_fwd_gb300 as pkg
from context_ring_attention_fwd_gb300 import inputs
from oracle import ref

BF16_MAX, BF16_MEAN = 2e-2, 2e-3
FAKE = ctypes.c_void_p(0x10000)


def _lib():
    if not os.path.exists(pkg.LIB_PATH):
        from context_ring_attention_fwd_gb300 import _build
        _build.build()
    return pkg.lib()


def test_noalloc_rejects_bad_arguments_on_host():
    f = _lib().cp_ring_attn_fwd_noalloc
    assert f(None, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 128, 4, 1, None, None) == -1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 250, 2, 128, 4, 1, None, None) == -2
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 96, 4, 1, None, None) == -3
    assert f(ctypes.c_void_p(0x10002), FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 128, 4, 1, None,
             None) == -4
    # the shape checks are cp_ring_attn_fwd's: B * H beyond the kernels' work counters
    g = _lib().cp_ring_attn_fwd
    for fn in (f, g):
        assert fn(FAKE, FAKE, FAKE, FAKE, FAKE, 65536, 1, 16384, 64, 1, 1, None, None) == -2


def _call_noalloc(lib, q, k, v, out, lse, N, causal, docs_t):
    B, S, H, d = q.shape
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = lib.cp_ring_attn_fwd_noalloc(p(q), p(k), p(v), p(out), p(lse), B, S, H, d, N,
                                      int(causal), p(docs_t),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, pkg.STATUS_NAMES.get(st, st)


def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib()
    torch.cuda.set_device(0)
    pkg.cp_get_last_status()                     # start from a clear error word
    return lib


@pytest.mark.gpu
def test_noalloc_equals_fused_forward_on_calls_in_a_row():
    lib = _gpu()
    B, S, H, d = 1, 2048, 4, 128
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, S, H, d, seed=31, dtype=torch.bfloat16))
    calls = [([0, 300, 301, 777, 1500, 2048], 4, True), ([0, 1024, 2048], 8, True),
             (None, 4, True), ([0, 5, 900, 2048], 1, False), ([0, 2047, 2048], 8, False)]
    for n, (docs, N, causal) in enumerate(calls):
        docs_t = pkg.doc_offsets_tensor(docs, q.device)
        want_o = torch.empty_like(q)
        want_l = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
        pkg.cp_ring_attn_fwd(q, k, v, want_o, want_l, N, causal, docs_t)
        out = torch.full_like(q, 5.0)
        lse = torch.full((B, H, S), 5.0, dtype=torch.float32, device=q.device)
        _call_noalloc(lib, q, k, v, out, lse, N, causal, docs_t)
        assert pkg.cp_get_last_status() == 0
        assert torch.equal(out, want_o) and torch.equal(lse, want_l), (docs, N, causal)
        if n == 0:
            wo, wl = ref.attention(q.float().cpu().numpy(), k.float().cpu().numpy(),
                                   v.float().cpu().numpy(), causal, docs)
            e = np.abs(out.float().cpu().numpy() - wo)
            assert e.max() <= BF16_MAX and e.mean() <= BF16_MEAN
            assert np.abs(lse.cpu().numpy() - wl).max() <= BF16_MAX


@pytest.mark.gpu
def test_noalloc_rejects_malformed_documents_and_keeps_outputs():
    lib = _gpu()
    B, S, H, d, N = 1, 2048, 2, 128, 4
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, S, H, d, seed=33, dtype=torch.bfloat16))
    for docs in ([0, 300, 300, 2048], [0, 700, 600, 2048], [1, 700, 2048], [0, 700, 4096]):
        docs_t = pkg.doc_offsets_tensor(docs, q.device)
        out = torch.full_like(q, 5.0)
        lse = torch.full((B, H, S), 5.0, dtype=torch.float32, device=q.device)
        _call_noalloc(lib, q, k, v, out, lse, N, True, docs_t)
        assert pkg.cp_get_last_status() == pkg.STATUS_CODES["CP_ERR_DOC_OFFSETS"], docs
        assert torch.all(out == 5.0) and torch.all(lse == 5.0), docs
    # the next well-formed call is unaffected
    docs_t = pkg.doc_offsets_tensor([0, 300, 2048], q.device)
    want_o, want_l = pkg.ring_attn_fwd(q, k, v, N, True, [0, 300, 2048])
    _call_noalloc(lib, q, k, v, out, lse, N, True, docs_t)
    assert pkg.cp_get_last_status() == 0
    assert torch.equal(out, want_o) and torch.equal(lse, want_l)


@pytest.mark.gpu
def test_noalloc_rejects_more_documents_than_its_scratch_holds():
    lib = _gpu()
    B, S, H, d, N = 1, 65540, 1, 64, 1
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, S, H, d, seed=32, dtype=torch.bfloat16))
    docs = list(range(0, 65537)) + [S]           # 65,537 documents: two more than the limit
    docs_t = pkg.doc_offsets_tensor(docs, q.device)
    out = torch.full_like(q, 5.0)
    lse = torch.full((B, H, S), 5.0, dtype=torch.float32, device=q.device)
    _call_noalloc(lib, q, k, v, out, lse, N, True, docs_t)
    assert pkg.cp_get_last_status() == pkg.STATUS_CODES["CP_ERR_SCRATCH"]
    assert torch.all(out == 5.0) and torch.all(lse == 5.0)
    # exactly the limit is accepted
    docs = list(range(0, 65535)) + [S]           # 65,535 documents
    docs_t = pkg.doc_offsets_tensor(docs, q.device)
    want_o, want_l = pkg.ring_attn_fwd(q, k, v, N, True, docs)
    _call_noalloc(lib, q, k, v, out, lse, N, True, docs_t)
    assert pkg.cp_get_last_status() == 0
    assert torch.equal(out, want_o) and torch.equal(lse, want_l)
    # the array is reusable right after a rejected call
    docs = [0, 40000, S]
    docs_t = pkg.doc_offsets_tensor(docs, q.device)
    want_o, want_l = pkg.ring_attn_fwd(q, k, v, N, True, docs)
    _call_noalloc(lib, q, k, v, out, lse, N, True, docs_t)
    assert pkg.cp_get_last_status() == 0
    assert torch.equal(out, want_o) and torch.equal(lse, want_l)
