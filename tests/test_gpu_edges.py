"""Degenerate shapes on the GPU paths against the fp64 oracle: a single
token, one token per shard (N = S), shards shorter than one 128-row tile,
ragged shards, single-token documents, and several batch rows with
documents.  Tolerances as in the other GPU parity files (bf16: max-abs 2e-2,
mean-abs 2e-3; backward: 2^-6 and 2^-10 of max|g|; FP8: 2^-4 and 2^-8 of
max|v|)."""
import os

import numpy as np
import pytest
import torch

import context_ring_attention_fwd_gb300 as pkg
from context_ring_attention_fwd_gb300 import inputs
from oracle import ref

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not os.path.exists(pkg.LIB_PATH):
        from context_ring_attention_fwd_gb300 import _build
        _build.build()
    pkg.lib()
    torch.cuda.set_device(0)
    yield
    assert pkg.cp_get_last_status() == 0


def _np(t):
    return t.detach().float().cpu().numpy()


EDGE = [
    # B, S, H, d, N, causal, docs
    (1, 1, 1, 128, 1, True, None),                 # a single token
    (1, 1, 2, 64, 1, False, None),
    (1, 7, 2, 64, 7, True, None),                  # one token per shard
    (1, 96, 3, 128, 3, False, None),               # 32-row shards
    (1, 130, 1, 128, 2, True, None),               # 65-row shards
    (3, 200, 1, 64, 4, True, [0, 1, 2, 3, 100, 200]),   # single-token documents
    (2, 384, 2, 128, 2, False, [0, 1, 129, 130, 384]),  # batch rows share the layout
]


@pytest.mark.parametrize("B,S,H,d,N,causal,docs", EDGE)
def test_forward_edges(B, S, H, d, N, causal, docs):
    q, k, v = (t.to(DEV) for t in inputs.make_qkv(B, S, H, d, 71, torch.bfloat16))
    out, lse = pkg.ring_attn_fwd(q, k, v, N, causal, docs)
    assert pkg.cp_get_last_status() == 0
    want_o, want_l = ref.attention(_np(q), _np(k), _np(v), causal, docs)
    e = np.abs(_np(out) - want_o)
    assert e.max() <= 2e-2 and e.mean() <= 2e-3, (e.max(), e.mean())
    assert np.abs(_np(lse) - want_l).max() <= 2e-2
    # the explicit ring of steps and merges gives the same result
    oc, lc = pkg.ring_attn_composed(q, k, v, N, causal, docs, order="ring")
    e2 = np.abs(_np(oc) - want_o)
    assert e2.max() <= 2e-2 and e2.mean() <= 2e-3


@pytest.mark.parametrize("B,S,H,d,N,causal,docs", EDGE)
def test_backward_edges(B, S, H, d, N, causal, docs):
    q, k, v = (t.to(DEV) for t in inputs.make_qkv(B, S, H, d, 72, torch.bfloat16))
    dout = inputs.make_qkv(B, S, H, d, 73, torch.bfloat16)[0].to(DEV)
    out, lse = pkg.ring_attn_fwd(q, k, v, N, causal, docs)
    got = pkg.ring_attn_bwd(q, k, v, out, lse, dout, N, causal, docs)
    assert pkg.cp_get_last_status() == 0
    want = ref.attention_bwd(_np(q), _np(k), _np(v), _np(dout), causal, docs)
    for name, a, b in zip(("dq", "dk", "dv"), got, want):
        # a gradient that vanishes exactly (one visible key makes dS = 0)
        # is held to the same bounds on an absolute scale of 1e-3
        gm = max(np.abs(b).max(), 1e-3)
        e = np.abs(_np(a) - b)
        assert e.max() <= 2.0 ** -6 * gm and e.mean() <= 2.0 ** -10 * gm, (name, e.max(), gm)


@pytest.mark.parametrize("B,S,H,N,causal,docs", [(1, 32, 1, 2, True, None),
                                                 (1, 48, 2, 3, False, None),
                                                 (2, 64, 1, 4, True, [0, 1, 17, 64])])
def test_fp8_edges(B, S, H, N, causal, docs):
    q, k, v = (t.to(DEV) for t in inputs.make_qkv(B, S, H, 128, 74, torch.bfloat16))
    f8 = pkg.fp8_quantize_qkv(q, k, v)
    out, lse = pkg.ring_attn_fwd_fp8(f8, N, causal, docs)
    assert pkg.cp_get_last_status() == 0
    q8, k8, v8t, qd, kd, vd = f8
    val = lambda c: c.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()  # noqa: E731
    v8 = np.ascontiguousarray(val(v8t).transpose(0, 3, 1, 2))
    want_o, want_l = ref.attention_fp8(val(q8), val(k8), v8, _np(qd), _np(kd), _np(vd), causal, docs)
    vmax = np.abs(ref.fp8_dequantize(v8, _np(vd))).max()
    e = np.abs(_np(out) - want_o)
    assert e.max() <= 2.0 ** -4 * vmax and e.mean() <= 2.0 ** -8 * vmax
    assert np.abs(_np(lse) - want_l).max() <= 2e-2
