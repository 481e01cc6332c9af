"""GPU parity of the FP8 (E4M3) form against the fp64 oracle, through the C ABI.

Quantisation (cp_fp8_quantize) is integer-valued work decided by exactly
rounded fp32 operations, so its codes and descales must equal the oracle's bit
for bit.

The FP8 forward is compared with the exact attention of the dequantized
inputs (oracle.attention_fp8 on the codes the GPU produced).  Its own error
comes from rounding P to E4M3 before the PV product: a relative error of at
most 2^-4 per element (3 mantissa bits, nearest), so |O - O_exact| is at most
2^-4 * max|v| row by row, a p-weighted average of the per-element errors
times v; entries of P below E4M3's normal range (2^-6 of the row's
reference) carry a larger relative error but a negligible weight.  The
tolerance is that bound on the maximum, 2^-4 * max|v|, and 2^-8 * max|v| on
the mean.  A numpy model of the same tile loop (128-key tiles, the same lazy
reference, P rounded to E4M3) on seeded N(0, s^2) inputs, s = 0.7 .. 3,
reached 0.040 * max|v| and 0.0018 * max|v|; peaked attention (large s),
where a few keys carry the row, comes closest.  The log-sum-exp is formed
from the unrounded P and keeps the bf16 bound, 2e-2.  Q = 0 makes every P
exactly 1 in E4M3, so that case keeps the bf16 output bounds.
"""
import os

import numpy as np
import pytest
import torch

import context_ring_attention_fwd_gb300 as pkg
from context_ring_attention_fwd_gb300 import inputs
from oracle import ref

pytestmark = pytest.mark.gpu

DEV = "cuda"
LSE_MAX = 2e-2
BF16_MAX, BF16_MEAN = 2e-2, 2e-3
FP8_MAX_REL, FP8_MEAN_REL = 2.0 ** -4, 2.0 ** -8   # times max|v| of the dequantized V


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


def _values(codes: torch.Tensor) -> np.ndarray:
    """E4M3 codes (uint8) decoded to float64 on the host."""
    return codes.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _np(t):
    return t.detach().float().cpu().numpy()


def _fp8_inputs(B, S, H, d, seed, scale=1.0):
    q, k, v = (t.to(DEV) for t in inputs.make_qkv(B, S, H, d, seed, torch.bfloat16, scale))
    return (q, k, v), pkg.fp8_quantize_qkv(q, k, v)


def _oracle_operands(fp8):
    """Decoded codes in the oracle's [B, S, H, d] layout and the descales."""
    q8, k8, v8t, qd, kd, vd = fp8
    v8 = np.ascontiguousarray(_values(v8t).transpose(0, 3, 1, 2))
    return _values(q8), _values(k8), v8, _np(qd), _np(kd), _np(vd)


def _check_fp8(out, lse, want_o, want_l, vmax, what=""):
    o = _np(out)
    assert np.all(np.isfinite(o)), what
    e = np.abs(o - want_o)
    assert e.max() <= FP8_MAX_REL * vmax, (what, e.max(), vmax)
    assert e.mean() <= FP8_MEAN_REL * vmax, (what, e.mean(), vmax)
    assert np.abs(_np(lse) - want_l).max() <= LSE_MAX, what


# ----------------------------------------------------------- quantisation
@pytest.mark.parametrize("B,S,H,d", [(2, 208, 3, 128), (1, 96, 2, 64), (1, 1040, 4, 128)])
@pytest.mark.parametrize("transpose", [False, True])
def test_fp8_quantize_bit_exact(B, S, H, d, transpose):
    x = inputs.make_qkv(B, S, H, d, seed=41, dtype=torch.bfloat16)[0]
    x[0, :, H - 1, :] = 0                     # an all-zero head
    x[B - 1, :, 0, :] *= 37.0                 # a head with a large range
    xd = x.to(DEV)
    shape = (B, H, d, S) if transpose else (B, S, H, d)
    x8 = torch.full(shape, 0x7F, dtype=torch.uint8, device=DEV)
    desc = torch.full((B, H), -1.0, dtype=torch.float32, device=DEV)
    pkg.cp_fp8_quantize(xd, x8, desc, transpose)
    want_v, want_d = ref.fp8_quantize(x.float().numpy())
    got = _values(x8)
    if transpose:
        got = got.transpose(0, 3, 1, 2)
    np.testing.assert_array_equal(got, want_v)
    np.testing.assert_array_equal(_np(desc), want_d)
    # the same codes twice in a row (the descale buffer doubles as scratch)
    x8b = torch.empty_like(x8)
    pkg.cp_fp8_quantize(xd, x8b, desc, transpose)
    assert torch.equal(x8, x8b)
    np.testing.assert_array_equal(_np(desc), want_d)


# ----------------------------------------------------------- forward
FP8_CASES = [
    # B, S, H, N, causal, docs, input scale
    (1, 1024, 2, 4, True, None, 1.0),
    (2, 2080, 2, 2, True, None, 1.0),           # shard of 1040 rows: a ragged last tile
    (1, 768, 3, 3, False, None, 2.0),
    (1, 1536, 2, 4, True, [0, 300, 301, 777, 1200, 1536], 1.0),
    (1, 512, 2, 1, False, [0, 100, 512], 0.7071),
]


@pytest.mark.parametrize("B,S,H,N,causal,docs,scale", FP8_CASES)
def test_fp8_fused_against_oracle(B, S, H, N, causal, docs, scale):
    d = 128
    _, fp8 = _fp8_inputs(B, S, H, d, seed=43, scale=scale)
    out, lse = pkg.ring_attn_fwd_fp8(fp8, N, causal, docs)
    assert pkg.cp_get_last_status() == 0
    q8, k8, v8, qd, kd, vd = _oracle_operands(fp8)
    want_o, want_l = ref.attention_fp8(q8, k8, v8, qd, kd, vd, causal, docs)
    vmax = np.abs(ref.fp8_dequantize(v8, vd)).max()
    _check_fp8(out, lse, want_o, want_l, vmax, (B, S, H, N, causal, docs))


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("blocks", [(128, 384), (192, 448)], ids=["first-half", "second-half"])
@pytest.mark.parametrize("bumps", [(1.0, 2.0), (0.75, 0.875)], ids=["past-f16", "inside-f16"])
def test_fp8_scores_jump_past_the_reference(causal, blocks, bumps):
    """Blocks of keys whose scores rise by about 16 and 32 (or 12 and 14) as
    base-2 exponents over the first key tile's: past the FP8 pass's 2^8
    guard, so the kernel must move its reference point (keeping every P
    inside E4M3's range) instead of saturating.  The fast pass exponentiates
    in half precision: the larger jumps overflow it to +inf, the smaller ones
    stay finite with a row sum above the guard; both must reach the redo."""
    B, S, H, d = 1, 768, 2, 128
    q, k, v = inputs.make_qkv(B, S, H, d, seed=72, dtype=torch.bfloat16)
    q = (q.float() * 0.25 + 1.0).to(torch.bfloat16)
    k = k.float() * 0.25
    for a, bump in zip(blocks, bumps):
        k[:, a:a + 32] += bump
    fp8 = pkg.fp8_quantize_qkv(q.to(DEV), k.to(torch.bfloat16).to(DEV), v.to(DEV))
    out, lse = pkg.ring_attn_fwd_fp8(fp8, 2, causal)
    assert pkg.cp_get_last_status() == 0
    q8, k8, v8, qd, kd, vd = _oracle_operands(fp8)
    want_o, want_l = ref.attention_fp8(q8, k8, v8, qd, kd, vd, causal)
    vmax = np.abs(ref.fp8_dequantize(v8, vd)).max()
    _check_fp8(out, lse, want_o, want_l, vmax, (causal, blocks))


def test_fp8_zero_query_is_the_prefix_mean():
    B, S, H, d, N = 1, 1024, 2, 128, 4
    (q, k, v), _ = _fp8_inputs(B, S, H, d, seed=44)
    fp8 = pkg.fp8_quantize_qkv(torch.zeros_like(q), k, v)
    out, lse = pkg.ring_attn_fwd_fp8(fp8, N, True)
    _, _, v8, _, _, vd = _oracle_operands(fp8)
    cf_o, cf_l = ref.zero_query_closed_form(ref.fp8_dequantize(v8, vd), True)
    e = np.abs(_np(out) - cf_o)
    assert e.max() <= BF16_MAX and e.mean() <= BF16_MEAN
    assert np.abs(_np(lse) - cf_l).max() <= LSE_MAX


def test_fp8_deterministic_and_shard_count_within_tolerance():
    B, S, H, d = 1, 2048, 2, 128
    _, fp8 = _fp8_inputs(B, S, H, d, seed=45)
    a = pkg.ring_attn_fwd_fp8(fp8, 4, True)
    b = pkg.ring_attn_fwd_fp8(fp8, 4, True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    q8, k8, v8, qd, kd, vd = _oracle_operands(fp8)
    want_o, want_l = ref.attention_fp8(q8, k8, v8, qd, kd, vd, True)
    vmax = np.abs(ref.fp8_dequantize(v8, vd)).max()
    for N in (1, 2, 8):
        _check_fp8(*pkg.ring_attn_fwd_fp8(fp8, N, True), want_o, want_l, vmax, N)


def test_fp8_workload_causal_128k_sampled():
    """bf16 causal 128K (B=1 S=131072 H=32 d=128 N=4) stored as FP8: 512
    seeded query rows of every head against the oracle, and Q = 0 against the
    prefix mean on every row of every fourth head."""
    w = inputs.BY_NAME["bf16_causal_128k"]
    q, k, v = inputs.make_qkv(w.B, w.S, w.H, w.d, w.seed, torch.bfloat16, w.scale, device=DEV)
    fp8 = pkg.fp8_quantize_qkv(q, k, v)
    out, lse = pkg.ring_attn_fwd_fp8(fp8, w.n_shards, w.causal)
    assert pkg.cp_get_last_status() == 0
    q8, k8, v8t, qd, kd, vd = fp8
    zero = pkg.fp8_quantize_qkv(torch.zeros_like(q), k, v)
    out0, lse0 = pkg.ring_attn_fwd_fp8(zero, w.n_shards, w.causal)
    on, ln, on0, ln0 = _np(out), _np(lse), _np(out0), _np(lse0)
    qdn, kdn, vdn = _np(qd), _np(kd), _np(vd)
    del q, k, v, zero
    errs_l = []
    for h in range(w.H):
        one = lambda x8, s: ref.fp8_dequantize(x8[None, :, None, :], np.array([[s]], np.float32))
        qh = one(_values(q8[0, :, h, :]), qdn[0, h])
        kh = one(_values(k8[0, :, h, :]), kdn[0, h])
        vh = one(np.ascontiguousarray(_values(v8t[0, h]).T), vdn[0, h])
        rows = inputs.sample_rows(w.S, 512, seed=w.seed * 100 + h)
        wo, wl = ref.attention_rows(qh, kh, vh, 0, 0, rows, w.causal, None)
        vmax = np.abs(vh).max()
        e = np.abs(on[0, rows, h] - wo)
        assert e.max() <= FP8_MAX_REL * vmax and e.mean() <= FP8_MEAN_REL * vmax, (h, e.max())
        errs_l.append(np.abs(ln[0, h, rows] - wl).max())
        if h % 4:
            continue
        cf_o, cf_l = ref.zero_query_closed_form(vh, w.causal, None)
        e0 = np.abs(on0[0, :, h] - cf_o[0, :, 0])
        assert e0.max() <= BF16_MAX and e0.mean() <= BF16_MEAN, (h, e0.max())
        assert np.abs(ln0[0, h] - cf_l[0, 0]).max() <= LSE_MAX
    assert max(errs_l) <= LSE_MAX
