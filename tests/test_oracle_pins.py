"""Pins of the fp64 oracle against things other than itself.

Each test ties an oracle function to a library routine, a closed form, brute
force on tiny inputs, or a worked example printed on the pages (fixtures
under tests/golden/, each citing its page and section).  All CPU.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import ref
from context_ring_attention_fwd_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _qkv(B, S, H, d, seed, scale=1.0):
    q, k, v = inputs.make_qkv(B, S, H, d, seed, torch.float64, scale)
    return q.numpy(), k.numpy(), v.numpy()


def _sdpa(q, k, v, causal, doc_offsets):
    """torch's scaled_dot_product_attention in fp64 on CPU ([B,S,H,d] in/out)."""
    B, S, H, d = q.shape
    tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
    if doc_offsets is None:
        o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal)
    else:
        doc = torch.zeros(S, dtype=torch.long)
        for t, (a, b) in enumerate(zip(doc_offsets[:-1], doc_offsets[1:])):
            doc[a:b] = t
        mask = doc[:, None] == doc[None, :]
        if causal:
            mask &= torch.ones(S, S, dtype=torch.bool).tril()
        o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)
    return o.permute(0, 2, 1, 3).numpy()


def _lse_scipy(q, k, causal, doc_offsets):
    """log-sum-exp of the visible scores via scipy.special.logsumexp."""
    B, S, H, d = q.shape
    doc = np.zeros(S, dtype=int)
    if doc_offsets is not None:
        for t, (a, b) in enumerate(zip(doc_offsets[:-1], doc_offsets[1:])):
            doc[a:b] = t
    out = np.empty((B, H, S))
    for b in range(B):
        for h in range(H):
            s = np.einsum("qd,kd->qk", q[b, :, h], k[b, :, h]) / math.sqrt(d)
            for r in range(S):
                keys = [c for c in range(S) if doc[c] == doc[r] and (not causal or c <= r)]
                out[b, h, r] = scipy.special.logsumexp(s[r, keys])
    return out


CASES = [
    (True, None), (False, None),
    (True, [0, 5, 13, 24]), (False, [0, 7, 8, 24]),
]


# P-1: N = 1, no documents, is textbook attention; with documents it is
# attention under a block-diagonal mask.  Library cross-check.
@pytest.mark.parametrize("causal,docs", CASES)
def test_attention_matches_torch_sdpa(causal, docs):
    q, k, v = _qkv(2, 24, 3, 8, seed=11)
    out, lse = ref.attention(q, k, v, causal, docs, q_block=7)
    np.testing.assert_allclose(out, _sdpa(q, k, v, causal, docs), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, _lse_scipy(q, k, causal, docs), rtol=0, atol=1e-12)


def test_attention_rows_matches_full():
    q, k, v = _qkv(1, 40, 2, 8, seed=12)
    docs = [0, 9, 31, 40]
    out, lse = ref.attention(q, k, v, True, docs)
    rows = np.array([0, 3, 9, 10, 30, 31, 39])
    o_r, l_r = ref.attention_rows(q, k, v, 0, 1, rows, True, docs, q_block=3)
    np.testing.assert_allclose(o_r, out[0, rows, 1], rtol=0, atol=1e-13)
    np.testing.assert_allclose(l_r, lse[0, 1, rows], rtol=0, atol=1e-13)


# P-2 / P-7: the ring + blockwise algorithm equals the naive definition for
# every shard count, every visiting order (N <= 4), with and without
# causality and documents, with and without skipping of masked steps.
def _divisors(S, cap=8):
    return [n for n in range(1, cap + 1) if S % n == 0]


@pytest.mark.parametrize("S", [8, 12, 16, 64])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("with_docs", [False, True])
def test_ring_blockwise_equals_naive(S, causal, with_docs):
    q, k, v = _qkv(1, S, 2, 4, seed=S)
    docs = inputs.random_doc_offsets(S, 3, seed=S) if with_docs else None
    want_o, want_l = ref.attention(q, k, v, causal, docs)
    for N in _divisors(S):
        orders = list(ref.all_orders(N)) if N <= 4 else ["ascending", "ring"]
        for order in orders:
            for skip in (True, False):
                o, l = ref.ring_forward(q, k, v, N, causal, docs, order, skip)
                np.testing.assert_allclose(o, want_o, rtol=0, atol=1e-12)
                np.testing.assert_allclose(l, want_l, rtol=0, atol=1e-12)


def test_ring_order_ring_kind():
    # at step t rank i holds the shard of rank (i - t) mod N
    assert ref.ring_order(1, 4, "ring") == [1, 0, 3, 2]
    assert ref.ring_order(0, 4, "ascending") == [0, 1, 2, 3]


# The partial step itself, against library routines: log(l_ij) + m_ij is
# the log-sum-exp of the shard's visible scores, and O_ij / l_ij is SDPA
# restricted to that shard's keys.
@pytest.mark.parametrize("causal,docs", CASES)
def test_partial_step_against_library(causal, docs):
    S, N = 24, 3
    q, k, v = _qkv(1, S, 2, 8, seed=21)
    L = S // N
    doc = ref.doc_of(S, docs)
    for i in range(N):
        for j in range(N):
            O, m, l = ref.partial_step(q, k, v, N, i, j, causal, docs)
            for h in range(2):
                for r in range(L):
                    qr = i * L + r
                    keys = [c for c in range(j * L, (j + 1) * L)
                            if doc[c] == doc[qr] and (not causal or c <= qr)]
                    if not keys:
                        assert m[0, h, r] == -np.inf and l[0, h, r] == 0
                        assert np.all(O[0, r, h] == 0)
                        continue
                    s = k[0, keys, h] @ q[0, qr, h] / math.sqrt(8)
                    assert abs(np.log(l[0, h, r]) + m[0, h, r] - scipy.special.logsumexp(s)) < 1e-12
                    tq = torch.from_numpy(q[0, qr, h][None, None, None])
                    tk = torch.from_numpy(k[0, keys, h][None, None])
                    tv = torch.from_numpy(v[0, keys, h][None, None])
                    want = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)[0, 0, 0].numpy()
                    np.testing.assert_allclose(O[0, r, h] / l[0, h, r], want, rtol=0, atol=1e-12)


def test_merge_identity_and_symmetry():
    S, N = 16, 2
    q, k, v = _qkv(1, S, 2, 4, seed=5)
    a = ref.partial_step(q, k, v, N, 1, 0, True)
    b = ref.partial_step(q, k, v, N, 1, 1, True)
    empty = (np.zeros_like(a[0]), np.full_like(a[1], -np.inf), np.zeros_like(a[2]))
    for x, y in ((empty, a), (a, empty)):
        got = ref.merge(*x, *y)
        for g, w in zip(got, a):
            assert np.array_equal(g, w)
    e2 = ref.merge(*empty, *empty)
    assert np.all(e2[1] == -np.inf) and np.all(e2[2] == 0) and np.all(e2[0] == 0)
    ab = ref.merge(*a, *b)
    ba = ref.merge(*b, *a)
    for g, w in zip(ab, ba):
        np.testing.assert_allclose(g, w, rtol=0, atol=1e-14)


# P-3: the streaming identity, without max subtraction.
@pytest.mark.parametrize("causal,docs", CASES)
def test_streaming_identity(causal, docs):
    S = 24
    q, k, v = _qkv(1, S, 1, 8, seed=31)
    out, lse = ref.attention(q, k, v, causal, docs)
    doc = ref.doc_of(S, docs)
    for r in range(S):
        keys = [c for c in range(S) if doc[c] == doc[r] and (not causal or c <= r)]
        o, ls = ref.streaming_unsafe(q[0, r, 0], k[0, keys, 0], v[0, keys, 0])
        np.testing.assert_allclose(out[0, r, 0], o, rtol=0, atol=1e-12)
        assert abs(lse[0, 0, r] - ls) < 1e-12


# P-4: with Q = 0 every score is zero: each output row is the mean of V over
# its visible keys and lse = log(count).  Checked against an explicit
# per-row mean.
@pytest.mark.parametrize("causal,docs", CASES)
def test_zero_query_closed_form(causal, docs):
    S = 24
    _, k, v = _qkv(2, S, 2, 4, seed=41)
    q = np.zeros_like(k)
    out, lse = ref.attention(q, k, v, causal, docs)
    cf_o, cf_l = ref.zero_query_closed_form(v, causal, docs)
    doc = ref.doc_of(S, docs)
    for r in range(S):
        keys = [c for c in range(S) if doc[c] == doc[r] and (not causal or c <= r)]
        np.testing.assert_allclose(cf_o[:, r], v[:, keys].mean(axis=1), rtol=0, atol=1e-13)
        assert np.allclose(cf_l[:, :, r], math.log(len(keys)), rtol=0, atol=1e-15)
    np.testing.assert_allclose(out, cf_o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, cf_l, rtol=0, atol=1e-13)


# P-5: rows of the softmax sum to one, so a constant V comes back unchanged.
def test_constant_v():
    q, k, _ = _qkv(1, 32, 2, 8, seed=51)
    v = np.full_like(q, 0.375)
    out, _ = ref.attention(q, k, v, True, [0, 10, 32])
    np.testing.assert_allclose(out, 0.375, rtol=0, atol=1e-15)


# P-6: under causality rank i needs no K/V of shards > i; poisoning them
# with NaN leaves rows of shards 0..i untouched.  With documents, keys
# before the first query's document start are poisoned too.
def test_causal_independence_poison():
    S, N = 32, 4
    q, k, v = _qkv(1, S, 2, 4, seed=61)
    docs = [0, 6, 19, 32]
    for use_docs in (None, docs):
        out, _ = ref.attention(q, k, v, True, use_docs)
        L = S // N
        for i in range(N):
            kp, vp = k.copy(), v.copy()
            kp[:, (i + 1) * L:] = np.nan
            vp[:, (i + 1) * L:] = np.nan
            lo = 0
            if use_docs is not None:
                lo = max(o for o in use_docs if o <= i * L)
                kp[:, :lo] = np.nan
                vp[:, :lo] = np.nan
            rows = np.arange(max(lo, i * L), (i + 1) * L)
            o_r, _ = ref.attention_rows(q, kp, vp, 0, 1, rows, True, use_docs)
            assert np.all(np.isfinite(o_r))
            np.testing.assert_allclose(o_r, out[0, rows, 1], rtol=0, atol=1e-12)


# P-8: the skip schedule.  Closed forms without documents; block-diagonal
# triangles when documents align with tiles; the causal-needs statement of
# the "Context Parallelism" page (golden fixture).
def test_shard_schedule_causal_closed_form():
    for N in (1, 2, 3, 4, 8):
        S = 8 * N
        pairs = ref.tile_schedule(S, N, S // N, S // N, True)
        assert len(pairs) == N * (N + 1) // 2
        for i in range(N):
            assert [j for (qi, j) in pairs if qi == i] == list(range(i + 1))
        assert [p for p in pairs if p[0] == 0] == [(0, 0)]
        full = ref.tile_schedule(S, N, S // N, S // N, False)
        assert len(full) == N * N


def test_causal_needs_golden():
    lines = [l.split() for l in open(os.path.join(GOLDEN, "causal_needs_n4.txt"))
             if l.strip() and not l.startswith("#")]
    N = int(lines[0][1])
    want = {int(r[0]): [int(x) for x in r[1:]] for r in lines[1:]}
    S = 16 * N
    pairs = ref.tile_schedule(S, N, S // N, S // N, True)
    got = {i: [j for (qi, j) in pairs if qi == i] for i in range(N)}
    assert got == want
    for i in range(N):
        for j in range(N):
            assert ref.shard_needed(i, j, S, N, True) == (j in want[i])


@pytest.mark.parametrize("T,N", [(4, 1), (4, 2), (8, 2), (2, 4)])
def test_tile_schedule_closed_forms(T, N):
    S = 64
    pairs = ref.tile_schedule(S, N, T, T, True)
    nt = S // T
    assert len(pairs) == nt * (nt + 1) // 2
    # documents aligned with tile boundaries: one triangle per document
    docs = [0, 3 * T, 4 * T, S]
    pairs = ref.tile_schedule(S, N, T, T, True, docs)
    tri = sum((b - a) // T * ((b - a) // T + 1) // 2 for a, b in zip(docs[:-1], docs[1:]))
    assert len(pairs) == tri
    sq = sum(((b - a) // T) ** 2 for a, b in zip(docs[:-1], docs[1:]))
    assert len(ref.tile_schedule(S, N, T, T, False, docs)) == sq


def test_tile_spans_respect_shards():
    spans = ref.tile_spans(48, 4, 5)          # shards of 12: tiles 5, 5, 2
    assert spans[:3] == [(0, 5), (5, 10), (10, 12)]
    assert len(spans) == 12 and spans[-1] == (46, 48)


def test_visible_pair_counts():
    S = 40
    assert ref.visible_pair_count(S, True, block=7) == S * (S + 1) // 2
    assert ref.visible_pair_count(S, False, block=7) == S * S
    docs = [0, 3, 17, 40]
    lens = [b - a for a, b in zip(docs[:-1], docs[1:])]
    assert ref.visible_pair_count(S, True, docs, block=6) == sum(L * (L + 1) // 2 for L in lens)
    assert ref.visible_pair_count(S, False, docs, block=6) == sum(L * L for L in lens)


# P-9: ring traffic.  The step-by-step simulation reproduces the per-rank
# total 2 (G/N) (N-1) of "大语言模型并行策略（五）" §通信模式, with G the K and V
# bytes of the whole sequence, and the per-step block of
# (S/N) x H x d x dtype_bytes per tensor of the "Context Parallelism"
# §關鍵指標 table; under causality rank i receives exactly i blocks.
@pytest.mark.parametrize("N", [1, 2, 3, 4, 8])
def test_ring_traffic_simulation(N):
    B, S, H, d, nb = 2, 64 * N, 3, 16, 2
    G = 2 * B * S * H * d * nb
    tot = ref.ring_traffic_simulated(B, S, H, d, nb, N, causal=False)
    assert tot == [2 * (G // N) * (N - 1)] * N
    block = 2 * B * (S // N) * H * d * nb
    assert block == 2 * ((S // N) * H * d * nb) * B
    sent, recv = ref.ring_traffic_simulated(B, S, H, d, nb, N, causal=True, split=True)
    assert recv == [i * (G // N) for i in range(N)]
    assert recv[0] == 0 and (N == 1 or recv[-1] == (N - 1) * G // N)
    assert sum(sent) == sum(recv)


# Golden: the 128K / 4-GPU walk-through of "大语言模型并行策略（五）" §Ring Attention.
def test_walkthrough_128k_golden():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "walkthrough_128k_4gpu.txt"))
            if l.strip() and not l.startswith("#")]
    S = int(rows[0][1]) * 1024
    N = int(rows[1][1])
    stages = [[int(x) for x in r] for r in rows[2:]]
    bounds = ref.shard_bounds(S, N)
    w = inputs.BY_NAME["bf16_causal_128k"]
    assert (w.S, w.n_shards) == (S, N)
    order = ref.ring_order(0, N, "ascending")
    for (stage, qlo, qhi, klo, khi), j in zip(stages, order):
        assert bounds[0] == (qlo * 1024, qhi * 1024)
        assert bounds[j] == (klo * 1024, khi * 1024)
    assert len(stages) == N


def test_shard_bounds_errors():
    with pytest.raises(ValueError):
        ref.shard_bounds(10, 3)
    with pytest.raises(ValueError):
        ref.shard_bounds(10, 0)
    with pytest.raises(ValueError):
        ref.doc_of(10, [0, 4, 4, 10])


def test_effective_flops():
    # 4 d per visible pair (2 d for Q K^T, 2 d for P V)
    assert ref.effective_flops(1, 1, 64, 10) == 2560
    w = inputs.BY_NAME["bf16_causal_128k"]
    pairs = ref.visible_pair_count(4096, True)
    assert pairs == 4096 * 4097 // 2


# ---------------------------------------------------------------------------
# FP8 (E4M3) storage: rounding, quantisation, attention over dequantized values
# ---------------------------------------------------------------------------

def _torch_e4m3(x32: np.ndarray) -> np.ndarray:
    """torch's float32 -> float8_e4m3fn conversion, decoded back to float64."""
    return torch.from_numpy(x32).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_round_matches_torch_conversion():
    rng = np.random.default_rng(7)
    mag = np.exp2(rng.uniform(-13, 8.8, 200_000)).astype(np.float32)     # subnormals..448
    x = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32)
    np.testing.assert_array_equal(ref.e4m3_round(x), _torch_e4m3(x))


def test_e4m3_round_fixed_points_and_ties():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = vals[np.isfinite(vals)]
    assert finite.size == 254 and finite.max() == 448.0 and finite.min() == -448.0
    np.testing.assert_array_equal(ref.e4m3_round(finite), finite)
    # every midpoint between neighbouring positive codes rounds to the even one
    grid = np.unique(finite[finite >= 0])
    mids = (grid[:-1] + grid[1:]) / 2
    got = ref.e4m3_round(mids)
    even_code = lambda v: int(torch.tensor([v]).to(torch.float8_e4m3fn).view(torch.uint8)) % 2 == 0
    for lo, hi, g in zip(grid[:-1], grid[1:], got):
        assert g == (lo if even_code(lo) else hi)
        assert even_code(g)


def test_e4m3_round_closed_forms():
    cases = {448.0: 448.0, 460.0: 448.0, 1e6: 448.0, -1e6: -448.0,   # saturation
             2.0 ** -10: 0.0, 1.5 * 2.0 ** -10: 2.0 ** -9,            # below the subnormals
             1.0625: 1.0, 1.1875: 1.25, 3.0 * 2 ** -8: 3.0 * 2 ** -8,  # ties to even; a subnormal
             0.0: 0.0, 2.0 ** -6: 2.0 ** -6, 240.0: 240.0, 250.0: 256.0}
    for x, want in cases.items():
        assert ref.e4m3_round(np.float32(x)) == want, x
    assert np.isnan(ref.e4m3_round(np.float32("nan")))


def test_fp8_quantize_scales_and_range():
    B, S, H, d = 2, 96, 3, 64
    x = torch.randn(B, S, H, d, generator=torch.Generator().manual_seed(11), dtype=torch.float32)
    x[1, :, 2, :] = 0.0                                # an all-zero (b, h)
    x[0, 17, 1, 5] = -9.5                              # a known extreme
    x8, desc = ref.fp8_quantize(x.numpy())
    assert desc.dtype == np.float32 and desc.shape == (B, H)
    assert desc[1, 2] == 1.0 and np.all(x8[1, :, 2, :] == 0.0)
    assert x8[0, 17, 1, 5] == -448.0                   # amax maps to the largest code
    assert desc[0, 1] == np.float32(9.5) / np.float32(448.0)
    np.testing.assert_array_equal(ref.e4m3_round(x8), x8)            # on the grid
    assert np.abs(x8).max() <= 448.0
    # dequantisation error: within half a quantum of the E4M3 grid, scaled
    deq = ref.fp8_dequantize(x8, desc)
    a = np.abs(x.numpy().astype(np.float64) / desc[:, None, :, None].astype(np.float64))
    half_q = np.ldexp(1.0, np.maximum(np.frexp(a)[1] - 5, -10))
    assert np.all(np.abs(deq - x.numpy()) <= (half_q * 1.0001 + 1e-7) * desc[:, None, :, None])


@pytest.mark.parametrize("causal,docs", [(True, None), (False, [0, 40, 41, 128]),
                                         (True, [0, 70, 128])])
def test_attention_fp8_is_attention_of_dequantized_inputs(causal, docs):
    B, S, H, d = 1, 128, 2, 64
    q, k, v = _qkv(B, S, H, d, 23)
    (q8, qd), (k8, kd), (v8, vd) = (ref.fp8_quantize(t) for t in (q, k, v))
    o, lse = ref.attention_fp8(q8, k8, v8, qd, kd, vd, causal, docs)
    deq = [torch.from_numpy(ref.fp8_dequantize(a, s)) for a, s in ((q8, qd), (k8, kd), (v8, vd))]
    want = _sdpa(*(t.numpy() for t in deq), causal, docs)
    np.testing.assert_allclose(o, want, atol=1e-12, rtol=0)
    # Q = 0: each query averages the dequantized V over its visible keys
    o0, lse0 = ref.attention_fp8(np.zeros_like(q8), k8, v8, qd, kd, vd, causal, docs)
    c_o, c_l = ref.zero_query_closed_form(ref.fp8_dequantize(v8, vd), causal, docs)
    np.testing.assert_allclose(o0, c_o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse0, c_l, atol=1e-12, rtol=0)


# ---------------------------------------------------------------------------
# Backward
# ---------------------------------------------------------------------------

def _autograd_bwd(q, k, v, dout, causal, docs):
    """torch autograd of SDPA in fp64 ([B,S,H,d] in/out)."""
    tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3).clone().requires_grad_(True)
                  for x in (q, k, v))
    B, S, H, d = q.shape
    if docs is None:
        o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal)
    else:
        doc = torch.zeros(S, dtype=torch.long)
        for t, (a, b) in enumerate(zip(docs[:-1], docs[1:])):
            doc[a:b] = t
        mask = doc[:, None] == doc[None, :]
        if causal:
            mask &= torch.ones(S, S, dtype=torch.bool).tril()
        o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)
    (o * torch.from_numpy(dout).permute(0, 2, 1, 3)).sum().backward()
    return tuple(t.grad.permute(0, 2, 1, 3).numpy() for t in (tq, tk, tv))


BWD_CASES = [(True, None), (False, None), (True, [0, 9, 10, 31, 48]), (False, [0, 20, 48])]


@pytest.mark.parametrize("causal,docs", BWD_CASES)
def test_attention_bwd_matches_autograd(causal, docs):
    q, k, v = _qkv(2, 48, 2, 16, 31)
    dout = _qkv(2, 48, 2, 16, 32)[0]
    got = ref.attention_bwd(q, k, v, dout, causal, docs)
    want = _autograd_bwd(q, k, v, dout, causal, docs)
    for g, w_ in zip(got, want):
        np.testing.assert_allclose(g, w_, atol=1e-12, rtol=0)


def test_attention_bwd_finite_differences():
    q, k, v = _qkv(1, 6, 1, 3, 33)
    dout = _qkv(1, 6, 1, 3, 34)[0]
    grads = ref.attention_bwd(q, k, v, dout, True, [0, 4, 6])
    eps = 1e-6
    for which, g in enumerate(grads):
        for idx in itertools.product(range(6), range(3)):
            arrs = [q.copy(), k.copy(), v.copy()]
            arrs[which][0, idx[0], 0, idx[1]] += eps
            up = (ref.attention(*arrs, True, [0, 4, 6])[0] * dout).sum()
            arrs[which][0, idx[0], 0, idx[1]] -= 2 * eps
            dn = (ref.attention(*arrs, True, [0, 4, 6])[0] * dout).sum()
            assert abs((up - dn) / (2 * eps) - g[0, idx[0], 0, idx[1]]) < 1e-7


@pytest.mark.parametrize("causal,docs", BWD_CASES)
@pytest.mark.parametrize("N,order", [(1, "ascending"), (4, "ascending"), (4, "ring"),
                                     (3, [2, 0, 1])])
def test_ring_backward_equals_the_gradient(causal, docs, N, order):
    q, k, v = _qkv(1, 48, 2, 8, 35)
    dout = _qkv(1, 48, 2, 8, 36)[0]
    got = ref.ring_backward(q, k, v, dout, N, causal, docs, order)
    want = ref.attention_bwd(q, k, v, dout, causal, docs)
    for g, w_ in zip(got, want):
        np.testing.assert_allclose(g, w_, atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal,docs", BWD_CASES)
def test_attention_bwd_closed_forms_and_invariants(causal, docs):
    q, k, v = _qkv(1, 48, 2, 8, 37)
    dout = _qkv(1, 48, 2, 8, 38)[0]
    # constant V: out is constant, so dQ = dK = 0 (dS vanishes)
    vc = np.broadcast_to(v[:, :1], v.shape).copy()
    dq, dk, _ = ref.attention_bwd(q, k, vc, dout, causal, docs)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    # Q = 0: dV is the suffix (causal) or document sum of dO / count
    _, _, dv0 = ref.attention_bwd(np.zeros_like(q), k, v, dout, causal, docs)
    np.testing.assert_allclose(dv0, ref.zero_query_dv_closed_form(dout, causal, docs),
                               atol=1e-12, rtol=0)
    # rows of P sum to 1 and rows of dS sum to 0
    dq, dk, dv = ref.attention_bwd(q, k, v, dout, causal, docs)
    np.testing.assert_allclose(dv.sum(axis=1), dout.sum(axis=1), atol=1e-12)
    assert np.abs(dk.sum(axis=1)).max() < 1e-12
    # the row form of dQ
    rows = np.array([0, 5, 17, 47])
    np.testing.assert_allclose(ref.attention_bwd_rows(q, k, v, dout, 0, 1, rows, causal, docs),
                               dq[0, rows, 1], atol=1e-12, rtol=0)
