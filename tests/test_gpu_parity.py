"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerances (fixed for this hot path): fp32 inputs within max-abs 1e-4 of the
oracle; bf16 inputs with fp32 accumulation within max-abs 2e-2 and mean-abs
2e-3, applied to the output and, with the same max-abs bound, to the
log-sum-exp.  Full-size workloads are checked on seeded samples of query
rows (512 per head) plus the Q = 0 closed form over every row.
"""
import os

import numpy as np
import pytest
import torch

import context_ring_attention_fwd_gb300 as pkg
from context_ring_attention_fwd_gb300 import inputs
from oracle import ref

pytestmark = pytest.mark.gpu

F32_TOL = 1e-4
BF16_MAX, BF16_MEAN = 2e-2, 2e-3


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


DEV = "cuda"


def _np(t):
    return t.detach().float().cpu().numpy()


def _check_bf16(out, lse, want_o, want_l, what=""):
    e = np.abs(_np(out) - want_o)
    el = np.abs(_np(lse) - want_l)
    assert np.all(np.isfinite(_np(out))), what
    assert e.max() <= BF16_MAX, (what, e.max())
    assert e.mean() <= BF16_MEAN, (what, e.mean())
    assert el.max() <= BF16_MAX, (what, el.max())


def _check_f32(out, lse, want_o, want_l, what=""):
    assert np.abs(_np(out) - want_o).max() <= F32_TOL, what
    assert np.abs(_np(lse) - want_l).max() <= F32_TOL, what


# ----------------------------------------------------------------- fp32 path
def test_tiny_f32_workload():
    w = inputs.BY_NAME["tiny_f32_causal"]
    q, k, v, docs = inputs.workload_inputs(w)
    out, lse = pkg.ring_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), w.n_shards, w.causal, docs)
    want_o, want_l = ref.attention(q.numpy(), k.numpy(), v.numpy(), w.causal, docs)
    _check_f32(out, lse, want_o, want_l)
    assert pkg.cp_get_last_status() == 0


@pytest.mark.parametrize("causal,docs", [(True, None), (False, None), (True, [0, 37, 100, 192]),
                                         (False, [0, 60, 61, 192])])
def test_f32_steps_and_merge_against_oracle(causal, docs):
    B, S, H, d, N = 2, 192, 2, 48, 3
    q, k, v = inputs.make_qkv(B, S, H, d, seed=3, dtype=torch.float32)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    dd = pkg.doc_offsets_tensor(docs, DEV)
    L = S // N
    for i in range(N):
        for j in range(N):
            o = torch.empty((B, L, H, d), device=DEV)
            m = torch.empty((B, H, L), device=DEV)
            l = torch.empty((B, H, L), device=DEV)
            pkg.cp_ring_step(qd, kd, vd, o, m, l, N, i, j, causal, dd)
            wo, wm, wl = ref.partial_step(q.numpy(), k.numpy(), v.numpy(), N, i, j, causal, docs)
            empty = ~np.isfinite(wm)
            assert np.array_equal(~np.isfinite(_np(m)), empty)
            assert np.all(_np(l)[empty] == 0)
            np.testing.assert_allclose(_np(m)[~empty], wm[~empty], rtol=0, atol=F32_TOL)
            np.testing.assert_allclose(_np(l), wl, rtol=1e-5, atol=F32_TOL)
            np.testing.assert_allclose(_np(o), wo, rtol=1e-5, atol=F32_TOL)
    want_o, want_l = ref.attention(q.numpy(), k.numpy(), v.numpy(), causal, docs)
    for order in ("ascending", "ring", [2, 0, 1]):
        out, lse = pkg.ring_attn_composed(qd, kd, vd, N, causal, docs, order)
        _check_f32(out, lse, want_o, want_l, order)
    out, lse = pkg.ring_attn_fwd(qd, kd, vd, N, causal, docs)
    _check_f32(out, lse, want_o, want_l, "fused")


# ----------------------------------------------------------------- bf16 path
BF16_CASES = [
    # B, S, H, d, N, causal, docs
    (1, 128, 1, 128, 1, True, None),          # one tile
    (1, 128, 1, 128, 1, False, None),
    (1, 512, 2, 128, 1, True, None),          # several tiles, one pair of q tiles
    (2, 768, 3, 128, 3, True, None),          # shards of 256
    (1, 640, 2, 128, 2, False, None),         # shards of 320: ragged tiles inside shards
    (1, 1000, 2, 64, 5, True, None),          # d = 64, shards of 200
    (1, 1000, 2, 128, 4, False, None),        # S not a multiple of the tile
    (1, 1024, 2, 128, 4, True, [0, 100, 101, 300, 777, 1024]),
    (2, 896, 2, 64, 7, False, [0, 128, 500, 896]),
]


@pytest.mark.parametrize("B,S,H,d,N,causal,docs", BF16_CASES)
def test_bf16_fused_against_oracle(B, S, H, d, N, causal, docs):
    q, k, v = inputs.make_qkv(B, S, H, d, seed=S + d + N, dtype=torch.bfloat16)
    out, lse = pkg.ring_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), N, causal, docs)
    assert pkg.cp_get_last_status() == 0
    want_o, want_l = ref.attention(_np(q), _np(k), _np(v), causal, docs)
    _check_bf16(out, lse, want_o, want_l)


def _jump_inputs(seed, bumps, blocks, B=1, S=768, H=2, d=128):
    """Small keys (scores of order 1) except blocks of 32 keys raised by the
    given amounts, so a row's scores jump far past its running maximum."""
    q, k, v = inputs.make_qkv(B, S, H, d, seed=seed, dtype=torch.bfloat16)
    q = (q.float() * 0.25 + 1.0).to(torch.bfloat16)
    k = (k.float() * 0.25)
    for a, bump in zip(blocks, bumps):
        k[:, a:a + 32] += bump
    return q, k.to(torch.bfloat16), v


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("blocks", [(128, 384), (192, 448), (176, 432)],
                         ids=["first-half", "second-half", "straddling"])
def test_bf16_scores_jump_past_the_reference(causal, blocks):
    """Scores that rise by about 2^98 and then 2^196 (as base-2 exponents)
    over the first key tile's: the kernel's no-max pass must see it (through
    the first 64 keys' row sum or the last 64 keys' row max, depending on
    where the block sits) and redo the tile against a new reference point."""
    q, k, v = _jump_inputs(71, (6.0, 12.0), blocks)
    out, lse = pkg.ring_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), 2, causal)
    assert pkg.cp_get_last_status() == 0
    want_o, want_l = ref.attention(_np(q), _np(k), _np(v), causal)
    _check_bf16(out, lse, want_o, want_l, (causal, blocks))


@pytest.mark.parametrize("causal,docs", [(True, None), (False, None),
                                         (True, [0, 300, 301, 700, 1024])])
def test_bf16_steps_against_oracle(causal, docs):
    B, S, H, d, N = 1, 1024, 2, 128, 4
    q, k, v = inputs.make_qkv(B, S, H, d, seed=77, dtype=torch.bfloat16)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    dd = pkg.doc_offsets_tensor(docs, DEV)
    L = S // N
    qn, kn, vn = _np(q), _np(k), _np(v)
    for i in range(N):
        for j in range(N):
            o = torch.full((B, L, H, d), 7.0, device=DEV)
            m = torch.full((B, H, L), 7.0, device=DEV)
            l = torch.full((B, H, L), 7.0, device=DEV)
            pkg.cp_ring_step(qd, kd, vd, o, m, l, N, i, j, causal, dd)
            wo, wm, wl = ref.partial_step(qn, kn, vn, N, i, j, causal, docs)
            empty = ~np.isfinite(wm)
            assert np.array_equal(~np.isfinite(_np(m)), empty), (i, j)
            assert np.all(_np(l)[empty] == 0) and np.all(_np(o)[np.transpose(empty, (0, 2, 1))] == 0)
            # m and l exactly as the pages define them (true row max); P in bf16
            np.testing.assert_allclose(_np(m)[~empty], wm[~empty], rtol=0, atol=1e-3)
            rel_l = np.abs(_np(l) - wl) / np.maximum(wl, 1.0)
            assert rel_l.max() <= 1e-2, (i, j, rel_l.max())
            # compare the normalised partial O_ij / l_ij
            lw = np.transpose(np.where(empty, 1.0, wl), (0, 2, 1))[..., None]
            lg = np.transpose(np.where(empty, 1.0, _np(l)), (0, 2, 1))[..., None]
            e = np.abs(_np(o) / lg - wo / lw)
            assert e.max() <= BF16_MAX and e.mean() <= BF16_MEAN, (i, j, e.max())


@pytest.mark.parametrize("order", ["ascending", "ring", [3, 1, 0, 2]])
def test_bf16_composed_ring_any_order(order):
    B, S, H, d, N = 1, 1024, 2, 128, 4
    q, k, v = inputs.make_qkv(B, S, H, d, seed=78, dtype=torch.bfloat16)
    out, lse = pkg.ring_attn_composed(q.to(DEV), k.to(DEV), v.to(DEV), N, True, None, order)
    want_o, want_l = ref.attention(_np(q), _np(k), _np(v), True, None)
    _check_bf16(out, lse, want_o, want_l, str(order))


def test_bf16_deterministic_and_guard_bands():
    B, S, H, d, N = 1, 1536, 4, 128, 3
    q, k, v = (t.to(DEV) for t in inputs.make_qkv(B, S, H, d, seed=5, dtype=torch.bfloat16))
    pad = 4096
    out_buf = torch.full((B * S * H * d + 2 * pad,), 3.0, dtype=torch.bfloat16, device=DEV)
    lse_buf = torch.full((B * H * S + 2 * pad,), 3.0, dtype=torch.float32, device=DEV)
    out = out_buf[pad:pad + B * S * H * d].view(B, S, H, d)
    lse = lse_buf[pad:pad + B * H * S].view(B, H, S)
    pkg.cp_ring_attn_fwd(q, k, v, out, lse, N, True)
    o1, l1 = out.clone(), lse.clone()
    for _ in range(3):
        pkg.cp_ring_attn_fwd(q, k, v, out, lse, N, True)
        assert torch.equal(out, o1) and torch.equal(lse, l1)
    assert torch.all(out_buf[:pad] == 3.0) and torch.all(out_buf[-pad:] == 3.0)
    assert torch.all(lse_buf[:pad] == 3.0) and torch.all(lse_buf[-pad:] == 3.0)


def test_bf16_causal_poisoning_of_unneeded_shards():
    # Rows of shard i never read K/V of shards > i: NaN there changes nothing.
    B, S, H, d, N = 1, 2048, 2, 128, 4
    q, k, v = (t.to(DEV) for t in inputs.make_qkv(B, S, H, d, seed=9, dtype=torch.bfloat16))
    out, lse = pkg.ring_attn_fwd(q, k, v, N, True)
    L = S // N
    for i in range(N - 1):
        kp, vp = k.clone(), v.clone()
        kp[:, (i + 1) * L:] = float("nan")
        vp[:, (i + 1) * L:] = float("nan")
        o2, l2 = pkg.ring_attn_fwd(q, kp, vp, N, True)
        rows = slice(0, (i + 1) * L)
        assert torch.equal(o2[:, rows], out[:, rows]), i
        assert torch.equal(l2[:, :, rows], lse[:, :, rows]), i
    # with documents: whole tiles before the first document start of a shard
    docs = [0, 700, 1300, 2048]
    out, lse = pkg.ring_attn_fwd(q, k, v, N, True, docs)
    i = 2                                            # shard [1024, 1536): first doc starts at 700
    cut = (700 // 128) * 128
    kp, vp = k.clone(), v.clone()
    kp[:, :cut] = float("nan")
    vp[:, :cut] = float("nan")
    kp[:, (i + 1) * L:] = float("nan")
    vp[:, (i + 1) * L:] = float("nan")
    o2, l2 = pkg.ring_attn_fwd(q, kp, vp, N, True, docs)
    rows = slice(i * L, (i + 1) * L)
    assert torch.equal(o2[:, rows], out[:, rows])
    assert torch.equal(l2[:, :, rows], lse[:, :, rows])


def test_bf16_empty_step_is_identity():
    B, S, H, d, N = 1, 512, 2, 128, 4
    q, k, v = (t.to(DEV) for t in inputs.make_qkv(B, S, H, d, seed=2, dtype=torch.bfloat16))
    L = S // N
    o = torch.full((B, L, H, d), 5.0, device=DEV)
    m = torch.full((B, H, L), 5.0, device=DEV)
    l = torch.full((B, H, L), 5.0, device=DEV)
    pkg.cp_ring_step(q, k, v, o, m, l, N, 1, 3, True)      # j > i: fully masked
    assert torch.all(o == 0) and torch.all(l == 0) and torch.all(torch.isneginf(m))


def test_malformed_doc_offsets_reported():
    B, S, H, d, N = 1, 256, 1, 128, 2
    q, k, v = (t.to(DEV) for t in inputs.make_qkv(B, S, H, d, seed=2, dtype=torch.bfloat16))
    out = torch.full_like(q, 9.0)
    lse = torch.full((B, H, S), 9.0, device=DEV)
    for bad in ([0, 100, 100, 256], [1, 256], [0, 300], [0, 50, 20, 256]):
        dd = torch.tensor(bad, dtype=torch.int32, device=DEV)
        pkg.cp_ring_attn_fwd(q, k, v, out, lse, N, True, dd)
        assert pkg.cp_get_last_status() == pkg.STATUS_CODES["CP_ERR_DOC_OFFSETS"], bad
        assert torch.all(out == 9.0) and torch.all(lse == 9.0)
    assert pkg.cp_get_last_status() == 0


def test_bounded_wait_runs_out_and_context_recovers():
    # A K tile that is never loaded (a flag nothing sets): the MMA thread's
    # wait gives up after 0.3 s, the CTA drains and exits, the host reads
    # CP_ERR_TIMEOUT, and the next call on the same context is correct.
    B, S, H, d, N = 1, 1024, 2, 128, 2
    q, k, v = inputs.make_qkv(B, S, H, d, seed=17, dtype=torch.bfloat16)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    assert pkg.cp_get_last_status() == 0
    try:
        pkg.test_set_wait_fault(True, 300_000_000)
        out = torch.empty_like(qd)
        lse = torch.empty((B, H, S), dtype=torch.float32, device=DEV)
        pkg.cp_ring_attn_fwd(qd, kd, vd, out, lse, N, True)
        assert pkg.cp_get_last_status() == pkg.STATUS_CODES["CP_ERR_TIMEOUT"]
    finally:
        pkg.test_set_wait_fault(False, 0)
    assert pkg.cp_get_last_status() == 0
    out, lse = pkg.ring_attn_fwd(qd, kd, vd, N, True)
    assert pkg.cp_get_last_status() == 0
    want_o, want_l = ref.attention(_np(q), _np(k), _np(v), True, None)
    _check_bf16(out, lse, want_o, want_l)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("overlap", [True, False])
@pytest.mark.parametrize("B,S,H,d,N", [(2, 1024, 2, 128, 4), (1, 768, 3, 64, 3)])
def test_ring_emulation_explicit_buffers(causal, overlap, B, S, H, d, N):
    # The ring with per-rank K/V buffers and copy-engine transfers gives the
    # fused result, and each rank receives exactly the blocks the traffic
    # count says: i blocks under causality, N - 1 otherwise.
    q, k, v = inputs.make_qkv(B, S, H, d, seed=S + N, dtype=torch.bfloat16)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    out = torch.full_like(qd, 9.0)
    lse = torch.full((B, H, S), 9.0, dtype=torch.float32, device=DEV)
    cs = torch.cuda.Stream() if overlap else None
    recv = pkg.cp_ring_attn_fwd_emulated(qd, kd, vd, out, lse, N, causal, copy_stream=cs)
    torch.cuda.synchronize()
    assert pkg.cp_get_last_status() == 0
    want_o, want_l = ref.attention(_np(q), _np(k), _np(v), causal, None)
    _check_bf16(out, lse, want_o, want_l)
    fo, fl = pkg.ring_attn_fwd(qd, kd, vd, N, causal)
    e = (out.float() - fo.float()).abs()
    assert e.max().item() <= BF16_MAX and e.mean().item() <= BF16_MEAN
    L = S // N
    block = 2 * B * L * H * d * 2  # K and V of one shard, bf16
    want_recv = [i * block for i in range(N)] if causal else [(N - 1) * block] * N
    assert recv == want_recv
    sent = [recv[(i + 1) % N] if (not causal or i < N - 1) else 0 for i in range(N)]
    assert [s_ + r_ for s_, r_ in zip(sent, recv)] == pkg.cp_ring_traffic(B, S, H, d, 2, N, causal)


@pytest.mark.parametrize("causal,docs,N", [(True, [0, 300, 301, 777, 1500, 2048], 8),
                                           (False, [0, 128, 900, 2048], 4),
                                           (True, [0, 2000, 2048], 2)])
def test_ring_emulation_with_documents(causal, docs, N):
    # Packed documents through the per-rank ring: boundaries anywhere,
    # including inside shards and tiles and one-token documents.  Every step
    # masks by document, so the ring gives the oracle's result and the
    # fused kernel's within the bf16 bounds; rows of one document never see
    # another's keys.
    B, S, H, d = 1, 2048, 2, 128
    q, k, v = inputs.make_qkv(B, S, H, d, seed=S + N + 7, dtype=torch.bfloat16)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    out = torch.full_like(qd, 9.0)
    lse = torch.full((B, H, S), 9.0, dtype=torch.float32, device=DEV)
    dd = pkg.doc_offsets_tensor(docs, DEV)
    recv = pkg.cp_ring_attn_fwd_emulated(qd, kd, vd, out, lse, N, causal,
                                         copy_stream=torch.cuda.Stream(), doc_offsets=dd)
    torch.cuda.synchronize()
    assert pkg.cp_get_last_status() == 0
    want_o, want_l = ref.attention(_np(q), _np(k), _np(v), causal, docs)
    _check_bf16(out, lse, want_o, want_l)
    fo, fl = pkg.ring_attn_fwd(qd, kd, vd, N, causal, docs)
    e = (out.float() - fo.float()).abs()
    assert e.max().item() <= BF16_MAX and e.mean().item() <= BF16_MEAN
    assert (lse - fl).abs().max().item() <= BF16_MAX
    L = S // N
    block = 2 * B * L * H * d * 2
    assert recv == ([i * block for i in range(N)] if causal else [(N - 1) * block] * N)


@pytest.mark.parametrize("causal,docs", [(True, None), (False, None),
                                         (True, [0, 300, 301, 777, 1024])])
def test_ulysses_all_to_all_form(causal, docs):
    # Head-split attention between two all-to-all permutations gives the
    # ring's result; with shards of whole 256-row tile pairs the same tiles
    # meet in the same order, so it is bit-identical to the fused kernel.
    B, S, H, d, N = 2, 1024, 8, 128, 4
    q, k, v = inputs.make_qkv(B, S, H, d, seed=55, dtype=torch.bfloat16)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    out = torch.full_like(qd, 9.0)
    lse = torch.full((B, H, S), 9.0, dtype=torch.float32, device=DEV)
    dd = pkg.doc_offsets_tensor(docs, DEV)
    moved = pkg.cp_ulysses_attn_fwd(qd, kd, vd, out, lse, N, causal, dd)
    assert pkg.cp_get_last_status() == 0
    fo, fl = pkg.ring_attn_fwd(qd, kd, vd, N, causal, docs)
    assert torch.equal(out, fo) and torch.equal(lse, fl)
    want_o, want_l = ref.attention(_np(q), _np(k), _np(v), causal, docs)
    _check_bf16(out, lse, want_o, want_l)
    shard = B * (S // N) * H * d * 2
    assert moved == 8 * shard * (N - 1)


@pytest.mark.parametrize("S,N,causal,ndocs", [(1024, 4, True, 0), (1040, 2, True, 0),
                                              (768, 3, False, 0), (2048, 4, True, 5),
                                              (2048, 1, False, 3), (4096, 8, True, 12)])
def test_device_schedule_matches_host_schedule(S, N, causal, ndocs):
    """The key-tile range the fused kernel walks for each 128-row query tile
    (its own decoding, run on the device) is exactly the contiguous range of
    the host schedule, which the oracle pins bit for bit."""
    docs = None if ndocs == 0 else inputs.random_doc_offsets(S, ndocs, seed=S + ndocs)
    dev = pkg.cp_ring_schedule_device(S, N, causal, pkg.doc_offsets_tensor(docs, DEV)).cpu()
    pairs = pkg.cp_ring_schedule(S, N, 128, 128, causal, docs)
    by_q = {}
    for qt, kt in pairs:
        by_q.setdefault(qt, []).append(kt)
    assert sorted(by_q) == list(range(dev.shape[0]))
    for qt, kts in by_q.items():
        lo, hi = min(kts), max(kts)
        assert len(kts) == hi - lo + 1                     # contiguous
        assert dev[qt].tolist() == [lo, hi], (qt, dev[qt].tolist(), lo, hi)


@pytest.mark.parametrize("B,S,H,d,N,causal,docs", [(1, 1024, 2, 128, 4, True, None),
                                                    (2, 768, 2, 64, 3, False, None),
                                                    (1, 1536, 2, 128, 4, True, [0, 300, 301, 777, 1536])])
def test_rank_calls_and_host_path_equal_the_fused_call(B, S, H, d, N, causal, docs):
    """cp_ring_attn_fwd_rank for every rank, and the pipelined host-buffer
    path built on it, give bitwise the result of one cp_ring_attn_fwd call;
    one rank writes only its own rows."""
    q, k, v = (t.to(DEV) for t in inputs.make_qkv(B, S, H, d, 61, torch.bfloat16))
    dd = pkg.doc_offsets_tensor(docs, DEV)
    want_o, want_l = pkg.ring_attn_fwd(q, k, v, N, causal, docs)
    out = torch.full_like(q, 3.0)
    lse = torch.full((B, H, S), 3.0, dtype=torch.float32, device=DEV)
    L = S // N
    pkg.cp_ring_attn_fwd_rank(q, k, v, out, lse, N, 1, causal, dd)
    assert torch.equal(out[:, L:2 * L], want_o[:, L:2 * L])
    assert torch.equal(lse[:, :, L:2 * L], want_l[:, :, L:2 * L])
    assert torch.all(out[:, :L] == 3.0) and torch.all(out[:, 2 * L:] == 3.0)
    assert torch.all(lse[:, :, :L] == 3.0) and torch.all(lse[:, :, 2 * L:] == 3.0)
    for r in range(N):
        pkg.cp_ring_attn_fwd_rank(q, k, v, out, lse, N, r, causal, dd)
    assert torch.equal(out, want_o) and torch.equal(lse, want_l)
    ho, hl = pkg.ring_attn_fwd_host(*(t.cpu().pin_memory() for t in (q, k, v)), N, causal, docs)
    assert torch.equal(ho, want_o.cpu()) and torch.equal(hl, want_l.cpu())
    assert pkg.cp_get_last_status() == 0
    oo, ol = ref.attention(_np(q), _np(k), _np(v), causal, docs)
    _check_bf16(ho, hl, oo, ol, "host path")


def test_host_entry_through_the_c_abi_twice_and_fp32():
    """cp_ring_attn_fwd_host called directly through ctypes with pageable
    and page-locked host buffers, twice in a row on the same workspace: both
    calls equal cp_ring_attn_fwd bit for bit.  The fp32 form equals the fp32
    fused call bit for bit and is within 1e-4 of the oracle."""
    import ctypes
    B, S, H, d, N = 2, 1280, 2, 128, 5
    lib = pkg.lib()
    stream = torch.cuda.current_stream()
    for dt in (torch.bfloat16, torch.float32):
        esz = 2 if dt == torch.bfloat16 else 4
        ws = torch.empty(pkg.cp_ring_attn_fwd_host_workspace_bytes(B, S, H, d, N, esz),
                         dtype=torch.uint8, device=DEV)
        for seed, pinned in ((71, True), (72, False)):
            q, k, v = inputs.make_qkv(B, S, H, d, seed, dt)
            if pinned:
                q, k, v = (t.pin_memory() for t in (q, k, v))
            ho = torch.full((B, S, H, d), 7.0, dtype=dt)
            hl = torch.full((B, H, S), 7.0, dtype=torch.float32)
            name = "cp_ring_attn_fwd_host" if esz == 2 else "cp_ring_attn_fwd_host_f32"
            p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
            st = getattr(lib, name)(p(q), p(k), p(v), p(ho), p(hl), B, S, H, d, N, 1, None,
                                    p(ws), ws.numel(), ctypes.c_void_p(stream.cuda_stream))
            assert st == 0, pkg.STATUS_NAMES.get(st, st)
            stream.synchronize()
            assert pkg.cp_get_last_status() == 0
            fo, fl = pkg.ring_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), N, True)
            assert torch.equal(ho, fo.cpu()) and torch.equal(hl, fl.cpu()), (dt, seed)
            if dt == torch.float32:
                wo, wl = ref.attention(q.numpy(), k.numpy(), v.numpy(), True, None)
                _check_f32(ho, hl, wo, wl)


def test_host_entry_with_documents_and_without_mask_equals_fused():
    """cp_ring_attn_fwd_host on packed documents and without the causal mask
    (every rank then waits for every shard): bf16 and fp32 outputs equal the
    fused call with the same shard count bit for bit."""
    import ctypes
    B, S, H, d, N = 2, 4096, 2, 128, 2
    lib = pkg.lib()
    stream = torch.cuda.current_stream()
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    for dt in (torch.bfloat16, torch.float32):
        esz = 2 if dt == torch.bfloat16 else 4
        name = "cp_ring_attn_fwd_host" if esz == 2 else "cp_ring_attn_fwd_host_f32"
        ws = torch.empty(pkg.cp_ring_attn_fwd_host_workspace_bytes(B, S, H, d, N, esz),
                         dtype=torch.uint8, device=DEV)
        q, k, v = (t.pin_memory() for t in inputs.make_qkv(B, S, H, d, 73, dt))
        for causal, docs in ((True, None), (True, [0, 700, 701, 2500, 4096]), (False, None)):
            docs_t = pkg.doc_offsets_tensor(docs, DEV)
            ho = torch.full((B, S, H, d), 7.0, dtype=dt)
            hl = torch.full((B, H, S), 7.0, dtype=torch.float32)
            st = getattr(lib, name)(p(q), p(k), p(v), p(ho), p(hl), B, S, H, d, N, int(causal),
                                    p(docs_t), p(ws), ws.numel(),
                                    ctypes.c_void_p(stream.cuda_stream))
            assert st == 0, pkg.STATUS_NAMES.get(st, st)
            stream.synchronize()
            assert pkg.cp_get_last_status() == 0
            fo, fl = pkg.ring_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), N, causal, docs)
            assert torch.equal(ho, fo.cpu()) and torch.equal(hl, fl.cpu()), (dt, causal, docs)


@pytest.mark.parametrize("B,S,H,d,N,causal", [(1, 2048, 4, 128, 4, True), (2, 1280, 3, 128, 5, False),
                                               (1, 1000, 2, 64, 4, True),
                                               (1, 16384, 32, 128, 4, True)])  # grouped heads
def test_claimed_items_equal_the_fixed_deal(B, S, H, d, N, causal):
    """One document covering the whole sequence ([0, S]) sends the launch
    down the claimed-items path (work queue, item ring, items published with
    their Q loads, slots ranked by cost) with the arithmetic of the launch
    without documents, which takes the fixed deal: the two must agree bit
    for bit, whole-sequence and rank by rank, so no item is lost, repeated
    or given the wrong rows by either deal."""
    q, k, v = (t.to(DEV) for t in inputs.make_qkv(B, S, H, d, seed=S + N, dtype=torch.bfloat16))
    fo, fl = pkg.ring_attn_fwd(q, k, v, N, causal, None)
    co, cl = pkg.ring_attn_fwd(q, k, v, N, causal, [0, S])
    assert pkg.cp_get_last_status() == 0
    assert torch.equal(fo, co) and torch.equal(fl, cl)
    docs_t = pkg.doc_offsets_tensor([0, S], DEV)
    ro = torch.full_like(q, 7.0)
    rl = torch.full((B, H, S), 7.0, dtype=torch.float32, device=DEV)
    for i in range(N):
        pkg.cp_ring_attn_fwd_rank(q, k, v, ro, rl, N, i, causal, docs_t)
    assert pkg.cp_get_last_status() == 0
    assert torch.equal(ro, fo) and torch.equal(rl, fl)


def test_native_kernels_launch():
    before = pkg.launch_counts()
    q, k, v = (t.to(DEV) for t in inputs.make_qkv(1, 256, 1, 128, seed=1, dtype=torch.bfloat16))
    pkg.ring_attn_fwd(q, k, v, 2, True)
    pkg.ring_attn_fwd(q.float(), k.float(), v.float(), 2, True)
    after = pkg.launch_counts()
    assert after[0] == before[0] + 1 and after[1] == before[1] + 1


# ------------------------------------------------------------ full workloads
def _device_inputs(w):
    q, k, v = inputs.make_qkv(w.B, w.S, w.H, w.d, w.seed, w.torch_dtype, w.scale, device=DEV)
    docs = (inputs.make_doc_offsets(w.S, w.seed + 1, w.doc_min, w.doc_max)
            if w.packed_docs else None)
    return q, k, v, docs


def _check_rows(w, q, k, v, docs, out, lse, n_rows=512):
    """Every (b, h) on a seeded sample of n_rows query rows, plus the first
    and last row of every shard, against the oracle row by row."""
    qn, kn, vn = _np(q), _np(k), _np(v)
    on, ln = _np(out), _np(lse)
    L = w.S // w.n_shards
    edges = np.array(sorted({r for i in range(w.n_shards) for r in (i * L, (i + 1) * L - 1)}))
    errs, errs_l = [], []
    for b in range(w.B):
        for h in range(w.H):
            rows = inputs.sample_rows(w.S, n_rows, seed=w.seed * 100 + b * w.H + h)
            rows = np.union1d(rows, edges)
            wo, wl = ref.attention_rows(qn, kn, vn, b, h, rows, w.causal, docs)
            errs.append(np.abs(on[b, rows, h] - wo))
            errs_l.append(np.abs(ln[b, h, rows] - wl))
    e = np.concatenate([x.ravel() for x in errs])
    el = np.concatenate([x.ravel() for x in errs_l])
    assert np.all(np.isfinite(e)) and np.all(np.isfinite(el)), w.name
    assert e.max() <= BF16_MAX and e.mean() <= BF16_MEAN, (w.name, e.max(), e.mean())
    assert el.max() <= BF16_MAX, (w.name, el.max())


def _zero_q_check(w, k, v, docs):
    q0 = torch.zeros_like(k)
    out, lse = pkg.ring_attn_fwd(q0, k, v, w.n_shards, w.causal, docs)
    cf_o, cf_l = ref.zero_query_closed_form(_np(v), w.causal, docs)
    e = np.abs(_np(out) - cf_o)
    assert e.max() <= BF16_MAX and e.mean() <= BF16_MEAN, (w.name, e.max(), e.mean())
    assert np.abs(_np(lse) - cf_l).max() <= BF16_MAX


def test_workload_causal_8k_and_shard_invariance():
    """Every row of every head against the oracle, at N = 1, 2, 4 and 8
    shards; the outputs and log-sum-exps of the four shard counts also agree
    with each other within the same bounds."""
    w = inputs.BY_NAME["bf16_causal_8k"]
    q, k, v, docs = _device_inputs(w)
    want_o, want_l = ref.attention(_np(q), _np(k), _np(v), w.causal, docs)
    outs = {}
    for N in (1, 2, 4, 8):
        outs[N] = pkg.ring_attn_fwd(q, k, v, N, w.causal, docs)
        assert pkg.cp_get_last_status() == 0
        _check_bf16(*outs[N], want_o, want_l, f"N={N}")
    for N in (1, 2, 8):
        e = (outs[N][0].float() - outs[w.n_shards][0].float()).abs()
        assert e.max().item() <= BF16_MAX and e.mean().item() <= BF16_MEAN, N
        el = (outs[N][1] - outs[w.n_shards][1]).abs()
        assert el.max().item() <= BF16_MAX, N
    _zero_q_check(w, k, v, docs)


def test_workload_full_32k():
    w = inputs.BY_NAME["bf16_full_32k"]
    q, k, v, docs = _device_inputs(w)
    out, lse = pkg.ring_attn_fwd(q, k, v, w.n_shards, w.causal, docs)
    assert pkg.cp_get_last_status() == 0
    _check_rows(w, q, k, v, docs, out, lse, n_rows=512)
    _zero_q_check(w, k, v, docs)


def test_workload_causal_128k():
    w = inputs.BY_NAME["bf16_causal_128k"]
    q, k, v, docs = _device_inputs(w)
    out, lse = pkg.ring_attn_fwd(q, k, v, w.n_shards, w.causal, docs)
    assert pkg.cp_get_last_status() == 0
    _check_rows(w, q, k, v, docs, out, lse, n_rows=512)
    _zero_q_check(w, k, v, docs)


def test_workload_packed_docs_64k():
    w = inputs.BY_NAME["bf16_causal_packed_64k"]
    q, k, v, docs = _device_inputs(w)
    out, lse = pkg.ring_attn_fwd(q, k, v, w.n_shards, w.causal, docs)
    assert pkg.cp_get_last_status() == 0
    _check_rows(w, q, k, v, docs, out, lse, n_rows=512)
    _zero_q_check(w, k, v, docs)
