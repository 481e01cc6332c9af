"""Host-side checks of the C ABI (no GPU needed).

* libcpring.so loads and exports every function include/cpring.h declares;
* arguments are rejected on the host, before any CUDA call, with the
  documented status codes;
* the integer skip schedule equals the oracle's brute-force enumeration,
  bit for bit, and the ring traffic equals the oracle's simulation.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import context_ring_attention_fwd_gb300 as pkg
from context_ring_attention_fwd_gb300 import inputs
from oracle import ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cpring.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(pkg.LIB_PATH):
        from context_ring_attention_fwd_gb300 import _build
        _build.build()
    return pkg.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cp_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    # and the binding wraps every one of them
    from context_ring_attention_fwd_gb300 import _binding
    assert set(names) <= set(_binding._SIGS)


def test_ring_emulation_workspace_and_checks(lib):
    n = pkg.cp_ring_emulated_workspace_bytes(2, 1024, 2, 128, 4)
    # 4 ranks x 2 slots x (K, V) blocks of 2*256*2*128 bf16, plus 5 fp32 states
    blk = 2 * 256 * 2 * 128
    assert n >= 4 * 2 * 2 * blk * 2 + 5 * blk * 4
    assert pkg.cp_ring_emulated_workspace_bytes(2, 1000, 2, 128, 3) == -1
    f = lib.cp_ring_attn_fwd_emulated
    assert f(None, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 128, 4, 1, None, FAKE, 1 << 30, None, None,
             None) == -1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 96, 4, 1, None, FAKE, 1 << 30, None, None,
             None) == -3
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 128, 4, 1, None, FAKE, 16, None, None,
             None) == -6
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 128, 4, 1, ctypes.c_void_p(0x10002), FAKE,
             1 << 30, None, None, None) == -4


def test_ulysses_checks(lib):
    assert pkg.cp_ulysses_workspace_bytes(1, 1024, 6, 128, 4) == -1   # 6 heads over 4 ranks
    n = pkg.cp_ulysses_workspace_bytes(1, 1024, 8, 128, 4)
    assert n >= 4 * 1024 * 8 * 128 * 2 + 8 * 1024 * 4
    f = lib.cp_ulysses_attn_fwd
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1024, 6, 128, 4, 1, None, FAKE, 1 << 30, None,
             None) == -2
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1024, 8, 128, 4, 1, None, FAKE, 16, None,
             None) == -6


def test_status_strings(lib):
    for code, name in pkg.STATUS_NAMES.items():
        s = pkg.cp_status_string(code)
        assert isinstance(s, str) and s
    assert pkg.cp_status_string(123) == "unknown status"


V = ctypes.c_void_p
FAKE = V(0x10000)        # 16-byte aligned, never dereferenced: checks fail first
ODD = V(0x10002)         # misaligned


def test_rejects_before_any_launch(lib):
    f = lib.cp_ring_attn_fwd
    # null pointers
    assert f(None, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 128, 4, 1, None, None) == -1
    # S % N != 0, N > S, N < 1, bad causal flag
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 250, 2, 128, 4, 1, None, None) == -2
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 128, 8, 1, None, None) == -2
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 128, 0, 1, None, None) == -2
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 128, 4, 2, None, None) == -2
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 256, 2, 128, 4, 1, None, None) == -2
    # unsupported head dims on the tensor-core path
    for d in (32, 96, 256):
        assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, d, 4, 1, None, None) == -3
    # misaligned operand
    assert f(ODD, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 128, 4, 1, None, None) == -4
    g = lib.cp_ring_attn_fwd_f32
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 129, 4, 1, None, None) == -3
    assert g(FAKE, FAKE, FAKE, FAKE, V(0x10001), 1, 256, 2, 64, 4, 1, None, None) == -4
    s = lib.cp_ring_step
    assert s(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 128, 4, 4, 0, 1, None, None) == -2
    assert s(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 128, 4, 0, -1, 1, None, None) == -2
    assert s(FAKE, FAKE, FAKE, None, FAKE, FAKE, 1, 256, 2, 128, 4, 0, 0, 1, None, None) == -1
    m = lib.cp_lse_merge
    assert m(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 0, 2, 64, None) == -2
    assert m(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 2, 129, None) == -3
    assert m(FAKE, FAKE, FAKE, None, FAKE, FAKE, 1, 8, 2, 64, None) == -1
    z = lib.cp_lse_finalize
    assert z(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 2, 64, 2, None) == -2
    assert z(FAKE, FAKE, FAKE, FAKE, ODD, 1, 8, 2, 64, 1, None) == -4


def test_rank_entry_point_rejects_before_any_launch(lib):
    f = lib.cp_ring_attn_fwd_rank
    assert f(None, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 128, 4, 0, 1, None, None) == -1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 128, 4, 4, 1, None, None) == -2
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 128, 4, -1, 1, None, None) == -2
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 96, 4, 0, 1, None, None) == -3
    assert f(ODD, FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 128, 4, 0, 1, None, None) == -4


def test_fp8_entry_points_reject_before_any_launch(lib):
    f = lib.cp_ring_attn_fwd_fp8
    ok = (FAKE,) * 8
    assert f(None, *ok[1:], 1, 1024, 2, 128, 4, 1, None, None) == -1
    assert f(*ok[:4], None, *ok[5:], 1, 1024, 2, 128, 4, 1, None, None) == -1   # a descale
    assert f(*ok, 1, 1024, 2, 64, 4, 1, None, None) == -3            # d = 128 only
    assert f(*ok, 1, 1000, 2, 128, 4, 1, None, None) == -2           # S % N != 0
    assert f(*ok, 1, 1000, 2, 128, 5, 1, None, None) == -2           # 200-row shards: % 16
    assert f(*ok, 1, 1024, 2, 128, 4, 3, None, None) == -2           # causal flag
    assert f(ODD, *ok[1:], 1, 1024, 2, 128, 4, 1, None, None) == -4
    assert f(*ok[:3], V(0x10001), *ok[4:], 1, 1024, 2, 128, 4, 1, None, None) == -4
    g = lib.cp_fp8_quantize
    assert g(None, FAKE, FAKE, 1, 64, 2, 128, 0, None) == -1
    assert g(FAKE, FAKE, FAKE, 1, 64, 2, 96, 0, None) == -3
    assert g(FAKE, FAKE, FAKE, 1, 40, 2, 128, 1, None) == -2          # V^T needs S % 16 == 0
    assert g(FAKE, FAKE, FAKE, 1, 64, 2, 128, 2, None) == -2
    assert g(FAKE, ODD, FAKE, 1, 64, 2, 128, 0, None) == -4


@pytest.mark.parametrize("S,N,T", [(64, 4, 16), (96, 3, 8), (48, 4, 5), (40, 2, 7), (32, 8, 4)])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("ndocs", [0, 1, 3, 6])
def test_schedule_bit_exact_vs_oracle(lib, S, N, T, causal, ndocs):
    docs = None if ndocs == 0 else inputs.random_doc_offsets(S, ndocs, seed=S * 7 + ndocs)
    got = pkg.cp_ring_schedule(S, N, T, T, causal, docs)
    want = ref.tile_schedule(S, N, T, T, causal, docs)
    assert got == want
    # rectangular tiles too
    got2 = pkg.cp_ring_schedule(S, N, T, T + 3, causal, docs)
    assert got2 == ref.tile_schedule(S, N, T, T + 3, causal, docs)


def test_schedule_shard_pairs_and_tile_closed_forms(lib):
    for N in (1, 2, 4, 8):
        pairs = pkg.cp_ring_schedule(64 * N, N, 64, 64, True)
        assert len(pairs) == N * (N + 1) // 2
        assert [p for p in pairs if p[0] == 0] == [(0, 0)]
    # the 128K workload at 128-row tiles: T(T+1)/2 tile pairs per (b, h)
    w = inputs.BY_NAME["bf16_causal_128k"]
    n = ctypes.c_int64(0)
    assert lib.cp_ring_schedule(w.S, w.n_shards, 128, 128, 1, None, None, 0, ctypes.byref(n)) == 0
    T = w.S // 128
    assert n.value == T * (T + 1) // 2


def test_schedule_errors(lib):
    n = ctypes.c_int64(0)
    assert lib.cp_ring_schedule(10, 3, 2, 2, 1, None, None, 0, ctypes.byref(n)) == -2
    bad = (ctypes.c_int32 * 3)(0, 5, 5)
    assert lib.cp_ring_schedule(10, 2, 2, 2, 1, ctypes.cast(bad, V), None, 0, ctypes.byref(n)) == -7
    buf = (ctypes.c_int32 * 4)()
    assert lib.cp_ring_schedule(16, 4, 4, 4, 1, None, ctypes.cast(buf, V), 2,
                                ctypes.byref(n)) == -6
    assert n.value == 10 and list(buf) == [0, 0, 1, 0]


@pytest.mark.parametrize("N", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_traffic_matches_simulation(lib, N, causal):
    B, S, H, d, nb = 2, 96 * N, 3, 64, 2
    got = pkg.cp_ring_traffic(B, S, H, d, nb, N, causal)
    assert got == ref.ring_traffic_simulated(B, S, H, d, nb, N, causal)


def test_traffic_at_workload_sizes(lib):
    # 2 (G/N)(N-1) with G = K + V bytes of the whole sequence
    for w in inputs.WORKLOADS[1:]:
        nb = 2
        got = pkg.cp_ring_traffic(w.B, w.S, w.H, w.d, nb, w.n_shards, False)
        G = 2 * w.B * w.S * w.H * w.d * nb
        assert got == [2 * (G // w.n_shards) * (w.n_shards - 1)] * w.n_shards


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    from context_ring_attention_fwd_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        _binding.lib()
