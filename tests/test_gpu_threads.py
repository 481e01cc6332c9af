"""The library's per-device shared state under concurrent host threads.

The library keeps a few things per device for the process's life: the cached
scratch that launches with documents lease (the doc-scan word and the
cost-ranked slot order), the backward's second stream for its dQ launch, and
the host-buffer entry's copy streams.  Two host threads here drive every one
of those on their own streams at the same time, several calls each, and
every result must equal the same call made alone, bit for bit: a lease
handed to one thread while another's kernels still read it, or an event of
one call waited on by another, would show as a difference.
"""
import os
import threading

import pytest
import torch

import context_ring_attention_fwd_gb300 as pkg
from context_ring_attention_fwd_gb300 import inputs

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


def _case(seed, S, docs):
    B, H, d, N = 1, 2, 128, 4
    q, k, v = (t.to(DEV) for t in inputs.make_qkv(B, S, H, d, seed=seed, dtype=torch.bfloat16))
    dout = inputs.make_qkv(B, S, H, d, seed=seed + 1, dtype=torch.bfloat16)[0].to(DEV)
    return dict(q=q, k=k, v=v, dout=dout, N=N, docs=docs, S=S)


def _run(c, stream):
    """Forward with documents, backward, and the host-buffer entry, all on
    `stream`; returns host copies of every output."""
    q, k, v, N, docs = c["q"], c["k"], c["v"], c["N"], c["docs"]
    with torch.cuda.stream(stream):
        out, lse = pkg.ring_attn_fwd(q, k, v, N, True, docs, stream=stream)
        dq, dk, dv = pkg.ring_attn_bwd(q, k, v, out, lse, c["dout"], N, True, docs, stream=stream)
        ho, hl = pkg.ring_attn_fwd_host(q.cpu().pin_memory(), k.cpu().pin_memory(),
                                        v.cpu().pin_memory(), N, True, docs, stream=stream)
    stream.synchronize()
    return [t.cpu() for t in (out, lse, dq, dk, dv)] + [ho.clone(), hl.clone()]


def test_two_threads_share_the_library_state():
    cases = [_case(81, 2048, [0, 300, 301, 1500, 2048]), _case(82, 4096, [0, 2000, 4096])]
    alone = [_run(c, torch.cuda.Stream()) for c in cases]
    errors, results = [], [[None] * 4 for _ in cases]

    def worker(i):
        try:
            torch.cuda.set_device(0)
            st = torch.cuda.Stream()
            for rep in range(4):
                results[i][rep] = _run(cases[i], st)
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    assert pkg.cp_get_last_status() == 0
    for i in range(len(cases)):
        for rep in range(4):
            got = results[i][rep]
            assert got is not None, (i, rep)
            for a, b in zip(got, alone[i]):
                assert torch.equal(a, b), (i, rep)
