"""Host logic of bench.py: the FLOP count, the max-over-ranks timing on two
gloo ranks (CPU), and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

import bench
from context_ring_attention_fwd_gb300 import inputs
from oracle import ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_visible_pairs_match_oracle_counts():
    for S, causal, docs in [(97, True, None), (97, False, None), (97, True, [0, 10, 50, 97]),
                            (64, False, [0, 1, 63, 64])]:
        assert bench.visible_pairs(S, causal, docs) == ref.visible_pair_count(S, causal, docs)
    w = inputs.BY_NAME["bf16_causal_128k"]
    assert bench.effective_flops(w, None) == 4 * 128 * (131072 * 131073 // 2) * 32


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.dist_init(world, "gloo")
    bench.barrier(world)
    m = bench.max_over_ranks(10.0 + rank, world)
    bench.barrier(world)
    q.put((rank, m))
    torch.distributed.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 11.0, 1: 11.0}


def test_reference_arm_line_under_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--workload", "tiny_f32_causal", "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1                     # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_recorded_traffic_holds_only_for_its_kernel_sources(monkeypatch):
    """A recorded DRAM figure is reported only while the kernel sources it
    was captured on are unchanged (their digest matches); any other digest,
    or a workload with no record, gives None, so a stale figure never
    reaches a bench line."""
    for name, rec in bench.NCU_TRAFFIC.items():
        files = rec.get("files", bench.KERNEL_SOURCES)
        if rec["bytes"] is not None and rec["sources"] == bench.kernel_sources_digest(files):
            assert bench.ncu_traffic(name) == rec["bytes"]
        else:
            assert bench.ncu_traffic(name) is None
    assert bench.ncu_traffic("no_such_workload") is None
    stale = {k: dict(v, sources="0000000000000000") for k, v in bench.NCU_TRAFFIC.items()}
    monkeypatch.setattr(bench, "NCU_TRAFFIC", stale)
    assert all(bench.ncu_traffic(k) is None for k in stale)
    # the digest covers every listed file: changing one byte of any changes it
    real = bench.kernel_sources_digest()
    assert len(real) == 16 and real != bench.kernel_sources_digest(bench.BWD_KERNEL_SOURCES)

