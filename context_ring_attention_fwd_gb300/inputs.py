"""Seeded synthetic inputs shared by the tests, the bench and the oracle's callers.

This module holds no attention arithmetic: it only draws random tensors and
document boundaries with fixed seeds, so that the CUDA path and the fp64 CPU
oracle can be fed the very same stored-dtype values.

Workloads follow the shapes named for this hot path: Q/K/V laid out as
[B, S, H, d] with d contiguous (the per-token Q, K, V in R^{S x H x d} of the
"Context Parallelism" page on compassingai.com, section 數學基礎, with the
batch dimension of the "Context Parallel" page on process-cxr.github.io,
section 为什么需要 Context Parallel).  The pages name no dataset; the draws
below are i.i.d. normal, as the workload definitions state.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    H: int
    d: int
    n_shards: int
    causal: bool
    dtype: str            # "f32" or "bf16": the stored input dtype
    scale: float          # multiplier applied to the N(0,1) draws
    seed: int
    packed_docs: bool = False
    doc_min: int = 512
    doc_max: int = 16384

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def describe(self) -> str:
        docs = ", packed documents" if self.packed_docs else ""
        kind = "causal" if self.causal else "non-causal"
        return (f"{self.dtype} {kind}{docs}: B={self.B} S={self.S} H={self.H} "
                f"d={self.d} N={self.n_shards}")


# The five workloads of this hot path.  Seeds are 1000 + position in the list.
WORKLOADS: List[Workload] = [
    Workload("tiny_f32_causal", B=1, S=256, H=2, d=64, n_shards=4, causal=True,
             dtype="f32", scale=1.0, seed=1000),
    Workload("bf16_causal_8k", B=1, S=8192, H=32, d=128, n_shards=4, causal=True,
             dtype="bf16", scale=2.0 ** -0.5, seed=1001),
    Workload("bf16_full_32k", B=2, S=32768, H=16, d=128, n_shards=8, causal=False,
             dtype="bf16", scale=1.0, seed=1002),
    Workload("bf16_causal_128k", B=1, S=131072, H=32, d=128, n_shards=4, causal=True,
             dtype="bf16", scale=1.0, seed=1003),
    Workload("bf16_causal_packed_64k", B=1, S=65536, H=16, d=128, n_shards=8,
             causal=True, dtype="bf16", scale=1.0, seed=1004, packed_docs=True),
]

BY_NAME = {w.name: w for w in WORKLOADS}


def make_qkv(B: int, S: int, H: int, d: int, seed: int, dtype=torch.float32,
             scale: float = 1.0, device: str = "cpu"):
    """Q, K, V of shape [B, S, H, d]: i.i.d. N(0, 1) fp32 draws times `scale`,
    then cast to `dtype`.  On "cpu" the draws come from a seeded CPU generator;
    on a CUDA device from a seeded generator of that device (different stream
    of numbers, same distribution)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = []
    for _ in range(3):
        t = torch.randn((B, S, H, d), generator=g, dtype=torch.float32, device=device)
        if scale != 1.0:
            t.mul_(scale)
        out.append(t.to(dtype))
    return tuple(out)


def make_doc_offsets(S: int, seed: int, doc_min: int = 512,
                     doc_max: int = 16384) -> List[int]:
    """Document boundaries for a packed sequence of S tokens.

    Lengths are drawn uniformly from {doc_min..doc_max} with a seeded numpy
    generator until they cover S; the last document is clipped to end at S
    (so it may be shorter than doc_min).  Returns the offsets
    [0, o_1, ..., S], strictly increasing, terminated by S.  Boundaries are
    free to fall anywhere, including inside a shard or a tile."""
    rng = np.random.default_rng(int(seed))
    offs = [0]
    while offs[-1] < S:
        L = int(rng.integers(doc_min, doc_max + 1))
        offs.append(min(S, offs[-1] + L))
    return offs


def workload_inputs(w: Workload, device: str = "cpu"):
    """(q, k, v, doc_offsets or None) for a workload."""
    q, k, v = make_qkv(w.B, w.S, w.H, w.d, w.seed, w.torch_dtype, w.scale, device)
    docs = (make_doc_offsets(w.S, w.seed + 1, w.doc_min, w.doc_max)
            if w.packed_docs else None)
    return q, k, v, docs


def sample_rows(S: int, n: int, seed: int, rows_lo: int = 0) -> np.ndarray:
    """A seeded, sorted sample of n distinct query rows from [rows_lo, S)."""
    rng = np.random.default_rng(int(seed))
    n = min(n, S - rows_lo)
    return np.sort(rng.choice(np.arange(rows_lo, S), size=n, replace=False))


def random_doc_offsets(S: int, n_docs: int, seed: int) -> List[int]:
    """n_docs documents with seeded random boundaries anywhere in (0, S)."""
    rng = np.random.default_rng(int(seed))
    n_docs = max(1, min(n_docs, S))
    cuts = np.sort(rng.choice(np.arange(1, S), size=n_docs - 1, replace=False)) if n_docs > 1 else []
    return [0] + [int(c) for c in cuts] + [S]
