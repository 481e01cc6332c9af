"""fp64 CPU oracle for the context-parallel ring-attention forward.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the bench's CPU
baseline leg may import this module.  It shares no code with the CUDA path:
it is plain numpy in float64, written from the pages' statement of the
method, and kept slow and obvious on purpose.

Sources (page title, site, section):
  * "上下文並行（Context Parallelism, CP）" (compassingai.com):
      - §數學基礎: Attn(Q,K,V) = softmax(QK^T/sqrt(d)) V with Q,K,V in
        R^{S x H x d}; each of N GPUs holds the contiguous shards
        Q_i, K_i, V_i in R^{(S/N) x H x d}.
      - §線上 Softmax, algorithm "Ring Attention + FlashAttention 分塊計算":
        per GPU i, start from O_i = 0, m_i = -inf, l_i = 0; for every K/V
        shard j form S_ij = Q_i K_j^T / sqrt(d), mask, m_ij = rowmax(S_ij),
        P_ij = exp(S_ij - m_ij), l_ij = rowsum(P_ij), fold into the running
        state with m_new = max(m_i, m_ij) and the two exp(. - m_new)
        rescalings, and finally O_i = O_i / l_i.
      - §因果掩碼的特殊處理: with an equal split into N shards, GPU i needs
        only the K/V of GPUs 0..i; GPU 0 needs no remote K/V.
  * "大语言模型并行策略（五）：上下文并行" (wangyu.me):
      - §Attention 的流式计算: Attention = sum_i s_i V_i / sum_j s_j with
        s_i = exp(Q K_i^T / sqrt(d_k)).
      - §Ring Attention: the 128K, 4-GPU walk-through (32K shards; GPU 0
        sees K/V [0-32K], [32K-64K], [64K-96K], [96K-128K] in stages 1-4).
      - §通信模式: every GPU sends and receives 2 x (G/N) x (N-1) in total.
  * "Context Parallel" (process-cxr.github.io):
      - §常见失败模式 / §配置关注点: packed samples keep their document
        boundaries across shards; a wrong causal or document mask leaks the
        future or mixes samples.
  * FP8 K/V: the communication-volume note of §通訊量分析 on the first page
    says the bytes moved depend on whether K/V travel in FP8; its timeline
    ties FP8 to FlashAttention-3.  Nothing more is given, so the FP8 form
    here is the plainest one: OCP E4M3 (bias 7, 3 mantissa bits, largest
    finite 448, no infinities) with one scale per (b, h), and attention over
    the dequantized values.

Readings where the pages are silent (each is listed in the design notes):
  * causal mask: key k is visible to query q iff k <= q (a token sees
    itself); shard pairs j > i are fully masked and skipped.
  * documents: key k is visible to q only if both lie in the same document;
    doc_offsets = [0, o_1, ..., S] (cu_seqlens style, ends with S).  Without
    causality a document is bidirectional.
  * shards are the half-open equal spans [i S/N, (i+1) S/N); S % N != 0 is
    an error.
  * log-sum-exp: natural log of sum over visible keys of exp(q.k/sqrt(d)),
    returned as [B, H, S].
  * a row with no visible key inside one step has m = -inf, l = 0, O = 0;
    the merge treats such a partial as the identity.
  * FP8 quantisation of a [B, S, H, d] tensor: amax = max |x| over (S, d) of
    each (b, h), in fp32; inv = 448 / amax and x8 = E4M3(x * inv), both fp32
    operations rounded to nearest, then rounded to the nearest E4M3 value
    (ties to even) and saturated at +-448; descale = amax / 448 (fp32).  An
    all-zero (b, h) gets inv = descale = 1.

Array conventions: q, k, v are [B, S, H, d] (any real dtype, upcast exactly
to float64); per-step partial state is O [B, L, H, d], m and l [B, H, L].
"""
from __future__ import annotations

import itertools
import math
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

NEG_INF = -np.inf


# ---------------------------------------------------------------------------
# Sharding and masks
# ---------------------------------------------------------------------------

def shard_bounds(S: int, n_shards: int) -> List[Tuple[int, int]]:
    """Contiguous equal shards [i*S/N, (i+1)*S/N) ("Context Parallelism",
    §數學基礎: Q_i, K_i, V_i in R^{(S/N) x H x d}; §因果掩碼的特殊處理: 等分)."""
    if n_shards < 1 or S % n_shards != 0:
        raise ValueError("S must split into n_shards equal shards")
    L = S // n_shards
    return [(i * L, (i + 1) * L) for i in range(n_shards)]


def doc_of(S: int, doc_offsets: Optional[Sequence[int]]) -> np.ndarray:
    """Document index of every token (all zero without doc_offsets)."""
    if doc_offsets is None:
        return np.zeros(S, dtype=np.int64)
    offs = [int(x) for x in doc_offsets]
    if offs[0] != 0 or offs[-1] != S or any(b <= a for a, b in zip(offs, offs[1:])):
        raise ValueError("doc_offsets must be 0 = o_0 < o_1 < ... < o_n = S")
    doc = np.empty(S, dtype=np.int64)
    for t in range(len(offs) - 1):
        doc[offs[t]:offs[t + 1]] = t
    return doc


def visible(q_idx: np.ndarray, k_idx: np.ndarray, causal: bool,
            doc: np.ndarray) -> np.ndarray:
    """Boolean mask [len(q_idx), len(k_idx)]: may query q look at key k?

    Causal part: k <= q ("Context Parallelism", §因果掩碼的特殊處理 and the
    masking comment of the §線上 Softmax algorithm).  Document part: same
    document ("Context Parallel", §常见失败模式, cross-sample contamination)."""
    q_idx = np.asarray(q_idx)[:, None]
    k_idx = np.asarray(k_idx)[None, :]
    m = doc[q_idx] == doc[k_idx]
    if causal:
        m = m & (k_idx <= q_idx)
    return m


# ---------------------------------------------------------------------------
# The definition: naive softmax(QK^T/sqrt(d)) V with explicit masks
# ---------------------------------------------------------------------------

def _row_block(qf, kf, vf, rows, causal, doc, d):
    """Exact masked softmax attention for query rows `rows` of one (b, h).

    Only keys inside the union of the rows' visible sets are touched, so
    keys that no row may see are never read (they may hold NaN)."""
    kk = np.arange(kf.shape[0])
    mask = visible(rows, kk, causal, doc)
    cols = np.nonzero(mask.any(axis=0))[0]
    if cols.size == 0:
        raise ValueError("a query row sees no key")
    lo, hi = cols[0], cols[-1] + 1
    mask = mask[:, lo:hi]
    s = (qf[rows] @ kf[lo:hi].T) / math.sqrt(d)
    s = np.where(mask, s, NEG_INF)
    m = s.max(axis=1)
    w = np.where(mask, np.exp(s - m[:, None]), 0.0)
    l = w.sum(axis=1)
    o = (w @ vf[lo:hi]) / l[:, None]
    return o, m + np.log(l)


def attention(q, k, v, causal: bool = True, doc_offsets=None, q_block: int = 256):
    """out [B,S,H,d] and lse [B,H,S] in float64: softmax(QK^T/sqrt(d))V over
    the visible keys of each query ("Context Parallelism", §數學基礎;
    "大语言模型并行策略（五）：上下文并行", §上下文并行的原理).

    lse[b,h,q] = log sum_{k visible} exp(q.k/sqrt(d))."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, S, H, d = q.shape
    doc = doc_of(S, doc_offsets)
    out = np.empty((B, S, H, d))
    lse = np.empty((B, H, S))
    for b in range(B):
        for h in range(H):
            qf, kf, vf = q[b, :, h, :], k[b, :, h, :], v[b, :, h, :]
            for r0 in range(0, S, q_block):
                rows = np.arange(r0, min(S, r0 + q_block))
                o, ls = _row_block(qf, kf, vf, rows, causal, doc, d)
                out[b, rows, h, :] = o
                lse[b, h, rows] = ls
    return out, lse


def attention_rows(q, k, v, b: int, h: int, rows, causal: bool = True,
                   doc_offsets=None, q_block: int = 128):
    """The same definition for a subset of query rows of one (b, h):
    returns out [len(rows), d] and lse [len(rows)]."""
    qf = np.asarray(q[b, :, h, :], dtype=np.float64)
    kf = np.asarray(k[b, :, h, :], dtype=np.float64)
    vf = np.asarray(v[b, :, h, :], dtype=np.float64)
    S, d = qf.shape
    doc = doc_of(S, doc_offsets)
    rows = np.asarray(rows)
    outs, lses = [], []
    for r0 in range(0, rows.size, q_block):
        o, ls = _row_block(qf, kf, vf, rows[r0:r0 + q_block], causal, doc, d)
        outs.append(o)
        lses.append(ls)
    return np.concatenate(outs), np.concatenate(lses)


# ---------------------------------------------------------------------------
# The ring + blockwise algorithm, step by step
# ---------------------------------------------------------------------------

def partial_step(q, k, v, n_shards: int, i: int, j: int, causal: bool = True,
                 doc_offsets=None):
    """One step of the §線上 Softmax algorithm ("Context Parallelism"):
    S_ij = Q_i K_j^T / sqrt(d), masked; m_ij = rowmax(S_ij);
    P_ij = exp(S_ij - m_ij); l_ij = rowsum(P_ij); returns the unnormalised
    O_ij = P_ij V_j [B, L, H, d], m_ij [B, H, L] and l_ij [B, H, L].

    Rows of Q_i that see no key of shard j get m = -inf, l = 0, O = 0."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, S, H, d = q.shape
    (qa, qb), (ka, kb) = shard_bounds(S, n_shards)[i], shard_bounds(S, n_shards)[j]
    L = qb - qa
    doc = doc_of(S, doc_offsets)
    mask = visible(np.arange(qa, qb), np.arange(ka, kb), causal, doc)
    any_vis = mask.any(axis=1)
    O = np.zeros((B, L, H, d))
    m = np.full((B, H, L), NEG_INF)
    l = np.zeros((B, H, L))
    if not mask.any():
        return O, m, l
    for b in range(B):
        for h in range(H):
            s = (q[b, qa:qb, h, :] @ k[b, ka:kb, h, :].T) / math.sqrt(d)
            s = np.where(mask, s, NEG_INF)
            mij = s.max(axis=1)
            msafe = np.where(any_vis, mij, 0.0)
            p = np.where(mask, np.exp(s - msafe[:, None]), 0.0)
            O[b, :, h, :] = p @ v[b, ka:kb, h, :]
            m[b, h, :] = mij
            l[b, h, :] = p.sum(axis=1)
    return O, m, l


def merge(O, m, l, O2, m2, l2):
    """The online merge of the §線上 Softmax algorithm ("Context Parallelism"):
    m_new = max(m, m2); O = O e^{m - m_new} + O2 e^{m2 - m_new};
    l = l e^{m - m_new} + l2 e^{m2 - m_new}.

    O is [B, L, H, d]; m, l are [B, H, L].  A partial with m = -inf is
    empty and acts as the identity (its factor is 0, never (-inf)-(-inf))."""
    m_new = np.maximum(m, m2)
    finite = np.isfinite(m_new)
    safe_new = np.where(finite, m_new, 0.0)
    a = np.where(np.isfinite(m), np.exp(np.where(np.isfinite(m), m, 0.0) - safe_new), 0.0)
    c = np.where(np.isfinite(m2), np.exp(np.where(np.isfinite(m2), m2, 0.0) - safe_new), 0.0)
    # a, c are [B, H, L]; broadcast onto O's [B, L, H, d]
    aO = np.transpose(a, (0, 2, 1))[..., None]
    cO = np.transpose(c, (0, 2, 1))[..., None]
    return O * aO + O2 * cO, m_new, l * a + l2 * c


def finalize(O, m, l):
    """O_i / l_i (last line of the §線上 Softmax algorithm) and the
    log-sum-exp m + log(l).  Returns out [B, L, H, d], lse [B, H, L]."""
    lO = np.transpose(l, (0, 2, 1))[..., None]
    return O / lO, m + np.log(l)


def ring_order(i: int, n_shards: int, kind="ascending") -> List[int]:
    """Visiting order of the K/V shards for rank i.

    "ascending": j = 0..N-1, as the §線上 Softmax loop and the 128K
    walk-through of "大语言模型并行策略（五）" (§Ring Attention) list it.
    "ring": at step t rank i holds the shard of rank (i - t) mod N, which is
    what "send to the next GPU, receive from the previous one" delivers.
    A list is taken as the order itself."""
    if kind == "ascending":
        return list(range(n_shards))
    if kind == "ring":
        return [(i - t) % n_shards for t in range(n_shards)]
    order = [int(x) for x in kind]
    if sorted(order) != list(range(n_shards)):
        raise ValueError("order must be a permutation of 0..N-1")
    return order


def shard_needed(i: int, j: int, S: int, n_shards: int, causal: bool,
                 doc_offsets=None) -> bool:
    """Does shard pair (i, j) hold at least one visible (q, k)?  For causal
    attention without documents this is j <= i ("Context Parallelism",
    §因果掩碼的特殊處理)."""
    (qa, qb), (ka, kb) = shard_bounds(S, n_shards)[i], shard_bounds(S, n_shards)[j]
    doc = doc_of(S, doc_offsets)
    return bool(visible(np.arange(qa, qb), np.arange(ka, kb), causal, doc).any())


def ring_forward(q, k, v, n_shards: int, causal: bool = True, doc_offsets=None,
                 order="ascending", skip_masked: bool = True):
    """The whole §線上 Softmax algorithm of "Context Parallelism", run for
    every virtual rank i: init (O, m, l) = (0, -inf, 0); for j in the
    visiting order, partial step (i, j) then merge; finally O / l.

    With skip_masked, shard pairs that hold no visible (q, k) are skipped,
    as §因果掩碼的特殊處理 allows.  Returns out [B,S,H,d], lse [B,H,S]."""
    q = np.asarray(q, dtype=np.float64)
    B, S, H, d = q.shape
    L = S // n_shards
    shard_bounds(S, n_shards)
    out = np.empty((B, S, H, d))
    lse = np.empty((B, H, S))
    for i in range(n_shards):
        O = np.zeros((B, L, H, d))
        m = np.full((B, H, L), NEG_INF)
        l = np.zeros((B, H, L))
        for j in ring_order(i, n_shards, order):
            if skip_masked and not shard_needed(i, j, S, n_shards, causal, doc_offsets):
                continue
            O2, m2, l2 = partial_step(q, k, v, n_shards, i, j, causal, doc_offsets)
            O, m, l = merge(O, m, l, O2, m2, l2)
        o_i, lse_i = finalize(O, m, l)
        out[:, i * L:(i + 1) * L] = o_i
        lse[:, :, i * L:(i + 1) * L] = lse_i
    return out, lse


def streaming_unsafe(q_row, k_rows, v_rows):
    """The streaming form of "大语言模型并行策略（五）：上下文并行"
    (§Attention 的流式计算): accumulate s_i = exp(q.k_i/sqrt(d)) into a
    denominator and s_i v_i into a numerator, one key at a time, with no
    max subtraction (the page notes it leaves safe softmax out); divide once
    at the end.  Only valid where exp does not overflow."""
    q_row = np.asarray(q_row, dtype=np.float64)
    d = q_row.shape[-1]
    num = np.zeros(d)
    den = 0.0
    for kr, vr in zip(np.asarray(k_rows, dtype=np.float64), np.asarray(v_rows, dtype=np.float64)):
        s = math.exp(float(q_row @ kr) / math.sqrt(d))
        den += s
        num += s * vr
    return num / den, math.log(den)


# ---------------------------------------------------------------------------
# Integer side: schedules, pair counts, traffic
# ---------------------------------------------------------------------------

def tile_spans(S: int, n_shards: int, tile: int) -> List[Tuple[int, int]]:
    """Tiles of `tile` rows laid over each shard from its first row; a tile
    never crosses a shard boundary (the last tile of a shard may be short).
    Tiles are numbered in order across shards."""
    spans = []
    for a, b in shard_bounds(S, n_shards):
        for t0 in range(a, b, tile):
            spans.append((t0, min(b, t0 + tile)))
    return spans


def tile_schedule(S: int, n_shards: int, tile_q: int, tile_k: int,
                  causal: bool = True, doc_offsets=None) -> List[Tuple[int, int]]:
    """Brute-force set of (q tile, kv tile) pairs that hold at least one
    visible (q, k): the blockwise skip of "Context Parallelism"
    (§因果掩碼的特殊處理: fully masked steps are skipped).  Enumerated per q
    tile in ascending order, kv tiles in ascending (shard, tile) order.
    With tile_q = tile_k = S/N it is the shard-pair schedule."""
    doc = doc_of(S, doc_offsets)
    qs = tile_spans(S, n_shards, tile_q)
    ks = tile_spans(S, n_shards, tile_k)
    full = visible(np.arange(S), np.arange(S), causal, doc)
    pairs = []
    for qi, (qa, qb) in enumerate(qs):
        for ki, (ka, kb) in enumerate(ks):
            if full[qa:qb, ka:kb].any():
                pairs.append((qi, ki))
    return pairs


def visible_pair_count(S: int, causal: bool = True, doc_offsets=None,
                       block: int = 4096) -> int:
    """Number of visible (q, k) pairs of one (b, h), counted from the mask
    row block by row block."""
    doc = doc_of(S, doc_offsets)
    total = 0
    kk = np.arange(S)
    for r0 in range(0, S, block):
        rows = np.arange(r0, min(S, r0 + block))
        total += int(visible(rows, kk, causal, doc).sum())
    return total


def ring_traffic_simulated(B: int, S: int, H: int, d: int, dtype_bytes: int,
                           n_shards: int, causal: bool, split: bool = False):
    """Bytes each rank sends plus receives when the K/V blocks travel the
    ring ("大语言模型并行策略（五）", §通信模式; block size (S/N) x H x d x
    dtype_bytes per tensor as in the "Context Parallelism" §關鍵指標 table).

    The ring is simulated step by step: at step t (1..N-1) rank r receives
    from rank r-1 the block that rank r-1 held at step t-1.  Without
    causality every block is forwarded.  With causality a block of shard s
    is only forwarded to a rank that needs it, i.e. rank r > s
    (§因果掩碼的特殊處理).  Returns send + receive bytes per rank, or the
    (sent, received) lists with split=True."""
    N = n_shards
    block = 2 * B * (S // N) * H * d * dtype_bytes          # K and V of one shard
    held = list(range(N))                                     # shard held by rank r
    sent = [0] * N
    recv = [0] * N
    for _t in range(1, N):
        new_held = [None] * N
        for r in range(N):
            src = (r - 1) % N
            s = held[src]
            if s is None:
                continue
            if causal and not (r > s):
                continue
            sent[src] += block
            recv[r] += block
            new_held[r] = s
        held = new_held
    if split:
        return sent, recv
    return [a + b for a, b in zip(sent, recv)]


def effective_flops(B: int, H: int, d: int, pairs_per_head: int) -> int:
    """Algorithmic FLOPs of the forward: 2 d per visible pair for Q K^T and
    2 d for P V, i.e. 4 d per pair, summed over (b, h)."""
    return 4 * d * pairs_per_head * B * H


# ---------------------------------------------------------------------------
# Closed forms used as pins
# ---------------------------------------------------------------------------

def zero_query_closed_form(v, causal: bool = True, doc_offsets=None):
    """With Q = 0 every score is 0, so each query averages V over its visible
    keys and lse = log(count).  Computed with prefix sums in O(S d) per
    (b, h): out [B,S,H,d], lse [B,H,S]."""
    v = np.asarray(v, dtype=np.float64)
    B, S, H, d = v.shape
    doc = doc_of(S, doc_offsets)
    offs = [0, S] if doc_offsets is None else [int(x) for x in doc_offsets]
    start = np.asarray(offs)[doc]
    end = np.asarray(offs)[doc + 1]
    q = np.arange(S)
    hi = q + 1 if causal else end
    cnt = (hi - start).astype(np.float64)
    csum = np.concatenate([np.zeros((B, 1, H, d)), np.cumsum(v, axis=1)], axis=1)
    out = (csum[:, hi] - csum[:, start]) / cnt[None, :, None, None]
    lse = np.broadcast_to(np.log(cnt)[None, None, :], (B, H, S)).copy()
    return out, lse


def all_orders(n_shards: int) -> Iterable[Tuple[int, ...]]:
    """Every visiting order of n_shards shards."""
    return itertools.permutations(range(n_shards))


# ---------------------------------------------------------------------------
# FP8 (E4M3) storage of Q, K, V
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_round(x) -> np.ndarray:
    """Nearest OCP E4M3 value to each element (ties to even), saturated at
    +-448, as float64.  The grid: in the binade [2^e, 2^(e+1)) with e >= -6
    three mantissa bits give a spacing of 2^(e-3); below 2^-6 the subnormals
    are the multiples of 2^-9.  Inputs are float32 or float64; NaN stays NaN."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)                       # a = f * 2^e, f in [0.5, 1)
    quantum = np.ldexp(1.0, np.maximum(e - 4, -9))
    r = np.rint(a / quantum) * quantum       # np.rint rounds halves to even
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, x)


def fp8_quantize(x):
    """Per-(b, h) E4M3 quantisation of x [B, S, H, d] (read as float32).
    Returns (x8, descale): x8 [B, S, H, d] float64 holding E4M3 values and
    descale [B, H] float32, so that x ~ x8 * descale."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.abs(x32).max(axis=(1, 3)).astype(np.float32)      # [B, H]
    nz = amax > 0
    safe = np.where(nz, amax, np.float32(1.0)).astype(np.float32)
    inv = np.where(nz, np.float32(E4M3_MAX) / safe, np.float32(1.0)).astype(np.float32)
    descale = np.where(nz, safe / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    scaled = (x32 * inv[:, None, :, None]).astype(np.float32)
    return e4m3_round(scaled), descale


def fp8_dequantize(x8, descale) -> np.ndarray:
    """x8 * descale in float64 (exact: an E4M3 value times an fp32 scale)."""
    x8 = np.asarray(x8, dtype=np.float64)
    return x8 * np.asarray(descale, dtype=np.float64)[:, None, :, None]


def attention_fp8(q8, k8, v8, q_descale, k_descale, v_descale, causal: bool = True,
                  doc_offsets=None):
    """The forward over FP8-stored inputs: the exact masked softmax attention
    of the dequantized Q, K, V.  Returns (out [B,S,H,d], lse [B,H,S])."""
    return attention(fp8_dequantize(q8, q_descale), fp8_dequantize(k8, k_descale),
                     fp8_dequantize(v8, v_descale), causal, doc_offsets)


# ---------------------------------------------------------------------------
# Backward
# ---------------------------------------------------------------------------
#
# "上下文並行" (§反向傳播) says only that the backward walks the K/V blocks of
# the ring again, with about 2-3x the forward's traffic; "大语言模型并行策略（五）"
# adds that dK/dV travel with their blocks.  The plainest reading: the exact
# gradient of the forward, accumulated block by block over the same shard
# pairs, with the forward's log-sum-exp saved (so P is recomputed, never
# stored).  With L = sum(out * dout) and, per (b, h), P = softmax of the
# visible scores S = Q K^T / sqrt(d):
#   dV = P^T dO;  dP = dO V^T;  D = rowsum(P * dP) = rowsum(dO * O);
#   dS = P * (dP - D);  dQ = dS K / sqrt(d);  dK = dS^T Q / sqrt(d).

def attention_bwd(q, k, v, dout, causal: bool = True, doc_offsets=None):
    """(dq, dk, dv), each [B,S,H,d] float64: the gradient of sum(out * dout)
    for out = attention(q, k, v).  Dense per (b, h): for small S."""
    q, k, v, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dout))
    B, S, H, d = q.shape
    doc = doc_of(S, doc_offsets)
    mask = visible(np.arange(S), np.arange(S), causal, doc)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            s = np.where(mask, q[b, :, h] @ k[b, :, h].T / math.sqrt(d), NEG_INF)
            m = s.max(axis=1, keepdims=True)
            p = np.where(mask, np.exp(s - m), 0.0)
            p /= p.sum(axis=1, keepdims=True)
            do = dout[b, :, h]
            dv[b, :, h] = p.T @ do
            dp = do @ v[b, :, h].T
            ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dq[b, :, h] = ds @ k[b, :, h] / math.sqrt(d)
            dk[b, :, h] = ds.T @ q[b, :, h] / math.sqrt(d)
    return dq, dk, dv


def attention_bwd_rows(q, k, v, dout, b: int, h: int, rows, causal: bool = True,
                       doc_offsets=None):
    """dq [len(rows), d] of one (b, h): row q of dQ needs only row q of P and
    D_q = dO_q . O_q, so this is O(S d) per row."""
    qf, kf, vf, dof = (np.asarray(x[b, :, h, :], dtype=np.float64) for x in (q, k, v, dout))
    S, d = qf.shape
    doc = doc_of(S, doc_offsets)
    rows = np.asarray(rows)
    mask = visible(rows, np.arange(S), causal, doc)
    s = np.where(mask, qf[rows] @ kf.T / math.sqrt(d), NEG_INF)
    p = np.where(mask, np.exp(s - s.max(axis=1, keepdims=True)), 0.0)
    p /= p.sum(axis=1, keepdims=True)
    dp = dof[rows] @ vf.T
    ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    return ds @ kf / math.sqrt(d)


def ring_backward(q, k, v, dout, n_shards: int, causal: bool = True, doc_offsets=None,
                  order="ascending"):
    """The backward walked over the ring's shard pairs: rank i holds Q_i, dO_i
    and the forward's O_i, lse_i; for every needed j in its visiting order it
    recomputes P_ij = exp(S_ij - lse_i), adds P_ij^T dO_i to dV_j and
    dS_ij^T Q_i / sqrt(d) to dK_j (the accumulators that travel with K_j, V_j)
    and dS_ij K_j / sqrt(d) to dQ_i, with dS_ij = P_ij (dO_i V_j^T - D_i) and
    D_i = rowsum(dO_i * O_i).  Returns (dq, dk, dv) [B,S,H,d]."""
    q, k, v, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dout))
    B, S, H, d = q.shape
    bounds = shard_bounds(S, n_shards)
    out, lse = ring_forward(q, k, v, n_shards, causal, doc_offsets)
    doc = doc_of(S, doc_offsets)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for i in range(n_shards):
        qa, qb = bounds[i]
        for j in ring_order(i, n_shards, order):
            if not shard_needed(i, j, S, n_shards, causal, doc_offsets):
                continue
            ka, kb = bounds[j]
            mask = visible(np.arange(qa, qb), np.arange(ka, kb), causal, doc)
            for b in range(B):
                for h in range(H):
                    s = q[b, qa:qb, h] @ k[b, ka:kb, h].T / math.sqrt(d)
                    p = np.where(mask, np.exp(np.where(mask, s, 0.0) - lse[b, h, qa:qb, None]), 0.0)
                    do = dout[b, qa:qb, h]
                    D = (do * out[b, qa:qb, h]).sum(axis=1, keepdims=True)
                    ds = p * (do @ v[b, ka:kb, h].T - D)
                    dv[b, ka:kb, h] += p.T @ do
                    dk[b, ka:kb, h] += ds.T @ q[b, qa:qb, h] / math.sqrt(d)
                    dq[b, qa:qb, h] += ds @ k[b, ka:kb, h] / math.sqrt(d)
    return dq, dk, dv


def zero_query_dv_closed_form(dout, causal: bool = True, doc_offsets=None):
    """With Q = 0, P is uniform over each query's visible keys, so
    dV_k = sum over the queries q that see k of dO_q / count_q.  Causal: the
    queries of k's document from k on (a suffix sum); otherwise the whole
    document.  O(S d) per (b, h).  Returns dv [B,S,H,d]."""
    dout = np.asarray(dout, dtype=np.float64)
    B, S, H, d = dout.shape
    doc = doc_of(S, doc_offsets)
    offs = [0, S] if doc_offsets is None else [int(x) for x in doc_offsets]
    start = np.asarray(offs)[doc]
    end = np.asarray(offs)[doc + 1]
    pos = np.arange(S)
    cnt = ((pos + 1 if causal else end) - start).astype(np.float64)
    w = dout / cnt[None, :, None, None]
    csum = np.concatenate([np.zeros((B, 1, H, d)), np.cumsum(w, axis=1)], axis=1)
    lo = pos if causal else start
    return csum[:, end] - csum[:, lo]
