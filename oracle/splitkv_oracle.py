"""Plain, slow, fp64 CPU oracle for split-KV paged decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code with
the CUDA library (``split_kv_paged_splitkv_gb300``) and never imports it.

What it computes, and where each step comes from:

* ``attention_direct`` -- the plain definition of decode attention over a paged
  KV cache: gather each visible key/value through the block table, score it
  against the query, softmax, weight the values.  Split-KV reaches this same
  result (up to rounding order), so the direct definition is the oracle.
  ("vLLM 0.30.0 FA4 SplitKV Bug: H100 Decode Can Be 48% Slower", section
  "Why the result is still correct": splitting changes where the work runs,
  not the answer.)
* ``split_ranges`` / ``plan_items`` -- the split planner: the KV range of a
  sequence is divided into ``num_splits`` ranges, one per CTA (same page,
  section "What SplitKV is trying to do"), every launched split getting a
  non-empty range (the failure dissected in "The actual bug is one missing
  constructor argument").  The partition formula and the automatic split
  choice are this library's readings; they are restated here step by step.
* ``partial_attention`` -- what one split computes: attention restricted to its
  KV range, returned as (normalised output, log-sum-exp); an empty range
  returns (0, -inf) ("Why the result is still correct": empty splits
  contribute zero weight).
* ``combine`` -- the log-sum-exp merge of partials (same section).
* ``attention_split_mode`` -- planner + partials + combine, end to end.
* ``e4m3_to_float`` -- OCP FP8 e4m3fn decoding from the format definition
  (exponent bias 7, 3 mantissa bits, subnormals, S.1111.111 = NaN, no inf),
  for the FP8 KV cache with BF16 queries ("Xqa decode kernels", section
  "Purpose": the decode path keeps BF16/FP16 queries over an FP8 KV cache).

Conventions (readings of points the pages leave open):

* ``seq_lens[b]`` counts all visible keys including the current ``T`` query
  tokens; query token ``t`` sees keys ``0 .. L - T + t`` (bottom-right causal).
* Query head ``h`` reads KV head ``h // G`` with ``G = Hq / Hkv``.
* Pages are HND, ``pages[phys][h_kv][slot][dim]``, or NHD,
  ``pages[phys][slot][h_kv][dim]`` (``layout="NHD"``); key ``j`` of sequence
  ``b`` lives in page ``block_table[b][j // P]``, slot ``j % P``.  ("Xqa decode
  kernels", section "Test Plan", runs its decode path with the cache layout
  set to HND; NHD is the other value of that setting.)
* FP8 dequantisation is ``code_value * kv_scale`` for both K and V, or, with
  per-head scales, ``code_value * k_scale[h_kv]`` for K and
  ``code_value * v_scale[h_kv]`` for V.
* With ``v_shares_k`` (MLA latent cache) ``V_j`` is the first ``Dv`` columns of
  ``K_j``.
* The LSE is the natural log of ``sum_j exp(s_j)`` where ``s_j`` already
  includes ``scale`` (and ``kv_scale`` through the dequantised keys).
* A row with no visible key has output 0 and LSE -inf.
"""
from __future__ import annotations

import heapq
import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

NEG_INF = -math.inf


# --------------------------------------------------------------------------
# Element decoding
# --------------------------------------------------------------------------

def bf16_to_float(raw: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64.  bf16 is the upper half of fp32."""
    raw = np.asarray(raw, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (raw.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def e4m3_to_float(codes: np.ndarray) -> np.ndarray:
    """OCP FP8 e4m3fn codes (uint8) -> float64, from the format definition.

    sign = bit 7, exponent E = bits 6..3 (bias 7), mantissa M = bits 2..0.
    E == 0: subnormal, value = M/8 * 2^(1-7).  Otherwise value =
    (1 + M/8) * 2^(E-7).  E == 15 with M == 7 is NaN; there is no infinity.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    E = (c >> 3) & 0xF
    M = c & 0x7
    normal = (1.0 + M / 8.0) * np.power(2.0, E - 7)
    subnormal = (M / 8.0) * 2.0 ** (1 - 7)
    val = sign * np.where(E == 0, subnormal, normal)
    return np.where((E == 15) & (M == 7), np.nan, val)


def dequant(raw: np.ndarray, kv_dtype: str, kv_scale: float) -> np.ndarray:
    if kv_dtype == "bf16":
        return bf16_to_float(raw)
    if kv_dtype == "fp8_e4m3":
        return e4m3_to_float(raw) * float(kv_scale)
    raise ValueError(kv_dtype)


# --------------------------------------------------------------------------
# Paged gather
# --------------------------------------------------------------------------

def page_size_of(pages: np.ndarray, layout: str = "HND") -> int:
    """P: axis 2 of HND pages ``[N][Hkv][P][D]``, axis 1 of NHD ``[N][P][Hkv][D]``."""
    return pages.shape[2] if layout == "HND" else pages.shape[1]


def kv_heads_of(pages: np.ndarray, layout: str = "HND") -> int:
    """Hkv: axis 1 of HND pages, axis 2 of NHD pages."""
    return pages.shape[1] if layout == "HND" else pages.shape[2]


def gather_keys(pages: np.ndarray, table_row: Sequence[int], n_keys: int,
                head: int, layout: str = "HND") -> np.ndarray:
    """Raw rows ``0 .. n_keys-1`` of one KV head, read through the block table.

    ``pages[phys][h_kv][slot][dim]`` (HND) or ``pages[phys][slot][h_kv][dim]``
    (NHD), raw storage; ``table_row[j // P]`` gives the physical page of key
    ``j``.  Returns ``[n_keys][dim]`` raw values.
    """
    if layout not in ("HND", "NHD"):
        raise ValueError(layout)
    P = page_size_of(pages, layout)
    out = np.empty((n_keys, pages.shape[3]), dtype=pages.dtype)
    for j in range(0, n_keys, P):  # one page (slots 0 .. take-1) at a time
        phys = int(table_row[j // P])
        take = min(P, n_keys - j)
        if layout == "HND":
            out[j:j + take] = pages[phys, head, :take, :]
        else:
            out[j:j + take] = pages[phys, :take, head, :]
    return out


# --------------------------------------------------------------------------
# Direct attention (the definition)
# --------------------------------------------------------------------------

def _softmax_attend(q_row: np.ndarray, K: np.ndarray, V: np.ndarray,
                    scale: float) -> Tuple[np.ndarray, float]:
    """out = sum_j softmax(scale * q.K_j) V_j and lse = ln sum_j exp(scale * q.K_j)."""
    if K.shape[0] == 0:
        return np.zeros(V.shape[1]), NEG_INF
    s = scale * (K @ q_row)
    m = s.max()
    w = np.exp(s - m)
    tot = w.sum()
    return (w @ V) / tot, float(m + math.log(tot))


def attention_direct(q, k_pages, v_pages, block_table, seq_lens, *, scale,
                     kv_dtype="bf16", kv_scale=1.0, v_dim=None,
                     v_shares_k=False, rows=None, k_scale=None, v_scale=None,
                     layout="HND"):
    """Decode attention by definition, in fp64.

    ``q``: bf16 bits ``[B][T][Hq][Dk]``; ``k_pages``/``v_pages``: raw pages
    ``[N][Hkv][P][D]`` (``layout`` HND) or ``[N][P][Hkv][D]`` (NHD), bf16 bits
    or e4m3 codes; ``block_table`` ``[B][max]``;
    ``seq_lens`` ``[B]``.  ``rows``: optional list of ``(b, t, h)`` to compute
    (all rows otherwise).  ``k_scale`` / ``v_scale``: optional per-KV-head
    dequantisation scales of an e4m3 cache, used for K / V in place of
    ``kv_scale``.  Returns ``(out[B][T][Hq][Dv], lse[B][T][Hq])`` in float64
    (rows not computed are NaN).
    """
    q = np.asarray(q)
    B, T, Hq, Dk = q.shape
    Hkv = kv_heads_of(k_pages, layout)
    G = Hq // Hkv
    if v_dim is None:
        v_dim = k_pages.shape[3] if v_shares_k else v_pages.shape[3]
    out = np.full((B, T, Hq, v_dim), np.nan)
    lse = np.full((B, T, Hq), np.nan)
    if rows is None:
        rows = [(b, t, h) for b in range(B) for t in range(T) for h in range(Hq)]
    rows = sorted(rows, key=lambda r: (r[0], r[2] // G, r[1], r[2]))
    cache = {}
    for (b, t, h) in rows:
        L = int(seq_lens[b])
        hk = h // G
        key = (b, hk)
        if key not in cache:
            ks = kv_scale if k_scale is None else float(k_scale[hk])
            vs = kv_scale if v_scale is None else float(v_scale[hk])
            Kr = gather_keys(k_pages, block_table[b], L, hk, layout)
            K = dequant(Kr, kv_dtype, ks)
            if v_shares_k:
                V = K[:, :v_dim]
            else:
                V = dequant(gather_keys(v_pages, block_table[b], L, hk, layout), kv_dtype, vs)
            cache = {key: (K, V)}  # one (b, h_kv) at a time keeps memory bounded
        K, V = cache[key]
        lim = L - T + t  # last visible key index for this query token
        n_vis = max(0, min(L, lim + 1))
        qr = bf16_to_float(q[b, t, h])
        o, l = _softmax_attend(qr, K[:n_vis], V[:n_vis], scale)
        out[b, t, h] = o
        lse[b, t, h] = l
    return out, lse


# --------------------------------------------------------------------------
# Split planner (restated from the library's reading)
# --------------------------------------------------------------------------

MAX_SPLITS = 64          # cap on splits per sequence
ITEM_OVERHEAD = 96       # fixed cost of one work item, in 1/16-page units (6 pages)
COMBINE_COST = 2         # cost per split of the merge, in 1/16-page units
MAX_WAVES = 8            # candidate granularities: 1 .. MAX_WAVES items per machine


def pages_of(L: int, P: int) -> int:
    return (int(L) + P - 1) // P


def split_ranges(n: int, S: int) -> List[Tuple[int, int]]:
    """Balanced page-granular partition of ``[0, n)`` into ``S`` ranges.

    Range ``s`` is ``[floor(s*n/S), floor((s+1)*n/S))``; with ``1 <= S <= n``
    every range holds at least one page and together they tile ``[0, n)``.
    """
    return [((s * n) // S, ((s + 1) * n) // S) for s in range(S)]


def _splits_for(n_pages: Sequence[int], chunk: int, round_up: bool) -> List[int]:
    """``S_b = clamp(n_b / chunk rounded up or down, 1, min(n_b, MAX_SPLITS))``."""
    out = []
    for n in n_pages:
        if n <= 0:
            out.append(1)
            continue
        q = -(-n // chunk) if round_up else n // chunk
        out.append(max(1, min(MAX_SPLITS, n, q)))
    return out


def _makespan(costs: List[int], machines: int) -> int:
    """Longest-processing-time-first list scheduling; returns the largest load."""
    loads = [0] * machines
    heapq.heapify(loads)
    for c in sorted(costs, reverse=True):
        heapq.heappush(loads, heapq.heappop(loads) + c)
    return max(loads)


def choose_splits(n_pages: Sequence[int], num_kv_heads: int, num_sms: int,
                  ctas_per_item: int = 1, ctas_per_sm: int = 1,
                  heads_per_item: int = 1) -> List[int]:
    """Automatic split count per sequence (``num_splits == 0``).

    The machine model: ``M = max(1, num_sms * ctas_per_sm // ctas_per_item)``
    work items run at once (a kernel with several resident CTAs per SM offers
    that many slots per SM; an item that launches several CTAs takes that many).
    A split of sequence b is ``U = Hkv / heads_per_item`` items (each covers
    ``heads_per_item`` KV heads), an item over ``p`` pages costs
    ``16 * p * heads_per_item + ITEM_OVERHEAD``.

    One chunk size ``c`` (pages per split) is used for all sequences.
    Candidates are ``c_k = ceil(total / (k * M))`` for ``k = 1 .. MAX_WAVES``
    (``total = U * sum n_b``), each with ``S_b = n_b / c_k`` rounded up and
    rounded down (then clamped to ``[1, min(n_b, MAX_SPLITS)]``), and last
    "no split".  A candidate scores the LPT makespan of its items over ``M``
    machines plus ``COMBINE_COST * max_b S_b``; the lowest score wins and ties
    go to the earlier candidate.
    """
    machines = max(1, (num_sms * ctas_per_sm) // ctas_per_item)
    units = num_kv_heads // heads_per_item
    total = sum(int(n) for n in n_pages) * units
    nmax = max([int(n) for n in n_pages] + [1])
    cands = []
    for k in range(1, MAX_WAVES + 1):
        c = max(1, -(-total // (k * machines)))
        cands += [(c, True), (c, False)]
    cands.append((nmax, True))
    best, best_S = None, None
    for c, up in cands:
        S = _splits_for(n_pages, c, up)
        costs = []
        for n, s_b in zip(n_pages, S):
            for (p0, p1) in split_ranges(n, s_b) if n > 0 else [(0, 0)]:
                costs.extend([16 * (p1 - p0) * heads_per_item + ITEM_OVERHEAD] * units)
        score = _makespan(costs, machines) + COMBINE_COST * max(S)
        if best is None or score < best:
            best, best_S = score, S
    return best_S


def plan_items(seq_lens: Sequence[int], page_size: int, num_kv_heads: int,
               num_splits: int, num_sms: int, ctas_per_item: int = 1,
               ctas_per_sm: int = 1,
               heads_per_item: int = 1) -> List[Tuple[int, int, int, int, int, int]]:
    """Work list ``[(b, h0, s, S_b, p0, p1)]`` in launch order.

    An item covers KV heads ``[h0, h0 + heads_per_item)`` of sequence b over
    pages ``[p0, p1)``.  ``num_splits > 0``: ``S_b = min(num_splits, n_b)`` --
    the requested count is honoured whenever the sequence has that many pages.
    ``num_splits == 0``: ``choose_splits``.  A sequence with no keys gets one
    empty item per head group (it only writes out = 0, lse = -inf).  Launch
    order: longest range first, ties by ``(b, h0, s)``.
    """
    n_pages = [pages_of(L, page_size) for L in seq_lens]
    if num_splits > 0:
        S = [max(1, min(num_splits, n)) if n > 0 else 1 for n in n_pages]
    else:
        S = choose_splits(n_pages, num_kv_heads, num_sms, ctas_per_item, ctas_per_sm,
                          heads_per_item)
    items = []
    for b, (n, s_b) in enumerate(zip(n_pages, S)):
        rngs = split_ranges(n, s_b) if n > 0 else [(0, 0)]
        for h in range(0, num_kv_heads, heads_per_item):
            for s, (p0, p1) in enumerate(rngs):
                items.append((b, h, s, s_b, p0, p1))
    items.sort(key=lambda it: (-(it[5] - it[4]), it[0], it[1], it[2]))
    return items


# --------------------------------------------------------------------------
# Split mode: partials and the log-sum-exp combine
# --------------------------------------------------------------------------

def partial_attention(q_row: np.ndarray, K: np.ndarray, V: np.ndarray, lo: int,
                      hi: int, lim: int, scale: float) -> Tuple[np.ndarray, float]:
    """One split's result over keys ``[lo, hi)`` that are also ``<= lim``.

    Returns ``(O_s, lse_s)`` with ``O_s`` normalised by the split's own
    softmax sum; an empty range returns ``(0, -inf)``.
    """
    hi = min(hi, lim + 1)
    if hi <= lo:
        return np.zeros(V.shape[1]), NEG_INF
    return _softmax_attend(q_row, K[lo:hi], V[lo:hi], scale)


def combine(parts: Sequence[Tuple[np.ndarray, float]]) -> Tuple[np.ndarray, float]:
    """Log-sum-exp merge: ``lse = ln sum_s exp(lse_s)``, ``out = sum_s exp(lse_s - lse) O_s``.

    Splits with ``lse_s = -inf`` get weight 0; if all are empty the result is
    ``(0, -inf)``.
    """
    lses = np.array([p[1] for p in parts], dtype=np.float64)
    dim = parts[0][0].shape[0]
    if lses.size == 0 or np.all(lses == NEG_INF):
        return np.zeros(dim), NEG_INF
    M = lses.max()
    w = np.exp(lses - M)
    tot = w.sum()
    out = sum(wi * p[0] for wi, p in zip(w, parts) if wi > 0) / tot
    return out, float(M + math.log(tot))


def attention_split_mode(q, k_pages, v_pages, block_table, seq_lens, *, scale,
                         num_splits, num_sms=148, kv_dtype="bf16", kv_scale=1.0,
                         v_dim=None, v_shares_k=False, layout="HND"):
    """Planner + per-split partials + combine, in fp64, for every row."""
    q = np.asarray(q)
    B, T, Hq, Dk = q.shape
    Hkv = kv_heads_of(k_pages, layout)
    P = page_size_of(k_pages, layout)
    G = Hq // Hkv
    if v_dim is None:
        v_dim = k_pages.shape[3] if v_shares_k else v_pages.shape[3]
    items = plan_items(seq_lens, P, Hkv, num_splits, num_sms)
    by_bh = {}
    for (b, h, s, s_b, p0, p1) in items:
        by_bh.setdefault((b, h), []).append((s, p0, p1))
    out = np.zeros((B, T, Hq, v_dim))
    lse = np.zeros((B, T, Hq))
    for (b, hk), splits in by_bh.items():
        L = int(seq_lens[b])
        K = dequant(gather_keys(k_pages, block_table[b], L, hk, layout), kv_dtype, kv_scale)
        V = K[:, :v_dim] if v_shares_k else dequant(
            gather_keys(v_pages, block_table[b], L, hk, layout), kv_dtype, kv_scale)
        splits.sort()
        for t in range(T):
            lim = L - T + t
            for g in range(G):
                h = hk * G + g
                qr = bf16_to_float(q[b, t, h])
                parts = [partial_attention(qr, K, V, p0 * P, min(p1 * P, L), lim, scale)
                         for (_, p0, p1) in splits]
                out[b, t, h], lse[b, t, h] = combine(parts)
    return out, lse
