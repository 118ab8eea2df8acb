"""Plain fp64 CPU oracle for coverage-selected sparse decode over a paged KV cache.

TEST INFRASTRUCTURE. This module is the parity reference, not part of the
product. Only the test suite (``tests/``), ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or call it. It shares no code with
the CUDA library and imports nothing from the product package.

Everything here is deliberately slow and direct: one (request, KV head)
segment at a time, numpy fp64, library primitives only for a sort, a matmul
and exp/log. There is no blocking, fusion or reordering beyond what each
definition states.

Sources (cited by page and section; no page prints code, equations or tables):

* [MOIRA] the abstract on the page "Adaptive DHiSparse: Speculative Decoding
  over a Load-Adaptive KV Hierarchy" (thelatestinai.com/papers/2610.13708).
  It fixes: decode reads the KV cache in pages; for each request, layer, KV
  head and step a *coverage rule* keeps the smallest set of pages whose
  *estimated attention mass* reaches a fraction gamma; attention then runs
  over those per-head page lists.
* [HiSparse] the abstract on the page "HiSparse: scaling sparse attention
  decoding with hierarchical KV cache" (scholarbro.com/p/47450-...), which
  names Quest among the sparse-attention families. Quest scores a page by an
  upper bound of the query-key product built from the page's channel-wise
  key minimum and maximum.

Readings taken where the pages are silent (each one is also listed in the
design notes):

1. Estimated attention mass of a page = softmax over the segment's pages of a
   Quest-style upper bound of the scaled logit q.k/sqrt(d).
2. The upper bound for one query head h and page p is
   sum_i max(q_hi * mn_pi, q_hi * mx_pi), where mn/mx are the channel-wise
   min/max of K over the page's valid tokens: the largest value q_h.k can take
   for any k inside the box [mn_p, mx_p].
3. With grouped-query attention the g query heads that share a KV head form
   one page score: the maximum of their bounds (a bound for every head in the
   group), times 1/sqrt(d), the attention temperature.
4. Every page is one softmax entry; the last, partial page is summarised over
   its valid tokens only and gets no token-count weighting.
5. Order: score descending, ties broken by the lower logical page id. The
   selected count k is the smallest with cumulative mass >= gamma ("reaches").
   gamma >= 1 keeps every page. No sink or recent pages are forced.
6. Fixed-budget comparison mode keeps the top min(budget, N) pages in the
   same order.
7. Lists are emitted as ascending logical page ids.

Parity pins for every function live in tests/test_oracle_pins.py and
tests/golden/; none of them re-types a formula from this file.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "bf16_bits_to_f64",
    "num_pages",
    "page_summaries",
    "page_scores",
    "page_mass",
    "coverage_select",
    "gather_tokens",
    "attend",
    "decode_segment",
    "segment_pages",
    "decode_step",
    "append_token",
]


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact conversion of raw bf16 bit patterns (uint16/int16) to float64.

    A bf16 value is the upper half of an IEEE fp32 word, so widening the bits
    and reinterpreting is exact.
    """
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def num_pages(seq_len: int, page_size: int) -> int:
    """Pages a request of ``seq_len`` tokens occupies: ceil(seq_len / page_size)."""
    return (int(seq_len) + page_size - 1) // page_size


def page_summaries(k_pages: np.ndarray, seq_len: int):
    """Channel-wise min and max of K over each page's valid tokens.

    [MOIRA] reads the cache in pages; reading 2 takes the Quest page summary.
    ``k_pages``: float64 [N, P, d], the pages of one (request, KV head) in
    logical order. Tokens at positions >= ``seq_len`` are not part of the
    context and are ignored. Returns (mn, mx), each [N, d].
    """
    n, p_size, d = k_pages.shape
    assert n == num_pages(seq_len, p_size), "page count does not match seq_len"
    mn = np.empty((n, d))
    mx = np.empty((n, d))
    for p in range(n):
        valid = min(p_size, seq_len - p * p_size)
        rows = k_pages[p, :valid]
        mn[p] = rows.min(axis=0)
        mx[p] = rows.max(axis=0)
    return mn, mx


def page_scores(q_group: np.ndarray, mn: np.ndarray, mx: np.ndarray) -> np.ndarray:
    """Per-page score s[p] (readings 2 and 3).

    For each head h of the group and page p, the largest q_h.k over the box
    [mn_p, mx_p] is reached channel by channel: sum_i max(q_hi*mn_pi,
    q_hi*mx_pi). The group's score is the maximum over its heads, scaled by
    1/sqrt(d). ``q_group``: [g, d]. Returns [N].
    """
    g, d = q_group.shape
    bound = np.empty((g, mn.shape[0]))
    for h in range(g):
        lo = q_group[h][None, :] * mn
        hi = q_group[h][None, :] * mx
        bound[h] = np.maximum(lo, hi).sum(axis=1)
    return bound.max(axis=0) / math.sqrt(d)


def page_mass(scores: np.ndarray) -> np.ndarray:
    """Estimated attention mass of each page: softmax of the scores over pages (reading 1)."""
    w = np.exp(scores - scores.max())
    return w / w.sum()


def _rank_order(scores: np.ndarray) -> np.ndarray:
    """Page ids by score descending, ties by lower page id (reading 5)."""
    ids = np.arange(len(scores))
    return np.lexsort((ids, -scores))


def coverage_select(scores: np.ndarray, gamma: float, budget: int = 0) -> np.ndarray:
    """The coverage rule of [MOIRA]: the smallest page set reaching mass gamma.

    Pages are ranked (reading 5) and the first k are kept, k being the
    smallest count whose cumulative softmax weight is >= gamma times the
    total. The total Z is the last entry of the same running sum, so some
    prefix always reaches gamma*Z when gamma <= 1. gamma >= 1 keeps all
    pages. ``budget`` > 0 switches to the fixed top-k comparison mode
    (reading 6). Returns ascending logical page ids (reading 7).
    """
    n = len(scores)
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    order = _rank_order(scores)
    if budget > 0:
        k = min(int(budget), n)
    elif gamma >= 1.0:
        k = n
    else:
        w = np.exp(scores - scores.max())
        cum = np.cumsum(w[order])
        target = gamma * cum[-1]
        k = int(np.argmax(cum >= target)) + 1
    return np.sort(order[:k])


def gather_tokens(pages: np.ndarray, ids, seq_len: int) -> np.ndarray:
    """Valid token rows of the listed pages, concatenated: [t, d]."""
    n, p_size, d = pages.shape
    rows = []
    for p in ids:
        p = int(p)
        valid = min(p_size, seq_len - p * p_size)
        rows.append(pages[p, :valid])
    if not rows:
        return np.zeros((0, d))
    return np.concatenate(rows, axis=0)


def attend(q_group: np.ndarray, k_tok: np.ndarray, v_tok: np.ndarray, scale: float):
    """Exact softmax attention of each query head over the given tokens.

    o_h = sum_t softmax_t(scale * q_h.k_t) v_t and lse_h = log sum_t
    exp(scale * q_h.k_t). With no tokens the output is zero and lse is -inf.
    Returns (o [g, d], lse [g]).
    """
    g, d = q_group.shape
    if k_tok.shape[0] == 0:
        return np.zeros((g, v_tok.shape[1] if v_tok.ndim == 2 else d)), np.full(g, -np.inf)
    logits = (q_group @ k_tok.T) * scale
    top = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - top)
    denom = e.sum(axis=1)
    o = (e @ v_tok) / denom[:, None]
    lse = top[:, 0] + np.log(denom)
    return o, lse


def decode_segment(q_group, k_pages, v_pages, seq_len, gamma, budget=0,
                   scale=None, ids=None):
    """One (request, layer, KV head) segment of the decode step, in order.

    summaries -> scores -> coverage selection -> attention over the valid
    tokens of the selected pages. ``ids`` may be given to rerun the attention
    on an externally chosen list (e.g. the GPU's own list). Returns a dict
    with ``ids``, ``o``, ``lse``, ``scores``, ``mn``, ``mx``.
    """
    d = q_group.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    n = k_pages.shape[0]
    if n == 0:
        o, lse = attend(q_group, np.zeros((0, d)), np.zeros((0, d)), scale)
        return {"ids": np.zeros(0, dtype=np.int64), "o": o, "lse": lse,
                "scores": np.zeros(0), "mn": np.zeros((0, d)), "mx": np.zeros((0, d))}
    mn, mx = page_summaries(k_pages, seq_len)
    s = page_scores(q_group, mn, mx)
    if ids is None:
        ids = coverage_select(s, gamma, budget)
    ids = np.asarray(ids, dtype=np.int64)
    o, lse = attend(q_group,
                    gather_tokens(k_pages, ids, seq_len),
                    gather_tokens(v_pages, ids, seq_len),
                    scale)
    return {"ids": ids, "o": o, "lse": lse, "scores": s, "mn": mn, "mx": mx}


def segment_pages(cache: np.ndarray, block_table: np.ndarray, b: int, kv_head: int,
                  seq_len: int) -> np.ndarray:
    """Logical-order pages [N, P, d] of one (request, KV head) from a paged cache.

    ``cache``: [num_phys_pages, Hkv, P, d]; ``block_table[b, p]`` is the
    physical page holding logical page p of request b.
    """
    p_size = cache.shape[2]
    n = num_pages(seq_len, p_size)
    return np.stack([cache[int(block_table[b, p]), kv_head] for p in range(n)]) if n else \
        np.zeros((0, p_size, cache.shape[3]))


def decode_step(k_cache, v_cache, block_table, seq_lens, q, num_kv_heads, gamma,
                budget=0, scale=None, lists=None, lens=None):
    """The whole step for one layer over a paged cache (small cases).

    ``k_cache``/``v_cache``: float64 [num_phys_pages, Hkv, P, d];
    ``q``: [B, Hq, d]; query head h reads KV head h // (Hq/Hkv).
    Optional ``lists`` [B, Hkv, max_pages] + ``lens`` [B, Hkv] replace the
    coverage selection. Returns dict of ``o`` [B, Hq, d], ``lse`` [B, Hq],
    ``ids`` (list of arrays per segment, request-major) and ``scores``.
    """
    B, hq, d = q.shape
    g = hq // num_kv_heads
    o = np.zeros((B, hq, d))
    lse = np.zeros((B, hq))
    all_ids, all_scores = [], []
    for b in range(B):
        T = int(seq_lens[b])
        for h in range(num_kv_heads):
            kp = segment_pages(k_cache, block_table, b, h, T)
            vp = segment_pages(v_cache, block_table, b, h, T)
            ext = None
            if lists is not None:
                ext = np.sort(np.asarray(lists[b, h, :int(lens[b, h])], dtype=np.int64))
            r = decode_segment(q[b, h * g:(h + 1) * g], kp, vp, T, gamma, budget, scale, ext)
            o[b, h * g:(h + 1) * g] = r["o"]
            lse[b, h * g:(h + 1) * g] = r["lse"]
            all_ids.append(r["ids"])
            all_scores.append(r["scores"])
    return {"o": o, "lse": lse, "ids": all_ids, "scores": all_scores}


def append_token(k_cache, v_cache, block_table, seq_lens_after, k_new, v_new):
    """Write one new token per request at position seq_len-1 (in place).

    ``seq_lens_after`` already counts the new token; ``k_new``/``v_new`` are
    [B, Hkv, d]. Returns the summaries of the touched pages, recomputed from
    their valid tokens: a dict (b, kv_head) -> (mn_row, mx_row).
    """
    p_size = k_cache.shape[2]
    out = {}
    for b in range(len(seq_lens_after)):
        T = int(seq_lens_after[b])
        if T <= 0:
            continue
        lp, slot = (T - 1) // p_size, (T - 1) % p_size
        phys = int(block_table[b, lp])
        k_cache[phys, :, slot] = k_new[b]
        v_cache[phys, :, slot] = v_new[b]
        for h in range(k_cache.shape[1]):
            rows = k_cache[phys, h, :slot + 1]
            out[(b, h)] = (rows.min(axis=0), rows.max(axis=0))
    return out
