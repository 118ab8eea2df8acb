"""Plant plausible mistakes in the oracle (on the CPU) and show the pins catch each.

A pin set that a dropped term, a wrong sign or index, or a swapped operand
passes would not pin anything; each case below mutates one oracle function
and requires at least one check from ``oracle_checks`` to fail.
"""
import math

import numpy as np
import pytest

import oracle.asp_oracle as O
from tests import oracle_checks as oc


def _no_scale(q_group, mn, mx):
    g, d = q_group.shape
    return np.stack([np.maximum(q_group[h] * mn, q_group[h] * mx).sum(1) for h in range(g)]).max(0)


def _lower_bound(q_group, mn, mx):
    g, d = q_group.shape
    return np.stack([np.minimum(q_group[h] * mn, q_group[h] * mx).sum(1)
                     for h in range(g)]).max(0) / math.sqrt(d)


def _group_min(q_group, mn, mx):
    g, d = q_group.shape
    return np.stack([np.maximum(q_group[h] * mn, q_group[h] * mx).sum(1)
                     for h in range(g)]).min(0) / math.sqrt(d)


def _mn_mx_swapped_signs(q_group, mn, mx):
    qp, qn = np.maximum(q_group, 0), np.minimum(q_group, 0)
    return (qp @ mn.T + qn @ mx.T).max(0) / math.sqrt(q_group.shape[1])


def _summaries_ignore_seq_len(k_pages, seq_len):
    return k_pages.min(axis=1), k_pages.max(axis=1)


def _select_strict(scores, gamma, budget=0):
    n = len(scores)
    order = np.lexsort((np.arange(n), -scores))
    if budget > 0:
        return np.sort(order[:min(budget, n)])
    if gamma >= 1:
        return np.arange(n)
    w = np.exp(scores - scores.max())
    cum = np.cumsum(w[order])
    k = min(int(np.argmax(cum > gamma * cum[-1])) + 1, n)
    return np.sort(order[:k])


def _select_ascending(scores, gamma, budget=0):
    return O.__dict__["_orig_coverage_select"](-scores, gamma, budget)


def _select_high_id_ties(scores, gamma, budget=0):
    n = len(scores)
    ids = np.arange(n)
    order = np.lexsort((-ids, -scores))
    if budget > 0:
        k = min(budget, n)
    elif gamma >= 1:
        k = n
    else:
        w = np.exp(scores - scores.max())
        cum = np.cumsum(w[order])
        k = int(np.argmax(cum >= gamma * cum[-1])) + 1
    return np.sort(order[:k])


def _attend_no_scale(q_group, k_tok, v_tok, scale):
    return O.__dict__["_orig_attend"](q_group, k_tok, v_tok, 1.0)


def _attend_k_for_v(q_group, k_tok, v_tok, scale):
    return O.__dict__["_orig_attend"](q_group, k_tok, k_tok, scale)


def _segment_pages_no_table(cache, block_table, b, kv_head, seq_len):
    p_size = cache.shape[2]
    n = (seq_len + p_size - 1) // p_size
    base = int(block_table[b, 0])
    return np.stack([cache[base + p, kv_head] for p in range(n)])


def _gather_whole_last_page(pages, ids, seq_len):
    """Takes all P rows of every listed page, the partial last one included."""
    rows = [pages[int(p)] for p in ids]
    return np.concatenate(rows, axis=0) if rows else np.zeros((0, pages.shape[2]))


def _num_pages_floor(seq_len, page_size):
    return int(seq_len) // page_size


def _page_mass_over_max(scores):
    return np.exp(scores - scores.max())


def _decode_step_interleaved_gqa(k_cache, v_cache, block_table, seq_lens, q, num_kv_heads,
                                 gamma, budget=0, scale=None, lists=None, lens=None):
    """Query head h reads KV head h % Hkv instead of h // g."""
    B, hq, d = q.shape
    o = np.zeros((B, hq, d))
    lse = np.zeros((B, hq))
    for b in range(B):
        T = int(seq_lens[b])
        for h in range(num_kv_heads):
            kp = O.segment_pages(k_cache, block_table, b, h, T)
            vp = O.segment_pages(v_cache, block_table, b, h, T)
            heads = list(range(h, hq, num_kv_heads))
            r = O.decode_segment(q[b, heads], kp, vp, T, gamma, budget, scale)
            o[b, heads] = r["o"]
            lse[b, heads] = r["lse"]
    return {"o": o, "lse": lse, "ids": [], "scores": []}


def _append_at_seq_len(k_cache, v_cache, block_table, seq_lens_after, k_new, v_new):
    """Writes the new token one slot too far (position seq_len instead of seq_len - 1)."""
    return O.__dict__["_orig_append_token"](k_cache, v_cache, block_table,
                                            np.asarray(seq_lens_after) + 1, k_new, v_new)


def _bf16_shift_15(bits):
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << 15
    return b.view(np.float32).astype(np.float64)


def _segment_ignores_ids(q_group, k_pages, v_pages, seq_len, gamma, budget=0, scale=None,
                         ids=None):
    return O.__dict__["_orig_decode_segment"](q_group, k_pages, v_pages, seq_len, gamma,
                                              budget, scale, None)


PLANTED = [
    ("page_scores", _no_scale),
    ("page_scores", _lower_bound),
    ("page_scores", _group_min),
    ("page_scores", _mn_mx_swapped_signs),
    ("page_summaries", _summaries_ignore_seq_len),
    ("coverage_select", _select_strict),
    ("coverage_select", _select_ascending),
    ("coverage_select", _select_high_id_ties),
    ("attend", _attend_no_scale),
    ("attend", _attend_k_for_v),
    ("segment_pages", _segment_pages_no_table),
    ("gather_tokens", _gather_whole_last_page),
    ("num_pages", _num_pages_floor),
    ("page_mass", _page_mass_over_max),
    ("decode_step", _decode_step_interleaved_gqa),
    ("append_token", _append_at_seq_len),
    ("bf16_bits_to_f64", _bf16_shift_15),
    ("decode_segment", _segment_ignores_ids),
]


@pytest.mark.parametrize("name,broken", PLANTED, ids=lambda x: getattr(x, "__name__", str(x)))
def test_planted_mistake_is_caught(monkeypatch, name, broken):
    monkeypatch.setitem(O.__dict__, "_orig_" + name, getattr(O, name))
    monkeypatch.setattr(O, name, broken)
    caught = []
    for check in oc.ALL_CHECKS:
        try:
            check(O)
        except (AssertionError, ValueError, IndexError):
            caught.append(check.__name__)
    assert caught, f"no pin catches a planted mistake in {name} ({broken.__name__})"
