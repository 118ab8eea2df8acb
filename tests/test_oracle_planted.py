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
