"""Pins for the fp64 oracle: checks against facts fixed outside the oracle.

Each ``check_*`` takes the oracle module and raises AssertionError on a
mismatch. ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_planted.py`` plants plausible mistakes in the oracle (on the
CPU) and confirms that at least one check catches each.

What pins what (none re-types an oracle formula):
* the hand-worked segment in golden/hand_worked_segment.json (closed form);
* the bound property q.k/sqrt(d) <= s[p] for every valid token, and its
  attainment at the box corner built independently from the sign of q;
* one-token pages, where the bound is an exact dot product;
* brute-force minimum-cardinality subset search on tiny inputs;
* closed forms of the selection (equal scores, gamma -> 0, gamma = 1, budget);
* attention against torch's scaled_dot_product_attention in fp64 and scipy's
  logsumexp (library routines), plus uniform-V and one-token cases;
* paged indexing against a relabelled physical layout and the GQA head map;
* the append path against a direct recount of the page's rows.
"""

from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bf16_values(rng, shape, scale=1.0):
    """Random values exactly representable in bf16 (as float64)."""
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    bits = (x.view(np.uint32) + 0x8000) >> 16  # round-half-up on the magnitude bits
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------- golden
def check_golden(o):
    with open(os.path.join(GOLDEN, "hand_worked_segment.json")) as f:
        gd = json.load(f)
    d, P, T = gd["d"], gd["page_size"], gd["seq_len"]
    k_rows = np.array(gd["k_rows"], dtype=np.float64)
    v_rows = np.array(gd["v_rows"], dtype=np.float64)
    q = np.array(gd["q_group"], dtype=np.float64)
    kp = k_rows.reshape(-1, P, d)
    vp = v_rows.reshape(-1, P, d)
    mn, mx = o.page_summaries(kp, T)
    assert np.array_equal(mn, np.array(gd["expected_mn"], float)), (mn, gd["expected_mn"])
    assert np.array_equal(mx, np.array(gd["expected_mx"], float)), (mx, gd["expected_mx"])
    for h in range(q.shape[0]):
        bound = o.page_scores(q[h:h + 1], mn, mx) * math.sqrt(d)
        assert np.allclose(bound, gd["expected_bound_per_head"][h], rtol=0, atol=1e-12), (h, bound)
    s = o.page_scores(q, mn, mx)
    assert np.allclose(s, gd["expected_scores"], rtol=0, atol=1e-12), s
    for g_str, want in gd["expected_selection"].items():
        got = o.coverage_select(s, float(g_str))
        assert list(got) == want, (g_str, list(got), want)
    for b_str, want in gd["expected_budget_selection"].items():
        got = o.coverage_select(s, 0.5, budget=int(b_str))
        assert list(got) == want, (b_str, list(got), want)
    # attention of q0 over pages {0,1}: softmax of the hand logits on unit V rows
    logits = gd["expected_logits_q0_over_pages_0_1"]
    z = sum(math.exp(x) for x in logits)
    r = o.decode_segment(q, kp, vp, T, gamma=0.9)
    assert list(r["ids"]) == [0, 1]
    want_o = [math.exp(x) / z for x in logits]
    assert np.allclose(r["o"][0], want_o, rtol=0, atol=1e-12), (r["o"][0], want_o)
    assert abs(r["lse"][0] - math.log(z)) < 1e-12


# ----------------------------------------------------------------------- summaries
def check_summaries_attain_and_bound(o, seed=1):
    rng = np.random.default_rng(seed)
    for (P, d, T) in [(16, 64, 16 * 7 + 5), (4, 8, 13), (16, 128, 16), (2, 4, 1)]:
        N = (T + P - 1) // P
        kp = _bf16_values(rng, (N, P, d))
        # tokens past seq_len hold values that would dominate any min/max
        flat = kp.reshape(N * P, d)
        flat[T:] = 1e30 * np.where(rng.random((N * P - T, d)) < 0.5, 1, -1)
        mn, mx = o.page_summaries(kp, T)
        assert mn.shape == (N, d) and mx.shape == (N, d)
        for p in range(N):
            valid = min(P, T - p * P)
            rows = kp[p, :valid]
            assert np.all(mn[p] <= rows) and np.all(rows <= mx[p])
            for i in range(d):
                assert np.any(rows[:, i] == mn[p, i]) and np.any(rows[:, i] == mx[p, i])


# --------------------------------------------------------------------------- scores
def check_scores_upper_bound(o, seed=2):
    rng = np.random.default_rng(seed)
    for (P, d, g, T) in [(16, 64, 4, 16 * 9 + 3), (4, 16, 8, 37), (16, 128, 1, 64)]:
        N = (T + P - 1) // P
        kp = _bf16_values(rng, (N, P, d))
        q = rng.standard_normal((g, d))
        mn, mx = o.page_summaries(kp, T)
        s = o.page_scores(q, mn, mx)
        for p in range(N):
            valid = min(P, T - p * P)
            for t in range(valid):
                for h in range(g):
                    logit = float(np.dot(q[h], kp[p, t])) / math.sqrt(d)
                    assert logit <= s[p] + 1e-9, (p, t, h, logit, s[p])


def check_scores_corner_attained(o, seed=3):
    """The bound equals q_h.k* at the box corner k* chosen by the sign of q_h."""
    rng = np.random.default_rng(seed)
    P, d, g, T = 8, 32, 4, 8 * 11 + 2
    N = (T + P - 1) // P
    kp = _bf16_values(rng, (N, P, d))
    q = rng.standard_normal((g, d))
    mn, mx = o.page_summaries(kp, T)
    s = o.page_scores(q, mn, mx)
    for p in range(N):
        best = -math.inf
        for h in range(g):
            corner = [mx[p, i] if q[h, i] >= 0 else mn[p, i] for i in range(d)]
            best = max(best, math.fsum(q[h, i] * corner[i] for i in range(d)))
        assert abs(s[p] - best / math.sqrt(d)) <= 1e-12 * max(1.0, abs(s[p])), (p, s[p], best)


def check_scores_one_token_pages(o, seed=4):
    rng = np.random.default_rng(seed)
    d, g, T = 16, 2, 9
    kp = _bf16_values(rng, (T, 1, d))
    q = rng.standard_normal((g, d))
    mn, mx = o.page_summaries(kp, T)
    s = o.page_scores(q, mn, mx)
    for p in range(T):
        want = max(math.fsum(q[h, i] * kp[p, 0, i] for i in range(d)) for h in range(g)) / math.sqrt(d)
        assert abs(s[p] - want) <= 1e-12 * max(1.0, abs(want)), (p, s[p], want)


def check_mass(o, seed=5):
    from scipy.special import softmax
    rng = np.random.default_rng(seed)
    s = rng.standard_normal(50) * 3
    m = o.page_mass(s)
    assert np.allclose(m, softmax(s), rtol=1e-12, atol=0)
    assert np.allclose(o.page_mass(s + 1000.0), m, rtol=1e-12, atol=0)


# ------------------------------------------------------------------------ selection
def _mass_of(w, subset):
    return math.fsum(w[i] for i in subset)


def check_select_bruteforce(o, seed=6, trials=300):
    rng = np.random.default_rng(seed)
    checked = 0
    for _ in range(trials):
        n = int(rng.integers(1, 10))
        s = np.round(rng.standard_normal(n) * 2, 1)  # rounding makes ties common
        gamma = float(rng.uniform(0.01, 0.999))
        w = [math.exp(x - float(s.max())) for x in s]
        Z = math.fsum(w)
        subsets_by_size = [list(itertools.combinations(range(n), k)) for k in range(n + 1)]
        best = [max(_mass_of(w, c) for c in subsets_by_size[k]) if k else 0.0 for k in range(n + 1)]
        # skip draws whose answer sits within float noise of gamma
        if any(abs(b - gamma * Z) < 1e-9 for b in best):
            continue
        k_star = next(k for k in range(1, n + 1) if best[k] >= gamma * Z)
        got = list(o.coverage_select(s, gamma))
        assert len(got) == k_star, (s, gamma, got, k_star)
        assert abs(_mass_of(w, got) - best[k_star]) < 1e-12, (s, gamma, got)
        ranked = sorted(range(n), key=lambda i: (-s[i], i))
        assert got == sorted(ranked[:k_star]), (s, gamma, got)
        checked += 1
    assert checked > trials // 2


def check_select_closed_forms(o):
    # equal scores: k = ceil(gamma * N)
    assert len(o.coverage_select(np.zeros(128), 0.99)) == 127
    assert len(o.coverage_select(np.full(1000, 3.25), 0.3)) == 300
    # ">= gamma": exactly reaching counts (100 equal pages, gamma 1/2 -> 50)
    got = o.coverage_select(np.zeros(100), 0.5)
    assert len(got) == 50 and list(got) == list(range(50))
    # single page, gamma = 1, gamma -> 0
    assert list(o.coverage_select(np.array([-7.0]), 0.5)) == [0]
    s = np.array([0.3, 2.0, -1.0, 2.0, 0.1])
    assert list(o.coverage_select(s, 1.0)) == [0, 1, 2, 3, 4]
    assert list(o.coverage_select(s, 1e-12)) == [1]          # argmax, lower id on a tie
    # budget mode: top-k, ties to the lower id, ascending output
    assert list(o.coverage_select(s, 0.5, budget=1)) == [1]
    assert list(o.coverage_select(s, 0.5, budget=2)) == [1, 3]
    assert list(o.coverage_select(s, 0.5, budget=3)) == [0, 1, 3]
    assert list(o.coverage_select(s, 0.5, budget=99)) == [0, 1, 2, 3, 4]
    # one dominant page
    s2 = np.array([0.0, 50.0, 0.0, 0.0])
    assert list(o.coverage_select(s2, 0.99)) == [1]
    assert len(o.coverage_select(np.zeros(0), 0.9)) == 0


# ------------------------------------------------------------------------ attention
def check_attention_matches_sdpa(o, seed=7):
    import torch
    from scipy.special import logsumexp
    rng = np.random.default_rng(seed)
    for (P, d, g, T) in [(16, 64, 4, 16 * 5 + 7), (4, 32, 2, 29), (16, 128, 8, 48)]:
        N = (T + P - 1) // P
        kp = _bf16_values(rng, (N, P, d))
        vp = _bf16_values(rng, (N, P, d))
        q = rng.standard_normal((g, d))
        r = o.decode_segment(q, kp, vp, T, gamma=1.0)
        assert list(r["ids"]) == list(range(N))
        K = torch.from_numpy(kp.reshape(N * P, d)[:T])
        V = torch.from_numpy(vp.reshape(N * P, d)[:T])
        Q = torch.from_numpy(q)
        want = torch.nn.functional.scaled_dot_product_attention(
            Q[:, None, :], K[None].expand(g, T, d), V[None].expand(g, T, d))[:, 0]
        assert np.allclose(r["o"], want.numpy(), rtol=0, atol=1e-12)
        logits = (Q @ K.T).numpy() / math.sqrt(d)
        assert np.allclose(r["lse"], logsumexp(logits, axis=1), rtol=0, atol=1e-12)


def check_attention_special_cases(o, seed=8):
    rng = np.random.default_rng(seed)
    P, d, g, T = 8, 16, 4, 8 * 6 + 3
    N = (T + P - 1) // P
    kp = _bf16_values(rng, (N, P, d))
    vp = np.broadcast_to(_bf16_values(rng, (d,)), (N, P, d)).copy()
    q = rng.standard_normal((g, d))
    r = o.decode_segment(q, kp, vp, T, gamma=0.9)
    assert np.allclose(r["o"], vp[0, 0][None].repeat(g, 0), rtol=0, atol=1e-12)
    # one selected token: P = 1 and a page far above the rest
    kp1 = _bf16_values(rng, (5, 1, d)) * 0.01
    vp1 = _bf16_values(rng, (5, 1, d))
    q1 = np.zeros((1, d)); q1[0, 0] = 1.0
    kp1[3, 0, 0] = 64.0
    r1 = o.decode_segment(q1, kp1, vp1, 5, gamma=0.5)
    assert list(r1["ids"]) == [3]
    assert np.allclose(r1["o"][0], vp1[3, 0], rtol=0, atol=1e-12)
    assert abs(r1["lse"][0] - 64.0 / math.sqrt(d)) < 1e-12


# ------------------------------------------------------------------- paged indexing
def check_paged_indexing(o, seed=9):
    rng = np.random.default_rng(seed)
    B, Hkv, g, P, d = 3, 2, 2, 4, 8
    seq = np.array([13, 4, 9])
    Ns = [(t + P - 1) // P for t in seq]
    max_pages = max(Ns)
    n_phys = sum(Ns) + 3
    k_log = [_bf16_values(rng, (Ns[b], Hkv, P, d)) for b in range(B)]
    v_log = [_bf16_values(rng, (Ns[b], Hkv, P, d)) for b in range(B)]
    q = rng.standard_normal((B, Hkv * g, d))

    def layout(perm):
        kc = np.full((n_phys, Hkv, P, d), np.nan)
        vc = np.full((n_phys, Hkv, P, d), np.nan)
        bt = np.full((B, max_pages), -1, dtype=np.int64)
        i = 0
        for b in range(B):
            for p in range(Ns[b]):
                kc[perm[i]] = k_log[b][p]
                vc[perm[i]] = v_log[b][p]
                bt[b, p] = perm[i]
                i += 1
        return kc, vc, bt

    a = o.decode_step(*layout(np.arange(n_phys)), seq, q, Hkv, gamma=0.8)
    b_ = o.decode_step(*layout(rng.permutation(n_phys)), seq, q, Hkv, gamma=0.8)
    assert np.array_equal(a["o"], b_["o"]) and np.array_equal(a["lse"], b_["lse"])
    # GQA map: query head h reads KV head h // g
    kc, vc, bt = layout(np.arange(n_phys))
    vc[:, 0] = 2.0
    vc[:, 1] = -3.0
    r = o.decode_step(kc, vc, bt, seq, q, Hkv, gamma=0.8)
    assert np.allclose(r["o"][:, :g], 2.0) and np.allclose(r["o"][:, g:], -3.0)


def check_append(o, seed=10):
    rng = np.random.default_rng(seed)
    B, Hkv, P, d = 2, 2, 4, 8
    kc = _bf16_values(rng, (6, Hkv, P, d))
    vc = _bf16_values(rng, (6, Hkv, P, d))
    bt = np.array([[4, 1, 0], [2, 5, 3]])
    seq_after = np.array([6, 9])  # request 0 appends at slot 1 of page 1, request 1 opens page 2
    k_new = _bf16_values(rng, (B, Hkv, d)) * 10
    v_new = _bf16_values(rng, (B, Hkv, d))
    summ = o.append_token(kc, vc, bt, seq_after, k_new, v_new)
    assert np.array_equal(kc[1, :, 1], k_new[0]) and np.array_equal(vc[3, :, 0], v_new[1])
    for h in range(Hkv):
        rows = [kc[1, h, 0], k_new[0, h]]
        assert np.array_equal(summ[(0, h)][0], np.minimum(*rows))
        assert np.array_equal(summ[(0, h)][1], np.maximum(*rows))
        assert np.array_equal(summ[(1, h)][0], k_new[1, h]) and np.array_equal(summ[(1, h)][1], k_new[1, h])


def check_bf16_decode(o, seed=11):
    """bf16 bit patterns -> values: IEEE-defined patterns, and torch's own
    bf16 -> fp32 widening (independent of the oracle's bit shift) on random
    non-NaN patterns."""
    fixed = {0x0000: 0.0, 0x3F80: 1.0, 0xBF80: -1.0, 0x4000: 2.0, 0xC000: -2.0,
             0x3F81: 1.0 + 2.0 ** -7, 0x4049: 3.140625, 0x0001: 2.0 ** -133,
             0x0080: 2.0 ** -126, 0x7F7F: (2.0 - 2.0 ** -7) * 2.0 ** 127,
             0x7F80: math.inf, 0xFF80: -math.inf}
    bits = np.array(list(fixed), dtype=np.uint16)
    got = o.bf16_bits_to_f64(bits)
    assert np.array_equal(got, np.array(list(fixed.values()))), got
    neg0 = o.bf16_bits_to_f64(np.array([0x8000], dtype=np.uint16))[0]
    assert neg0 == 0.0 and math.copysign(1.0, neg0) < 0
    assert np.isnan(o.bf16_bits_to_f64(np.array([0x7FC0], dtype=np.uint16))[0])
    import torch
    rng = np.random.default_rng(seed)
    rb = rng.integers(0, 1 << 16, 4096).astype(np.uint16)
    rb = rb[(rb & 0x7F80) != 0x7F80]  # finite patterns only
    want = torch.from_numpy(rb.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert np.array_equal(o.bf16_bits_to_f64(rb), want)
    assert np.array_equal(o.bf16_bits_to_f64(rb.view(np.int16)), want)  # signed input too


def check_segment_external_ids(o, seed=12):
    """decode_segment with a given list attends over exactly that list: every
    page given equals gamma = 1, an empty list gives 0 and -inf."""
    rng = np.random.default_rng(seed)
    P, d, T = 4, 8, 4 * 6 + 3
    kp = _bf16_values(rng, (7, P, d))
    vp = _bf16_values(rng, (7, P, d))
    kp[2] += 3.0  # one page far above the rest, so gamma = 0.5 keeps fewer pages
    q = np.abs(rng.standard_normal((2, d)))
    own = o.decode_segment(q, kp, vp, T, gamma=0.5)
    assert len(own["ids"]) < 7
    full = o.decode_segment(q, kp, vp, T, gamma=0.5, ids=np.arange(7))
    dense = o.decode_segment(q, kp, vp, T, gamma=1.0)
    assert np.array_equal(full["o"], dense["o"]) and np.array_equal(full["lse"], dense["lse"])
    none = o.decode_segment(q, kp, vp, T, gamma=0.5, ids=np.zeros(0, dtype=np.int64))
    assert np.all(none["o"] == 0) and np.all(np.isneginf(none["lse"]))


ALL_CHECKS = [
    check_bf16_decode,
    check_segment_external_ids,
    check_golden,
    check_summaries_attain_and_bound,
    check_scores_upper_bound,
    check_scores_corner_attained,
    check_scores_one_token_pages,
    check_mass,
    check_select_bruteforce,
    check_select_closed_forms,
    check_attention_matches_sdpa,
    check_attention_special_cases,
    check_paged_indexing,
    check_append,
]
