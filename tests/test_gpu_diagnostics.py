"""Budget diagnostics on the GPU: required fractions per gamma and a fixed budget.

Checks properties the coverage rule fixes: required fractions lie in (0, 1]
and grow with gamma; every coverage-rule list captures at least gamma of the
estimated mass (softmax of the page scores) while being minimal; a fixed
budget of the same total size captures the mean amount it reports.
"""

import numpy as np
import pytest
import torch

from adaptive_sparse_paged_gb300 import binding as B
from adaptive_sparse_paged_gb300 import diagnostics as Dg
from tests import guards
from tests.test_gpu_parity import Case, small

pytestmark = pytest.mark.gpu


def test_budget_diagnostics_properties(cuda_device):
    w = small("diag", 4, 16, 4, 128, 16, 16 * 300 + 9, layers=3, hot=("frac", 0.005, 0.5))
    case = Case(w, seed=12, device=cuda_device)
    q_all = torch.stack([lay.q for lay in case.layers])
    d = Dg.budget_diagnostics(case.kvs, q_all, gammas=(0.9, 0.99, 0.999), ref_gamma=0.99)
    means = [d["by_gamma"][g]["mean"] for g in ("0.9", "0.99", "0.999")]
    assert all(0 < m <= 1 for m in means) and means[0] <= means[1] <= means[2]
    assert sum(d["by_gamma"]["0.99"]["counts"]) == d["segments"]
    fb = d["fixed_budget_equal_bytes"]
    assert fb["pages_per_segment"] >= 1 and 0 < fb["captured_mass"]["mean"] <= 1 + 1e-9
    # the coverage rule's own lists reach gamma of the estimated mass, minimally
    kv, q = case.kvs[0], case.layers[0].q
    lists = guards.guarded((w.batch, w.num_kv_heads, case.sh.max_pages), torch.int32,
                           cuda_device, fill=0, what="lists")
    lens = guards.guarded((w.batch, w.num_kv_heads), torch.int32, cuda_device, fill=0,
                          what="lens")
    scores = guards.guarded((w.batch, w.num_kv_heads, case.sh.max_pages), torch.float32,
                            cuda_device, fill=0, what="scores")
    B.asp_coverage_select(kv, q, 0.99, 0, lists, lens, case.ws)
    B.asp_page_scores(kv, q, scores, case.ws)
    assert B.asp_get_device_error(case.ws) == 0
    n = case.sh.num_pages[0]
    for h in range(w.num_kv_heads):
        s = scores[0, h, :n].double()
        m = torch.softmax(s, 0)
        ids = lists[0, h, :int(lens[0, h])].long()
        got = float(m[ids].sum())
        low = float(m[ids].min())
        assert got >= 0.99 - 1e-6 and got - low < 0.99 + 1e-6


def test_budget_diagnostics_against_oracle(cuda_device):
    """Every number the diagnostics report, recomputed by the oracle.

    On every segment of a 3-layer case (48 segments): the required fraction
    len / N_b per gamma equals the oracle's selection count over N_b (each GPU
    list judged by the acceptance rule; a mass tie is the only way a count
    may differ), the fraction histograms equal the oracle's, the fixed budget
    k is the oracle's equal-bytes k, and each segment's captured mass of the
    top min(k, N_b) pages is within the bound that the GPU's fp32 scores
    allow of the oracle's fp64 value. A subset's softmax mass moves by at
    most half the largest score error, and the scores carry the bound of
    tests/test_gpu_scores.py (4.6e-6 of the sum of absolute terms, / sqrt(d)).
    """
    import math

    import oracle.asp_oracle as O
    from tests import parity

    gammas = (0.9, 0.99, 0.999)
    w = small("diag_oracle", 4, 16, 4, 128, 16, 16 * 300 + 9, layers=3, hot=("frac", 0.005, 0.5))
    case = Case(w, seed=13, device=cuda_device)
    q_all = torch.stack([lay.q for lay in case.layers])
    d = Dg.budget_diagnostics(case.kvs, q_all, gammas=gammas, ref_gamma=0.99, detail=True)
    det = d["detail"]
    g = w.num_q_heads // w.num_kv_heads
    n = case.sh.num_pages[0]
    oracle_lens = {gm: np.zeros_like(det["lens"][gm]) for gm in gammas}
    tally = parity.VerdictCounts("budget diagnostics, 3 layers, every segment")
    scores_of = {}
    for l, (lay, kv) in enumerate(zip(case.layers, case.kvs)):
        q = lay.q.double().cpu().numpy()
        for b in range(w.batch):
            for h in range(w.num_kv_heads):
                kp, _ = parity.segment_kv(lay.k_cache, lay.v_cache, case.sh.block_table, b, h,
                                          int(case.sh.seq_lens[b]))
                mn, mx = O.page_summaries(kp, int(case.sh.seq_lens[b]))
                qg = q[b, h * g:(h + 1) * g]
                scores_of[(l, b, h)] = (O.page_scores(qg, mn, mx), qg, mn, mx)
        for gm in gammas:
            lists = torch.zeros((w.batch, w.num_kv_heads, case.sh.max_pages), dtype=torch.int32,
                                device=cuda_device)
            lens = torch.zeros((w.batch, w.num_kv_heads), dtype=torch.int32, device=cuda_device)
            B.asp_coverage_select(kv, lay.q, gm, 0, lists, lens, case.ws)
            assert np.array_equal(lens.cpu().numpy(), det["lens"][gm][l])
            lc = lists.cpu().numpy()
            for b in range(w.batch):
                for h in range(w.num_kv_heads):
                    s = scores_of[(l, b, h)][0]
                    oracle_lens[gm][l, b, h] = len(O.coverage_select(s, float(np.float32(gm))))
                    k = int(lens[b, h])
                    tally.add(parity.list_verdict(lc[b, h, :k], s, gm), where=f"{(l, b, h, gm)}")
    assert B.asp_get_device_error(case.ws) == 0
    counts = tally.finish()
    ties = counts["mass_tie"]
    for gm in gammas:
        differ = int((det["lens"][gm] != oracle_lens[gm]).sum())
        assert differ <= ties, f"gamma {gm}: {differ} counts differ, {ties} mass ties"
        want = Dg.fraction_histogram(oracle_lens[gm].ravel() / n)
        got = d["by_gamma"][f"{gm:g}"]
        if differ == 0:
            assert got["counts"] == want["counts"]
            for key in ("mean", "p10", "p50", "p90", "min", "max"):
                assert abs(got[key] - want[key]) <= 1e-12, key
    # the fixed budget: equal bytes to the oracle's selections at gamma 0.99
    n_seg = 3 * w.batch * w.num_kv_heads
    k = max(1, int(round(float(oracle_lens[0.99].sum()) / n_seg)))
    assert d["fixed_budget_equal_bytes"]["pages_per_segment"] == k
    caps = []
    for (l, b, h), (s, qg, mn, mx) in scores_of.items():
        want = float(O.page_mass(s)[O.coverage_select(s, 0.5, budget=k)].sum())
        absx = np.maximum(np.abs(mn), np.abs(mx))
        bound = 4.6e-6 / math.sqrt(w.head_dim) * (np.abs(qg) @ absx.T).max()
        got = float(det["captured"][l, b, h])
        assert abs(got - want) <= 0.5 * bound + 1e-12, (l, b, h, got, want, bound)
        caps.append(want)
    caps = np.array(caps)
    fb = d["fixed_budget_equal_bytes"]
    assert abs(fb["captured_mass"]["mean"] - caps.mean()) <= 1e-5
    assert abs(fb["captured_mass"]["min"] - caps.min()) <= 1e-5
    assert abs(fb["segments_below_ref_gamma"] - float((caps < 0.99).mean())) <= 1.0 / n_seg
