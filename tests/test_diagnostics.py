"""Host logic of the budget diagnostics (no GPU): fractions, histograms, top-k mass."""

import numpy as np
import torch

from adaptive_sparse_paged_gb300 import diagnostics as Dg


def test_required_fractions_skip_empty_requests():
    lens = np.array([[[2, 4], [0, 0], [5, 1]]])  # L1, B3, Hkv2
    fr = Dg.required_fractions(lens, [8, 0, 10])
    assert np.allclose(sorted(fr), sorted([0.25, 0.5, 0.5, 0.1]))


def test_fraction_histogram_counts_and_quantiles():
    fr = np.array([0.005, 0.015, 0.04, 0.4, 0.9, 1.0])
    h = Dg.fraction_histogram(fr)
    assert sum(h["counts"]) == len(fr)
    assert h["counts"][0] == 1 and h["counts"][1] == 1 and h["counts"][2] == 1
    assert h["counts"][-1] == 2  # [0.8, 1.0] closed on the right
    assert h["min"] == 0.005 and h["max"] == 1.0


def test_captured_mass_topk_matches_direct_sum():
    rng = np.random.default_rng(0)
    s = rng.normal(size=(2, 3, 12))
    n = np.array([12, 5])
    got = Dg.captured_mass_topk(torch.tensor(s, dtype=torch.float32), torch.tensor(n), 4).numpy()
    for b in range(2):
        for h in range(3):
            x = s[b, h, :n[b]].astype(np.float32).astype(np.float64)
            m = np.exp(x - x.max())
            m /= m.sum()
            want = np.sort(m)[::-1][:min(4, n[b])].sum()
            assert abs(got[b, h] - want) < 1e-12
