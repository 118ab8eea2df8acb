"""Coverage selection on the paths ordinary workloads do not reach.

The select kernel finds the cutoff in one histogram round whose bins are
linear in the distance from the top score, then resolves the crossing bin
exactly: one warp with one candidate per lane (a handful of candidates), one
warp running radix rounds (up to 4096), or block-wide radix rounds (more).
Segments of more than 8192 pages take the general path, which reads scores
from global memory. Ordinary data lands in the first case, so these tests
build the others on purpose:

- a long segment (N > 8192 pages) through the whole step, against the oracle;
- clustered scores: summaries written directly so that every page but one
  lies inside a single linear bin, with one outlier far below (near-zero
  mass) that widens the bin range; gamma = 0.5 then puts the cutoff inside
  the cluster with thousands of candidates.

Lists are checked with the acceptance rule of tests/parity.py against the
oracle's fp64 scores of the same summaries.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.asp_oracle as O
from adaptive_sparse_paged_gb300 import binding as B
from tests import guards, parity
from tests.test_gpu_parity import Case, check_case, small

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("gamma,budget", [(0.9, 0), (0.99, 0), (0.5, 3000)])
def test_long_segment_general_path(cuda_device, gamma, budget):
    # request 0 has 9001 pages (general path), request 1 exactly 8192 (fast path)
    w = small("long_general", 2, 2, 1, 64, 16, 16 * 9000 + 3)
    case = Case(w, seed=21, device=cuda_device, seq_lens=[16 * 9000 + 3, 16 * 8192])
    res = case.run(0, gamma, budget)
    check_case(case, 0, gamma, budget, *res)


def _clustered_case(device, n_pages, seed):
    """One segment (B=1, Hkv=1, g=2, d=64, P=16) whose summaries are written directly."""
    w = small("cluster", 1, 2, 1, 64, 16, 16 * n_pages)
    case = Case(w, seed=seed, device=device)
    gen = np.random.default_rng(seed)
    d = w.head_dim
    q = np.abs(gen.normal(0.0, 1e-4, size=(1, 2, d))).astype(np.float32) + 1e-5  # q- = 0
    mx = gen.normal(0.0, 1.0, size=(n_pages, d))
    mx[0, :] = -40000.0  # the outlier: about 29 below the cluster after 1/sqrt(d)
    mn = mx - 1.0
    summ = np.stack([mn, mx], axis=1)  # [N, 2, d]
    kv = case.kvs[0]
    kv.summaries.zero_()
    kv.summaries[0, 0, :n_pages] = torch.from_numpy(summ).to(torch.bfloat16).to(device)
    case.layers[0].q.copy_(torch.from_numpy(q))
    # oracle scores from the exact bf16 values that the GPU reads
    s_bf = parity.bf16_np(kv.summaries[0, 0, :n_pages])
    scores = O.page_scores(q[0].astype(np.float64), s_bf[:, 0], s_bf[:, 1])
    return case, kv, scores


@pytest.mark.parametrize("n_pages", [1500, 7000, 12000])
@pytest.mark.parametrize("gamma,budget", [(0.5, 0), (0.9, 0), (0.5, 700)])
def test_clustered_scores(cuda_device, n_pages, gamma, budget):
    case, kv, scores = _clustered_case(cuda_device, n_pages, seed=n_pages)
    # the construction does what it says: one page far below, the rest packed
    spread = np.ptp(scores[1:])
    assert scores[0] < scores[1:].min() - 20.0 and spread < 24.0 / 4096
    lists = guards.guarded((1, 1, case.sh.max_pages), torch.int32, cuda_device, fill=-7,
                           what="lists")
    lens = guards.guarded((1, 1), torch.int32, cuda_device, fill=-7, what="lens")
    B.asp_coverage_select(kv, case.layers[0].q, gamma, budget, lists, lens, case.ws)
    assert B.asp_get_device_error(case.ws) == 0
    k = int(lens[0, 0])
    ids = lists[0, 0, :k].cpu().numpy()
    assert np.all(np.diff(ids) > 0)
    verdict = parity.list_verdict(ids, scores, gamma, budget)
    tally = parity.VerdictCounts(f"clustered {n_pages} pages gamma {gamma} budget {budget}")
    tally.add(verdict)
    tally.finish()
    if budget == 0:  # thousands of pages share the cutoff bin
        assert k > 32
