"""asp_page_scores against the oracle's fp64 page scores, element by element.

The score kernel splits each fp32 query into three bf16 terms (residual below
2^-27 of the query), multiplies them exactly by the bf16 summaries and
accumulates in fp32 on the tensor cores: 2 * 16 k-steps of at most 16
products each, then a few additions over split terms and heads. Its error is
therefore bounded by about (32 + 6) fp32 rounding steps of the partial sums,
i.e. 38 * 2^-24 < 2.3e-6 of the sum of absolute terms. The test allows twice
that per page:

    |gpu - ref| <= 4.6e-6 * (1/sqrt(d)) * max_h sum_i |q_hi| * max(|mn_i|, |mx_i|)
"""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle.asp_oracle as O
from adaptive_sparse_paged_gb300 import binding as B
from tests import guards, parity
from tests.test_gpu_parity import SMALL, Case

pytestmark = pytest.mark.gpu

REL = 4.6e-6


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_scores_match_oracle(cuda_device, w):
    case = Case(w, seed=3, device=cuda_device)
    kv, lay = case.kvs[0], case.layers[0]
    scores = guards.guarded((w.batch, w.num_kv_heads, case.sh.max_pages), torch.float32,
                            cuda_device, fill=float("nan"), what="scores")
    B.asp_page_scores(kv, lay.q, scores, case.ws)
    assert B.asp_get_device_error(case.ws) == 0
    sc = scores.cpu().numpy()
    summ = parity.bf16_np(kv.summaries)
    q = lay.q.double().cpu().numpy()
    g = w.num_q_heads // w.num_kv_heads
    inv = 1.0 / math.sqrt(w.head_dim)
    for b in range(w.batch):
        n = case.sh.num_pages[b]
        for h in range(w.num_kv_heads):
            qg = q[b, h * g:(h + 1) * g]
            mn, mx = summ[b, h, :n, 0], summ[b, h, :n, 1]
            ref = O.page_scores(qg, mn, mx)
            absx = np.maximum(np.abs(mn), np.abs(mx))
            bound = REL * inv * (np.abs(qg) @ absx.T).max(axis=0)
            err = np.abs(sc[b, h, :n] - ref)
            assert np.all(err <= bound + 1e-30), \
                f"segment {(b, h)}: max err {err.max()} vs bound {bound[np.argmax(err)]}"
            assert np.all(np.isnan(sc[b, h, n:])), "entries past N_b must stay untouched"
