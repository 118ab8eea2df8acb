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
