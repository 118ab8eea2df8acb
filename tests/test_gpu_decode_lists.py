"""asp_sparse_decode on lists that the selection did not write, and gamma just below 1.

The decode's contract is exact attention over the valid tokens of whatever
pages a list names, in any order within the list. These tests hand it
lists built on the host: random page subsets (ascending, descending and
shuffled, one page, every page, empty rows) and the selection's own lists
reversed. Each output is checked against the oracle's attention over the
same pages. The selection is also run with gamma = 1 - 2^-24 (the largest
fp32 below 1), where the target ceil(gamma * Z) is within one part in 10^7
of the total mass.
"""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle.asp_oracle as O
from adaptive_sparse_paged_gb300 import binding as B
from tests import guards, parity
from tests.test_gpu_parity import SMALL, Case, check_case, small

pytestmark = pytest.mark.gpu


def _decode_host_lists(case, rows, cuda_device):
    """rows[(b, h)] -> page ids; returns (out, lse) of asp_sparse_decode on them."""
    w, kv, lay = case.w, case.kvs[0], case.layers[0]
    lists = guards.guarded((w.batch, w.num_kv_heads, case.sh.max_pages), torch.int32,
                           cuda_device, fill=-5, what="lists")
    lens = guards.guarded((w.batch, w.num_kv_heads), torch.int32, cuda_device, fill=0,
                          what="lens")
    for (b, h), ids in rows.items():
        if len(ids):
            lists[b, h, :len(ids)] = torch.as_tensor(np.asarray(ids), dtype=torch.int32)
        lens[b, h] = len(ids)
    out = guards.guarded((w.batch, w.num_q_heads, w.head_dim), torch.float32, cuda_device,
                         fill=float("nan"), what="out")
    lse = guards.guarded((w.batch, w.num_q_heads), torch.float32, cuda_device,
                         fill=float("nan"), what="lse")
    B.asp_sparse_decode(kv, lay.q, lists, lens, 1.0 / math.sqrt(w.head_dim), out, lse, case.ws)
    assert B.asp_get_device_error(case.ws) == 0
    return out.cpu().numpy(), lse.cpu().numpy()


def _check_rows(case, rows, out, lse):
    w, lay = case.w, case.layers[0]
    g = w.num_q_heads // w.num_kv_heads
    q = lay.q.double().cpu().numpy()
    seq = case.sh.seq_lens.cpu().tolist()
    for (b, h), ids in rows.items():
        kp, vp = parity.segment_kv(lay.k_cache, lay.v_cache, case.sh.block_table, b, h, seq[b])
        qg = q[b, h * g:(h + 1) * g]
        o_ref, lse_ref = O.attend(qg, O.gather_tokens(kp, ids, seq[b]),
                                  O.gather_tokens(vp, ids, seq[b]), 1.0 / math.sqrt(w.head_dim))
        parity.check_outputs(out[b, h * g:(h + 1) * g], lse[b, h * g:(h + 1) * g], o_ref,
                             lse_ref, what=f"segment {(b, h)} ({len(ids)} pages)")


@pytest.mark.parametrize("w", [SMALL[0], SMALL[2], SMALL[3]], ids=lambda w: w.name)
def test_host_lists_any_order(cuda_device, w):
    case = Case(w, seed=61, device=cuda_device)
    rng = np.random.default_rng(62)
    rows = {}
    kinds = ["ascending", "descending", "shuffled", "one", "all", "empty"]
    for i, (b, h) in enumerate((b, h) for b in range(w.batch) for h in range(w.num_kv_heads)):
        n = case.sh.num_pages[b]
        kind = kinds[i % len(kinds)]
        if kind == "one":
            ids = [int(rng.integers(0, n))]
        elif kind == "all":
            ids = list(range(n))
        elif kind == "empty":
            ids = []
        else:
            k = int(rng.integers(1, n + 1))
            ids = sorted(int(x) for x in rng.choice(n, k, replace=False))
            if kind == "descending":
                ids = ids[::-1]
            elif kind == "shuffled":
                rng.shuffle(ids)
        rows[(b, h)] = ids
    out, lse = _decode_host_lists(case, rows, cuda_device)
    _check_rows(case, rows, out, lse)
    for (b, h), ids in rows.items():  # an empty row gives zeros and -inf
        if not ids:
            g = w.num_q_heads // w.num_kv_heads
            assert np.all(out[b, h * g:(h + 1) * g] == 0)
            assert np.all(np.isneginf(lse[b, h * g:(h + 1) * g]))


def test_selection_lists_reversed_give_the_same_outputs(cuda_device):
    w = SMALL[1]
    case = Case(w, seed=63, device=cuda_device)
    lists, lens, out_fwd, lse_fwd = case.run(0, 0.95)
    ln = lens.cpu().numpy()
    ls = lists.cpu().numpy()
    rows = {(b, h): [int(x) for x in ls[b, h, :ln[b, h]][::-1]]
            for b in range(w.batch) for h in range(w.num_kv_heads)}
    out, lse = _decode_host_lists(case, rows, cuda_device)
    _check_rows(case, rows, out, lse)
    # the same pages in the other order: equal up to the order of the additions
    # and the bf16 rounding of probabilities taken against other running maxima
    parity.check_outputs(out, lse, out_fwd.cpu().numpy(), lse_fwd.cpu().numpy(),
                         what="reversed lists vs selection order")


@pytest.mark.parametrize("budget", [0, 1])
def test_gamma_just_below_one(cuda_device, budget):
    gamma = float(np.nextafter(np.float32(1.0), np.float32(0.0)))  # 1 - 2^-24
    w = small("near_one", 2, 8, 2, 64, 16, 16 * 150 + 9, hot=("frac", 0.005, 0.05))
    case = Case(w, seed=64, device=cuda_device)
    res = case.run(0, gamma, budget)
    check_case(case, 0, gamma, budget, *res)
