"""The largest page count one request may have: max_pages = 2^20 pages.

One segment (B = 1, Hkv = 1, g = 2, d = 64, P = 16) of 2^20 pages, the last
one partial (11 of 16 tokens), i.e. 16.8M tokens and 4 GiB of K/V. At this
size page-space offsets, score-buffer offsets and TMA row coordinates are at
their largest, and the selection takes its general path (scores read from
global memory). The oracle cannot redo the whole step at this size, so the
checks are:

- summaries bit-exact on 2000 sampled pages plus the first and last two;
- asp_page_scores against the oracle's fp64 scores of every page (the same
  bound as tests/test_gpu_scores.py), the oracle scoring the GPU's own bf16
  summaries;
- lists in mass and budget mode under the acceptance rule of tests/parity.py
  against the oracle's scores of every page, and at gamma = 1 every id in
  order;
- outputs against the oracle's attention over the GPU's own (short) lists;
- the no-allocation entry point, whose capacity is exactly these 2^20
  scores, equal to the workspace path.
"""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle.asp_oracle as O
from adaptive_sparse_paged_gb300 import binding as B
from tests import guards, parity
from tests.test_gpu_parity import Case, small

pytestmark = pytest.mark.gpu

N_MAX = 1 << 20
P = 16
T = N_MAX * P - 5
REL = 4.6e-6


@pytest.fixture(scope="module")
def big(cuda_device):
    # a few hot pages far above the rest, so mass-mode lists stay short
    w = small("max_pages", 1, 2, 1, 64, P, T, hot=("count", 4, 48), shift=(6.0, 8.0))
    case = Case(w, seed=51, device=cuda_device, max_pages=N_MAX)
    assert case.sh.max_pages == N_MAX and case.sh.num_pages == [N_MAX]
    kv = case.kvs[0]
    summ = parity.bf16_np(kv.summaries[0, 0])  # [N, 2, d], exact
    q = case.layers[0].q.double().cpu().numpy()[0]  # [g, d]
    scores = O.page_scores(q, summ[:, 0], summ[:, 1])
    entries = guards.take()  # these buffers outlive each test: re-armed per test
    yield case, kv, summ, q, scores, entries


@pytest.fixture(autouse=True)
def _rearm_guards(big):
    guards.register(big[-1])
    yield


def test_summaries_sampled(big, cuda_device):
    case, kv, summ, _, _, _ = big
    rng = np.random.default_rng(52)
    ids = sorted(set(int(x) for x in rng.integers(0, N_MAX, 2000)) | {0, 1, N_MAX - 2, N_MAX - 1})
    phys = case.sh.block_table[0, torch.tensor(ids, device=cuda_device)].long()
    k_pages = parity.bf16_np(case.layers[0].k_cache[phys, 0])  # [n, P, d]
    for j, p in enumerate(ids):
        valid = min(P, T - p * P)
        mn, mx = O.page_summaries(k_pages[j][None], valid)
        assert np.array_equal(summ[p, 0], mn[0]) and np.array_equal(summ[p, 1], mx[0]), p


def test_scores_every_page(big, cuda_device):
    case, kv, summ, q, scores, _ = big
    out = guards.guarded((1, 1, N_MAX), torch.float32, cuda_device, fill=float("nan"),
                         what="scores")
    B.asp_page_scores(kv, case.layers[0].q, out, case.ws)
    assert B.asp_get_device_error(case.ws) == 0
    got = out[0, 0].double().cpu().numpy()
    absx = np.maximum(np.abs(summ[:, 0]), np.abs(summ[:, 1]))
    bound = REL / math.sqrt(64) * (np.abs(q) @ absx.T).max(axis=0)
    err = np.abs(got - scores)
    assert np.all(err <= bound + 1e-30), f"max err {err.max()} at page {int(np.argmax(err))}"


@pytest.mark.parametrize("gamma,budget", [(0.9, 0), (0.99, 0), (0.5, 4096), (1.0, 0)])
def test_lists_and_outputs(big, gamma, budget):
    case, kv, summ, q, scores, _ = big
    lists, lens, out, lse = case.run(0, gamma, budget)
    k = int(lens[0, 0])
    ids = lists[0, 0, :k].cpu().numpy()
    if gamma >= 1.0 and budget == 0:
        assert k == N_MAX and np.array_equal(ids, np.arange(N_MAX))
        return
    assert np.all(np.diff(ids) > 0)
    v = parity.list_verdict(ids, scores, gamma, budget)
    tally = parity.VerdictCounts(f"2^20 pages gamma {gamma} budget {budget}")
    tally.add(v)
    tally.finish()
    assert k <= 20000, "the construction keeps the mass-mode lists short"
    phys = case.sh.block_table[0, torch.as_tensor(ids, device=lists.device).long()].long()
    kp = parity.bf16_np(case.layers[0].k_cache[phys, 0])
    vp = parity.bf16_np(case.layers[0].v_cache[phys, 0])
    valid = [min(P, T - int(p) * P) for p in ids]
    k_tok = np.concatenate([kp[j, :n] for j, n in enumerate(valid)])
    v_tok = np.concatenate([vp[j, :n] for j, n in enumerate(valid)])
    o_ref, lse_ref = O.attend(q, k_tok, v_tok, 1.0 / math.sqrt(64))
    parity.check_outputs(out[0].cpu().numpy(), lse[0].cpu().numpy(), o_ref, lse_ref,
                         what=f"gamma {gamma} budget {budget}")


def test_noalloc_at_capacity(big, cuda_device):
    case, kv, _, _, _, _ = big
    assert kv.batch * kv.num_kv_heads * kv.max_pages == 1 << 20  # ASP_NOALLOC_MAX_SCORES
    want_l, want_n, _, _ = case.run(0, 0.95)
    lists = guards.guarded((1, 1, N_MAX), torch.int32, cuda_device, fill=-1, what="lists")
    lens = guards.guarded((1, 1), torch.int32, cuda_device, fill=-1, what="lens")
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    B.asp_coverage_select_noalloc(kv, case.layers[0].q, 0.95, 0, lists, lens, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(lens, want_n)
    k = int(want_n[0, 0])
    assert torch.equal(lists[0, 0, :k], want_l[0, 0, :k])


def test_flat_scores_half_mass(big, cuda_device):
    """Queries scaled by 0.02 flatten the scores (hot pages < 1 unit above the
    rest), so gamma = 0.5 keeps about half of the 2^20 pages and the cutoff
    lands among many near-equal keys (block radix rounds on the general path)."""
    case, kv, summ, _, _, _ = big
    q_small = (case.layers[0].q * 0.02).contiguous()
    lists = guards.guarded((1, 1, N_MAX), torch.int32, cuda_device, fill=-1, what="lists")
    lens = guards.guarded((1, 1), torch.int32, cuda_device, fill=-1, what="lens")
    B.asp_coverage_select(kv, q_small, 0.5, 0, lists, lens, case.ws)
    assert B.asp_get_device_error(case.ws) == 0
    k = int(lens[0, 0])
    assert N_MAX // 8 < k < N_MAX
    ids = lists[0, 0, :k].cpu().numpy()
    assert np.all(np.diff(ids) > 0)
    scores = O.page_scores(q_small.double().cpu().numpy()[0], summ[:, 0], summ[:, 1])
    tally = parity.VerdictCounts("2^20 pages, flat scores, gamma 0.5")
    tally.add(parity.list_verdict(ids, scores, 0.5))
    tally.finish()


def test_cutoff_among_near_zero_mass_pages(big, cuda_device):
    """One hot page and 2^20 - 1 pages 26.5 score units below it, each of mass
    e^-26.5 = 3.1e-12 of the hot page's, 3.25e-6 of the total between them;
    gamma = 1 - 1.6e-6 puts the cutoff about half way through those tied pages.

    Each near-zero weight is below half a unit of a 2^-37 fixed point (it
    would round to zero, losing 3.25e-6 of the mass and keeping the hot page
    alone); the general path's 2^-42 unit keeps the rounding of all 2^20
    weights within 2^20 * 2^-43 = 1.2e-7 of the total, inside the rule's 1e-6
    mass tolerance. Summaries are written directly (a separate buffer, so the
    module's other tests keep theirs): channel 0 holds 212 on the hot page and
    0 elsewhere, every other channel 0, and the queries are e_0, so the scores
    are 212 / 8 = 26.5 and 0 exactly.
    """
    case, kv, _, _, _, _ = big
    d = 64
    summ = guards.guarded((1, 1, N_MAX, 2, d), torch.bfloat16, cuda_device, fill=0,
                          what="summaries (near-zero mass)")
    hot = 777_777
    summ[0, 0, hot, :, 0] = 212.0
    kv2 = B.PagedKV(kv.k_cache, kv.v_cache, summ, kv.block_table, kv.seq_lens, kv.num_q_heads)
    q = torch.zeros((1, 2, d), dtype=torch.float32, device=cuda_device)
    q[0, :, 0] = 1.0
    gamma = float(np.float32(1.0 - 1.6e-6))
    lists = guards.guarded((1, 1, N_MAX), torch.int32, cuda_device, fill=-1, what="lists")
    lens = guards.guarded((1, 1), torch.int32, cuda_device, fill=-1, what="lens")
    B.asp_coverage_select(kv2, q, gamma, 0, lists, lens, case.ws)
    assert B.asp_get_device_error(case.ws) == 0
    k = int(lens[0, 0])
    ids = lists[0, 0, :k].cpu().numpy()
    assert np.all(np.diff(ids) > 0)
    s_np = parity.bf16_np(summ[0, 0])
    scores = O.page_scores(q.double().cpu().numpy()[0], s_np[:, 0], s_np[:, 1])
    assert scores[hot] == 26.5 and np.count_nonzero(scores) == 1
    want = O.coverage_select(scores, gamma)
    # the oracle keeps the hot page and about half of the tied near-zero pages
    assert hot in want and 300_000 < len(want) < 800_000
    assert hot in ids and 300_000 < k < 800_000, f"{k} pages kept"
    tally = parity.VerdictCounts("2^20 pages, cutoff among near-zero-mass pages")
    tally.add(parity.list_verdict(ids, scores, gamma))
    tally.finish()
    m = O.page_mass(scores)
    print(f"near-zero cutoff: gpu {k} pages, oracle {len(want)}, "
          f"mass gpu {m[ids].sum():.9f} oracle {m[want].sum():.9f} gamma {gamma:.9f}")
