"""CUDA path (through the C ABI) against the fp64 oracle, element by element.

Summaries: bit-exact. Page lists: the acceptance rule in tests/parity.py
(exact, or equal up to 1e-6 score/mass ties). Outputs and lse: max-abs 2e-2,
mean-abs 2e-3 against the oracle rerun on the GPU's own lists.
"""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle.asp_oracle as O
from adaptive_sparse_paged_gb300 import binding as B
from adaptive_sparse_paged_gb300 import synth
from adaptive_sparse_paged_gb300.step import DecodeStep
from tests import guards, parity

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ fixtures
GUARD_CACHE_BYTES = 256 << 20  # K/V caches up to this size get guard bands too


def guard_outputs(step):
    """Moves a DecodeStep's or DecodeLoop's outputs and workspace into guarded buffers."""
    for name in ("lists", "lens", "out", "lse"):
        t = getattr(step, name)
        setattr(step, name, guards.guarded(t.shape, t.dtype, t.device, fill=0, what=name))
    step.ws = guards.guarded_workspace(step.kvs[0] if not isinstance(step.kvs[0], list)
                                       else step.kvs[0][0])


class Case:
    """A workload built on the GPU: shared tables, layers, PagedKVs (BULK-summarised).

    Every buffer a kernel writes (summaries, workspace, outputs, and the K/V
    caches of small cases, which APPEND writes) sits between guard bands that
    tests/conftest.py checks when the test ends.
    """

    def __init__(self, w: synth.Workload, seed: int, device, seq_lens=None, max_pages=None,
                 layers=None):
        self.w = w
        self.sh = synth.make_shared(w, seed, device, max_pages=max_pages, seq_lens=seq_lens)
        self.layer_ids = list(range(w.layers)) if layers is None else list(layers)
        self.layers, self.kvs = [], []
        for l in self.layer_ids:
            lay = synth.make_layer(w, self.sh, seed, l, device)
            if lay.k_cache.numel() * 2 <= GUARD_CACHE_BYTES:
                lay.k_cache = guards.guarded_like(lay.k_cache, what=f"k_cache[{l}]")
                lay.v_cache = guards.guarded_like(lay.v_cache, what=f"v_cache[{l}]")
            summ = guards.guarded((w.batch, w.num_kv_heads, self.sh.max_pages, 2, w.head_dim),
                                  torch.bfloat16, device, fill=0, what=f"summaries[{l}]")
            kv = B.PagedKV(lay.k_cache, lay.v_cache, summ, self.sh.block_table, self.sh.seq_lens,
                           w.num_q_heads)
            self.layers.append(lay)
            self.kvs.append(kv)
        self.ws = guards.guarded_workspace(self.kvs[0])
        for kv in self.kvs:
            B.asp_page_summarize(kv, B.ASP_SUMMARIZE_BULK, None, None, self.ws)
        assert B.asp_get_device_error(self.ws) == 0

    @property
    def g(self):
        return self.w.num_q_heads // self.w.num_kv_heads

    def run(self, i, gamma, budget=0):
        kv, lay = self.kvs[i], self.layers[i]
        w = self.w
        dev = kv.device
        lists = guards.guarded((w.batch, w.num_kv_heads, self.sh.max_pages), torch.int32, dev,
                               fill=-7, what="lists")
        lens = guards.guarded((w.batch, w.num_kv_heads), torch.int32, dev, fill=-7, what="lens")
        out = guards.guarded((w.batch, w.num_q_heads, w.head_dim), torch.float32, dev,
                             fill=float("nan"), what="out")
        lse = guards.guarded((w.batch, w.num_q_heads), torch.float32, dev, fill=float("nan"),
                             what="lse")
        B.asp_coverage_select(kv, lay.q, gamma, budget, lists, lens, self.ws)
        B.asp_sparse_decode(kv, lay.q, lists, lens, 1.0 / math.sqrt(w.head_dim), out, lse, self.ws)
        assert B.asp_get_device_error(self.ws) == 0
        return lists, lens, out, lse


def check_case(case: Case, i, gamma, budget, lists, lens, out, lse, segs=None, tally=None,
               check_summaries=True, what=None):
    """Summaries, lists and outputs of layer i against the oracle, per segment.

    Lists are judged by parity.list_verdict and tallied in `tally` (a
    parity.VerdictCounts; a new one, finished here, when None)."""
    w, sh, lay, kv = case.w, case.sh, case.layers[i], case.kvs[i]
    g = case.g
    lists_c, lens_c = lists.cpu().numpy(), lens.cpu().numpy()
    out_c, lse_c = out.cpu().numpy(), lse.cpu().numpy()
    q_c = lay.q.double().cpu().numpy()
    summ = kv.summaries
    seq = sh.seq_lens.cpu().tolist()
    if segs is None:
        segs = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    own = tally is None
    if own:
        tally = parity.VerdictCounts(what or f"{w.name} layer {i} gamma {gamma} budget {budget}")
    for (b, h) in segs:
        T = seq[b]
        kp, vp = parity.segment_kv(lay.k_cache, lay.v_cache, sh.block_table, b, h, T)
        n = kp.shape[0]
        qg = q_c[b, h * g:(h + 1) * g]
        if n:
            mn, mx = O.page_summaries(kp, T)
            scores = O.page_scores(qg, mn, mx)
        if check_summaries and n:
            gmn = parity.bf16_np(summ[b, h, :n, 0])
            gmx = parity.bf16_np(summ[b, h, :n, 1])
            assert np.array_equal(gmn, mn) and np.array_equal(gmx, mx), \
                f"summaries differ at segment {(b, h)}"
        k = int(lens_c[b, h])
        assert 0 <= k <= n, f"len {k} outside [0, {n}] at {(b, h)}"
        ids = lists_c[b, h, :k]
        assert np.all(np.diff(ids) > 0), f"list not ascending at {(b, h)}"
        v = parity.list_verdict(ids, scores, gamma, budget) if n else (
            "exact" if k == 0 else "nonempty")
        tally.add(v, where=f"segment {(b, h)}")
        tally.pages += k
        tally.total += n
        o_ref, lse_ref = O.attend(qg, O.gather_tokens(kp, ids, T), O.gather_tokens(vp, ids, T),
                                  1.0 / math.sqrt(w.head_dim))
        parity.check_outputs(out_c[b, h * g:(h + 1) * g], lse_c[b, h * g:(h + 1) * g],
                             o_ref, lse_ref, what=f"segment {(b, h)}")
    if own:
        tally.finish()
    return tally


def small(name, B_, Hq, Hkv, d, P, T, layers=1, hot=("frac", 0.005, 0.5), shift=(1.0, 4.0)):
    return synth.Workload(name, B_, layers, Hq, Hkv, d, P, seq_len=T, hot=hot, shift=shift)


SMALL = [
    small("g4_d64_p16", 2, 8, 2, 64, 16, 16 * 37 + 5),
    small("g4_d128_p16", 2, 16, 4, 128, 16, 16 * 80 + 11),
    small("g8_d128_p64", 2, 64, 8, 128, 64, 64 * 21 + 63),
    small("g1_d128_p32", 3, 4, 4, 128, 32, 32 * 40 + 1),
    small("g2_d64_p64", 2, 4, 2, 64, 64, 64 * 9 + 17),
    small("g8_d64_p32", 1, 8, 1, 64, 32, 32 * 50),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("gamma", [0.5, 0.9, 0.99, 1.0])
def test_small_shapes(cuda_device, w, gamma):
    case = Case(w, seed=0, device=cuda_device)
    res = case.run(0, gamma)
    check_case(case, 0, gamma, 0, *res)


@pytest.mark.parametrize("budget", [1, 7, 10_000])
def test_budget_mode_small(cuda_device, budget):
    case = Case(SMALL[1], seed=1, device=cuda_device)
    res = case.run(0, 0.5, budget)
    check_case(case, 0, 0.5, budget, *res)


def test_ragged_lengths_and_edges(cuda_device):
    """seq_len 0, 1, P, P+1, mixed lengths, all in one batch."""
    P = 16
    lens = [0, 1, P, P + 1, 5 * P + 3, 33 * P, 2]
    w = synth.Workload("edges", len(lens), 1, 8, 2, 128, P, seq_len=1)
    case = Case(w, seed=2, device=cuda_device, seq_lens=lens, max_pages=40)
    for gamma in (0.3, 0.99, 1.0):
        lists, lens_t, out, lse = case.run(0, gamma)
        check_case(case, 0, gamma, 0, lists, lens_t, out, lse)
        ln = lens_t.cpu()
        assert ln[0].tolist() == [0, 0]
        assert torch.all(out[0] == 0) and torch.all(torch.isinf(lse[0]))
        assert ln[1].tolist() == [1, 1]


def test_single_hot_page_and_tiny_gamma(cuda_device):
    w = small("onehot", 1, 8, 2, 64, 16, 16 * 64, hot=("count", 1, 1), shift=(4.0, 4.0))
    case = Case(w, seed=3, device=cuda_device)
    lists, lens, out, lse = case.run(0, 0.99)
    check_case(case, 0, 0.99, 0, lists, lens, out, lse)
    assert lens.cpu().tolist() == [[1, 1]]
    lists, lens, out, lse = case.run(0, 1e-6)
    check_case(case, 0, 1e-6, 0, lists, lens, out, lse)
    assert lens.cpu().tolist() == [[1, 1]]


def test_all_pages_tied(cuda_device):
    """Constant keys: every score ties, so the lowest ids win and k = ceil(gamma*N)."""
    w = small("tied", 1, 4, 1, 64, 16, 16 * 128)
    case = Case(w, seed=4, device=cuda_device)
    case.layers[0].k_cache.fill_(0.5)
    B.asp_page_summarize(case.kvs[0], B.ASP_SUMMARIZE_BULK, None, None, case.ws)
    for gamma, want in ((0.99, 127), (0.5, 64), (0.3, 39)):
        lists, lens, out, lse = case.run(0, gamma)
        assert int(lens[0, 0]) == want
        assert lists[0, 0, :want].cpu().tolist() == list(range(want))
        check_case(case, 0, gamma, 0, lists, lens, out, lse)


def test_determinism(cuda_device):
    case = Case(SMALL[2], seed=5, device=cuda_device)
    a = case.run(0, 0.95)
    b = case.run(0, 0.95)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("name", ["tiny", "llama8b_32k", "mixed64", "wide70b_64k"])
def test_full_configs(cuda_device, name):
    w = synth.CONFIGS[name]
    case = Case(w, seed=0, device=cuda_device)
    runs = [(g, 0) for g in w.gammas]
    if w.budget_frac > 0:
        n = case.sh.num_pages[0]
        runs.append((0.5, int(math.ceil(w.budget_frac * n))))
    rng = np.random.default_rng(0)
    all_segs = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    for gamma, budget in runs:
        res = case.run(0, gamma, budget)
        segs = all_segs
        if len(all_segs) > 96:  # mixed64: every request's first head + 64 random segments
            pick = rng.choice(len(all_segs), 64, replace=False)
            segs = sorted({(b, 0) for b in range(w.batch)} | {all_segs[i] for i in pick})
        t = check_case(case, 0, gamma, budget, *res, segs=segs,
                       what=f"{name} gamma {gamma} budget {budget}")
        print(f"{name} gamma={gamma} budget={budget}: {t.counts}")


@pytest.fixture(scope="module")
def long128k(cuda_device):
    """The bench's 128k workload (B4 L32 Hq32 Hkv8 d128 P16, 68 GiB resident), built once."""
    case = Case(synth.CONFIGS["long128k"], seed=0, device=cuda_device)
    entries = guards.take()  # the case's buffers outlive each test: re-armed per test
    yield case, entries


@pytest.mark.parametrize("gamma", [0.98, 0.99, 1.0])
def test_long128k_graph_sampled(long128k, gamma):
    """The bench's 128k step (32 layers in one CUDA graph) at each configured gamma,
    checked against the oracle on every segment of layers 0 and 31 plus 16 sampled
    (layer, request, KV head) segments; gamma = 1 is the dense reference the bench times."""
    case, entries = long128k
    guards.register(entries)
    w = case.w
    q = torch.stack([lay.q for lay in case.layers])
    step = DecodeStep(case.kvs, q, gamma=gamma)
    guard_outputs(step)
    step.capture()
    step.replay()
    torch.cuda.synchronize()
    assert B.asp_get_device_error(step.ws) == 0
    rng = np.random.default_rng(1)
    samples = {(0, b, h) for b in range(w.batch) for h in range(w.num_kv_heads)}
    samples |= {(31, b, h) for b in range(w.batch) for h in range(w.num_kv_heads)}
    samples |= {(int(rng.integers(1, 31)), int(rng.integers(0, w.batch)),
                 int(rng.integers(0, w.num_kv_heads))) for _ in range(16)}
    tally = parity.VerdictCounts(f"long128k gamma {gamma} (graph, sampled segments)")
    for l in sorted({s[0] for s in samples}):
        segs = sorted((b, h) for (ll, b, h) in samples if ll == l)
        check_case(case, l, gamma, 0, step.lists[l], step.lens[l], step.out[l], step.lse[l],
                   segs=segs, tally=tally, check_summaries=(l in (0, 31) and gamma == 0.99))
    tally.finish()
    if gamma >= 1.0:
        n = np.array(case.sh.num_pages)
        assert np.array_equal(step.lens.cpu().numpy(),
                              np.broadcast_to(n[None, :, None], tuple(step.lens.shape)))
    print(f"long128k gamma={gamma}: {tally.counts} pages {tally.pages}/{tally.total}")


def test_graph_replay_matches_eager(cuda_device):
    w = small("graph", 2, 16, 4, 128, 16, 16 * 50 + 7, layers=3)
    case = Case(w, seed=6, device=cuda_device)
    q = torch.stack([lay.q for lay in case.layers])
    step = DecodeStep(case.kvs, q, gamma=0.97)
    guard_outputs(step)
    step.run()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (step.lists, step.lens, step.out, step.lse)]
    for t in (step.lists, step.lens, step.out, step.lse):
        t.zero_()
    step.capture()
    for _ in range(3):
        step.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, (step.lists, step.lens, step.out, step.lse)):
        assert torch.equal(a, b)
    for l in range(3):
        check_case(case, l, 0.97, 0, step.lists[l], step.lens[l], step.out[l], step.lse[l])


def test_append_matches_oracle(cuda_device):
    P = 16
    w = small("append", 3, 8, 2, 128, P, 1)
    lens0 = [P * 4, P * 2 + 5, 0]
    # tables sized for the lengths after the append; summaries built before it
    case = Case(w, seed=7, device=cuda_device, seq_lens=[t + 1 for t in lens0], max_pages=8)
    kv = case.kvs[0]
    case.sh.seq_lens.copy_(torch.tensor(lens0, dtype=torch.int32))
    B.asp_page_summarize(kv, B.ASP_SUMMARIZE_BULK, None, None, case.ws)
    case.sh.seq_lens.copy_(torch.tensor([t + 1 for t in lens0], dtype=torch.int32))
    k_ref = parity.bf16_np(kv.k_cache).copy()
    v_ref = parity.bf16_np(kv.v_cache).copy()
    gen = torch.Generator(device=cuda_device).manual_seed(9)
    k_new = torch.randn((3, 2, 128), generator=gen, device=cuda_device).to(torch.bfloat16)
    v_new = torch.randn((3, 2, 128), generator=gen, device=cuda_device).to(torch.bfloat16)
    for _ in range(2):  # idempotent: replaying the append changes nothing
        B.asp_page_summarize(kv, B.ASP_SUMMARIZE_APPEND, k_new, v_new, case.ws)
    assert B.asp_get_device_error(case.ws) == 0
    bt = case.sh.block_table.cpu().numpy()
    want = O.append_token(k_ref, v_ref, bt, np.array([t + 1 for t in lens0]),
                          parity.bf16_np(k_new), parity.bf16_np(v_new))
    assert np.array_equal(parity.bf16_np(kv.k_cache), k_ref)
    assert np.array_equal(parity.bf16_np(kv.v_cache), v_ref)
    summ = parity.bf16_np(kv.summaries)
    for (b, h), (mn, mx) in want.items():
        lp = lens0[b] // P  # logical page of the appended token
        assert np.array_equal(summ[b, h, lp, 0], mn) and np.array_equal(summ[b, h, lp, 1], mx)
    # after the append the whole step still matches the oracle
    res = case.run(0, 0.9)
    check_case(case, 0, 0.9, 0, *res)


def test_device_error_on_bad_page(cuda_device):
    """A corrupt block-table entry sets a device error bit; nothing traps."""
    w = small("bad", 2, 8, 2, 64, 16, 16 * 10)
    case = Case(w, seed=8, device=cuda_device)
    case.sh.block_table[1, 3] = case.sh.num_phys_pages + 1000
    lists = guards.guarded((2, 2, case.sh.max_pages), torch.int32, cuda_device, fill=0)
    lens = guards.guarded((2, 2), torch.int32, cuda_device, fill=0)
    out = guards.guarded((2, 8, 64), torch.float32, cuda_device, fill=0)
    lse = guards.guarded((2, 8), torch.float32, cuda_device, fill=0)
    B.asp_coverage_select(case.kvs[0], case.layers[0].q, 1.0, 0, lists, lens, case.ws)
    B.asp_sparse_decode(case.kvs[0], case.layers[0].q, lists, lens, 0.125, out, lse, case.ws)
    code = B.asp_get_device_error(case.ws)
    assert code & B.ASP_DEVERR_PAGE_RANGE
    assert B.asp_get_device_error(case.ws) == 0  # cleared
    # a list entry past the request and an oversized length
    case.sh.block_table[1, 3] = 0
    lists[0, 0, 0] = 999
    lens[1, 1] = 10_000
    B.asp_workspace_init(case.ws)
    B.asp_sparse_decode(case.kvs[0], case.layers[0].q, lists, lens, 0.125, out, lse, case.ws)
    code = B.asp_get_device_error(case.ws)
    assert code & B.ASP_DEVERR_LIST_RANGE and code & B.ASP_DEVERR_LEN_RANGE
    # the context is still usable: a clean run passes
    B.asp_workspace_init(case.ws)
    case.sh.block_table.copy_(synth.make_shared(w, 8, cuda_device).block_table)
    res = case.run(0, 0.9)
    check_case(case, 0, 0.9, 0, *res)


def test_maximum_segment_count(cuda_device):
    """4096 segments (512 requests x 8 KV heads), the most one call accepts.

    The decode's per-CTA prefix of list lengths then takes 16 KiB of shared
    memory, which leaves the regular (two-slot) ring; the select grid has 4096
    CTAs and the score kernel's request prefix 512 entries. Lengths are drawn
    from 0 to 400 tokens (empty requests and partial pages included); 300
    seeded segments are checked against the oracle, every length for range.
    """
    rng = np.random.default_rng(41)
    lens = [int(x) for x in rng.integers(0, 401, size=512)]
    lens[:3] = [0, 1, 16]
    w = small("max_segments", 512, 32, 8, 64, 16, 1)
    case = Case(w, seed=41, device=cuda_device, seq_lens=lens)
    res = case.run(0, 0.9)
    n_pages = np.array(case.sh.num_pages)
    ln = res[1].cpu().numpy()
    assert np.all(ln >= 0) and np.all(ln <= n_pages[:, None])
    assert np.all((ln == 0) == (n_pages[:, None] == 0))
    segs = [(int(b), int(h)) for b, h in zip(rng.integers(0, 512, 300), rng.integers(0, 8, 300))]
    segs += [(0, 0), (1, 3), (2, 7)]
    check_case(case, 0, 0.9, 0, *res, segs=segs)
