"""asp_coverage_select_append = APPEND then asp_coverage_select, bit for bit.

The fused call does the append inside the score kernel: the warp that
streams a segment's last page writes the new K/V rows and folds the key into
that page's summary before copying it. Two identical workloads are run, one
through the two separate calls and one through the fused call; K and V
caches, summaries, lists and lengths must be identical (all integer or
exactly rounded bf16 data), for appends into a partial page, into slot 0 of a
fresh page, into a one-token request and with an empty request, in mass and
budget mode (a budget of every page included) and at gamma = 1 (scores
skipped, append still done), on both selection paths.
"""

import pytest
import torch

from adaptive_sparse_paged_gb300 import binding as B
from adaptive_sparse_paged_gb300 import synth
from tests import guards
from tests.test_gpu_parity import Case, small

pytestmark = pytest.mark.gpu


def _pair(dev, w, lens_before, seed):
    cases = []
    for _ in range(2):
        c = Case(w, seed=seed, device=dev, seq_lens=[t + 1 if t > 0 else 0 for t in lens_before])
        c.sh.seq_lens.copy_(torch.tensor(lens_before, dtype=torch.int32))
        for kv in c.kvs:
            B.asp_page_summarize(kv, B.ASP_SUMMARIZE_BULK, None, None, c.ws)
        c.sh.seq_lens.copy_(torch.tensor([t + 1 if t > 0 else 0 for t in lens_before],
                                         dtype=torch.int32))
        assert B.asp_get_device_error(c.ws) == 0
        cases.append(c)
    return cases


@pytest.mark.parametrize("d,P,g,lens", [
    (128, 16, 4, [16 * 40 + 7, 16 * 12 - 1 + 16, 0]),  # partial page; next-to-full; empty request
    (128, 16, 4, [16 * 31, 1, 16 * 5 + 3]),            # slot 0 of a fresh page; 1 -> 2 tokens
    (64, 32, 2, [32 * 9 + 31, 32 * 3, 77]),
    (128, 64, 8, [64 * 7 + 10, 64 * 2, 63]),
    # 64 pages or more: the cluster kernel scores, appends and selects
    (128, 16, 4, [16 * 300 + 7, 16 * 100, 0]),
    (64, 16, 2, [16 * 2100 + 5, 16 * 70, 9]),
])
@pytest.mark.parametrize("gamma,budget", [(0.9, 0), (0.5, 5), (1.0, 0), (0.5, 100_000)])
def test_fused_append_equals_separate_calls(cuda_device, d, P, g, lens, gamma, budget):
    Hkv = 2
    w = small(f"fused_d{d}_p{P}", len(lens), g * Hkv, Hkv, d, P, 1)
    a, b = _pair(cuda_device, w, lens, seed=d + P)
    gen = torch.Generator(device=cuda_device).manual_seed(31)
    k_new = torch.randn((len(lens), Hkv, d), generator=gen, device=cuda_device).to(torch.bfloat16)
    v_new = torch.randn((len(lens), Hkv, d), generator=gen, device=cuda_device).to(torch.bfloat16)
    outs = []
    for c, fused in ((a, False), (b, True)):
        kv, q = c.kvs[0], c.layers[0].q
        lists = guards.guarded((w.batch, Hkv, c.sh.max_pages), torch.int32, cuda_device,
                               fill=-3, what="lists")
        ln = guards.guarded((w.batch, Hkv), torch.int32, cuda_device, fill=-3, what="lens")
        for _ in range(2):  # idempotent: a second pass changes nothing
            if fused:
                B.asp_coverage_select_append(kv, k_new, v_new, q, gamma, budget, lists, ln, c.ws)
            else:
                B.asp_page_summarize(kv, B.ASP_SUMMARIZE_APPEND, k_new, v_new, c.ws)
                B.asp_coverage_select(kv, q, gamma, budget, lists, ln, c.ws)
        assert B.asp_get_device_error(c.ws) == 0
        outs.append((kv.k_cache, kv.v_cache, kv.summaries, lists, ln))
    for x, y, name in zip(outs[0], outs[1], ("k_cache", "v_cache", "summaries", "lists", "lens")):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y), name
