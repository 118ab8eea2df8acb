"""Several decode steps in one CUDA graph, each appending a token, against the oracle.

Step i of the loop appends one token per request at position T0_b + i
(APPEND: its K/V rows and the fold into its page summary), then runs every
layer's coverage selection and attention with its own queries. Appends only
ever write positions past the previous step's, so the final cache restricted
to the first T0_b + i + 1 tokens is exactly the cache step i saw, and the
oracle reruns step i from it (summaries recomputed over those tokens).

Checked: the appended K/V rows and the final summaries bit-exact; every
step's lists under the acceptance rule of tests/parity.py; every step's
outputs against the oracle rerun on the GPU's own lists.
"""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle.asp_oracle as O
from adaptive_sparse_paged_gb300 import binding as B
from adaptive_sparse_paged_gb300 import synth
from adaptive_sparse_paged_gb300.step import DecodeLoop
from tests import parity
from tests.test_gpu_parity import Case, guard_outputs, small

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("gamma,budget", [(0.9, 0), (0.99, 0), (0.5, 6)])
def test_decode_loop_matches_oracle(cuda_device, gamma, budget):
    P, n = 16, 5
    # ragged starts: a partial page, a page one token from full (step 1 opens a
    # fresh page), a three-token request
    T0 = [P * 20 + 13, P * 9 + 15, 3]
    final = [t + n for t in T0]
    w = small("loop", 3, 8, 2, 128, P, 1, layers=2)
    case = Case(w, seed=5, device=cuda_device, seq_lens=final)
    # summaries must describe the first T0 tokens when the loop starts
    case.sh.seq_lens.copy_(torch.tensor(T0, dtype=torch.int32))
    for kv in case.kvs:
        B.asp_page_summarize(kv, B.ASP_SUMMARIZE_BULK, None, None, case.ws)
    assert B.asp_get_device_error(case.ws) == 0
    steps = synth.make_steps(w, [lay.q for lay in case.layers], n, seed=6, device=cuda_device)
    loop = DecodeLoop(case.kvs, case.sh.seq_lens.clone(), steps.q, steps.k_new, steps.v_new,
                      gamma, budget)
    guard_outputs(loop)
    loop.capture()
    loop.replay()  # the first launch of the loop: fresh steps
    torch.cuda.synchronize()
    assert B.asp_get_device_error(loop.ws) == 0

    g = w.num_q_heads // w.num_kv_heads
    bt = case.sh.block_table.cpu().numpy()
    scale = 1.0 / math.sqrt(w.head_dim)
    q_all = steps.q.double().cpu().numpy()
    kn, vn = parity.bf16_np(steps.k_new), parity.bf16_np(steps.v_new)
    lists, lens = loop.lists.cpu().numpy(), loop.lens.cpu().numpy()
    out, lse = loop.out.cpu().numpy(), loop.lse.cpu().numpy()
    tally = parity.VerdictCounts(f"multistep {w.name} gamma {gamma} budget {budget}")
    for l, (lay, kv) in enumerate(zip(case.layers, case.kvs)):
        k_all, v_all = parity.bf16_np(kv.k_cache), parity.bf16_np(kv.v_cache)
        summ = parity.bf16_np(kv.summaries)
        for b in range(w.batch):
            for h in range(w.num_kv_heads):
                # appended rows landed where APPEND puts them
                for i in range(n):
                    t = T0[b] + i
                    phys = bt[b, t // P]
                    assert np.array_equal(k_all[phys, h, t % P], kn[i, l, b, h])
                    assert np.array_equal(v_all[phys, h, t % P], vn[i, l, b, h])
                kp, vp = parity.segment_kv(kv.k_cache, kv.v_cache, case.sh.block_table, b, h,
                                           final[b])
                mn, mx = O.page_summaries(kp, final[b])
                npg = kp.shape[0]
                assert np.array_equal(summ[b, h, :npg, 0], mn)
                assert np.array_equal(summ[b, h, :npg, 1], mx)
                for i in range(n):
                    T = T0[b] + i + 1
                    npi = (T + P - 1) // P  # pages of step i's context
                    kpi, vpi = kp[:npi], vp[:npi]
                    qg = q_all[i, l, b, h * g:(h + 1) * g]
                    ref = O.decode_segment(qg, kpi, vpi, T, gamma, budget, scale)
                    k = int(lens[i, l, b, h])
                    ids = lists[i, l, b, h, :k]
                    v = parity.list_verdict(ids, ref["scores"], gamma, budget)
                    tally.add(v, where=f"step {i} layer {l} segment {(b, h)}")
                    o_ref, lse_ref = O.attend(qg, O.gather_tokens(kpi, ids, T),
                                              O.gather_tokens(vpi, ids, T), scale)
                    parity.check_outputs(out[i, l, b, h * g:(h + 1) * g],
                                         lse[i, l, b, h * g:(h + 1) * g], o_ref, lse_ref,
                                         what=f"step {i} layer {l} segment {(b, h)}")
    assert tally.finish()["exact"] > 0


def test_decode_loop_replay_is_stable(cuda_device):
    """Replays re-time the same work: appended rows, lengths and shapes stay put."""
    P, n = 16, 3
    T0 = [P * 8 + 2, P * 4]
    w = small("loop_replay", 2, 4, 1, 64, P, 1, layers=1)
    case = Case(w, seed=9, device=cuda_device, seq_lens=[t + n for t in T0])
    case.sh.seq_lens.copy_(torch.tensor(T0, dtype=torch.int32))
    B.asp_page_summarize(case.kvs[0], B.ASP_SUMMARIZE_BULK, None, None, case.ws)
    steps = synth.make_steps(w, [case.layers[0].q], n, seed=10, device=cuda_device)
    loop = DecodeLoop(case.kvs, case.sh.seq_lens.clone(), steps.q, steps.k_new, steps.v_new,
                      0.9)
    guard_outputs(loop)
    loop.capture()
    loop.replay()
    torch.cuda.synchronize()
    k1 = case.kvs[0].k_cache.clone()
    for _ in range(3):
        loop.replay()
    torch.cuda.synchronize()
    assert B.asp_get_device_error(loop.ws) == 0
    assert torch.equal(case.kvs[0].k_cache, k1)
    assert loop.launches == n * 1 * 3  # fused append: score, select, decode
    assert [int(x[0]) for x in loop.seq_lens] == [T0[0] + i + 1 for i in range(n)]
