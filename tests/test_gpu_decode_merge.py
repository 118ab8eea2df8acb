"""The decode's merge of split segments, done by the last of their CTAs.

Each CTA that holds part of a segment counts itself in with one atomic after
its stream; the CTA that completes the count folds the segment's partials in
CTA order, writes out/lse and puts the count back to zero. The counts live
in the workspace right after its 256-byte header, one int32 per segment
(B * Hkv). These tests check that contract directly: the counts are zero
after every call, repeated calls give bit-identical outputs, a segment held
by every CTA of the grid (more pieces than one fold batch of eight) matches
the oracle, and so do many short segments of mixed lengths, where CTAs hold
several pieces and may complete two segments each.
"""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle.asp_oracle as O
from adaptive_sparse_paged_gb300 import binding as B
from tests import guards, parity
from tests.test_gpu_parity import Case, check_case, small

pytestmark = pytest.mark.gpu

ARRIVALS_OFF = 256  # after the workspace header (error word)


def _arrivals(case) -> np.ndarray:
    S = case.w.batch * case.w.num_kv_heads
    raw = case.ws[ARRIVALS_OFF:ARRIVALS_OFF + 4 * S].clone()
    return raw.view(torch.int32).cpu().numpy()


def _decode(case, lists, lens):
    w, kv, lay = case.w, case.kvs[0], case.layers[0]
    out = guards.guarded((w.batch, w.num_q_heads, w.head_dim), torch.float32, kv.device,
                         fill=float("nan"), what="out")
    lse = guards.guarded((w.batch, w.num_q_heads), torch.float32, kv.device,
                         fill=float("nan"), what="lse")
    B.asp_sparse_decode(kv, lay.q, lists, lens, 1.0 / math.sqrt(w.head_dim), out, lse, case.ws)
    assert B.asp_get_device_error(case.ws) == 0
    return out, lse


def test_one_segment_held_by_every_cta(cuda_device):
    """4096 pages of one segment: every CTA holds a piece, 152 partials folded
    in batches of eight by the last CTA to finish."""
    w = small("one_segment", 1, 8, 1, 128, 16, 16 * 4096)
    case = Case(w, seed=71, device=cuda_device)
    n = case.sh.num_pages[0]
    lists = guards.guarded((1, 1, case.sh.max_pages), torch.int32, cuda_device, fill=-3,
                           what="lists")
    lists[0, 0, :n] = torch.arange(n, dtype=torch.int32, device=cuda_device)
    lens = guards.guarded((1, 1), torch.int32, cuda_device, fill=n, what="lens")
    assert not _arrivals(case).any()
    out, lse = _decode(case, lists, lens)
    assert not _arrivals(case).any(), "arrival count left non-zero"
    lay = case.layers[0]
    seq = int(case.sh.seq_lens[0])
    kp, vp = parity.segment_kv(lay.k_cache, lay.v_cache, case.sh.block_table, 0, 0, seq)
    ids = list(range(n))
    o_ref, lse_ref = O.attend(lay.q.double().cpu().numpy()[0], O.gather_tokens(kp, ids, seq),
                              O.gather_tokens(vp, ids, seq), 1.0 / math.sqrt(w.head_dim))
    parity.check_outputs(out.cpu().numpy()[0], lse.cpu().numpy()[0], o_ref, lse_ref,
                         what="one segment over every CTA")
    out2, lse2 = _decode(case, lists, lens)
    assert torch.equal(out, out2) and torch.equal(lse, lse2), "repeat differs"
    assert not _arrivals(case).any()


@pytest.mark.parametrize("d,gamma", [(64, 0.9), (64, 0.99), (128, 0.99)])
def test_many_short_segments_of_mixed_lengths(cuda_device, d, gamma):
    """256 segments of 1 to 700 pages: CTAs hold several pieces and complete
    up to two segments each; lists and outputs against the oracle, counts
    back to zero, a repeat bit-identical. At d = 128 the prefix of 256
    segment lengths no longer fits beside the deep ring, so the decode runs
    its shallower ring."""
    rng = np.random.default_rng(72)
    seq_lens = [int(x) for x in rng.integers(1, 16 * 700, size=64)]
    seq_lens[3] = 0
    seq_lens[7] = 16
    w = small(f"mixed_short_d{d}", 64, 8, 4, d, 16, max(seq_lens))
    case = Case(w, seed=73, device=cuda_device, seq_lens=seq_lens)
    lists, lens, out, lse = case.run(0, gamma)
    assert not _arrivals(case).any(), "arrival count left non-zero"
    check_case(case, 0, gamma, 0, lists, lens, out, lse, what=f"mixed_short d{d} gamma {gamma}")
    out2, lse2 = _decode(case, lists, lens)
    assert torch.equal(out, out2) and torch.equal(lse, lse2), "repeat differs"
    assert not _arrivals(case).any()
