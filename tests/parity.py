"""Helpers that compare the CUDA path with the fp64 oracle.

List acceptance (coverage rule of the MOIRA abstract: per request, layer, KV
head and step, the smallest page set whose estimated attention mass reaches
gamma). The GPU list G of one segment is compared with the oracle's set W,
k_W = |W| pages, using the oracle's fp64 scores s and masses (softmax of s):

* ``exact``: G == W.
* ``score_tie``: |G| == |W| and G equals W after swapping pages tied with
  the cutoff, with the tie width taken relative to the cutoff score s_cut
  (the lowest score in W), as the decode-path specification states:
    1. every page in the symmetric difference of G and W scores within
       1e-6 * max(|s_cut|, 1e-30) of s_cut;
    2. mass(G) >= gamma - 1e-6;
    3. mass(G without its lowest-scored page) < gamma + 1e-6.
  Budget mode keeps condition 1 and |G| == min(budget, N).
* ``mass_tie``: |G| != |W|, but G is the oracle's top |G| pages (up to pages
  tied, in the same sense, with that set's own cutoff score) and conditions
  2 and 3 hold: the oracle's running mass crosses gamma within 1e-6 of where
  the two counts differ. The GPU decides that crossing on fp32 scores, whose
  rounding (about 1e-7 of a score) moves masses by about as much. It is not
  a score tie, so every test counts these lists separately and bounds how
  many it accepts (``mass_tie_max``).

Anything else is a failure, returned as a reason string. gamma is taken at
float32, the precision the C ABI passes it in.

Attention outputs are compared against the oracle rerun on the GPU's own
lists (so selection and arithmetic errors stay apart): max-abs 2e-2 and
mean-abs 2e-3 over fp32 outputs and lse, for bf16 K/V with fp32 accumulation.
"""

from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle.asp_oracle as O

TIE_REL = 1e-6
MASS_TOL = 1e-6
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
ACCEPTED = ("exact", "score_tie", "mass_tie")


def mass_tie_max(segments: int) -> int:
    """Mass ties a test accepts over `segments` checked lists: one per 256
    lists, at least one. Each needs the oracle's running mass to land within
    about 1e-7 of gamma at the cutoff; on the benchmark workloads that is
    about one segment in a thousand."""
    return max(1, segments // 256)


def bf16_np(t: torch.Tensor) -> np.ndarray:
    """Exact fp64 copy of a bf16 tensor (any device)."""
    return O.bf16_bits_to_f64(t.detach().contiguous().view(torch.int16).cpu().numpy())


def segment_kv(layer_k, layer_v, block_table, b, h, seq_len):
    """Gather one segment's pages [N, P, d] (logical order) as exact fp64."""
    P = layer_k.shape[2]
    n = (seq_len + P - 1) // P
    if n == 0:
        d = layer_k.shape[3]
        return np.zeros((0, P, d)), np.zeros((0, P, d))
    idx = block_table[b, :n].to(torch.long)
    return bf16_np(layer_k[idx, h]), bf16_np(layer_v[idx, h])


def _rank(scores):
    """Oracle order: score descending, ties to the lower page id."""
    return np.lexsort((np.arange(len(scores)), -scores))


def _tied_with(scores, pages, s_c):
    w = TIE_REL * max(abs(float(s_c)), 1e-30)
    return all(abs(float(scores[p]) - float(s_c)) <= w for p in pages)


def list_verdict(gpu_ids, scores, gamma, budget=0):
    """'exact', 'score_tie', 'mass_tie' or a failure reason string."""
    gamma = float(np.float32(gamma))
    n = len(scores)
    G = sorted(int(x) for x in gpu_ids)
    want = sorted(int(x) for x in O.coverage_select(scores, gamma, budget))
    if G == want:
        return "exact"
    if len(set(G)) != len(G) or any(p < 0 or p >= n for p in G):
        return f"invalid ids {G[:8]}..."
    if not G:
        return "empty list"
    if budget > 0 and len(G) != min(budget, n):
        return f"budget count {len(G)}"
    if budget <= 0 and gamma >= 1.0:
        return f"gamma=1 count {len(G)}"
    order = _rank(scores)
    gs = set(G)
    # G against the oracle's top |G| pages, up to pages tied with that set's cutoff
    top = set(int(p) for p in order[:len(G)])
    if not _tied_with(scores, gs ^ top, scores[order[len(G) - 1]]):
        return f"not a top set within the tie width ({len(G)} pages, oracle {len(want)})"
    kind = "score_tie" if len(G) == len(want) else "mass_tie"
    if budget > 0:
        return kind
    mass = O.page_mass(scores)
    m_all = float(mass[G].sum())
    low = G[int(np.argmin(scores[G]))]
    m_less = m_all - float(mass[low])
    if m_all < gamma - MASS_TOL:
        return f"mass {m_all} below gamma {gamma}"
    if m_less >= gamma + MASS_TOL:
        return f"not minimal: {m_less} without the lowest page"
    return kind


class VerdictCounts:
    """Per-test tally of list verdicts; enforces the mass-tie bound."""

    def __init__(self, what: str):
        self.what = what
        self.counts = {k: 0 for k in ACCEPTED}
        self.pages = 0
        self.total = 0

    def add(self, verdict: str, where=""):
        assert verdict in ACCEPTED, f"{self.what} {where}: {verdict}"
        self.counts[verdict] += 1

    @property
    def segments(self) -> int:
        return sum(self.counts.values())

    def finish(self):
        """Asserts the mass-tie bound and records the tally (see record())."""
        record(self.what, dict(self.counts, segments=self.segments,
                               pages=self.pages, total_pages=self.total))
        cap = mass_tie_max(self.segments)
        assert self.counts["mass_tie"] <= cap, \
            f"{self.what}: {self.counts['mass_tie']} mass ties in {self.segments} lists (max {cap})"
        return self.counts


_RECORDS: dict = {}


def record(what: str, counts: dict):
    """Keeps a verdict tally for the session report (ASP_PARITY_REPORT=path
    writes every tally as JSON when the session ends)."""
    _RECORDS[what] = counts


def write_report():
    path = os.environ.get("ASP_PARITY_REPORT")
    if path and _RECORDS:
        os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
        with open(path, "w") as f:
            json.dump(_RECORDS, f, indent=1, sort_keys=True)


def check_outputs(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    err = np.abs(o_gpu - o_ref)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    assert err.max() <= OUT_MAX_ABS, f"{what}: max-abs {err.max():.3e}"
    assert err.mean() <= OUT_MEAN_ABS, f"{what}: mean-abs {err.mean():.3e}"
    lg, lr = np.asarray(lse_gpu, np.float64), np.asarray(lse_ref, np.float64)
    fin = np.isfinite(lr)
    assert np.array_equal(np.isfinite(lg), fin), f"{what}: lse finiteness differs"
    if fin.any():
        le = np.abs(lg[fin] - lr[fin])
        assert le.max() <= OUT_MAX_ABS, f"{what}: lse max-abs {le.max():.3e}"
        assert le.mean() <= OUT_MEAN_ABS, f"{what}: lse mean-abs {le.mean():.3e}"
    return float(err.max()), float(err.mean())
