"""Helpers that compare the CUDA path with the fp64 oracle.

List acceptance (coverage rule of the MOIRA abstract): a GPU list G for one
segment is accepted when it equals the oracle's set, or when both
  (a) G is a top set up to score ties: every page in G scores at least every
      page outside G, within 1e-6 relative, and
  (b) G reaches gamma and is minimal up to mass ties: mass(G) >= gamma - 1e-6
      and mass(G without its lowest-scored page) < gamma + 1e-6,
with scores and masses from the oracle in fp64. Budget mode replaces (b) by
|G| = min(budget, N). The 1e-6 is the tie width the selection is specified
to; each accepted-but-different list is counted and reported.

Attention outputs are compared against the oracle rerun on the GPU's own
lists (so selection and arithmetic errors stay apart): max-abs 2e-2 and
mean-abs 2e-3 over fp32 outputs and lse, for bf16 K/V with fp32 accumulation.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle.asp_oracle as O

TIE_REL = 1e-6
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3


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


def list_verdict(gpu_ids, scores, gamma, budget=0):
    """'exact', 'accepted' or a failure reason string."""
    n = len(scores)
    G = sorted(int(x) for x in gpu_ids)
    want = sorted(int(x) for x in O.coverage_select(scores, gamma, budget))
    if G == want:
        return "exact"
    if len(set(G)) != len(G) or any(p < 0 or p >= n for p in G):
        return f"invalid ids {G[:8]}..."
    inside = np.zeros(n, dtype=bool)
    inside[G] = True
    if not inside.any():
        return "empty list"
    scale = max(float(np.max(np.abs(scores))), 1e-30)
    lo_in = float(scores[inside].min())
    hi_out = float(scores[~inside].max()) if (~inside).any() else -np.inf
    if lo_in < hi_out - TIE_REL * scale:
        return f"not a top set: min in {lo_in} < max out {hi_out}"
    if budget > 0:
        return "accepted" if len(G) == min(budget, n) else f"budget count {len(G)}"
    if gamma >= 1.0:
        return "accepted" if len(G) == n else f"gamma=1 count {len(G)}"
    mass = O.page_mass(scores)
    m_all = float(mass[inside].sum())
    low = G[int(np.argmin(scores[G]))]
    m_less = m_all - float(mass[low])
    if m_all < gamma - TIE_REL:
        return f"mass {m_all} below gamma {gamma}"
    if m_less >= gamma + TIE_REL:
        return f"not minimal: {m_less} without the lowest page"
    return "accepted"


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
