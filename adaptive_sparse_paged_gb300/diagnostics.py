"""Budget diagnostics: how many pages the coverage rule needs, against a fixed budget.

The MOIRA abstract (page "Adaptive DHiSparse: Speculative Decoding over a
Load-Adaptive KV Hierarchy") argues that the pages attention needs vary
widely across requests, layers, KV heads and steps, so a fixed page budget
sized for demanding heads wastes bytes on easy ones and still falls short on
hard ones. This module measures that on a workload:

* for each gamma, the distribution over (layer, request, KV head) segments of
  the required fraction len / N_b that the coverage rule selects;
* a fixed top-k budget with the same total bytes as the coverage rule at a
  reference gamma (the same k pages for every segment, capped at N_b), and
  the estimated mass it captures per segment, beside the gamma every
  coverage-rule list reaches by construction.

Selections come from asp_coverage_select and the estimate from
asp_page_scores (the library's kernels); the aggregation (softmax over a
segment's page scores, sorting, histograms) runs as plain tensor operations,
outside the decode path.
"""

from __future__ import annotations

import numpy as np
import torch

from . import binding as B

FRACTION_EDGES = (0.0, 0.01, 0.02, 0.05, 0.1, 0.2, 0.3, 0.5, 0.8, 1.0)


def required_fractions(lens: np.ndarray, num_pages) -> np.ndarray:
    """lens [L, B, Hkv] and N_b per request -> len / N_b for segments with N_b > 0."""
    lens = np.asarray(lens, dtype=np.float64)
    n = np.asarray(num_pages, dtype=np.float64)[None, :, None]
    n = np.broadcast_to(n, lens.shape)
    keep = n > 0
    return lens[keep] / n[keep]


def fraction_histogram(fracs: np.ndarray, edges=FRACTION_EDGES) -> dict:
    """Counts per [edge_i, edge_i+1) bin (the last bin closed) plus summary quantiles."""
    fracs = np.asarray(fracs, dtype=np.float64)
    counts, _ = np.histogram(fracs, bins=np.asarray(edges))
    q = np.quantile(fracs, [0.1, 0.5, 0.9]) if fracs.size else np.zeros(3)
    return {"edges": list(edges), "counts": [int(c) for c in counts],
            "mean": float(fracs.mean()) if fracs.size else 0.0,
            "p10": float(q[0]), "p50": float(q[1]), "p90": float(q[2]),
            "min": float(fracs.min()) if fracs.size else 0.0,
            "max": float(fracs.max()) if fracs.size else 0.0}


def captured_mass_topk(scores: torch.Tensor, num_pages: torch.Tensor, k: int) -> torch.Tensor:
    """Estimated mass (softmax of page scores) that the top min(k, N_b) pages of
    each segment capture. scores [B, Hkv, max_pages]; num_pages int [B]."""
    Bn, H, M = scores.shape
    idx = torch.arange(M, device=scores.device)
    valid = idx[None, None, :] < num_pages.to(scores.device)[:, None, None]
    s = torch.where(valid, scores.double(), torch.full_like(scores, float("-inf"), dtype=torch.float64))
    mass = torch.softmax(s, dim=-1)
    srt, _ = torch.sort(mass, dim=-1, descending=True)
    cum = torch.cumsum(srt, dim=-1)
    kk = torch.clamp(num_pages.to(scores.device).long(), max=k).clamp(min=1) - 1
    return cum.gather(-1, kk[:, None, None].expand(Bn, H, 1)).squeeze(-1)


def budget_diagnostics(kvs, q_all, gammas=(0.95, 0.98, 0.99, 0.995, 0.999),
                       ref_gamma: float = 0.99, detail: bool = False) -> dict:
    """kvs: PagedKV per layer; q_all fp32 [L, B, Hq, d]. Returns a JSON-ready dict.

    detail=True adds the per-segment arrays behind the summaries under
    "detail": "lens" {gamma: int [L, B, Hkv]} and "captured" (float64
    [L, B, Hkv], the fixed budget's captured mass; NaN where N_b = 0)."""
    kv0 = kvs[0]
    L, dev = len(kvs), kv0.device
    ws = B.new_workspace(kv0)
    seq = kv0.seq_lens.cpu().numpy().astype(np.int64)
    n_pages = (seq + kv0.page_size - 1) // kv0.page_size
    lists = torch.empty((kv0.batch, kv0.num_kv_heads, kv0.max_pages), dtype=torch.int32,
                        device=dev)
    out = {"segments": int(L * kv0.batch * kv0.num_kv_heads), "by_gamma": {}}
    lens_ref = None
    lens_all = {}
    for gm in sorted(set(list(gammas) + [ref_gamma])):
        lens = torch.empty((L, kv0.batch, kv0.num_kv_heads), dtype=torch.int32, device=dev)
        for l, kv in enumerate(kvs):
            B.asp_coverage_select(kv, q_all[l], gm, 0, lists, lens[l], ws)
        ln = lens.cpu().numpy()
        lens_all[gm] = ln
        if gm == ref_gamma:
            lens_ref = ln
        if gm in gammas:
            out["by_gamma"][f"{gm:g}"] = fraction_histogram(required_fractions(ln, n_pages))
    assert B.asp_get_device_error(ws) == 0
    # fixed budget with the same total pages as the coverage rule at ref_gamma
    n_seg = int((n_pages > 0).sum()) * kv0.num_kv_heads * L
    k = max(1, int(round(float(lens_ref.sum()) / max(1, n_seg))))
    scores = torch.empty((kv0.batch, kv0.num_kv_heads, kv0.max_pages), dtype=torch.float32,
                         device=dev)
    n_dev = torch.as_tensor(n_pages, device=dev)
    caps = []
    cap_full = np.full((L, kv0.batch, kv0.num_kv_heads), np.nan)
    for l, kv in enumerate(kvs):
        B.asp_page_scores(kv, q_all[l], scores, ws)
        cap = captured_mass_topk(scores, n_dev, k)
        caps.append(cap[n_dev > 0].flatten())
        cap_full[l][n_pages > 0] = cap[n_dev > 0].cpu().numpy()
    assert B.asp_get_device_error(ws) == 0
    cap = torch.cat(caps).cpu().numpy()
    out["fixed_budget_equal_bytes"] = {
        "pages_per_segment": k,
        "ref_gamma": ref_gamma,
        "captured_mass": {"mean": float(cap.mean()), "min": float(cap.min()),
                          "p10": float(np.quantile(cap, 0.1)),
                          "p50": float(np.quantile(cap, 0.5))},
        "segments_below_ref_gamma": float((cap < ref_gamma).mean()),
    }
    if detail:
        out["detail"] = {"lens": lens_all, "captured": cap_full}
    return out
