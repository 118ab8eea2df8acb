"""Seeded synthetic decode workloads (inputs only; none of the method's arithmetic).

This module is the one piece of code that both the CUDA path's tests/bench
and the CPU oracle consume: it draws the paged K/V caches, block tables,
sequence lengths and queries. It imports nothing from the rest of the package
and computes no summary, score, selection or attention.

The shapes mirror the long-context decode workloads the MOIRA abstract (page
"Adaptive DHiSparse: Speculative Decoding over a Load-Adaptive KV
Hierarchy") measures on RULER at 128k context; RULER itself and model weights
are not used, these seeded draws stand in for them:

* K and V are N(0, 1), stored as bf16. Queries are fp32 N(0, 1).
* Each (layer, request, KV head) gets its own set of "hot" pages, drawn
  uniformly without replacement among the request's pages; every key of a hot
  page is moved by  shift * sqrt(d) * q_hat,  q_hat the unit mean of the
  group's queries. The sqrt(d) makes `shift` a multiple of the typical key
  norm; with a unit-norm shift the page bounds barely move and every head
  would need ~95% of its pages, against the spread of needed fractions the
  workloads are meant to have. Hot keys are shifted in fp32 and rounded to
  bf16 once more.
* Physical pages are a seeded permutation, so consecutive logical pages are
  scattered in memory. A few physical pages stay unmapped.
* Hot-page count: "count" draws round(exp(U * ln 32)) in [1, 32];
  "frac" draws a fraction log-uniform in [0.5%, 50%] of N_b (at least 1).
* Sequence lengths: fixed, or log-normal (median 16384, sigma 1) clipped to
  [4096, 131072] and not rounded to the page size (partial last pages).
* Multi-step decoding: step i's queries are the layer's queries plus
  sigma * N(0, 1) noise (sigma 0.25), so consecutive steps stay correlated
  while their page lists vary; each step appends one token per request whose
  key and value are N(0, 1) in bf16.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    seq_len: int = 0                # fixed context, or 0 with lognormal_lens
    lognormal_lens: bool = False
    hot: tuple = ("frac", 0.005, 0.5)
    shift: tuple = (1.0, 4.0)       # uniform range of the hot-page shift
    gammas: tuple = (0.99,)
    budget_frac: float = 0.0        # > 0: also run the fixed top-k comparison
    extra_phys_pages: int = 8


CONFIGS = {
    "tiny": Workload("tiny", 1, 1, 8, 2, 64, 16, seq_len=2048, hot=("count", 1, 32),
                     shift=(3.0, 3.0), gammas=(0.99, 1.0)),
    "llama8b_32k": Workload("llama8b_32k", 8, 1, 32, 8, 128, 16, seq_len=32768,
                            gammas=(0.98, 0.99)),
    "long128k": Workload("long128k", 4, 32, 32, 8, 128, 16, seq_len=131072,
                         gammas=(0.98, 0.99, 1.0)),
    "mixed64": Workload("mixed64", 64, 1, 32, 8, 128, 16, lognormal_lens=True,
                        gammas=(0.99,)),
    "wide70b_64k": Workload("wide70b_64k", 16, 1, 64, 8, 128, 64, seq_len=65536,
                            gammas=(0.99,), budget_frac=0.3),
}


def _gen(seed: int, *salt: int, device) -> torch.Generator:
    """A torch generator on `device` seeded from (seed, *salt)."""
    h = 0x9E3779B97F4A7C15 ^ (seed & 0xFFFFFFFF)
    for s in salt:
        h = (h * 0x100000001B3) ^ (int(s) & 0xFFFFFFFF)
        h &= 0xFFFFFFFFFFFFFFFF
    g = torch.Generator(device=device)
    g.manual_seed(h & 0x7FFFFFFFFFFFFFFF)
    return g


def seq_lens_for(w: Workload, seed: int):
    if not w.lognormal_lens:
        return [w.seq_len] * w.batch
    g = _gen(seed, 1, device="cpu")
    z = torch.randn(w.batch, generator=g, dtype=torch.float64)
    return [int(min(131072, max(4096, round(16384 * math.exp(float(x)))))) for x in z]


@dataclass
class Shared:
    """Layer-independent inputs: lengths, block table, page counts."""
    seq_lens: torch.Tensor        # int32 [B]
    block_table: torch.Tensor     # int32 [B, max_pages]
    num_pages: list               # N_b
    max_pages: int
    num_phys_pages: int


def make_shared(w: Workload, seed: int, device, max_pages: int | None = None,
                seq_lens=None) -> Shared:
    lens = list(seq_lens) if seq_lens is not None else seq_lens_for(w, seed)
    P = w.page_size
    n_pages = [(t + P - 1) // P for t in lens]
    mp = max_pages if max_pages is not None else max(1, max(n_pages))
    n_phys = sum(n_pages) + w.extra_phys_pages
    g = _gen(seed, 2, device="cpu")
    perm = torch.randperm(n_phys, generator=g).to(torch.int32)
    bt = torch.full((w.batch, mp), -1, dtype=torch.int32)
    i = 0
    for b, n in enumerate(n_pages):
        bt[b, :n] = perm[i:i + n]
        i += n
    return Shared(torch.tensor(lens, dtype=torch.int32, device=device), bt.to(device),
                  n_pages, mp, n_phys)


@dataclass
class Layer:
    k_cache: torch.Tensor   # bf16 [num_phys, Hkv, P, d]
    v_cache: torch.Tensor
    q: torch.Tensor         # fp32 [B, Hq, d]
    hot: dict = field(default_factory=dict)  # (b, kv_head) -> list of hot logical pages


def make_layer(w: Workload, sh: Shared, seed: int, layer: int, device,
               unit_shift: bool = False) -> Layer:
    """Draws one layer's caches and queries (on `device`).

    unit_shift: move hot keys by shift * q_hat (the literal unit-norm reading
    of the configs) instead of shift * sqrt(d) * q_hat; the draws are otherwise
    the same."""
    B, Hq, Hkv, d, P = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size
    g_grp = Hq // Hkv
    gk = _gen(seed, 10, layer, device=device)
    gv = _gen(seed, 11, layer, device=device)
    gq = _gen(seed, 12, layer, device=device)
    shape = (sh.num_phys_pages, Hkv, P, d)
    k = torch.randn(shape, generator=gk, device=device, dtype=torch.bfloat16)
    v = torch.randn(shape, generator=gv, device=device, dtype=torch.bfloat16)
    q = torch.randn((B, Hq, d), generator=gq, device=device, dtype=torch.float32)
    gh = _gen(seed, 13, layer, device="cpu")
    bt_cpu = sh.block_table.cpu()
    hot = {}
    for b in range(B):
        n = sh.num_pages[b]
        if n == 0:
            continue
        for h in range(Hkv):
            u = float(torch.rand(1, generator=gh, dtype=torch.float64))
            if w.hot[0] == "count":
                cnt = int(round(math.exp(u * math.log(w.hot[2])))) if w.hot[2] > 1 else 1
                cnt = max(int(w.hot[1]), cnt)
            else:
                lo, hi = math.log(w.hot[1]), math.log(w.hot[2])
                cnt = max(1, int(round(math.exp(lo + u * (hi - lo)) * n)))
            cnt = min(cnt, n)
            lo_s, hi_s = w.shift
            s = lo_s + float(torch.rand(1, generator=gh, dtype=torch.float64)) * (hi_s - lo_s)
            pages = torch.randperm(n, generator=gh)[:cnt]
            qg = q[b, h * g_grp:(h + 1) * g_grp].mean(0)
            qhat = qg / qg.norm()
            phys = bt_cpu[b, pages].to(torch.long).to(device)
            blk = k[phys, h].float() + (s * (1.0 if unit_shift else math.sqrt(d))) * qhat
            k[phys, h] = blk.to(torch.bfloat16)
            hot[(b, h)] = sorted(int(x) for x in pages)
    return Layer(k, v, q, hot)


@dataclass
class Steps:
    q: torch.Tensor       # fp32 [n, L, B, Hq, d]
    k_new: torch.Tensor   # bf16 [n, L, B, Hkv, d]
    v_new: torch.Tensor


def make_steps(w: Workload, layer_q, n: int, seed: int, device, sigma: float = 0.25) -> Steps:
    """Inputs of n consecutive decode steps: per-step queries (the layers'
    queries plus sigma * N(0, 1)) and the tokens each step appends."""
    L = len(layer_q)
    base = torch.stack(list(layer_q))  # [L, B, Hq, d]
    g = _gen(seed, 20, device=device)
    q = base.unsqueeze(0) + sigma * torch.randn((n,) + tuple(base.shape), generator=g,
                                                device=device, dtype=torch.float32)
    shape = (n, L, w.batch, w.num_kv_heads, w.head_dim)
    k_new = torch.randn(shape, generator=g, device=device, dtype=torch.bfloat16)
    v_new = torch.randn(shape, generator=g, device=device, dtype=torch.bfloat16)
    return Steps(q.contiguous(), k_new, v_new)
