"""One decode step over L layers, optionally captured into a single CUDA graph.

Per layer: asp_coverage_select (score + select kernels) then asp_sparse_decode
(self-planning attention), and optionally asp_page_summarize in APPEND mode
first. The layers share one workspace; stream order serialises them. Nothing
returns to the host between layers, which is what lets the whole step live
inside one CUDA graph (MOIRA abstract, page "Adaptive DHiSparse: Speculative
Decoding over a Load-Adaptive KV Hierarchy").
"""

from __future__ import annotations

import math

import torch

from . import binding as B


class DecodeStep:
    def __init__(self, kvs, q, gamma: float, budget: int = 0, sm_scale: float | None = None,
                 append=None):
        """kvs: list of PagedKV (one per layer, same shape); q: fp32 [L, B, Hq, d].

        append: optional (k_new, v_new), bf16 [L, B, Hkv, d] each, written with
        APPEND before each layer's selection.
        """
        self.kvs = list(kvs)
        kv0 = self.kvs[0]
        L = len(self.kvs)
        dev = kv0.device
        assert q.shape == (L, kv0.batch, kv0.num_q_heads, kv0.head_dim)
        self.q = q
        self.gamma, self.budget = float(gamma), int(budget)
        self.sm_scale = sm_scale if sm_scale is not None else 1.0 / math.sqrt(kv0.head_dim)
        self.append = append
        self.lists = torch.zeros((L, kv0.batch, kv0.num_kv_heads, kv0.max_pages), dtype=torch.int32,
                                 device=dev)
        self.lens = torch.zeros((L, kv0.batch, kv0.num_kv_heads), dtype=torch.int32, device=dev)
        self.out = torch.zeros((L, kv0.batch, kv0.num_q_heads, kv0.head_dim), dtype=torch.float32,
                               device=dev)
        self.lse = torch.zeros((L, kv0.batch, kv0.num_q_heads), dtype=torch.float32, device=dev)
        self.ws = B.new_workspace(kv0)
        self.graph = None

    # kernel launches of one step, per layer: score + select (select alone at
    # gamma = 1), decode + merge, and the append kernel when enabled
    @property
    def launches_per_step(self) -> int:
        per = 2 if (self.budget > 0 or self.gamma < 1.0) else 1
        return len(self.kvs) * (per + 2 + (1 if self.append is not None else 0))

    def run_layer(self, l: int, stream=None, events=None):
        kv = self.kvs[l]
        if self.append is not None:
            B.asp_page_summarize(kv, B.ASP_SUMMARIZE_APPEND, self.append[0][l], self.append[1][l],
                                 self.ws, stream)
        if events is not None:
            events[0].record(stream)
        B.asp_coverage_select(kv, self.q[l], self.gamma, self.budget, self.lists[l],
                              self.lens[l], self.ws, stream)
        if events is not None:
            events[1].record(stream)
        B.asp_sparse_decode(kv, self.q[l], self.lists[l], self.lens[l], self.sm_scale,
                            self.out[l], self.lse[l], self.ws, stream)
        if events is not None:
            events[2].record(stream)

    def run(self, stream=None):
        for l in range(len(self.kvs)):
            self.run_layer(l, stream)

    def capture(self):
        """Captures one full step into a CUDA graph (warm up first)."""
        s = torch.cuda.Stream(device=self.kvs[0].device)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.run()  # warm-up outside capture: sets kernel attributes, loads modules
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run()
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()
