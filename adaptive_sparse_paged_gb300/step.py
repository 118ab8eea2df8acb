"""One decode step over L layers, optionally captured into a single CUDA graph.

Per layer: asp_coverage_select (one cluster kernel, or score + select kernels) then asp_sparse_decode
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


def _check_shape(name, t, shape):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


class DecodeStep:
    def __init__(self, kvs, q, gamma: float, budget: int = 0, sm_scale: float | None = None,
                 append=None):
        """kvs: list of PagedKV (one per layer, same shape); q: fp32 [L, B, Hq, d].

        append: optional (k_new, v_new), bf16 [L, B, Hkv, d] each, written with
        APPEND before each layer's selection.
        """
        self.kvs = list(kvs)
        if not self.kvs:
            raise ValueError("kvs must hold at least one layer")
        kv0 = self.kvs[0]
        L = len(self.kvs)
        dev = kv0.device
        _check_shape("q", q, (L, kv0.batch, kv0.num_q_heads, kv0.head_dim))
        if append is not None:
            shp = (L, kv0.batch, kv0.num_kv_heads, kv0.head_dim)
            _check_shape("append[0]", append[0], shp)
            _check_shape("append[1]", append[1], shp)
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

    # kernel launches of one step, per layer: the selection's (one cluster
    # kernel, or a score pass and a select kernel; select alone at gamma = 1),
    # the decode, and the append kernel when enabled
    @property
    def launches_per_step(self) -> int:
        per, _ = B.asp_select_plan(self.kvs[0], self.gamma, self.budget)
        return len(self.kvs) * (per + 1 + (1 if self.append is not None else 0))

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


class DecodeLoop:
    """n consecutive decode steps over L layers, captured into one CUDA graph.

    Step i appends one token per request at position T0_b + i (APPEND: its K
    and V rows, folded into its page's summary), then runs every layer's
    coverage selection and attention with that step's queries; the page lists
    change from step to step as the queries and the newest pages do (MOIRA
    abstract: lists per request, layer, KV head and step). Each step has its own
    length buffer (T0 + i + 1) and its own outputs, so the steps are unrolled
    in the graph rather than indexed by a device counter.

    The block tables must already map the pages of T0 + n tokens, and the
    summaries must describe the first T0 tokens when the loop first runs.
    Replaying the graph re-times the same work: the appends are idempotent,
    but a replayed step's last-page summary then already holds the later
    steps' tokens, so only the first run's lists are those of fresh steps.
    """

    def __init__(self, kvs, seq_lens0, q, k_new, v_new, gamma: float, budget: int = 0,
                 sm_scale: float | None = None, fused_append: bool = True):
        """kvs: PagedKV per layer; seq_lens0: int32 [B] (T0); q: fp32 [n, L, B, Hq, d];
        k_new, v_new: bf16 [n, L, B, Hkv, d]. fused_append: append inside the score
        pass (asp_coverage_select_append) instead of a separate APPEND launch."""
        if not kvs:
            raise ValueError("kvs must hold at least one layer")
        kv0 = kvs[0]
        n, L = q.shape[0], len(kvs)
        _check_shape("q", q, (n, L, kv0.batch, kv0.num_q_heads, kv0.head_dim))
        _check_shape("k_new", k_new, (n, L, kv0.batch, kv0.num_kv_heads, kv0.head_dim))
        _check_shape("v_new", v_new, tuple(k_new.shape))
        _check_shape("seq_lens0", seq_lens0, (kv0.batch,))
        dev = kv0.device
        self.n, self.L = n, L
        self.q, self.k_new, self.v_new = q, k_new, v_new
        self.gamma, self.budget = float(gamma), int(budget)
        self.sm_scale = sm_scale if sm_scale is not None else 1.0 / math.sqrt(kv0.head_dim)
        self.seq_lens = [(seq_lens0 + (i + 1)).to(torch.int32).contiguous() for i in range(n)]
        self.kvs = [[B.PagedKV(kv.k_cache, kv.v_cache, kv.summaries, kv.block_table,
                               self.seq_lens[i], kv.num_q_heads) for kv in kvs] for i in range(n)]
        self.lists = torch.zeros((n, L, kv0.batch, kv0.num_kv_heads, kv0.max_pages),
                                 dtype=torch.int32, device=dev)
        self.lens = torch.zeros((n, L, kv0.batch, kv0.num_kv_heads), dtype=torch.int32, device=dev)
        self.out = torch.zeros((n, L, kv0.batch, kv0.num_q_heads, kv0.head_dim),
                               dtype=torch.float32, device=dev)
        self.lse = torch.zeros((n, L, kv0.batch, kv0.num_q_heads), dtype=torch.float32,
                               device=dev)
        self.fused_append = bool(fused_append)
        self.ws = B.new_workspace(kv0)
        self.graph = None

    @property
    def launches(self) -> int:
        """Kernel launches of the whole loop: [append,] the selection's, the decode."""
        per, _ = B.asp_select_plan(self.kvs[0][0], self.gamma, self.budget,
                                   append=self.fused_append)
        return self.n * self.L * ((0 if self.fused_append else 1) + per + 1)

    def run(self, stream=None):
        for i in range(self.n):
            for l in range(self.L):
                kv = self.kvs[i][l]
                if self.fused_append:
                    B.asp_coverage_select_append(kv, self.k_new[i, l], self.v_new[i, l],
                                                 self.q[i, l], self.gamma, self.budget,
                                                 self.lists[i, l], self.lens[i, l], self.ws,
                                                 stream)
                else:
                    B.asp_page_summarize(kv, B.ASP_SUMMARIZE_APPEND, self.k_new[i, l],
                                         self.v_new[i, l], self.ws, stream)
                    B.asp_coverage_select(kv, self.q[i, l], self.gamma, self.budget,
                                          self.lists[i, l], self.lens[i, l], self.ws, stream)
                B.asp_sparse_decode(kv, self.q[i, l], self.lists[i, l], self.lens[i, l],
                                    self.sm_scale, self.out[i, l], self.lse[i, l], self.ws,
                                    stream)

    def capture(self):
        """Captures the loop into one CUDA graph. The capture itself launches
        nothing, so the first replay is the loop's first (fresh) run."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run()
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()
