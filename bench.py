#!/usr/bin/env python3
"""Decode-step benchmark: coverage-selected sparse attention over a paged KV cache.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl asp|reference]
                    [--config long128k] [--gamma 0.99] [--budget 0] [--seed 1]

--budget K > 0 keeps the top K pages per segment (the fixed-budget mode)
instead of the coverage rule at --gamma, in both arms.

One step = every layer of the workload through asp_coverage_select (score +
select kernels) and asp_sparse_decode, replayed from one CUDA graph, with all
inputs resident in HBM (64 GiB of K/V at 128k: far larger than L2, so no L2
flush is needed between steps). Prints one JSON line (rank 0).

Under torchrun each rank runs its own batch of requests (the path shards by
request with no collective); value = all ranks' steps / max-over-ranks time.

--impl reference times the fp64 CPU oracle (numpy, spawn pool over the host
cores) on a bounded sample of the same workload and scales it to steps/s.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode steps/s and selected-KV HBM GB/s (% of GB300 roofline) at 128k, γ=0.99"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ helpers
def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["asp", "reference"], default="asp")
    ap.add_argument("--config", default="long128k")
    ap.add_argument("--gamma", type=float, default=0.99)
    ap.add_argument("--budget", type=int, default=0,
                    help="keep the top BUDGET pages per segment instead of the coverage rule")
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-multistep", action="store_true")
    ap.add_argument("--no-diagnostics", action="store_true")
    ap.add_argument("--multistep-steps", type=int, default=8,
                    help="decode steps unrolled in the multi-step graph")
    ap.add_argument("--oracle-segments", type=int, default=0,
                    help="segments per oracle sample (default: host cores, at least 8)")
    return ap.parse_args(argv)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def max_over_ranks(x: float, dist, device=None) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


TRAFFIC_RECORD = os.path.join("profiles", "decode_kernel_traffic.json")


def source_digest(*names) -> str:
    """sha256[:16] over the named kernel sources (csrc/), in order."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "adaptive_sparse_paged_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def decode_traffic_per_page(cfg_name: str):
    """ncu DRAM bytes per selected (page, head) of the decode kernel from the
    committed profile record, if it was taken on the current kernel source
    (the record names the sources it hashed); else None."""
    try:
        with open(os.path.join(ROOT, TRAFFIC_RECORD)) as f:
            rec = json.load(f)
        if source_digest(*rec["sources"]) != rec["sources_sha256_16"]:
            return None
        return float(rec["dram_bytes_per_selected_page_head"])
    except (OSError, KeyError, ValueError, TypeError):
        return None


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.proc.stdout.readline()  # first sample: the sampler is running
        except (OSError, ValueError):
            self.proc = None

    def mark(self, which):
        if which == 0:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append(parts)
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i] == "Active"})
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((float(r[4]) for r in rows
                                    if r[4].replace(".", "").isdigit()), default=None)}


def workload_name(w, gamma, budget=0) -> str:
    """The workload both arms report in config.workload."""
    rule = f"budget{budget}" if budget > 0 else f"gamma{gamma}"
    return (f"{w.name}: B{w.batch} L{w.layers} Hq{w.num_q_heads} Hkv{w.num_kv_heads} "
            f"d{w.head_dim} P{w.page_size} T{w.seq_len or 'lognormal'} {rule}")


def bench_config(w, sh, gamma, budget) -> dict:
    """The config object, identical in both arms for the same arguments."""
    P, d, Hkv, L = w.page_size, w.head_dim, w.num_kv_heads, w.layers
    kv_gib = 2 * sh.num_phys_pages * Hkv * P * d * 2 * L / 2**30
    summ_gib = w.batch * Hkv * sh.max_pages * 4 * d * L / 2**30
    return {"workload": workload_name(w, gamma, budget), "gamma": gamma, "budget": budget,
            "l2": "inputs larger than L2 (K/V %.1f GiB, summaries %.2f GiB resident); no flush"
                  % (kv_gib, summ_gib)}


# ------------------------------------------------------------- oracle sample
def _oracle_worker(args):
    import numpy as np
    import oracle.asp_oracle as O
    qg, kbits, vbits, T, gamma, budget, scale = args
    kp = O.bf16_bits_to_f64(kbits)
    vp = O.bf16_bits_to_f64(vbits)
    r = O.decode_segment(qg, kp, vp, T, gamma, budget, scale)
    return np.asarray(r["ids"], dtype=np.int32), float(np.abs(r["o"]).sum())


def _pool_init():
    os.environ.setdefault("OMP_NUM_THREADS", "1")


def start_oracle_pool():
    n = os.cpu_count() or 1
    os.environ["OMP_NUM_THREADS"] = "1"
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    os.environ["MKL_NUM_THREADS"] = "1"
    ctx = mp.get_context("spawn")
    return ctx.Pool(n, initializer=_pool_init), n


def oracle_sample_tasks(w, sh, layer, nseg, gamma, budget, seed):
    """Seeded sample of (request, KV head) segments of one layer, as oracle inputs
    (every segment of the layer when nseg covers them all)."""
    import numpy as np
    import torch
    rng = np.random.default_rng(seed)
    segs = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    if nseg >= len(segs):
        pick = segs
    else:
        pick = [segs[i] for i in rng.choice(len(segs), nseg, replace=False)]
    g = w.num_q_heads // w.num_kv_heads
    q = layer.q.double().cpu().numpy()
    tasks = []
    for b, h in pick:
        T = int(sh.seq_lens[b])
        n = sh.num_pages[b]
        idx = sh.block_table[b, :n].long()
        kb = layer.k_cache[idx, h].contiguous().view(torch.int16).cpu().numpy()
        vb = layer.v_cache[idx, h].contiguous().view(torch.int16).cpu().numpy()
        tasks.append((q[b, h * g:(h + 1) * g], kb, vb, T, float(np.float32(gamma)), budget,
                      1.0 / math.sqrt(w.head_dim)))
    return tasks, pick


def time_oracle(pool, tasks):
    """Seconds for the oracle over `tasks`, and its results."""
    t0 = time.perf_counter()
    res = pool.map(_oracle_worker, tasks, chunksize=1)
    return time.perf_counter() - t0, res


# ------------------------------------------------------------------- asp arm
def run_asp(args):
    world, rank, local = dist_env()
    pool = cores = None
    if rank == 0 and not args.no_cpu_baseline:
        pool, cores = start_oracle_pool()  # spawn, before any CUDA call
    import numpy as np
    import torch

    from adaptive_sparse_paged_gb300 import binding as B
    from adaptive_sparse_paged_gb300 import synth
    from adaptive_sparse_paged_gb300.step import DecodeLoop, DecodeStep

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = dist_init(world, "nccl")
    w = synth.CONFIGS[args.config]
    seed = args.seed + 1000 * rank
    t_gen = time.perf_counter()
    sh = synth.make_shared(w, seed, dev)
    layers, kvs = [], []
    for l in range(w.layers):
        lay = synth.make_layer(w, sh, seed, l, dev)
        summ = B.new_summaries(lay.k_cache, sh.block_table)
        kv = B.PagedKV(lay.k_cache, lay.v_cache, summ, sh.block_table, sh.seq_lens, w.num_q_heads)
        layers.append(lay)
        kvs.append(kv)
    q_all = torch.stack([lay.q for lay in layers])
    ws0 = B.new_workspace(kvs[0])
    for kv in kvs:
        B.asp_page_summarize(kv, B.ASP_SUMMARIZE_BULK, None, None, ws0)
    assert B.asp_get_device_error(ws0) == 0
    torch.cuda.synchronize()
    gen_s = time.perf_counter() - t_gen

    step = DecodeStep(kvs, q_all, gamma=args.gamma, budget=args.budget)
    step.capture()
    stream = torch.cuda.current_stream()

    def timed_graph(st, K, W):
        for _ in range(W):
            st.replay()
        torch.cuda.synchronize()
        barrier(dist)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            st.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        return e0.elapsed_time(e1) / 1e3

    clocks = ClockSampler(dev.index)
    clocks.start()
    clocks.mark(0)
    t_loc = timed_graph(step, args.steps, max(3, args.warmup))
    clocks.mark(1)
    clk = clocks.stop()
    t_max = max_over_ranks(t_loc, dist, dev)
    assert B.asp_get_device_error(step.ws) == 0

    # selection statistics of this step (same every replay)
    lens = step.lens.cpu().numpy().astype(np.int64)     # [L, B, Hkv]
    n_pages = np.array(sh.num_pages, dtype=np.int64)     # [B]
    sel_pages = int(lens.sum())
    all_pages = int(n_pages.sum()) * w.num_kv_heads * w.layers
    P, d, Hq, Hkv, Bt, L = w.page_size, w.head_dim, w.num_q_heads, w.num_kv_heads, w.batch, w.layers
    page_bytes = 2 * P * d * 2                        # K + V of one (page, head)
    q_bytes = Bt * Hq * d * 4
    out_bytes = Bt * Hq * d * 4 + Bt * Hq * 4
    dec_bytes = [int(lens[l].sum()) * (page_bytes + 8) + q_bytes + Bt * Hkv * 4 + out_bytes
                 for l in range(L)]                  # pages + list/table entries + q + lens + out
    score_bytes = int(n_pages.sum()) * Hkv * (4 * d + 4) + q_bytes  # summaries + scores + q
    select_bytes = [int(n_pages.sum()) * Hkv * 4 + int(lens[l].sum()) * 4 + Bt * Hkv * 4
                    for l in range(L)]                # scores + lists + lens
    step_bytes = sum(dec_bytes) + L * score_bytes + sum(select_bytes)

    # per-kernel durations: eager pass with events on the launching stream
    K_e = max(3, min(args.steps, 20))
    for _ in range(2):
        step.run()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(L * K_e)]
    for k in range(K_e):
        for l in range(L):
            step.run_layer(l, stream, events=evs[k * L + l])
    torch.cuda.synchronize()
    sel_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(L * K_e)]
    dec_ms = [evs[i][1].elapsed_time(evs[i][2]) for i in range(L * K_e)]
    dec_avg_s = float(np.mean(dec_ms)) / 1e3
    sel_avg_s = float(np.mean(sel_ms)) / 1e3
    dec_bytes_avg = float(np.mean(dec_bytes))
    peak, peak_kind = measured_hbm_peak()
    dec_gbs = dec_bytes_avg / dec_avg_s / 1e9
    tpp = decode_traffic_per_page(args.config)
    traffic = None if tpp is None else tpp * float(lens.sum()) / L

    # dense comparison: the same kernels at gamma = 1
    dense = None
    if not args.no_dense:
        dstep = DecodeStep(kvs, q_all, gamma=1.0)
        dstep.capture()
        Kd = max(3, args.steps // 4)
        td = max_over_ranks(timed_graph(dstep, Kd, 3), dist, dev)
        dense = {"steps_per_s": world * Kd / td, "ms_per_step": 1e3 * td / Kd}
        del dstep

    # end to end: host q in, host out/lse back, every step
    q_host = q_all.cpu().pin_memory()
    out_host = torch.empty(step.out.shape, dtype=torch.float32).pin_memory()
    lse_host = torch.empty(step.lse.shape, dtype=torch.float32).pin_memory()
    K2 = args.steps
    for _ in range(3):
        step.q.copy_(q_host, non_blocking=True)
        step.replay()
        out_host.copy_(step.out, non_blocking=True)
        lse_host.copy_(step.lse, non_blocking=True)
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K2):
        step.q.copy_(q_host, non_blocking=True)
        step.replay()
        out_host.copy_(step.out, non_blocking=True)
        lse_host.copy_(step.lse, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3, dist, dev)
    e2e = {"value": world * K2 / t_e2e, "unit": "steps/s",
           "h2d_bytes_per_step": int(q_host.numel() * 4),
           "d2h_bytes_per_step": int(out_host.numel() * 4 + lse_host.numel() * 4)}

    # the same step at the pages' own sparsity: the top 30% of pages by score
    # (budget mode), so the fixed per-layer costs weigh as they would there
    at30 = None
    if not args.no_dense:
        k30 = int(math.ceil(0.3 * float(n_pages.max())))
        bstep = DecodeStep(kvs, q_all, gamma=args.gamma, budget=k30)
        bstep.capture()
        Kb = max(3, args.steps // 4)
        tb = max_over_ranks(timed_graph(bstep, Kb, 3), dist, dev)
        blens = bstep.lens.cpu().numpy().astype(np.int64)
        b_dec = sum(int(blens[l].sum()) * (page_bytes + 8) + q_bytes + Bt * Hkv * 4 + out_bytes
                    for l in range(L))
        b_sel = sum(int(n_pages.sum()) * Hkv * 4 + int(blens[l].sum()) * 4 + Bt * Hkv * 4
                    for l in range(L))
        b_bytes = b_dec + L * score_bytes + b_sel
        at30 = {"budget_pages": k30, "pages_read_frac": round(float(blens.sum()) / all_pages, 4),
                "steps_per_s": round(world * Kb / tb, 3), "ms_per_step": round(1e3 * tb / Kb, 4),
                "hbm_frac_of_measured": round(b_bytes / (tb / Kb) / 1e9 / peak, 4)}
        del bstep

    # Sensitivity to the generator's reading: the pages read when hot keys
    # move by shift * q_hat (unit norm, the configs' literal wording) instead
    # of shift * sqrt(d) * q_hat, on the first two layers of the same draws.
    literal = None
    if not args.no_diagnostics:
        nl = min(2, w.layers)
        lit_kvs, lit_q = [], []
        for l in range(nl):
            lay = synth.make_layer(w, sh, seed, l, dev, unit_shift=True)
            summ = B.new_summaries(lay.k_cache, sh.block_table)
            kv = B.PagedKV(lay.k_cache, lay.v_cache, summ, sh.block_table, sh.seq_lens,
                           w.num_q_heads)
            B.asp_page_summarize(kv, B.ASP_SUMMARIZE_BULK, None, None, ws0)
            lit_kvs.append(kv)
            lit_q.append(lay.q)
        lit_lens = torch.zeros((nl, w.batch, w.num_kv_heads), dtype=torch.int32, device=dev)
        lit_lists = torch.zeros((w.batch, w.num_kv_heads, sh.max_pages), dtype=torch.int32,
                                device=dev)
        for l in range(nl):
            B.asp_coverage_select(lit_kvs[l], lit_q[l], args.gamma, args.budget, lit_lists,
                                  lit_lens[l], ws0)
        assert B.asp_get_device_error(ws0) == 0
        lit_pages = float(lit_lens.sum())
        literal = {"shift": "shift * q_hat (unit norm)", "layers": nl,
                   "pages_read_frac": round(lit_pages / (float(n_pages.sum()) * Hkv * nl), 4),
                   "pages_read_frac_same_layers_sqrt_d_shift":
                       round(float(lens[:nl].sum()) / (float(n_pages.sum()) * Hkv * nl), 4)}
        del lit_kvs, lit_q, lit_lens, lit_lists

    # required page fractions per gamma, and a fixed budget of equal bytes
    diag = None
    if not args.no_diagnostics:
        from adaptive_sparse_paged_gb300 import diagnostics as Dg
        diag = Dg.budget_diagnostics(kvs, q_all, ref_gamma=args.gamma)

    # Several decode steps in one graph: step i appends one token per request
    # (the last n tokens of the context are replayed as n appends) and runs
    # every layer with its own queries, so the page lists vary from step to step.
    multi = None
    if not args.no_multistep and args.multistep_steps > 0:
        n_ms = args.multistep_steps
        full_lens = sh.seq_lens.clone()
        t0 = (full_lens - n_ms).clamp(min=0)
        sh.seq_lens.copy_(t0)
        for kv in kvs:  # summaries of the first T0 tokens
            B.asp_page_summarize(kv, B.ASP_SUMMARIZE_BULK, None, None, ws0)
        steps_in = synth.make_steps(w, [lay.q for lay in layers], n_ms, seed, dev)
        # the append fused into the score pass
        loop = DecodeLoop(kvs, t0.clone(), steps_in.q, steps_in.k_new, steps_in.v_new,
                          gamma=args.gamma, budget=args.budget)
        loop.capture()
        loop.replay()  # the first run: fresh steps
        torch.cuda.synchronize()
        assert B.asp_get_device_error(loop.ws) == 0
        lens_ms = loop.lens.cpu().numpy().astype(np.int64)  # [n, L, B, Hkv]
        Km = max(3, args.steps // 20)
        t_ms = max_over_ranks(timed_graph(loop, Km, 3), dist, dev)
        launches_ms = loop.launches
        del loop
        # the same loop with the append as its own kernel, for comparison
        sep = DecodeLoop(kvs, t0.clone(), steps_in.q, steps_in.k_new, steps_in.v_new,
                         gamma=args.gamma, budget=args.budget, fused_append=False)
        sep.capture()
        t_sep = max_over_ranks(timed_graph(sep, Km, 3), dist, dev)
        del sep
        sh.seq_lens.copy_(full_lens)  # the appended tokens are now the context's last ones
        torch.cuda.synchronize()
        tpot = t_ms / (Km * n_ms)
        frac = [round(float(lens_ms[i].sum()) / all_pages, 4) for i in range(n_ms)]
        multi = {"steps_in_graph": n_ms, "append": "fused into the score pass",
                 "tpot_ms": round(1e3 * tpot, 4), "steps_per_s": round(world / tpot, 3),
                 "tpot_ms_append_separate": round(1e3 * t_sep / (Km * n_ms), 4),
                 "replays": Km, "pages_read_frac_by_step": frac,
                 "launches_per_graph": launches_ms,
                 "query_change": "per step: layer queries + 0.25 * N(0, 1)"}
        del steps_in

    cpu = list_parity = None
    if pool is not None:
        # two whole layers (every segment of layers 0 and 1), scaled to all L layers
        nl = min(2, w.layers)
        seg_layer = w.batch * w.num_kv_heads
        tasks, where = [], []
        for l in range(nl):
            tk, pick = oracle_sample_tasks(w, sh, layers[l], seg_layer, args.gamma, args.budget,
                                           args.seed)
            tasks += tk
            where += [(l, b, h) for (b, h) in pick]
        time_oracle(pool, tasks[:min(len(tasks), cores)])  # warm the workers
        t_cpu, res = time_oracle(pool, tasks)
        segs_per_step = seg_layer * w.layers
        step_s = t_cpu * segs_per_step / len(tasks)
        cpu = {"value": 1.0 / step_s, "unit": "steps/s", "cores": cores, "kind": "oracle",
               "sample": f"layers 0-{nl - 1} in full ({len(tasks)} of {segs_per_step} "
                         f"(request, KV head, layer) segments, full context each), fp64 numpy, "
                         f"{cores} spawn workers x 1 thread, inputs pickled to the workers; "
                         f"{t_cpu:.1f} s, extrapolated x{w.layers / nl:g} to a full step"}
        pool.close()
        # the step's page lists on the same segments against the oracle's (one
        # more replay: the multi-step graph above appended tokens to the caches)
        step.replay()
        torch.cuda.synchronize()
        lists_c = step.lists.cpu().numpy()
        lens_c = step.lens.cpu().numpy()
        same = 0
        for (l, b, h), (ids, _) in zip(where, res):
            k = int(lens_c[l, b, h])
            same += int(np.array_equal(np.sort(lists_c[l, b, h, :k]), ids))
        list_parity = {"segments": len(res), "identical_to_oracle": same,
                       "different": len(res) - same,
                       "sample": "the cpu_baseline segments, lists of the step's graph"}

    if rank == 0:
        steps_per_s = world * args.steps / t_max
        ms = 1e3 * t_max / args.steps
        line = {
            "metric": METRIC,
            "value": round(steps_per_s, 3),
            "unit": "steps/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": max(3, args.warmup),
            "ms_per_step": round(ms, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": bench_config(w, sh, args.gamma, args.budget),
            "step": "all layers replayed from one CUDA graph",
            "parallelism": f"replica per GPU x{world} (requests shard, no collective)",
            "setup_s": round(gen_s, 1),
            "layer_us": round(1e3 * ms / L, 2),
            "selected_kv_gbs": round(world * step_bytes * args.steps / t_max / 1e9, 1),
            "hbm_frac_of_measured": round(step_bytes / (ms / 1e3) / 1e9 / peak, 4),
            "hbm_frac_of_nominal_8tbs": round(step_bytes / (ms / 1e3) / 1e12 / 8.0, 4),
            "pages_read_frac": round(sel_pages / all_pages, 4),
            "selected_page_heads_per_step": sel_pages,
            "bytes_per_step": step_bytes,
            "dense_gamma1": dense,
            "top30_budget": at30,
            "multi_step": multi,
            "budget_diagnostics": diag,
            "pages_read_literal_unit_shift": literal,
            "list_parity": list_parity,
            "kernels_ms": {"select_avg": round(sel_avg_s * 1e3, 4),
                           "decode_avg": round(dec_avg_s * 1e3, 4)},
            "roofline": {
                "kernel": "decode_kernel (asp_sparse_decode)",
                "bound": "hbm",
                "achieved": round(dec_gbs, 1),
                "peak": peak,
                "peak_kind": peak_kind,
                "unit": "GB/s",
                "frac": round(dec_gbs / peak, 4),
                "frac_of_nominal_8tbs": round(dec_gbs / 8000.0, 4),
                "traffic": None if traffic is None else round(traffic),
                "algorithmic_bytes_per_launch": round(dec_bytes_avg),
            },
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps * step.launches_per_step,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return  # the oracle arm runs once, on rank 0's host
    pool, cores = start_oracle_pool()
    import torch

    from adaptive_sparse_paged_gb300 import synth
    w = synth.CONFIGS[args.config]
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    sh = synth.make_shared(w, args.seed, dev)
    lay = synth.make_layer(w, sh, args.seed, 0, dev)
    nseg = args.oracle_segments or max(8, cores)
    segs_per_step = w.batch * w.num_kv_heads * w.layers
    tasks, _ = oracle_sample_tasks(w, sh, lay, nseg, args.gamma, args.budget, args.seed)
    del lay
    for _ in range(max(0, min(args.warmup, 1))):
        time_oracle(pool, tasks[:min(len(tasks), cores)])
    t = 0.0
    for _ in range(args.steps):
        t += time_oracle(pool, tasks)[0]
    pool.close()
    # Each timed step is the oracle over a sample of one layer's segments:
    # steps and ms_per_step describe that timed work; value, in the metric's
    # full decode steps per second, scales it to every segment of every layer.
    scale = segs_per_step / len(tasks)
    value = args.steps / (t * scale)
    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": bench_config(w, sh, args.gamma, args.budget),
        "step": f"fp64 oracle on the host cores over {len(tasks)} of the {segs_per_step} "
                f"segments of a full step",
        "extrapolation": {"segments_timed_per_step": len(tasks),
                          "segments_per_full_step": segs_per_step, "factor": scale,
                          "ms_per_full_step": 1e3 * t * scale / args.steps,
                          "value_is": "full steps per second = steps / (timed seconds x factor)"},
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {len(tasks)} of {segs_per_step} segments of "
                                   f"layer 0 through the fp64 oracle, scaled to a full step"},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_asp(args)


if __name__ == "__main__":
    main()
