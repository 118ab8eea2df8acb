"""Per-layer timeline of a captured decode step, from %globaltimer stamps.

A profiling tool, not part of the library's path: it copies the package to a
scratch directory, adds per-CTA %globaltimer stamps to the cluster selection
kernel and the decode kernel of the copy, builds it, replays the DecodeStep
graph of a synthetic workload once more after warm-up, and prints when each
phase begins and ends inside the graph, relative to the first selection CTA
of each layer (median over the middle layers). The library itself is never
modified and never loads the copy.

    python -m adaptive_sparse_paged_gb300.timeline --config long128k

Stamps are written by thread 0 of each CTA into a device array indexed by
launch (a per-kernel arrival counter divided by the grid size) and CTA; each
costs one global store. The cluster selection path is the one stamped: a
shape that takes the two-kernel path reports no selection phases.
"""

from __future__ import annotations

import argparse
import os
import shutil
import sys
import tempfile

PKG = "adaptive_sparse_paged_gb300"
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

SEL_SLOTS = ("start", "waited", "streamed", "barrier 1", "barrier 2", "barrier 3", "end", "cutoff", "candidates")
DEC_SLOTS = ("start", "waited", "planned", "first data", "streamed", "arrived", "merged", "smid",
             "lengths loaded", "prefix done")
N_LAUNCH, N_CTA = 64, 160  # launches kept (ring) and CTAs per launch recorded


def _decl(tag: str, n: int) -> str:
    return (f"__device__ unsigned int g_tl_arr_{tag};\n"
            f"__device__ unsigned long long g_tl_{tag}[{N_LAUNCH} * {N_CTA} * {n}];\n")


def _reader(tag: str, n: int) -> str:
    return f'''
extern "C" int asp_timeline_read_{tag}(void* dst) {{
  return (int)cudaMemcpyFromSymbol(dst, asp::g_tl_{tag}, sizeof(unsigned long long) * {N_LAUNCH} * {N_CTA} * {n});
}}
extern "C" int asp_timeline_reset_{tag}() {{
  static unsigned long long zeros[{N_LAUNCH} * {N_CTA} * {n}];
  unsigned int z = 0;
  cudaError_t e = cudaMemcpyToSymbol(asp::g_tl_{tag}, zeros, sizeof(zeros));
  if (e != cudaSuccess) return (int)e;
  return (int)cudaMemcpyToSymbol(asp::g_tl_arr_{tag}, &z, sizeof(z));
}}
'''


def _stamp(tag: str, n: int, slot: int, cond: str = "threadIdx.x == 0", value: str = "globaltimer_ns()") -> str:
    return (f"if ({cond}) g_tl_{tag}[((tl_L % {N_LAUNCH}) * {N_CTA} + blockIdx.x) * {n} + {slot}] = {value};")


def _launch_index(tag: str) -> str:
    return (f"unsigned tl_L = 0;\n  if (threadIdx.x == 0) tl_L = atomicAdd(&g_tl_arr_{tag}, 1u) / gridDim.x;\n  ")


def patches():
    """(file, [(anchor, replacement)], appended text) for the stamped copy."""
    ns = len(SEL_SLOTS)
    sel = [
        ("namespace asp {\nnamespace {\n", "namespace asp {\n" + _decl("sel", ns) + "namespace {\n"),
        ("  const int rank = (int)cluster.block_rank();\n",
         "  const int rank = (int)cluster.block_rank();\n  " + _launch_index("sel") + _stamp("sel", ns, 0) + "\n"),
        ("  pdl_wait_predecessor();\n\n  const int T = clamp_seq_len",
         "  pdl_wait_predecessor();\n  " + _stamp("sel", ns, 1) + "\n\n  const int T = clamp_seq_len"),
        ("  __syncthreads();  // every score of this CTA is in shared memory; the ring is free\n",
         "  __syncthreads();  // every score of this CTA is in shared memory; the ring is free\n  "
         + _stamp("sel", ns, 2) + "\n"),
        ("  cluster.sync();  // barrier 1\n", "  cluster.sync();  // barrier 1\n  " + _stamp("sel", ns, 3) + "\n"),
        ("  cluster.sync();  // barrier 2: every histogram of the cluster is complete\n",
         "  cluster.sync();  // barrier 2: every histogram of the cluster is complete\n  "
         + _stamp("sel", ns, 4) + "\n"),
        ("  cluster.sync();  // barrier 3: every CTA holds every candidate\n",
         "  cluster.sync();  // barrier 3: every CTA holds every candidate\n  " + _stamp("sel", ns, 5) + "\n"),
        ("  // ------------------------------------- 7. kept ids, ascending, per CTA\n",
         "  " + _stamp("sel", ns, 7) + "\n  " + _stamp("sel", ns, 8, value="1ull + nc")
         + "\n  // ------------------------------------- 7. kept ids, ascending, per CTA\n"),
        ("      }\n    }\n  }\n}\n\n// Pieces per warp fetched",
         "      }\n    }\n  }\n  __syncthreads();\n  " + _stamp("sel", ns, 6) + "\n}\n\n// Pieces per warp fetched"),
    ]
    nd = len(DEC_SLOTS)
    smid = ("if (threadIdx.x == 0) { unsigned r_; asm(\"mov.u32 %0, %%smid;\" : \"=r\"(r_)); "
            f"g_tl_dec[((tl_L % {N_LAUNCH}) * {N_CTA} + blockIdx.x) * {nd} + 7] = 1ull + r_; }}")
    dec = [
        ("namespace asp {\nnamespace {\n", "namespace asp {\n" + _decl("dec", nd) + "namespace {\n"),
        ("  const int G = gridDim.x, cta = blockIdx.x;\n",
         "  const int G = gridDim.x, cta = blockIdx.x;\n  " + _launch_index("dec") + _stamp("dec", nd, 0) + "\n"),
        ("  pdl_launch_dependents();\n  pdl_wait_predecessor();\n  // ---- self-plan",
         "  pdl_launch_dependents();\n  pdl_wait_predecessor();\n  " + _stamp("dec", nd, 1) + "\n  // ---- self-plan"),
        ("  __syncthreads();  // the weights are done with: the ring is free for copies\n",
         "  __syncthreads();  // the weights are done with: the ring is free for copies\n  "
         + _stamp("dec", nd, 2) + "\n"),
        ("        if (__all_sync(kFull, got)) {\n          waited = nc + 1;",
         "        if (__all_sync(kFull, got)) {\n          if (nc == 0) { "
         + _stamp("dec", nd, 3, "warp == 0 && lane == 0") + " }\n          waited = nc + 1;"),
        ("  if (bad) report(p.err, bad);\n", "  if (bad) report(p.err, bad);\n  " + _stamp("dec", nd, 8) + "\n"),
        ("  // Weighted split: page j of segment s weighs 1, plus X when j = prefix[s];\n",
         "  " + _stamp("dec", nd, 9) + "\n  // Weighted split: page j of segment s weighs 1, plus X when j = prefix[s];\n"),
        ("  // never leave the CTA with copies in flight",
         "  " + _stamp("dec", nd, 4) + "\n  " + smid + "\n  // never leave the CTA with copies in flight"),
        ("    flags[1] = np_b > 1 && ob == np_b - 1 ? 1 : 0;\n",
         "    flags[1] = np_b > 1 && ob == np_b - 1 ? 1 : 0;\n    " + _stamp("dec", nd, 5, "true") + "\n"),
        ("    if (tid == 0) p.arrivals[ms] = 0;\n  }\n}\n",
         "    if (tid == 0) p.arrivals[ms] = 0;\n    __syncthreads();\n    " + _stamp("dec", nd, 6) + "\n  }\n}\n"),
    ]
    return [("select_cluster.cu", sel, _reader("sel", ns)), ("decode.cu", dec, _reader("dec", nd))]


def make_copy(dest: str) -> str:
    """Copies the package and its header to dest and stamps the copy; returns dest."""
    for d in (PKG, "include"):
        shutil.copytree(os.path.join(ROOT, d), os.path.join(dest, d),
                        ignore=shutil.ignore_patterns("*.so", "*.o", "_build*", "__pycache__"))
    csrc = os.path.join(dest, PKG, "csrc")
    for name, reps, tail in patches():
        path = os.path.join(csrc, name)
        with open(path) as f:
            s = f.read()
        for anchor, new in reps:
            if s.count(anchor) != 1:
                raise RuntimeError(f"{name}: stamp anchor found {s.count(anchor)} times: {anchor[:60]!r}")
            s = s.replace(anchor, new)
        with open(path, "w") as f:
            f.write(s + tail)
    return dest


def _median_rows(sel, dec, layers):
    import numpy as np

    def col(a, i):
        x = a[:, i]
        return x[x > 0].astype(np.float64)

    rows, counts = {}, {}

    def add(k, v):  # a time in ns
        rows.setdefault(k, []).append(v)

    def add_count(k, v):  # a count or a fraction
        counts.setdefault(k, []).append(v)
    for l in range(min(4, layers // 4), layers - min(4, layers // 4) - 1):
        s, d, s_next = sel[l], dec[l], sel[l + 1]
        if not len(col(s, 0)):
            continue
        t0 = col(s, 0).min()
        w = np.median(col(s, 1))
        for i, name in enumerate(SEL_SLOTS[:8]):
            c = col(s, i)
            if len(c):
                add(f"select {name} (median CTA)", np.median(c) - t0)
        c = col(s, 8)
        if len(c):
            add_count("select CTAs with > 32 candidates (fraction)", float(np.mean(c - 1 > 32)))
            add_count("select candidates per cluster (median)", float(np.median(c - 1)))
        if len(col(s, 6)):
            add("select end (last CTA)", col(s, 6).max() - t0)
        for i in (0, 1, 8, 9, 2, 3, 4):
            c = col(d, i)
            if len(c):
                add(f"decode {DEC_SLOTS[i]} (median CTA)", np.median(c) - t0)
        if len(col(d, 4)):
            add("decode streamed (last CTA)", col(d, 4).max() - t0)
        if len(col(d, 6)):
            add("decode merged (last merge)", col(d, 6).max() - t0)
        if len(col(s_next, 1)):
            add("next select waited (median CTA)", np.median(col(s_next, 1)) - t0)
            add("layer period (select waited to next)", np.median(col(s_next, 1)) - w)
    out = {k: float(np.median(v)) / 1e3 for k, v in rows.items()}
    out.update({k: float(np.median(v)) for k, v in counts.items()})
    return out


def _sm_consistency(dec, layers):
    """Stream-end lateness (vs the layer median) by SM and by CTA index."""
    import numpy as np
    from collections import defaultdict
    by_sm, by_cta = defaultdict(list), defaultdict(list)
    for l in range(layers):
        d = dec[l]
        ok = (d[:, 4] > 0) & (d[:, 7] > 0)
        if ok.sum() < 8:
            continue
        se = d[ok, 4].astype(np.float64)
        rel = (se - np.median(se)) / 1e3
        for c, r, sm in zip(np.nonzero(ok)[0], rel, d[ok, 7] - 1):
            by_sm[int(sm)].append(r)
            by_cta[int(c)].append(r)

    def halves(dct):
        ks = [k for k in dct if len(dct[k]) >= 4]
        a = np.array([np.mean(dct[k][0::2]) for k in ks])
        b = np.array([np.mean(dct[k][1::2]) for k in ks])
        return float(np.corrcoef(a, b)[0, 1]), float(np.std([np.mean(dct[k]) for k in ks]))
    return halves(by_sm), halves(by_cta)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--config", default="long128k")
    ap.add_argument("--gamma", type=float, default=0.99)
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--keep", default=None, help="directory for the stamped copy (default: a temp dir)")
    args = ap.parse_args(argv)
    dest = args.keep or tempfile.mkdtemp(prefix="asp_timeline_")
    if os.path.exists(os.path.join(dest, PKG)):
        shutil.rmtree(os.path.join(dest, PKG))
        shutil.rmtree(os.path.join(dest, "include"), ignore_errors=True)
    make_copy(dest)
    # the stamped copy must be the package imported from here on
    for m in [m for m in sys.modules if m == PKG or m.startswith(PKG + ".")]:
        del sys.modules[m]
    sys.path.insert(0, dest)
    import importlib
    bld = importlib.import_module(PKG + ".build")
    bld.build(force=True)
    import ctypes
    import numpy as np
    import torch
    B = importlib.import_module(PKG + ".binding")
    synth = importlib.import_module(PKG + ".synth")
    step_mod = importlib.import_module(PKG + ".step")
    if not os.path.abspath(B.LIB_PATH).startswith(os.path.abspath(dest)):
        raise RuntimeError("the stamped copy was not the one loaded")

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = synth.CONFIGS[args.config]
    sh = synth.make_shared(w, args.seed, dev)
    kvs, qs = [], []
    for l in range(w.layers):
        lay = synth.make_layer(w, sh, args.seed, l, dev)
        kvs.append(B.PagedKV(lay.k_cache, lay.v_cache, B.new_summaries(lay.k_cache, sh.block_table),
                             sh.block_table, sh.seq_lens, w.num_q_heads))
        qs.append(lay.q)
    ws0 = B.new_workspace(kvs[0])
    for kv in kvs:
        B.asp_page_summarize(kv, B.ASP_SUMMARIZE_BULK, None, None, ws0)
    step = step_mod.DecodeStep(kvs, torch.stack(qs), gamma=args.gamma)
    step.capture()
    for _ in range(5):
        step.replay()
    torch.cuda.synchronize()
    lib = B.load_library()
    for tag in ("sel", "dec"):
        if getattr(lib, f"asp_timeline_reset_{tag}")() != 0:
            raise RuntimeError("reset failed")
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    step.replay()
    e1.record()
    torch.cuda.synchronize()
    arr = {}
    for tag, n in (("sel", len(SEL_SLOTS)), ("dec", len(DEC_SLOTS))):
        a = np.zeros((N_LAUNCH, N_CTA, n), dtype=np.uint64)
        if getattr(lib, f"asp_timeline_read_{tag}")(a.ctypes.data_as(ctypes.c_void_p)) != 0:
            raise RuntimeError("read failed")
        arr[tag] = a.astype(np.int64)
    L = min(w.layers, N_LAUNCH)
    print(f"{args.config}, gamma {args.gamma}: stamped step {e0.elapsed_time(e1):.3f} ms for {w.layers} layers")
    print("us from each layer's first selection CTA start (median over the middle layers):")
    for k, v in _median_rows(arr["sel"], arr["dec"], L).items():
        print(f"  {k:40s} {v:8.2f}")
    (c_sm, s_sm), (c_cta, s_cta) = _sm_consistency(arr["dec"], L)
    print(f"decode stream end vs layer median: by SM corr(even, odd layers) {c_sm:.3f}, "
          f"spread of SM means {s_sm:.2f} us; by CTA index corr {c_cta:.3f}, spread {s_cta:.2f} us")


if __name__ == "__main__":
    main()
