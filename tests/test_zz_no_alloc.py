"""asp_coverage_select_noalloc: coverage selection for callers that cannot allocate.

Callers such as an engine that owns all GPU memory through its own pool, or a
loop that must not allocate once running, cannot hand the library a
workspace. This entry point keeps its scratch in a fixed array inside the
library instead; these tests call it through the C ABI and require its page
lists and lengths to equal those of asp_coverage_select (integer outputs:
bit-exact) on two calls in a row, and an oversized shape to be rejected.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test; it also passes on its own.
"""
import ctypes

import pytest
import torch

from adaptive_sparse_paged_gb300 import binding as B
from adaptive_sparse_paged_gb300 import synth
from tests import guards

pytestmark = pytest.mark.gpu


def _case(dev, seed):
    w = synth.Workload("noalloc", 3, 2, 16, 4, 128, 16, seq_len=1)
    sh = synth.make_shared(w, seed, dev, seq_lens=[16 * 300 + 7, 16 * 41, 5], max_pages=320)
    layers = [synth.make_layer(w, sh, seed, l, dev) for l in range(2)]
    summ_shape = (w.batch, w.num_kv_heads, sh.max_pages, 2, w.head_dim)
    kvs = [B.PagedKV(lay.k_cache, lay.v_cache,
                     guards.guarded(summ_shape, torch.bfloat16, dev, fill=0, what="summaries"),
                     sh.block_table, sh.seq_lens,
                     w.num_q_heads) for lay in layers]
    ws = guards.guarded_workspace(kvs[0])
    for kv in kvs:
        B.asp_page_summarize(kv, B.ASP_SUMMARIZE_BULK, None, None, ws)
    assert B.asp_get_device_error(ws) == 0
    return w, sh, layers, kvs, ws


def test_noalloc_matches_workspace_path_twice(cuda_device):
    w, sh, layers, kvs, ws = _case(cuda_device, seed=11)
    shape_l = (w.batch, w.num_kv_heads, sh.max_pages)
    calls = [(kvs[0], layers[0].q, 0.95, 0), (kvs[1], layers[1].q, 0.6, 0),
             (kvs[1], layers[1].q, 0.5, 37)]
    want = []
    for kv, q, gamma, budget in calls:  # reference: the workspace entry point
        lists = torch.full(shape_l, -1, dtype=torch.int32, device=cuda_device)
        lens = torch.full(shape_l[:2], -1, dtype=torch.int32, device=cuda_device)
        B.asp_coverage_select(kv, q, gamma, budget, lists, lens, ws)
        want.append((lists, lens))
    assert B.asp_get_device_error(ws) == 0
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    got = []
    for kv, q, gamma, budget in calls:  # the no-allocation entry point, back to back
        lists = guards.guarded(shape_l, torch.int32, cuda_device, fill=-1, what="lists")
        lens = guards.guarded(shape_l[:2], torch.int32, cuda_device, fill=-1, what="lens")
        B.asp_coverage_select_noalloc(kv, q, gamma, budget, lists, lens, err)
        got.append((lists, lens))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for (wl, wn), (gl, gn) in zip(want, got):
        assert torch.equal(wn, gn)
        for b in range(w.batch):
            for h in range(w.num_kv_heads):
                n = int(wn[b, h])
                assert torch.equal(wl[b, h, :n], gl[b, h, :n])


def test_noalloc_rejects_oversized_shape(cuda_device):
    lib = B.load_library()
    fake = 0x100000  # never dereferenced: the call must return before any device work
    kv = B.AspPagedKVStruct(fake, fake, fake, fake, fake, 16, 64, 8, 128, 16, 8193, 1 << 16)
    assert 16 * 8 * 8193 > (1 << 20)
    st = lib.asp_coverage_select_noalloc(ctypes.byref(kv), fake, ctypes.c_float(0.9), 0, fake,
                                         fake, None, None)
    assert st == B.ASP_EUNSUPPORTED
