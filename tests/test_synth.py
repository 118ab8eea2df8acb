"""The seeded input generator: shapes, permutation, hot pages, lengths (CPU)."""
import math

import torch

from adaptive_sparse_paged_gb300 import synth


def test_shared_tables():
    w = synth.CONFIGS["mixed64"]
    sh = synth.make_shared(w, 3, "cpu")
    lens = sh.seq_lens.tolist()
    assert all(4096 <= t <= 131072 for t in lens)
    assert any(t % w.page_size for t in lens)  # partial last pages occur
    used = []
    for b, n in enumerate(sh.num_pages):
        row = sh.block_table[b]
        assert torch.all(row[:n] >= 0) and torch.all(row[n:] == -1)
        used += row[:n].tolist()
    assert len(set(used)) == len(used) and max(used) < sh.num_phys_pages
    assert sh.num_phys_pages > len(used)  # some pages stay unmapped
    sh2 = synth.make_shared(w, 3, "cpu")
    assert torch.equal(sh.block_table, sh2.block_table)


def test_layer_hot_pages_and_seeding():
    w = synth.Workload("t", 2, 1, 8, 2, 64, 16, seq_len=16 * 40 + 3)
    sh = synth.make_shared(w, 0, "cpu")
    a = synth.make_layer(w, sh, 0, 0, "cpu")
    b = synth.make_layer(w, sh, 0, 0, "cpu")
    assert torch.equal(a.k_cache, b.k_cache) and torch.equal(a.q, b.q)
    c = synth.make_layer(w, sh, 0, 1, "cpu")
    assert not torch.equal(a.k_cache, c.k_cache)
    g = w.num_q_heads // w.num_kv_heads
    for (bb, h), pages in a.hot.items():
        n = sh.num_pages[bb]
        assert 1 <= len(pages) <= n and len(set(pages)) == len(pages)
        qhat = a.q[bb, h * g:(h + 1) * g].mean(0)
        qhat = qhat / qhat.norm()
        phys = sh.block_table[bb, :n].long()
        proj = (a.k_cache[phys, h].float() @ qhat).mean(1)  # mean key projection per page
        hot = torch.zeros(n, dtype=torch.bool)
        hot[pages] = True
        # hot keys sit >= 1 * sqrt(d) further along q_hat than noise
        assert proj[hot].min() > proj[~hot].max() if (~hot).any() else True
        assert proj[hot].min() > 0.9 * math.sqrt(w.head_dim)
