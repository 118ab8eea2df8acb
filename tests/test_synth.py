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


def test_unit_shift_moves_hot_keys_by_q_hat_only():
    """unit_shift keeps every draw and moves hot keys by shift * q_hat instead of
    shift * sqrt(d) * q_hat: cold pages are identical, hot pages differ."""
    import math

    import torch

    from adaptive_sparse_paged_gb300 import synth
    w = synth.Workload("u", 1, 1, 4, 1, 64, 16, seq_len=16 * 20, hot=("count", 3, 3),
                       shift=(2.0, 2.0))
    sh = synth.make_shared(w, 0, "cpu")
    a = synth.make_layer(w, sh, 0, 0, "cpu")
    b = synth.make_layer(w, sh, 0, 0, "cpu", unit_shift=True)
    assert torch.equal(a.q, b.q) and torch.equal(a.v_cache, b.v_cache)
    hot = a.hot[(0, 0)]
    assert hot == b.hot[(0, 0)] and len(hot) == 3
    phys = sh.block_table[0, :sh.num_pages[0]].long()
    cold = [i for i in range(sh.num_pages[0]) if i not in hot]
    assert torch.equal(a.k_cache[phys[cold], 0], b.k_cache[phys[cold], 0])
    qh = a.q[0].mean(0)
    qh = qh / qh.norm()
    # the mean hot key moves along q_hat by about shift * sqrt(d) vs shift
    da = (a.k_cache[phys[hot], 0].float().mean((0, 1)) @ qh).item()
    db = (b.k_cache[phys[hot], 0].float().mean((0, 1)) @ qh).item()
    assert abs(da - 2.0 * math.sqrt(64)) < 1.0 and abs(db - 2.0) < 1.0
