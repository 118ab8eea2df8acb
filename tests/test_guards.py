"""The guard-band helper catches writes past either end of a tensor (CPU)."""

from __future__ import annotations

import pytest
import torch

from tests import guards


def _base(t, band_elems):
    """The whole allocation behind a guarded tensor, as t's dtype."""
    return t.view(-1).as_strided((t.numel() + 2 * band_elems,), (1,),
                                 t.storage_offset() - band_elems)


@pytest.mark.parametrize("dtype", [torch.int32, torch.float32, torch.bfloat16, torch.uint8])
def test_in_bounds_writes_pass(dtype):
    t = guards.guarded((3, 5, 7), dtype, "cpu", fill=0, what="t")
    assert t.is_contiguous() and t.shape == (3, 5, 7)
    t.fill_(1)
    t[0, 0, 0] = 2
    t[-1, -1, -1] = 3
    guards.check_guards()
    assert guards.registered() == 0


@pytest.mark.parametrize("where", ["head", "tail", "far_tail"])
def test_out_of_bounds_writes_fail(where):
    t = guards.guarded((4, 100), torch.int32, "cpu", fill=-7, what="lists")
    band = guards._band_bytes(t.numel() * 4) // 4
    base = _base(t, band)
    idx = {"head": band - 1, "tail": band + t.numel(), "far_tail": 2 * band + t.numel() - 1}[where]
    base[idx] = 123
    with pytest.raises(AssertionError, match="lists"):
        guards.check_guards()
    assert guards.registered() == 0


def test_band_sizes_keep_alignment():
    for nbytes in (1, 4095, 4096, 12345, 1 << 20, 1 << 24):
        b = guards._band_bytes(nbytes)
        assert b % 4096 == 0 and 4096 <= b <= (1 << 20) and (b >= nbytes or b == 1 << 20)


def test_guarded_like_copies():
    src = torch.arange(24, dtype=torch.float32).view(2, 3, 4)
    t = guards.guarded_like(src, what="copy")
    assert torch.equal(t, src) and t.data_ptr() != src.data_ptr()
    guards.check_guards()
