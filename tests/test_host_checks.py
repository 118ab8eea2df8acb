"""Host-side argument checks of the C ABI reject bad calls before any CUDA call.

Every call below returns from the library's validation code, which runs
before it touches the CUDA runtime, so these run on a machine without a GPU.
The pointers are non-null placeholders that are never dereferenced.
"""
import ctypes

import pytest

from adaptive_sparse_paged_gb300 import binding as B
from tests.test_abi_exports import lib  # noqa: F401  (fixture)

FAKE = 0x100000  # aligned, never dereferenced


def kv(**over):
    f = dict(k_cache=FAKE, v_cache=FAKE, summaries=FAKE, block_table=FAKE, seq_lens=FAKE,
             batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16, max_pages=64,
             num_phys_pages=128)
    f.update(over)
    return B.AspPagedKVStruct(*[f[n] for n, _ in B.AspPagedKVStruct._fields_])


@pytest.mark.parametrize("over,want", [
    (dict(k_cache=None), B.ASP_EINVAL),
    (dict(batch=0), B.ASP_EINVAL),
    (dict(num_q_heads=6, num_kv_heads=4), B.ASP_EINVAL),
    (dict(head_dim=96), B.ASP_EUNSUPPORTED),
    (dict(page_size=8), B.ASP_EUNSUPPORTED),
    (dict(num_kv_heads=3, num_q_heads=6), B.ASP_EUNSUPPORTED),
    (dict(num_q_heads=32, num_kv_heads=2), B.ASP_EUNSUPPORTED),  # group 16
    (dict(batch=1024, num_kv_heads=8, num_q_heads=8), B.ASP_EUNSUPPORTED),
    (dict(max_pages=(1 << 20) + 1), B.ASP_EUNSUPPORTED),
    (dict(k_cache=FAKE + 8), B.ASP_EINVAL),
])
def test_bad_shapes_rejected(lib, over, want):
    s = kv(**over)
    size = ctypes.c_size_t(0)
    assert lib.asp_workspace_size(ctypes.byref(s), ctypes.byref(size)) == want
    assert lib.asp_coverage_select(ctypes.byref(s), FAKE, 0.9, 0, FAKE, FAKE, FAKE, 1 << 20,
                                   None) == want
    assert lib.asp_sparse_decode(ctypes.byref(s), FAKE, FAKE, FAKE, 0.1, FAKE, FAKE, FAKE,
                                 1 << 20, None) == want
    assert lib.asp_page_summarize(ctypes.byref(s), 0, None, None, FAKE, 1 << 20, None) == want
    assert lib.asp_page_scores(ctypes.byref(s), FAKE, FAKE, FAKE, 1 << 20, None) == want


@pytest.mark.parametrize("gamma,budget", [(0.0, 0), (-0.5, 0), (1.5, 0), (float("nan"), 0),
                                          (0.9, -1)])
def test_bad_gamma_budget(lib, gamma, budget):
    s = kv()
    assert lib.asp_coverage_select(ctypes.byref(s), FAKE, gamma, budget, FAKE, FAKE, FAKE,
                                   1 << 20, None) == B.ASP_EINVAL


def test_null_outputs_and_modes(lib):
    s = kv()
    assert lib.asp_coverage_select(ctypes.byref(s), None, 0.9, 0, FAKE, FAKE, FAKE, 1, None) == B.ASP_EINVAL
    assert lib.asp_sparse_decode(ctypes.byref(s), FAKE, FAKE, FAKE, 0.1, None, FAKE, FAKE, 1,
                                 None) == B.ASP_EINVAL
    assert lib.asp_sparse_decode(ctypes.byref(s), FAKE, FAKE, FAKE, 0.0, FAKE, FAKE, FAKE, 1,
                                 None) == B.ASP_EINVAL
    assert lib.asp_page_summarize(ctypes.byref(s), 7, None, None, FAKE, 1, None) == B.ASP_EINVAL
    assert lib.asp_page_summarize(ctypes.byref(s), 1, None, None, FAKE, 1, None) == B.ASP_EINVAL
    assert lib.asp_page_summarize(ctypes.byref(s), 0, FAKE, FAKE, FAKE, 1, None) == B.ASP_EINVAL
    assert lib.asp_page_scores(ctypes.byref(s), None, FAKE, FAKE, 1, None) == B.ASP_EINVAL
    assert lib.asp_coverage_select_append(ctypes.byref(s), None, FAKE, FAKE, 0.9, 0, FAKE, FAKE,
                                          FAKE, 1, None) == B.ASP_EINVAL
    assert lib.asp_coverage_select_append(ctypes.byref(s), FAKE, FAKE + 8, FAKE, 0.9, 0, FAKE,
                                          FAKE, FAKE, 1, None) == B.ASP_EINVAL
    assert lib.asp_coverage_select_append(ctypes.byref(s), FAKE, FAKE, FAKE, 0.0, 0, FAKE, FAKE,
                                          FAKE, 1, None) == B.ASP_EINVAL
    assert lib.asp_page_scores(ctypes.byref(s), FAKE, None, FAKE, 1, None) == B.ASP_EINVAL
    assert lib.asp_page_scores(ctypes.byref(s), FAKE + 4, FAKE, FAKE, 1, None) == B.ASP_EINVAL


def test_workspace_pointer_checks(lib):
    assert lib.asp_workspace_init(None, 4096, None) == B.ASP_EWORKSPACE
    assert lib.asp_workspace_init(FAKE + 16, 4096, None) == B.ASP_EWORKSPACE
    assert lib.asp_workspace_init(FAKE, 16, None) == B.ASP_EWORKSPACE
    code = ctypes.c_uint32(0)
    assert lib.asp_get_device_error(None, ctypes.byref(code), None) == B.ASP_EINVAL


def test_step_shape_checks():
    """DecodeStep / DecodeLoop reject mis-shaped inputs before touching a device."""
    import torch
    from adaptive_sparse_paged_gb300.step import DecodeLoop, DecodeStep

    class FakeKV:  # the fields the constructors read before any allocation
        batch, num_q_heads, num_kv_heads, head_dim, max_pages = 2, 8, 2, 64, 4
        device = torch.device("cpu")

    kv = FakeKV()
    with pytest.raises(ValueError, match="q must have shape"):
        DecodeStep([kv], torch.zeros(1, 2, 8, 32), gamma=0.9)
    with pytest.raises(ValueError, match="at least one layer"):
        DecodeStep([], torch.zeros(1, 2, 8, 64), gamma=0.9)
    with pytest.raises(ValueError, match="append"):
        DecodeStep([kv], torch.zeros(1, 2, 8, 64), gamma=0.9,
                   append=(torch.zeros(1, 2, 2, 63), torch.zeros(1, 2, 2, 64)))
    q = torch.zeros(3, 1, 2, 8, 64)
    kn = torch.zeros(3, 1, 2, 2, 64)
    with pytest.raises(ValueError, match="v_new"):
        DecodeLoop([kv], torch.zeros(2, dtype=torch.int32), q, kn, torch.zeros(3, 1, 2, 2, 32),
                   gamma=0.9)
    with pytest.raises(ValueError, match="seq_lens0"):
        DecodeLoop([kv], torch.zeros(3, dtype=torch.int32), q, kn, kn, gamma=0.9)


@pytest.mark.parametrize("over", [
    dict(batch=512, num_q_heads=8, num_kv_heads=8, max_pages=1 << 20),  # page space >= 2^31
    dict(num_phys_pages=1 << 27, num_kv_heads=2, page_size=16),         # TMA rows >= 2^31
])
def test_int32_index_limits(lib, over):
    s = kv(**over)
    size = ctypes.c_size_t(0)
    assert lib.asp_workspace_size(ctypes.byref(s), ctypes.byref(size)) == B.ASP_EUNSUPPORTED


@pytest.mark.parametrize("scale", [float("nan"), float("inf"), -0.1])
def test_bad_decode_scale(lib, scale):
    s = kv()
    assert lib.asp_sparse_decode(ctypes.byref(s), FAKE, FAKE, FAKE, scale, FAKE, FAKE, FAKE,
                                 1 << 20, None) == B.ASP_EINVAL


def test_misaligned_decode_query(lib):
    s = kv()
    assert lib.asp_sparse_decode(ctypes.byref(s), FAKE + 4, FAKE, FAKE, 0.1, FAKE, FAKE, FAKE,
                                 1 << 20, None) == B.ASP_EINVAL


def test_noalloc_capacity_checked_first(lib):
    """Shapes beyond the fixed scratch are rejected before any device work."""
    s = kv(batch=4, num_q_heads=8, num_kv_heads=8, max_pages=(1 << 20) // 32 + 1)
    assert lib.asp_coverage_select_noalloc(ctypes.byref(s), FAKE, 0.9, 0, FAKE, FAKE, None,
                                           None) == B.ASP_EUNSUPPORTED
    assert lib.asp_coverage_select_noalloc(None, FAKE, 0.9, 0, FAKE, FAKE, None,
                                           None) == B.ASP_EINVAL
