"""The timeline profiling tool stamps a copy of the kernels: its anchors must
exist exactly once in the current sources, and the library never imports it."""
import os
import subprocess
import sys

from adaptive_sparse_paged_gb300 import timeline

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_stamp_anchors_apply(tmp_path):
    timeline.make_copy(str(tmp_path))
    csrc = tmp_path / "adaptive_sparse_paged_gb300" / "csrc"
    sel = (csrc / "select_cluster.cu").read_text()
    dec = (csrc / "decode.cu").read_text()
    assert sel.count("g_tl_sel[((tl_L") == len(timeline.SEL_SLOTS)
    assert dec.count("g_tl_dec[((tl_L") == len(timeline.DEC_SLOTS)
    assert "asp_timeline_read_sel" in sel and "asp_timeline_read_dec" in dec
    # the repository's own sources are untouched
    with open(os.path.join(ROOT, "adaptive_sparse_paged_gb300", "csrc", "decode.cu")) as f:
        assert "g_tl_dec" not in f.read()


def test_library_does_not_import_the_tool():
    code = ("import sys; import adaptive_sparse_paged_gb300.binding, adaptive_sparse_paged_gb300.step; "
            "assert 'adaptive_sparse_paged_gb300.timeline' not in sys.modules")
    subprocess.run([sys.executable, "-c", code], cwd=ROOT, check=True)
