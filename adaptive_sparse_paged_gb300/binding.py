"""ctypes binding of libasp.so: argument marshalling only.

Every function here has the name of the C entry point it wraps (see
include/asp.h) and does nothing but check tensor dtypes/devices/shapes,
collect pointers and sizes, pass the current torch stream, and raise on a
negative status. All arithmetic of the decode path runs in the library's
CUDA kernels; there is no CPU fallback. If libasp.so is missing the import of
any function fails loudly (build it with adaptive_sparse_paged_gb300.build).
"""

from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libasp.so")

ASP_OK, ASP_EINVAL, ASP_EUNSUPPORTED, ASP_EWORKSPACE, ASP_ECUDA, ASP_EDEVICE = 0, -1, -2, -3, -4, -5
ASP_SUMMARIZE_BULK, ASP_SUMMARIZE_APPEND = 0, 1
ASP_DEVERR_PAGE_RANGE, ASP_DEVERR_LIST_RANGE, ASP_DEVERR_LEN_RANGE = 0x1, 0x2, 0x4
ASP_DEVERR_SEQ_RANGE, ASP_DEVERR_TIMEOUT = 0x8, 0x10

#: every symbol include/asp.h declares
EXPORTED = (
    "asp_abi_version",
    "asp_status_string",
    "asp_workspace_size",
    "asp_workspace_init",
    "asp_page_summarize",
    "asp_coverage_select",
    "asp_coverage_select_append",
    "asp_select_plan",
    "asp_page_scores",
    "asp_sparse_decode",
    "asp_get_device_error",
    "asp_coverage_select_noalloc",
    "asp_selftest_wait_timeout",
)


class AspPagedKVStruct(ctypes.Structure):
    """Mirror of asp_paged_kv."""
    _fields_ = [
        ("k_cache", ctypes.c_void_p),
        ("v_cache", ctypes.c_void_p),
        ("summaries", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("seq_lens", ctypes.c_void_p),
        ("batch", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("max_pages", ctypes.c_int32),
        ("num_phys_pages", ctypes.c_int32),
    ]


class AspError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_status_string(status)} (status {status})")


_lib = None
_lock = threading.Lock()


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libasp.so once (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libasp.so not found at {path}; build it with "
                               "`python -m adaptive_sparse_paged_gb300.build`")
        lib = ctypes.CDLL(path)
        vp, sz, i32, u32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.POINTER(ctypes.c_uint32)
        kvp = ctypes.POINTER(AspPagedKVStruct)
        sig = {
            "asp_abi_version": ([], i32),
            "asp_status_string": ([i32], ctypes.c_char_p),
            "asp_workspace_size": ([kvp, ctypes.POINTER(sz)], i32),
            "asp_workspace_init": ([vp, sz, vp], i32),
            "asp_page_summarize": ([kvp, i32, vp, vp, vp, sz, vp], i32),
            "asp_coverage_select": ([kvp, vp, ctypes.c_float, i32, vp, vp, vp, sz, vp], i32),
            "asp_page_scores": ([kvp, vp, vp, vp, sz, vp], i32),
            "asp_select_plan": ([kvp, ctypes.c_float, i32, i32, ctypes.POINTER(i32),
                                 ctypes.POINTER(i32)], i32),
            "asp_coverage_select_append": ([kvp, vp, vp, vp, ctypes.c_float, i32, vp, vp, vp,
                                            sz, vp], i32),
            "asp_sparse_decode": ([kvp, vp, vp, vp, ctypes.c_float, vp, vp, vp, sz, vp], i32),
            "asp_get_device_error": ([vp, u32p, vp], i32),
            "asp_coverage_select_noalloc": ([kvp, vp, ctypes.c_float, i32, vp, vp, vp, vp], i32),
            "asp_selftest_wait_timeout": ([vp, sz, vp], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _status_string(status: int) -> str:
    try:
        return load_library().asp_status_string(int(status)).decode()
    except Exception:  # the library itself failed to load
        return "status"


def _check(status: int, where: str) -> None:
    if status != ASP_OK:
        raise AspError(status, where)


def _stream_ptr(device: torch.device, stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _need(t: torch.Tensor, name: str, dtype, device, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


@dataclass
class PagedKV:
    """One layer's paged cache (device tensors), mirrored into asp_paged_kv.

    k_cache, v_cache : bf16 [num_phys_pages, Hkv, P, d]
    summaries        : bf16 [B, Hkv, max_pages, 2, d], logical page order
    block_table      : int32 [B, max_pages]
    seq_lens         : int32 [B]
    num_q_heads      : Hq (query head h reads KV head h // (Hq // Hkv))
    """
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    summaries: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    num_q_heads: int

    def __post_init__(self):
        dev = self.k_cache.device
        if dev.type != "cuda":
            raise ValueError("PagedKV tensors must live on a CUDA device")
        n, hkv, p, d = self.k_cache.shape
        _need(self.k_cache, "k_cache", torch.bfloat16, dev)
        _need(self.v_cache, "v_cache", torch.bfloat16, dev, (n, hkv, p, d))
        _need(self.block_table, "block_table", torch.int32, dev)
        b, max_pages = self.block_table.shape
        _need(self.summaries, "summaries", torch.bfloat16, dev, (b, hkv, max_pages, 2, d))
        _need(self.seq_lens, "seq_lens", torch.int32, dev, (b,))
        self.device = dev
        self.batch, self.num_kv_heads, self.page_size, self.head_dim = b, hkv, p, d
        self.max_pages, self.num_phys_pages = max_pages, n
        self.struct = AspPagedKVStruct(
            self.k_cache.data_ptr(), self.v_cache.data_ptr(), self.summaries.data_ptr(),
            self.block_table.data_ptr(), self.seq_lens.data_ptr(), b, int(self.num_q_heads),
            hkv, d, p, max_pages, n)

    @property
    def ref(self):
        return ctypes.byref(self.struct)


def new_summaries(k_cache: torch.Tensor, block_table: torch.Tensor) -> torch.Tensor:
    """Zeroed summaries tensor [B, Hkv, max_pages, 2, d] for this cache and table."""
    _, hkv, _, d = k_cache.shape
    b, max_pages = block_table.shape
    return torch.zeros((b, hkv, max_pages, 2, d), dtype=torch.bfloat16, device=k_cache.device)


# ----------------------------------------------------------- C-ABI mirrors
def asp_abi_version() -> int:
    return int(load_library().asp_abi_version())


def asp_workspace_size(kv: PagedKV) -> int:
    out = ctypes.c_size_t(0)
    with torch.cuda.device(kv.device):
        _check(load_library().asp_workspace_size(kv.ref, ctypes.byref(out)), "asp_workspace_size")
    return int(out.value)


def asp_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _need(ws, "ws", torch.uint8, ws.device)
    with torch.cuda.device(ws.device):
        _check(load_library().asp_workspace_init(ws.data_ptr(), ws.numel(),
                                                 _stream_ptr(ws.device, stream)),
               "asp_workspace_init")


def asp_page_summarize(kv: PagedKV, mode: int, k_new, v_new, ws: torch.Tensor, stream=None) -> None:
    if mode == ASP_SUMMARIZE_APPEND:
        shape = (kv.batch, kv.num_kv_heads, kv.head_dim)
        _need(k_new, "k_new", torch.bfloat16, kv.device, shape)
        _need(v_new, "v_new", torch.bfloat16, kv.device, shape)
        kp, vp = k_new.data_ptr(), v_new.data_ptr()
    else:
        kp = vp = None
    _need(ws, "ws", torch.uint8, kv.device)
    with torch.cuda.device(kv.device):
        _check(load_library().asp_page_summarize(kv.ref, int(mode), kp, vp, ws.data_ptr(),
                                                 ws.numel(), _stream_ptr(kv.device, stream)),
               "asp_page_summarize")


def asp_coverage_select(kv: PagedKV, q: torch.Tensor, gamma: float, budget: int,
                        lists: torch.Tensor, lens: torch.Tensor, ws: torch.Tensor,
                        stream=None) -> None:
    _need(q, "q", torch.float32, kv.device, (kv.batch, kv.num_q_heads, kv.head_dim))
    _need(lists, "lists", torch.int32, kv.device, (kv.batch, kv.num_kv_heads, kv.max_pages))
    _need(lens, "lens", torch.int32, kv.device, (kv.batch, kv.num_kv_heads))
    _need(ws, "ws", torch.uint8, kv.device)
    with torch.cuda.device(kv.device):
        _check(load_library().asp_coverage_select(
            kv.ref, q.data_ptr(), ctypes.c_float(gamma), int(budget), lists.data_ptr(),
            lens.data_ptr(), ws.data_ptr(), ws.numel(), _stream_ptr(kv.device, stream)),
            "asp_coverage_select")


def asp_coverage_select_append(kv: PagedKV, k_new: torch.Tensor, v_new: torch.Tensor,
                               q: torch.Tensor, gamma: float, budget: int, lists: torch.Tensor,
                               lens: torch.Tensor, ws: torch.Tensor, stream=None) -> None:
    """APPEND (k_new, v_new: bf16 [B, Hkv, d]) and coverage selection in one pass."""
    shp = (kv.batch, kv.num_kv_heads, kv.head_dim)
    _need(k_new, "k_new", torch.bfloat16, kv.device, shp)
    _need(v_new, "v_new", torch.bfloat16, kv.device, shp)
    _need(q, "q", torch.float32, kv.device, (kv.batch, kv.num_q_heads, kv.head_dim))
    _need(lists, "lists", torch.int32, kv.device, (kv.batch, kv.num_kv_heads, kv.max_pages))
    _need(lens, "lens", torch.int32, kv.device, (kv.batch, kv.num_kv_heads))
    _need(ws, "ws", torch.uint8, kv.device)
    with torch.cuda.device(kv.device):
        _check(load_library().asp_coverage_select_append(
            kv.ref, k_new.data_ptr(), v_new.data_ptr(), q.data_ptr(), ctypes.c_float(gamma),
            int(budget), lists.data_ptr(), lens.data_ptr(), ws.data_ptr(), ws.numel(),
            _stream_ptr(kv.device, stream)), "asp_coverage_select_append")


def asp_select_plan(kv: PagedKV, gamma: float, budget: int = 0, append: bool = False):
    """(kernels one selection call launches, cluster CTAs per segment or 0)."""
    k, c = ctypes.c_int32(0), ctypes.c_int32(0)
    with torch.cuda.device(kv.device):
        _check(load_library().asp_select_plan(kv.ref, ctypes.c_float(gamma), int(budget),
                                              int(bool(append)), ctypes.byref(k),
                                              ctypes.byref(c)), "asp_select_plan")
    return int(k.value), int(c.value)


def asp_page_scores(kv: PagedKV, q: torch.Tensor, scores: torch.Tensor, ws: torch.Tensor,
                    stream=None) -> None:
    """Per-page scores [B, Hkv, max_pages] fp32 (entries past N_b untouched)."""
    _need(q, "q", torch.float32, kv.device, (kv.batch, kv.num_q_heads, kv.head_dim))
    _need(scores, "scores", torch.float32, kv.device,
          (kv.batch, kv.num_kv_heads, kv.max_pages))
    _need(ws, "ws", torch.uint8, kv.device)
    with torch.cuda.device(kv.device):
        _check(load_library().asp_page_scores(kv.ref, q.data_ptr(), scores.data_ptr(),
                                              ws.data_ptr(), ws.numel(),
                                              _stream_ptr(kv.device, stream)),
               "asp_page_scores")


def asp_sparse_decode(kv: PagedKV, q: torch.Tensor, lists: torch.Tensor, lens: torch.Tensor,
                      sm_scale: float, out: torch.Tensor, lse: torch.Tensor, ws: torch.Tensor,
                      stream=None) -> None:
    _need(q, "q", torch.float32, kv.device, (kv.batch, kv.num_q_heads, kv.head_dim))
    _need(lists, "lists", torch.int32, kv.device, (kv.batch, kv.num_kv_heads, kv.max_pages))
    _need(lens, "lens", torch.int32, kv.device, (kv.batch, kv.num_kv_heads))
    _need(out, "out", torch.float32, kv.device, (kv.batch, kv.num_q_heads, kv.head_dim))
    _need(lse, "lse", torch.float32, kv.device, (kv.batch, kv.num_q_heads))
    _need(ws, "ws", torch.uint8, kv.device)
    with torch.cuda.device(kv.device):
        _check(load_library().asp_sparse_decode(
            kv.ref, q.data_ptr(), lists.data_ptr(), lens.data_ptr(), ctypes.c_float(sm_scale),
            out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(),
            _stream_ptr(kv.device, stream)), "asp_sparse_decode")


def asp_coverage_select_noalloc(kv: PagedKV, q: torch.Tensor, gamma: float, budget: int,
                                lists: torch.Tensor, lens: torch.Tensor,
                                dev_error: torch.Tensor | None = None, stream=None) -> None:
    """asp_coverage_select with the library's own fixed scratch instead of a workspace.

    For callers that cannot allocate device memory; see include/asp.h for the
    size limit and the rule that overlapping calls must be serialised.
    dev_error: optional int32 [1] device tensor that collects device error bits.
    """
    _need(q, "q", torch.float32, kv.device, (kv.batch, kv.num_q_heads, kv.head_dim))
    _need(lists, "lists", torch.int32, kv.device, (kv.batch, kv.num_kv_heads, kv.max_pages))
    _need(lens, "lens", torch.int32, kv.device, (kv.batch, kv.num_kv_heads))
    err_ptr = None
    if dev_error is not None:
        _need(dev_error, "dev_error", torch.int32, kv.device, (1,))
        err_ptr = dev_error.data_ptr()
    with torch.cuda.device(kv.device):
        _check(load_library().asp_coverage_select_noalloc(
            kv.ref, q.data_ptr(), ctypes.c_float(gamma), int(budget), lists.data_ptr(),
            lens.data_ptr(), err_ptr, _stream_ptr(kv.device, stream)),
            "asp_coverage_select_noalloc")


def asp_selftest_wait_timeout(ws: torch.Tensor, stream=None) -> None:
    """Failure-detection self-test: a bounded on-chip wait that runs out (~2 s)
    and sets ASP_DEVERR_TIMEOUT in `ws`'s error word (read it with
    asp_get_device_error)."""
    _need(ws, "ws", torch.uint8, ws.device)
    with torch.cuda.device(ws.device):
        _check(load_library().asp_selftest_wait_timeout(ws.data_ptr(), ws.numel(),
                                                        _stream_ptr(ws.device, stream)),
               "asp_selftest_wait_timeout")


def asp_get_device_error(ws: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error mask."""
    code = ctypes.c_uint32(0)
    with torch.cuda.device(ws.device):
        st = load_library().asp_get_device_error(ws.data_ptr(), ctypes.byref(code),
                                                 _stream_ptr(ws.device, stream))
    if st not in (ASP_OK, ASP_EDEVICE):
        _check(st, "asp_get_device_error")
    return int(code.value)


def new_workspace(kv: PagedKV, stream=None) -> torch.Tensor:
    """Allocates (through torch) and zero-initialises a workspace for `kv`'s shape."""
    n = asp_workspace_size(kv)
    ws = torch.empty(n, dtype=torch.uint8, device=kv.device)
    asp_workspace_init(ws, stream)
    return ws
