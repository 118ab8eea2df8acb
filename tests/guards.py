"""Guard bands (canaries) around every buffer a kernel under test writes.

A guarded tensor is carved out of a larger allocation: the bytes before and
after it hold a fixed pattern, and `check_guards` fails when any of them
changed, i.e. when a kernel wrote past either end of the tensor it was
given. This stands in for a memory checker on the writes that matter most
(outputs, workspace, summaries and appended cache rows). The bands are as
large as the tensor itself, capped at 1 MiB and at least 4 KiB, so a write
one row (or one segment) too far still lands inside a band; being multiples
of 4 KiB they keep the tensor's alignment (the workspace needs 256 bytes).

tests/conftest.py checks every band registered during a test when the test
ends.
"""

from __future__ import annotations

import math

import torch

PATTERN = 0xA5
_MIN_BAND, _MAX_BAND = 4096, 1 << 20

_registry: list = []


def _band_bytes(nbytes: int) -> int:
    b = min(max(nbytes, _MIN_BAND), _MAX_BAND)
    return (b + _MIN_BAND - 1) // _MIN_BAND * _MIN_BAND


def guarded(shape, dtype, device, fill=None, what: str = "tensor") -> torch.Tensor:
    """A contiguous tensor of `shape` with pattern bands on both sides.

    fill: value written into the tensor itself (None leaves the pattern).
    """
    shape = tuple(int(s) for s in shape)
    n = math.prod(shape)
    isz = torch.empty((), dtype=dtype).element_size()
    band = _band_bytes(n * isz)
    raw = torch.full((2 * band + n * isz,), PATTERN, dtype=torch.uint8, device=device)
    t = raw[band:band + n * isz].view(dtype).view(shape)
    if fill is not None:
        t.fill_(fill)
    _registry.append((raw, band, n * isz, what))
    return t


def guarded_like(src: torch.Tensor, what: str = "tensor") -> torch.Tensor:
    """A guarded copy of `src`."""
    t = guarded(src.shape, src.dtype, src.device, what=what)
    t.copy_(src)
    return t


def guarded_workspace(kv, what: str = "workspace") -> torch.Tensor:
    """A guarded, initialised workspace for `kv` (the library's own size query)."""
    from adaptive_sparse_paged_gb300 import binding as B
    ws = guarded((B.asp_workspace_size(kv),), torch.uint8, kv.device, what=what)
    B.asp_workspace_init(ws)
    return ws


def violations() -> list:
    """Names (with the first bad offset) of every registered band that changed."""
    bad = []
    for raw, band, nbytes, what in _registry:
        if raw.is_cuda:
            torch.cuda.synchronize(raw.device)
        head = raw[:band] != PATTERN
        tail = raw[band + nbytes:] != PATTERN
        if bool(head.any()):
            first = int(torch.nonzero(head)[-1])
            bad.append(f"{what}: write {band - first} bytes before the start")
        if bool(tail.any()):
            first = int(torch.nonzero(tail)[0])
            bad.append(f"{what}: write {first} bytes past the end")
    return bad


def check_guards() -> None:
    """Fails if any band changed; forgets every registered band either way."""
    try:
        bad = violations()
    finally:
        _registry.clear()
    assert not bad, "out-of-bounds writes: " + "; ".join(bad)


def registered() -> int:
    return len(_registry)


def take() -> list:
    """Removes and returns every registered band (for buffers that outlive one
    test: hand them back with `register` at the start of each test)."""
    entries = list(_registry)
    _registry.clear()
    return entries


def register(entries) -> None:
    _registry.extend(entries)
