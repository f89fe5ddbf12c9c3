"""Page-locked host buffers of exact size (kvm_host_alloc).

PyTorch's pinned-memory allocator rounds every request up to a power of two,
so a 74 GB host repository would lock 128 GB.  These buffers come from
kvm_host_alloc: exactly the requested size, allocated by the CUDA driver as
portable, mapped, page-locked memory.  The library accepts them like any
pinned memory: its kernels address them through their device alias, and
copies to and from them run at the pinned-copy rate.

The GPU reads a repository's missed blocks at scattered places over the host
link.  From driver-allocated memory a 148 GB repository streams at the full
pinned-copy rate.  Ordinary host memory registered after allocation streamed
at 0.48 to 0.93 of it, depending on how its pages happened to be laid out.

The tensors do not own their memory: each buffer stays allocated until
``release`` frees it (or the process exits), and a tensor must not be used
after its buffer is released.
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi

# data_ptr -> (tensor, ctypes buffer): the live buffers
_LIVE: dict[int, tuple] = {}


def pinned_empty(shape, dtype) -> torch.Tensor:
    """An uninitialised host tensor of exactly ``shape`` x ``dtype`` bytes in
    page-locked memory that kernels can address."""
    shape = torch.Size(shape)
    n = shape.numel() * torch.empty((), dtype=dtype).element_size()
    if n == 0:
        return torch.empty(shape, dtype=dtype)
    lib = _abi.load()
    p = ctypes.c_void_p()
    st = lib.kvm_host_alloc(n, ctypes.byref(p))
    if st != 0:
        raise RuntimeError(f"kvm_host_alloc of {n} bytes failed: "
                           f"{lib.kvm_last_error().decode()}")
    buf = (ctypes.c_uint8 * n).from_address(p.value)
    t = torch.frombuffer(buf, dtype=torch.uint8, count=n).view(dtype).view(shape)
    _LIVE[t.data_ptr()] = (t, buf)
    return t


def pinned_copy(src: torch.Tensor) -> torch.Tensor:
    """A page-locked host copy of ``src`` (any device)."""
    h = pinned_empty(src.shape, src.dtype)
    h.copy_(src)
    return h


def release(t: torch.Tensor) -> None:
    """Free a buffer made by pinned_empty, after the device has finished all
    work.  Other tensors pass through untouched."""
    if _LIVE.pop(t.data_ptr(), None) is not None:
        torch.cuda.synchronize()
        _abi.load().kvm_host_free(t.data_ptr())
