"""Pinned host buffers for feeding the step from host memory.

A page-locked host buffer is read by the GPU's copy engines through the
system MMU.  With the 64 KiB base pages of the Arm hosts GB300 sits in, a
multi-GB buffer needs hundreds of thousands of translations, and repeated
host-to-device copies of it stall on translation misses (a 16 GB copy took
76 ms or 250-540 ms from one repeat to the next).  Backing the buffer with
transparent huge pages (512 MiB on such kernels) before registering it with
CUDA keeps every copy at the link rate.

``pinned_empty`` maps anonymous memory aligned to 2 MiB, asks the kernel for
huge pages (madvise MADV_HUGEPAGE), touches it, and page-locks it with
cudaHostRegister.  If huge pages are unavailable it still works, as a plain
registered buffer.
"""
from __future__ import annotations

import ctypes
import mmap

import numpy as np
import torch

_MADV_HUGEPAGE = 14
_ALIGN = 1 << 21


class PinnedHostBuffer:
    """Owns one registered mapping; ``tensor`` views it with the given dtype."""

    def __init__(self, numel: int, dtype: torch.dtype):
        self.nbytes = numel * torch.tensor([], dtype=dtype).element_size()
        self._mm = mmap.mmap(-1, self.nbytes + _ALIGN,
                             flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        base = ctypes.addressof(ctypes.c_char.from_buffer(self._mm))
        aligned = (base + _ALIGN - 1) & ~(_ALIGN - 1)
        libc = ctypes.CDLL(None)
        self.huge_pages = libc.madvise(ctypes.c_void_p(aligned), ctypes.c_size_t(self.nbytes),
                                       _MADV_HUGEPAGE) == 0
        raw = np.frombuffer(self._mm, dtype=np.uint8, count=self.nbytes, offset=aligned - base)
        raw[::4096] = 0                       # fault the pages in before locking them
        err = torch.cuda.cudart().cudaHostRegister(aligned, self.nbytes, 0)
        if int(err) != 0:
            raise RuntimeError(f"cudaHostRegister failed: {err}")
        self._ptr = aligned
        self.tensor = torch.from_numpy(raw).view(dtype)

    def close(self):
        if self._ptr:
            torch.cuda.cudart().cudaHostUnregister(self._ptr)
            self._ptr = 0
            self.tensor = None
            try:
                self._mm.close()
            except BufferError:       # a view is still alive; the GC unmaps later
                pass

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pinned_empty(numel: int, dtype: torch.dtype) -> PinnedHostBuffer:
    return PinnedHostBuffer(numel, dtype)
