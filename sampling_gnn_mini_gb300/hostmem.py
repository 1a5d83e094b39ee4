"""Host feature tables for zero-copy reads of cache misses.

A table of tens of GB read at random rows loses most of the host link's rate
to address translation when it is backed by small pages.  Measured on GB300
(Grace host, 64 KB base pages) with random 512-byte rows from a 60 GB table:

  cudaHostAlloc (torch pin_memory)                 10 GB/s random, 40 GB/s by region
  anonymous mmap with transparent huge pages,
  then cudaHostRegister (still pinned)             22 GB/s random, 67 GB/s by region

(a 16 GB table reads at ~208 GB/s either way).  pinned_table() therefore
backs large tables with transparent huge pages and pins them with
cudaHostRegister; small tables use torch's pinned allocator.

The GPU reaches a registered table through the host's page tables, and every
change the kernel makes to the table's entries (page aging clearing accessed
bits, huge-page collapse scans) invalidates the GPU's cached translations:
the gathers after it run cold, a single cold gather of 100K rows taking tens
of ms.  A large table's pages are therefore also locked (mlock: they leave the
reclaim lists, so aging skips them) and, once faulted in, marked no longer
eligible for huge-page collapse, so that the background scanner skips them.
"""
from __future__ import annotations

import ctypes
import mmap

import torch

HUGE_TABLE_BYTES = 32 << 30  # from this size on, back the table with huge pages


def huge_bytes_in(addr: int, smaps_lines) -> int:
    """AnonHugePages (bytes) of the mapping that starts at addr, from the
    lines of a /proc/<pid>/smaps listing; 0 if no mapping starts there."""
    found = False
    for line in smaps_lines:
        parts = line.split(None, 1)
        if not parts:
            continue
        head = parts[0]
        if "-" in head and not head.endswith(":"):
            found = int(head.split("-")[0], 16) == addr
        elif found and head == "AnonHugePages:":
            return int(line.split()[1]) * 1024
    return 0


def _huge_bytes(addr: int) -> int:
    try:
        with open("/proc/self/smaps") as f:
            return huge_bytes_in(addr, f)
    except (OSError, ValueError):
        return 0


def _lock_pages(addr: int, nbytes: int) -> bool:
    """mlock(2) of [addr, addr + nbytes); False where it is refused."""
    try:
        libc = ctypes.CDLL(None, use_errno=True)
        return int(libc.mlock(ctypes.c_void_p(addr), ctypes.c_size_t(nbytes))) == 0
    except (OSError, AttributeError):
        return False


class _Registered:
    """Owns a huge-page mapping pinned with cudaHostRegister (and locked
    where the process may lock it)."""

    def __init__(self, nbytes: int):
        self.registered = False
        self.map = mmap.mmap(-1, nbytes, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        if hasattr(mmap, "MADV_HUGEPAGE"):
            self.map.madvise(mmap.MADV_HUGEPAGE)
        self.nbytes = nbytes
        self.base = torch.frombuffer(self.map, dtype=torch.uint8)
        self.base.fill_(0)  # fault the pages in (as huge pages where the kernel allows)
        self.ptr = self.base.data_ptr()
        self.huge = _huge_bytes(self.ptr)
        self.locked = False
        if self.huge < 0.9 * nbytes:  # the kernel gave mostly small pages: not worth registering
            return
        self.locked = _lock_pages(self.ptr, nbytes)
        if hasattr(mmap, "MADV_NOHUGEPAGE"):
            self.map.madvise(mmap.MADV_NOHUGEPAGE)  # the pages are in: no collapse scans from here on
        err = torch.cuda.cudart().cudaHostRegister(self.ptr, nbytes, 0)
        if int(err) != 0:
            raise RuntimeError("cudaHostRegister of the host table failed: %s" % err)
        self.registered = True

    def __del__(self):
        if getattr(self, "registered", False):
            try:
                torch.cuda.cudart().cudaHostUnregister(self.ptr)
            except Exception:
                pass
            self.registered = False


def pinned_table(n_rows: int, dim: int, dtype: torch.dtype) -> torch.Tensor:
    """An uninitialised n_rows x dim page-locked host tensor suited to
    zero-copy row reads from the GPU (huge pages from HUGE_TABLE_BYTES on)."""
    elem = torch.empty((), dtype=dtype).element_size()
    nbytes = n_rows * dim * elem
    if nbytes < HUGE_TABLE_BYTES:
        return torch.empty((n_rows, dim), dtype=dtype, pin_memory=True)
    owner = _Registered(nbytes)
    if not owner.registered:
        # huge pages were not available (fragmented host memory): small-page
        # registered memory read slower than cudaHostAlloc's (measured 6 GB/s
        # against 10-40 GB/s on the 61 GB Wide table), so use the latter
        del owner
        return torch.empty((n_rows, dim), dtype=dtype, pin_memory=True)
    t = owner.base.view(dtype).view(n_rows, dim)
    t._sg_owner = owner  # keeps the mapping (and its registration) alive with the tensor
    return t
