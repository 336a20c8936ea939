"""Page-locked host buffers on transparent huge pages, for the gradients a
trainer copies to the device every step.

A host-to-device copy runs at full speed only from page-locked memory.  The
driver's own page-locked allocation (``torch.empty(..., pin_memory=True)``)
uses small pages; measured on a GB300 host, 3.5 GB uploads from such buffers
ran at 211 GB/s but a few in forty stalled for 130 to 540 ms on the copy
engine itself, while the same uploads from memory backed by 2 MB pages and
page-locked afterwards stalled for at most ~50 ms, and less often.  So
:func:`pinned_empty` maps anonymous memory, asks the kernel for huge pages
(``MADV_HUGEPAGE``; where transparent huge pages are off it gets small pages
and still works), touches every page, and page-locks the range for the
device with ``cudaHostRegister``.
"""

import mmap

import torch


class _Region:
    """An anonymous mapping page-locked for the device; unlocked and unmapped
    when the last tensor viewing it is gone."""

    def __init__(self, nbytes):
        self.nbytes = max(int(nbytes), 1)
        self.map = mmap.mmap(-1, self.nbytes, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        if hasattr(mmap, "MADV_HUGEPAGE"):
            try:
                self.map.madvise(mmap.MADV_HUGEPAGE)
            except OSError:
                pass  # huge pages unavailable: small pages, still page-locked below
        self.bytes = torch.frombuffer(self.map, dtype=torch.uint8)
        self.bytes.zero_()  # touch every page before locking it
        self.ptr = self.bytes.data_ptr()
        cudart = torch.cuda.cudart()
        err = cudart.cudaHostRegister(self.ptr, self.nbytes, 0)
        if err != cudart.cudaError.success:
            raise RuntimeError("cudaHostRegister of %d bytes failed: %s" % (self.nbytes, err))
        self.locked = True

    def __del__(self):
        if getattr(self, "locked", False):
            try:
                torch.cuda.cudart().cudaHostUnregister(self.ptr)
            except Exception:  # interpreter shutdown
                pass
            self.locked = False


def pinned_empty(numel, dtype):
    """A 1-D host tensor of ``numel`` elements of ``dtype`` in page-locked,
    huge-page-backed memory (see the module docstring); ``is_pinned()`` is
    true, so copies to the device with ``non_blocking=True`` are
    asynchronous.  The memory is released with the tensor."""
    es = torch.empty(0, dtype=dtype).element_size()
    region = _Region(numel * es)
    t = region.bytes[:numel * es].view(dtype)
    t._gbo_region = region  # keeps the mapping alive as long as the tensor
    return t
