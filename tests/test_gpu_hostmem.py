"""Page-locked, huge-page-backed host buffers (hostmem.pinned_empty): they
are page-locked for the device, asynchronous copies in both directions give
back the same bytes, and the memory goes away with the tensor."""

import gc

import pytest
import torch

from adamw_optimizer_step_gb300 import hostmem

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_pinned_round_trip(dtype):
    n = 3 * (1 << 20) + 7  # a few huge pages and a ragged tail
    h = hostmem.pinned_empty(n, dtype)
    assert h.is_pinned() and h.numel() == n and h.dtype == dtype
    src = torch.randn(n, device="cuda").to(dtype)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        h.copy_(src, non_blocking=True)
        back = torch.empty_like(src)
        back.copy_(h, non_blocking=True)
    s.synchronize()
    assert torch.equal(back, src)
    assert torch.equal(h, src.cpu())
    del h, back
    gc.collect()


@pytest.mark.parametrize("nbytes", [1, 15, 16, 17, 3 * 4096 + 7, (5 << 20) + 3, (64 << 20) + 48])
@pytest.mark.parametrize("alloc", ["hostmem", "pin_memory"])
@pytest.mark.parametrize("blocks", [0, 1, 4])
def test_h2d_copy_kernel(nbytes, alloc, blocks):
    """gbo_h2d_copy (SM loads of page-locked host memory) gives back the
    same bytes as the host buffer, for ragged sizes, from huge-page
    registered memory and from the driver's pinned allocation, on a side
    stream."""
    from adamw_optimizer_step_gb300 import _binding as B
    g = torch.Generator().manual_seed(nbytes)
    data = torch.randint(0, 256, (nbytes,), generator=g, dtype=torch.uint8)
    h = hostmem.pinned_empty(nbytes, torch.uint8) if alloc == "hostmem" else torch.empty(nbytes, dtype=torch.uint8,
                                                                                           pin_memory=True)
    h.copy_(data)
    d = torch.full((nbytes + 64,), 0xA5, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    launches = B.gbo_launch_count()
    B.gbo_h2d_copy(d[:nbytes], h, blocks=blocks, stream=s)
    s.synchronize()
    assert B.gbo_launch_count() == launches + 1
    assert torch.equal(d[:nbytes].cpu(), data)
    assert bool((d[nbytes:] == 0xA5).all())  # nothing past the end is written


def test_h2d_copy_refusals():
    """Pageable or device memory as the source, host memory as the
    destination and misaligned pointers are refused before any copy."""
    from adamw_optimizer_step_gb300 import _binding as B
    L = B.lib()
    n = 1 << 16
    d = torch.zeros(n, dtype=torch.uint8, device="cuda")
    pageable = torch.zeros(n, dtype=torch.uint8)
    pinned = hostmem.pinned_empty(n, torch.uint8)
    stream = torch.cuda.current_stream().cuda_stream
    assert L.gbo_h2d_copy(d.data_ptr(), pageable.data_ptr(), n, 0, stream) == -1
    assert L.gbo_h2d_copy(d.data_ptr(), d.data_ptr(), n, 0, stream) == -1
    assert L.gbo_h2d_copy(pinned.data_ptr(), pinned.data_ptr(), n, 0, stream) == -1
    assert L.gbo_h2d_copy(d.data_ptr() + 8, pinned.data_ptr(), 64, 0, stream) == -1
    # a source range that runs past its registration
    assert L.gbo_h2d_copy(d.data_ptr(), pinned.data_ptr(), n + (4 << 20), 0, stream) == -1
    torch.cuda.synchronize()
    assert bool((d == 0).all())
