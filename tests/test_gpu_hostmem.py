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
