"""Output buffers with guard canaries before and after them.

`guarded(shape, dtype)` allocates a device buffer with GUARD elements of a
canary value on each side of the region a call may write, fills the whole
allocation with the canary, and returns the inner region (contiguous, of
`shape`) and a check that fails when any guard element changed -- a write
before the start or past the end of an output buffer."""
from __future__ import annotations

import torch

GUARD = 64          # elements on each side
CANARY = -123456789  # int32 guard value (a bit pattern no kernel writes)


def guarded(shape, dtype=torch.int32, device="cuda:0", fill=None):
    n = 1
    for d in shape:
        n *= int(d)
    buf = torch.full((n + 2 * GUARD,), CANARY, dtype=dtype, device=device)
    inner = buf[GUARD:GUARD + n].view(*shape)
    if fill is not None:
        inner.fill_(fill)

    def check(what=""):
        head = buf[:GUARD].cpu()
        tail = buf[GUARD + n:].cpu()
        assert torch.all(head == CANARY), f"{what}: a write before the output buffer"
        assert torch.all(tail == CANARY), f"{what}: a write past the output buffer"
    return inner, check
