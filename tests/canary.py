"""Guard regions around device outputs, in place of a memory checker.

Every output tensor a GPU test hands to the library can be allocated inside a
larger byte buffer whose 4 KiB head and tail (and the padding up to the next
256-byte boundary) hold a fixed byte pattern.  After the call, `check()`
confirms that no kernel wrote outside the tensor: a TMA store or reduce-add
box that is not clipped at a ragged edge, or a plain store past the last row,
would change the pattern.
"""
from __future__ import annotations

GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """A device tensor of `shape` and `dtype` between two guard regions."""

    def __init__(self, shape, dtype, device="cuda", fill=None):
        import torch
        numel = 1
        for s in shape:
            numel *= int(s)
        item = torch.empty((), dtype=dtype).element_size()
        self.nbytes = numel * item
        padded = (self.nbytes + 255) // 256 * 256
        self.raw = torch.full((GUARD + padded + GUARD,), PATTERN, dtype=torch.uint8, device=device)
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(*shape)
        if fill is not None:
            if isinstance(fill, (int, float)):
                self.t.fill_(fill)
            else:
                self.t.copy_(fill)

    def check(self, what="output"):
        import torch
        torch.cuda.synchronize()
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        bad_head = int((head != PATTERN).sum().item())
        bad_tail = int((tail != PATTERN).sum().item())
        assert bad_head == 0 and bad_tail == 0, (
            f"{what}: {bad_head} guard bytes changed before the tensor, {bad_tail} after it")


def guarded(shape, dtype, fill=None):
    return Guarded(shape, dtype, fill=fill)


def check_all(*gs):
    for i, g in enumerate(gs):
        if g is not None:
            g.check(f"output {i}")
