"""Guard bands around the output buffers of the GPU tests.

compute-sanitizer is closed on this machine, so stray writes are caught the
plain way: every output a parity test hands to the library sits inside a
larger device allocation whose bytes before and after it hold a seeded
random pattern, and after the call the pattern must be unchanged.

Band sizes: a 2-D output [r, c] gets 32 rows' worth of bytes (32 * c *
itemsize, at least 256) on each side, one full 32-row tile-store box past
either edge; a 1-D output gets 16 KiB (one 32 KiB bf16 input chunk's worth
of 8-bit output) on each side.  The band in front is a multiple of 256
bytes plus `offset`, so an output keeps the alignment the caller asks for.
"""
from __future__ import annotations

import torch

_INTERIOR_FILL = 0xA5


class Guards:
    def __init__(self, seed: int = 0x5A17):
        self._gen = torch.Generator().manual_seed(seed)
        self._items = []

    @staticmethod
    def _band(shape, itemsize: int) -> int:
        if len(shape) >= 2:
            b = 32 * int(shape[-1]) * itemsize
        else:
            b = 16 * 1024
        return max(256, (b + 255) // 256 * 256)

    def empty(self, shape, dtype=torch.uint8, offset: int = 0) -> torch.Tensor:
        """A CUDA tensor of `shape` / `dtype` whose bytes start `offset`
        bytes past a 256-byte boundary, with guard bands on both sides."""
        if isinstance(shape, int):
            shape = (shape,)
        shape = tuple(int(s) for s in shape)
        itemsize = torch.empty(0, dtype=dtype).element_size()
        numel = 1
        for s in shape:
            numel *= s
        nbytes = numel * itemsize
        band = self._band(shape, itemsize)
        front = band + offset
        buf = torch.empty(front + nbytes + band, dtype=torch.uint8, device="cuda")
        pf = torch.randint(0, 256, (front,), generator=self._gen, dtype=torch.uint8)
        pb = torch.randint(0, 256, (band,), generator=self._gen, dtype=torch.uint8)
        buf[:front].copy_(pf)
        buf[front + nbytes:].copy_(pb)
        if nbytes:
            buf[front:front + nbytes].fill_(_INTERIOR_FILL)
        t = buf[front:front + nbytes].view(dtype).view(shape)
        self._items.append((buf, front, nbytes, pf, pb))
        return t

    def full(self, shape, value, dtype) -> torch.Tensor:
        t = self.empty(shape, dtype)
        t.fill_(value)
        return t

    def check(self, what="") -> None:
        """Assert every guard band is unchanged (synchronises the device)."""
        torch.cuda.synchronize()
        for k, (buf, front, nbytes, pf, pb) in enumerate(self._items):
            got_f = buf[:front].cpu()
            got_b = buf[front + nbytes:].cpu()
            if not torch.equal(got_f, pf):
                bad = int((got_f != pf).nonzero()[-1])
                raise AssertionError(f"write {front - bad} bytes before output #{k} ({nbytes} bytes) {what}")
            if not torch.equal(got_b, pb):
                bad = int((got_b != pb).nonzero()[0])
                raise AssertionError(f"write {bad} bytes past the end of output #{k} ({nbytes} bytes) {what}")

    def release(self) -> None:
        self._items.clear()

    def check_and_release(self, what="") -> None:
        try:
            self.check(what)
        finally:
            self.release()
