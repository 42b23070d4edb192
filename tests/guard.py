"""Guard bands around device tensors.

Each tensor of a call is placed inside a larger device allocation, with
GUARD_BYTES of canary bytes before and after it (plus any extra offset asked
for, to place a tensor at a deliberately misaligned address).  The canaries
hold a 16-bit pattern that reads as a NaN in binary16 and bfloat16 (and, twice
over, in binary32).  After the call every canary byte must still be in place,
so a store past either end of any tensor fails the test that made it.  This is
the memory-safety check the GPU tests use in place of a memory checker.
"""
import torch

GUARD_BYTES = 4096
CANARY = 0x7FA5  # int16 pattern: NaN as binary16, bfloat16 and (doubled) binary32


class Guards:
    """The guarded device tensors of one call."""

    def __init__(self, device="cuda"):
        self.device = device
        self._buffers = []  # (raw int16 buffer, first byte of the tensor, its bytes, name)

    def put(self, t: torch.Tensor, name: str = "", offset: int = 0) -> torch.Tensor:
        """A device copy of ``t`` inside a guarded buffer: a contiguous view
        whose first byte sits GUARD_BYTES + ``offset`` bytes into the buffer
        (the buffer itself is 512-byte aligned)."""
        t = t.detach().contiguous()
        nbytes = t.numel() * t.element_size()
        start = GUARD_BYTES + offset
        total = start + nbytes + GUARD_BYTES
        total += total % 2
        raw = torch.full((total // 2,), CANARY, dtype=torch.int16, device=self.device)
        view = raw.view(torch.uint8)[start:start + nbytes].view(t.dtype).view(t.shape)
        view.copy_(t.to(self.device))
        self._buffers.append((raw, start, nbytes, name))
        return view

    def empty(self, shape, dtype, name: str = "", offset: int = 0) -> torch.Tensor:
        """A guarded device tensor holding the canary pattern."""
        nbytes = int(torch.Size(shape).numel()) * torch.empty(0, dtype=dtype).element_size()
        return self.put(torch.full((nbytes // 2,), CANARY, dtype=torch.int16).view(dtype).view(shape), name, offset)

    def check(self) -> None:
        """Every canary byte of every guarded tensor is unchanged."""
        torch.cuda.synchronize()
        for raw, start, nbytes, name in self._buffers:
            got = raw.view(torch.uint8)
            ref = torch.full_like(raw, CANARY).view(torch.uint8)
            front = torch.equal(got[:start], ref[:start])
            back = torch.equal(got[start + nbytes:], ref[start + nbytes:])
            assert front and back, "guard band of %s overwritten (%s)" % (
                name or "a tensor", ", ".join(w for w, ok in (("before it", front), ("after it", back)) if not ok))
