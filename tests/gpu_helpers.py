"""Device-buffer helpers for the GPU parity tests (raw bytes in, raw bytes out).

Buffers travel as uint8 torch tensors so that every comparison is on bits.
`Canvas` surrounds an output with guard bands holding a canary pattern and
checks after each call that nothing outside the output was written.
"""
import numpy as np
import torch

CANARY = np.frombuffer(bytes.fromhex("ADDEC07F") * 4, np.uint8)  # 0x7FC0DEAD little-endian, repeated


def dev(a: np.ndarray) -> torch.Tensor:
    """Copy a numpy array's bytes to a new device buffer (uint8 tensor)."""
    flat = np.ascontiguousarray(a).reshape(-1).view(np.uint8)
    return torch.from_numpy(flat.copy()).to("cuda")


def host(t: torch.Tensor, dtype, shape) -> np.ndarray:
    return t.cpu().numpy().view(dtype).reshape(shape)


class Canvas:
    """An output buffer of `nbytes` inside guard bands of `guard` canary bytes."""

    def __init__(self, nbytes: int, guard: int = 4096, fill: np.ndarray | None = None):
        self.nbytes, self.guard = nbytes, guard
        total = nbytes + 2 * guard
        pattern = np.resize(CANARY, total)
        if fill is not None:
            fb = np.ascontiguousarray(fill).reshape(-1).view(np.uint8)
            assert fb.size == nbytes
            pattern[guard:guard + nbytes] = fb
        self.buf = torch.from_numpy(pattern.copy()).to("cuda")
        self._pattern = pattern

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr() + self.guard

    def inner(self, dtype, shape) -> np.ndarray:
        b = self.buf.cpu().numpy()
        return b[self.guard:self.guard + self.nbytes].view(dtype).reshape(shape)

    def original(self, dtype, shape) -> np.ndarray:
        """The bytes the output region held before the call."""
        g = self.guard
        return self._pattern[g:g + self.nbytes].view(dtype).reshape(shape)

    def guards_intact(self) -> bool:
        b = self.buf.cpu().numpy()
        g = self.guard
        return np.array_equal(b[:g], self._pattern[:g]) and np.array_equal(b[-g:], self._pattern[-g:])


def sync():
    torch.cuda.synchronize()
