"""Helpers for the GPU parity tests: host<->device transfer of bit patterns, ulp distances,
canary-guarded output buffers. No arithmetic of the method lives here."""
from __future__ import annotations

import numpy as np
import torch

GUARD = 4096  # bytes of canary before and after every guarded output
CANARY = 0xA5


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    """numpy uint16 bf16 bits -> CUDA bfloat16 tensor (same bits)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.uint8).cpu().numpy()


def dev_scale(s: float) -> torch.Tensor:
    return torch.tensor([s], dtype=torch.float32, device="cuda")


class Guarded:
    """A device output of `nbytes` bytes with canary bands on both sides."""

    def __init__(self, shape, dtype: torch.dtype):
        self.shape = tuple(shape)
        self.dtype = dtype
        n = int(np.prod(self.shape)) * torch.tensor([], dtype=dtype).element_size()
        self.nbytes = n
        self.raw = torch.full((GUARD + n + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        self.tensor = self.raw[GUARD:GUARD + n].view(dtype).view(self.shape)

    def intact(self) -> bool:
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        return bool((head == CANARY).all().item()) and bool((tail == CANARY).all().item())


def bf16_ordinal(b: np.ndarray) -> np.ndarray:
    """Monotone integer ordinal of bf16 bit patterns (+0 and -0 both map to 0)."""
    b = b.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(bf16_ordinal(a) - bf16_ordinal(b))


def e4m3_ordinal(c: np.ndarray) -> np.ndarray:
    c = c.astype(np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def e4m3_step_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(e4m3_ordinal(a) - e4m3_ordinal(b))


def bf16_as_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)
