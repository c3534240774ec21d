"""Shared test utilities: bit views, guard-banded device buffers, MXFP8 operand setup."""
import numpy as np
import torch

GUARD = 256          # bytes of canary before and after every guarded output
CANARY = 0xA5


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().numpy()


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class Guarded:
    """A device byte buffer with canary bands on both sides of the payload."""

    def __init__(self, nbytes: int, device="cuda"):
        self.n = int(nbytes)
        self.buf = torch.full((self.n + 2 * GUARD,), CANARY, dtype=torch.uint8, device=device)
        self.body = self.buf[GUARD:GUARD + self.n]

    def view(self, dtype=torch.uint8, shape=None):
        t = self.body.view(dtype)
        return t.view(shape) if shape is not None else t

    def intact(self) -> bool:
        b = self.buf.cpu()
        return bool((b[:GUARD] == CANARY).all()) and bool((b[GUARD + self.n:] == CANARY).all())


def rel_fro(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """ulp of the bf16 binade that holds |v| (subnormal floor 2^-133)."""
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.ldexp(1.0, (np.maximum(e, -126) - 7).astype(np.int64))
