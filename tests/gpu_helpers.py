"""Helpers for the GPU parity tests: run the CUDA library and the CPU oracle on
the same inputs and compare element by element (bit patterns).

Output buffers handed to the library are views of larger buffers filled with
a poison byte; the bytes past the view (canaries) must come back untouched, so
an out-of-bounds write fails the test.
"""
import numpy as np
import torch

POISON = 0xA5
PAD = 256  # canary bytes after every output


class Poisoned:
    """A CUDA output buffer of `numel` elements followed by PAD canary bytes."""

    def __init__(self, numel, dtype, device="cuda"):
        esize = torch.empty(0, dtype=dtype).element_size()
        nbytes = numel * esize
        total = (nbytes + PAD + 31) // 32 * 32
        self.raw = torch.full((total,), POISON, dtype=torch.uint8, device=device)
        self.nbytes = nbytes
        self.t = self.raw[:nbytes].view(dtype) if numel else torch.empty(0, dtype=dtype, device=device)

    def canary_ok(self):
        tail = self.raw[self.nbytes:].cpu().numpy()
        return bool(np.all(tail == POISON))


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a tensor as an unsigned numpy array."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.int32:
        return t.numpy().view(np.uint32)
    if t.dtype in (torch.int8, torch.uint8):
        return t.numpy().view(np.uint8)
    raise TypeError(t.dtype)


def oracle_input(x: torch.Tensor) -> np.ndarray:
    """CPU view the oracle reads: float32 values or bf16 bit patterns."""
    x = x.detach().cpu().contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    return x.numpy().reshape(-1)


def first_diff(a: np.ndarray, b: np.ndarray) -> str:
    a = np.asarray(a).reshape(-1)
    b = np.asarray(b).reshape(-1)
    if a.shape != b.shape:
        return f"shape {a.shape} vs {b.shape}"
    d = np.nonzero(a != b)[0]
    if d.size == 0:
        return "equal"
    i = d[0]
    return f"{d.size} differ, first at {i}: {a[i]!r} vs {b[i]!r}"


def obits(a: np.ndarray) -> np.ndarray:
    """Bit patterns of an oracle output (float32 viewed as uint32)."""
    a = np.ascontiguousarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a


def assert_same(gpu: np.ndarray, ref: np.ndarray, what: str):
    gpu = obits(np.asarray(gpu)).reshape(-1)
    ref = obits(np.asarray(ref)).reshape(-1)
    assert gpu.shape == ref.shape and np.array_equal(gpu, ref), f"{what}: {first_diff(gpu, ref)}"
