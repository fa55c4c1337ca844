"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
from __future__ import annotations

import numpy as np
import torch

# Float tolerance for y against the fp64 oracle: relative L2 error and max
# absolute error relative to the rms of the reference.
REL_L2 = 2e-3
MAX_ABS_RMS = 1e-2


def check_y(got: np.ndarray, ref: np.ndarray, what: str = "y") -> tuple[float, float]:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    nref = np.linalg.norm(ref)
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    if nref == 0.0:
        assert np.max(np.abs(got)) == 0.0, f"{what}: expected exact zeros"
        return 0.0, 0.0
    rel = float(np.linalg.norm(got - ref) / nref)
    mx = float(np.max(np.abs(got - ref)) / rms)
    assert rel <= REL_L2, f"{what}: relative L2 error {rel:.3e} > {REL_L2}"
    assert mx <= MAX_ABS_RMS, f"{what}: max abs error {mx:.3e} * rms > {MAX_ABS_RMS}"
    return rel, mx


def to_dev_bf16(bits: np.ndarray, dev="cuda") -> torch.Tensor:
    """uint16 bf16 bits (numpy) -> CUDA bfloat16 tensor with the same bits."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(dev).view(torch.bfloat16)


def to_dev_f32(a: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


def u16(t: torch.Tensor) -> np.ndarray:
    """Bit patterns of a 16-bit CUDA tensor as a numpy uint16 array."""
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def guarded(shape, dtype, dev="cuda", pad_bytes=4096, poison=0x5A):
    """A tensor view with poisoned guard bytes on both sides; returns
    (view, check) where check() asserts the guards are intact."""
    esize = torch.tensor([], dtype=dtype).element_size()
    n = int(np.prod(shape))
    pad = pad_bytes // esize
    raw = torch.empty(n + 2 * pad, dtype=dtype, device=dev)
    raw.view(torch.uint8).fill_(poison)
    view = raw[pad:pad + n].view(*shape)

    def check():
        b = raw.view(torch.uint8)
        pb = pad * esize
        head = b[:pb].cpu().numpy()
        tail = b[pb + n * esize:].cpu().numpy()
        assert np.all(head == poison) and np.all(tail == poison), "write outside the output buffer"

    return view, check
