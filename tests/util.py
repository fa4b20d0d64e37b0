"""Comparison helpers shared by the GPU parity tests."""
import numpy as np
import torch


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


# Tolerances (rel-L2 per tensor): float32 path 1e-4 everywhere; bf16 storage
# with float32 accumulation 1e-2 on outputs and 2e-2 on gradients; CE loss
# absolute error 1e-3.
TOL = {"f32": (1e-4, 1e-4), "bf16": (1e-2, 2e-2)}
CE_LOSS_ABS = 1e-3


class Guarded:
    """Out-of-bounds write detection (compute-sanitizer is not available):
    tensors placed inside one larger allocation between two guard regions of
    `guard` bytes filled with a byte pattern. `check()` asserts that no guard
    byte changed, i.e. no kernel wrote before the start or past the end of any
    of the tensors handed out. Views start 256-byte aligned (as the library's
    16-byte rule needs)."""

    PATTERN = 0xA7

    def __init__(self, guard: int = 4096):
        self.guard = guard
        self.bufs = []

    def empty(self, shape, dtype, fill=None):
        es = torch.empty((), dtype=dtype).element_size()
        n = 1
        for s in shape:
            n *= s
        body = (n * es + 255) // 256 * 256
        raw = torch.full((self.guard + body + self.guard,), self.PATTERN, dtype=torch.uint8,
                         device="cuda")
        view = raw[self.guard:self.guard + n * es].view(dtype).view(*shape)
        if fill is not None:
            view.fill_(fill)
        self.bufs.append((raw, n * es))
        return view

    def like(self, t: torch.Tensor, fill=None):
        return self.empty(tuple(t.shape), t.dtype, fill)

    def check(self):
        torch.cuda.synchronize()
        for i, (raw, nbytes) in enumerate(self.bufs):
            head = raw[:self.guard]
            tail = raw[self.guard + nbytes:]
            bad_h = int((head != self.PATTERN).sum())
            bad_t = int((tail != self.PATTERN).sum())
            assert bad_h == 0 and bad_t == 0, f"buffer {i}: {bad_h} bytes before, {bad_t} after it changed"
