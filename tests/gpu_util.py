"""Helpers for the GPU parity tests (host <-> device conversions, tolerances)."""
import numpy as np
import torch


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def to_host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def as_f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits; subnormal floor 2^-133)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.maximum(2.0 ** (e - 7), 2.0 ** -133)


def assert_psum(got: np.ndarray, ref64: np.ndarray, abs_sum: np.ndarray, what: str = "") -> None:
    """Partial-sum tolerance. float32: |got - ref| <= 1e-6 * sum_i |x_i| (a
    condition-aware relative bound; 8 sequential float32 additions stay below
    7 * 2^-24 of it). bf16: within one bf16 spacing of the exact sum."""
    g = as_f64(got)
    if got.dtype == np.uint16:
        bad = np.abs(g - ref64) > bf16_ulp(ref64)
    else:
        bad = np.abs(g - ref64) > 1e-6 * abs_sum
    if bad.any():
        i = np.flatnonzero(bad.reshape(-1))[0]
        raise AssertionError("%s: %d elements outside the bound; first at %d: got %r, exact %r, sum|x| %r"
                             % (what, bad.sum(), i, g.reshape(-1)[i], ref64.reshape(-1)[i], abs_sum.reshape(-1)[i]))


GUARD_BYTES = 4096
POISON = 0xA5


class Guarded:
    """Output buffers, each inside a larger device buffer whose bytes just
    before and just after it are poisoned (0xA5). A kernel that writes past a
    buffer's end, or before its start, changes a guard byte; check() finds it.
    compute-sanitizer does not run on these GPUs, so this is how the parity
    tests see out-of-bounds writes that no comparison would read. The buffers
    start 4096 bytes into their allocation (256-byte aligned, as cudaMalloc's
    are) and their own bytes start poisoned too."""

    def __init__(self):
        self.items = []

    def empty(self, shape, dtype, name="out"):
        shape = tuple(int(s) for s in shape)
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((GUARD_BYTES + n + GUARD_BYTES,), POISON, dtype=torch.uint8, device="cuda")
        view = raw[GUARD_BYTES:GUARD_BYTES + n].view(dtype).view(shape)
        self.items.append((raw, n, "%s%s" % (name, shape)))
        return view

    def many(self, shapes, dtype, name="out"):
        return [self.empty(s, dtype, "%s[%d]" % (name, i)) for i, s in enumerate(shapes)]

    def check(self, what=""):
        torch.cuda.synchronize()
        for raw, n, name in self.items:
            for side, part in (("before", raw[:GUARD_BYTES]), ("after", raw[GUARD_BYTES + n:])):
                bad = torch.nonzero(part != POISON)
                if bad.numel():
                    off = int(bad[0]) - (GUARD_BYTES if side == "before" else 0)
                    raise AssertionError("%s: %d guard bytes %s %s changed (first at byte %d %s it)"
                                         % (what, bad.numel(), side, name, off, side))
