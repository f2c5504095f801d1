"""Helpers shared by the GPU parity tests: storage <-> torch, tile-wise error, device pools."""
import numpy as np

from recurrent_state_update_gb300 import workloads as wl


def torch_dtype(dtype):
    import torch
    return {wl.F32: torch.float32, wl.BF16: torch.bfloat16}[dtype]


def to_dev(stored, dtype, device="cuda"):
    """numpy storage (float32, or uint16 bf16 bits) -> CUDA tensor of that dtype."""
    import torch
    if stored is None:
        return None
    a = np.ascontiguousarray(stored)
    if dtype == wl.BF16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a.astype(np.float32)).to(device)


def to_i32(a, device="cuda"):
    import torch
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def f64(t):
    """Exact float64 copy of a CUDA/CPU float tensor (bf16 and fp32 upcast exactly)."""
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def tile_rel_err(got, ref, tile_axes):
    """max over tiles of max|got-ref| / max|ref| (tile = the trailing ``tile_axes`` axes)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    axes = tuple(range(got.ndim - tile_axes, got.ndim))
    num = np.abs(got - ref).max(axis=axes)
    den = np.abs(ref).max(axis=axes)
    den = np.where(den == 0, 1.0, den)
    return float((num / den).max())


def device_normal_pool(shape, dtype, seed, std=0.1, device="cuda"):
    """Seeded N(0, std^2) pool generated on the device (for pools too large to draw on the host)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = torch.empty(shape, dtype=torch_dtype(dtype), device=device)
    flat = t.view(shape[0], -1)
    for s0 in range(0, shape[0], 64):
        blk = torch.randn(flat[s0:s0 + 64].shape, generator=g, device=device, dtype=torch.float32)
        flat[s0:s0 + 64].copy_(blk.mul_(std))
    return t


def tile_rms_err(got, ref, tile_axes):
    """max over tiles of ||got-ref||_2 / ||ref||_2 (tile = the trailing ``tile_axes`` axes)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    axes = tuple(range(got.ndim - tile_axes, got.ndim))
    num = np.sqrt(((got - ref) ** 2).sum(axis=axes))
    den = np.sqrt((ref ** 2).sum(axis=axes))
    den = np.where(den == 0, 1.0, den)
    return float((num / den).max())


GUARD_BYTES = 4096  # per side; a multiple of 256 so the guarded tensor keeps its alignment
GUARD_BYTE = 0x5A


class Guarded:
    """A device tensor placed between two guard zones of GUARD_BYTES bytes each, filled with
    GUARD_BYTE: after a library call, check() compares every guard byte exactly, so a write that
    runs off either end of a pool or an output (one vector past the last slot or row) fails."""

    def __init__(self, t):
        import torch
        nbytes = t.numel() * t.element_size()
        self.raw = torch.full((GUARD_BYTES + nbytes + GUARD_BYTES,), GUARD_BYTE, dtype=torch.uint8, device=t.device)
        inner = self.raw[GUARD_BYTES:GUARD_BYTES + nbytes].view(t.dtype).view(t.shape)
        inner.copy_(t)
        self.t = inner
        self.nbytes = nbytes

    def check(self, what=""):
        import torch
        lo = self.raw[:GUARD_BYTES]
        hi = self.raw[GUARD_BYTES + self.nbytes:]
        assert bool((lo == GUARD_BYTE).all()), f"guard bytes before {what} were written"
        assert bool((hi == GUARD_BYTE).all()), f"guard bytes after {what} were written"
        torch.cuda.synchronize()


def guarded(t):
    """Copy of device tensor t inside guard zones; returns the Guarded holder (use .t)."""
    return Guarded(t)
