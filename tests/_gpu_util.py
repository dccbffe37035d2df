"""Helpers for the GPU parity tests: guarded, poisoned device buffers and
plane comparisons against the CPU oracle."""
import numpy as np
import pytest
import torch

from quant_int8_quantized_gb300 import mq

POISON = 0xCD
GUARD = 256   # bytes of guard band on each side of a buffer


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from quant_int8_quantized_gb300 import build as B
    B.build()
    mq.lib()


class Guarded:
    """A device tensor carved out of a larger poisoned byte buffer.

    Every byte of the buffer starts as 0xCD; `check()` asserts that the guard
    bands before and after the tensor are untouched (no out-of-bounds write),
    and `untouched()` counts tensor bytes still equal to the poison (no write).
    """

    def __init__(self, shape, dtype, device="cuda"):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.nbytes = n
        self.raw = torch.full((n + 2 * GUARD,), POISON, dtype=torch.uint8, device=device)
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(shape) if n else torch.empty(shape, dtype=dtype, device=device)

    def check(self):
        raw = self.raw.cpu().numpy()
        assert np.all(raw[:GUARD] == POISON), "write before the buffer"
        assert np.all(raw[GUARD + self.nbytes:] == POISON), "write after the buffer"

    def untouched(self):
        """Number of 4-byte words of the tensor still equal to the poison (never written).
        For f32 outputs the poison word is -4.3e8, not a value these kernels produce."""
        words = self.raw[GUARD:GUARD + self.nbytes - self.nbytes % 4].view(torch.int32)
        poison = int(np.frombuffer(bytes([POISON] * 4), np.int32)[0])
        return int((words == poison).sum().item())


class GuardedPlane:
    def __init__(self, M, K, f16=True):
        self.g = [Guarded((M, K), torch.int8), Guarded((M, K // 32), torch.float32),
                  Guarded((M, K // 32), torch.int32)]
        if f16:
            self.g.append(Guarded((M, K), torch.float16))
        self.plane = mq.Plane(self.g[0].t, self.g[1].t, self.g[2].t, self.g[3].t if f16 else None)

    def check(self):
        for g in self.g:
            g.check()
        if self.plane.qh is not None:   # the f16 copy holds exactly the int8 quants
            qs = self.plane.qs.cpu().numpy().astype(np.float32)
            assert np.array_equal(self.plane.qh.cpu().numpy().astype(np.float32), qs), "qh != qs"

    def numpy(self):
        return (self.plane.qs.cpu().numpy(), self.plane.d.cpu().numpy(), self.plane.s.cpu().numpy())


def assert_plane_equal(got, ref, what=""):
    qs, d, s = got
    rq, rd, rs = ref
    assert qs.shape == rq.shape and d.shape == rd.shape
    bad = np.argwhere(qs != rq)
    assert bad.size == 0, f"{what}: {len(bad)} qs mismatches, first at {bad[:5].tolist()}"
    assert np.array_equal(d.view(np.uint32), rd.view(np.uint32)), f"{what}: d differs"
    assert np.array_equal(s, rs), f"{what}: s differs"
