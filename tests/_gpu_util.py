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

    Every byte of the buffer starts as the poison (0xCD; 0xFF for binary16
    tensors, whose 0xCDCD is an ordinary value but 0xFFFF a NaN the kernels never
    write); `check()` asserts that the guard bands before and after the tensor
    are untouched (no out-of-bounds write), and `untouched()` counts 4-byte words
    of the tensor still equal to the poison (no write).
    """

    def __init__(self, shape, dtype, device="cuda"):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.nbytes = n
        self.poison = 0xFF if dtype == torch.float16 else POISON
        self.raw = torch.full((n + 2 * GUARD,), self.poison, dtype=torch.uint8, device=device)
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(shape) if n else torch.empty(shape, dtype=dtype, device=device)

    def check(self):
        raw = self.raw.cpu().numpy()
        assert np.all(raw[:GUARD] == self.poison), "write before the buffer"
        assert np.all(raw[GUARD + self.nbytes:] == self.poison), "write after the buffer"

    def untouched(self):
        """Number of 4-byte words of the tensor still equal to the poison (never written).
        For f32 outputs the poison word is -4.3e8, not a value these kernels produce."""
        words = self.raw[GUARD:GUARD + self.nbytes - self.nbytes % 4].view(torch.int32)
        poison = int(np.frombuffer(bytes([self.poison] * 4), np.int32)[0])
        return int((words == poison).sum().item())


class GuardedPlane:
    """A plane whose arrays are all Guarded: the q8 arrays (q8=True) and/or the GEMM
    operand arrays (op=True)."""

    def __init__(self, M, K, q8=True, op=True):
        self.M, self.K = M, K
        self.g = {}
        if q8:
            self.g.update(qs=Guarded((M, K), torch.int8), d=Guarded((M, K // 32), torch.float32),
                          s=Guarded((M, K // 32), torch.int32))
        if op:
            self.g.update(ah=Guarded((M, K), torch.float16), ax=Guarded((M, K // 256, 16), torch.float16),
                          af=Guarded((K // 256, mq.Plane.af_stride(M)), torch.float32))
        self.plane = mq.Plane(**{k: v.t for k, v in self.g.items()})

    def check(self, ref=None):
        """Guard bands intact; with both groups, the operand arrays equal the oracle's
        operand form of this plane's own q8 arrays; with `ref` = (qs, d) from the oracle,
        they equal the operand form of that plane."""
        for g in self.g.values():
            g.check()
        if "ah" not in self.g:
            return
        if ref is None:
            if "qs" not in self.g:
                return
            ref = (self.plane.qs.cpu().numpy(), self.plane.d.cpu().numpy())
        assert_operand_form(self.plane, ref[0], ref[1])

    def numpy(self):
        return (self.plane.qs.cpu().numpy(), self.plane.d.cpu().numpy(), self.plane.s.cpu().numpy())


def assert_operand_form(plane, qs, d, rows=None, what="operand form"):
    """ah, ax and af of the device plane (rows `rows`, default all) equal, bit for bit, the
    oracle's operand form of the q8 plane (qs, d) (given for those rows)."""
    from oracle import mq_oracle as O
    ah, ax, af = O.operand_form(qs, d)
    idx = None if rows is None else torch.as_tensor(np.asarray(rows), device=plane.ah.device)
    gah = (plane.ah if idx is None else plane.ah[idx]).cpu().numpy()
    gax = (plane.ax if idx is None else plane.ax[idx]).cpu().numpy()
    gaf = plane.af.cpu().numpy()
    gaf = gaf[:, :plane.M] if rows is None else gaf[:, np.asarray(rows)]
    bad = np.argwhere(gah.view(np.uint16) != ah.view(np.uint16))
    assert bad.size == 0, f"{what}: {len(bad)} ah mismatches, first at {bad[:5].tolist()}"
    assert np.array_equal(gax.view(np.uint16), ax.view(np.uint16)), f"{what}: ax differs"
    assert np.array_equal(gaf.view(np.uint32), af.view(np.uint32)), f"{what}: af differs"


def assert_plane_equal(got, ref, what=""):
    qs, d, s = got
    rq, rd, rs = ref
    assert qs.shape == rq.shape and d.shape == rd.shape
    bad = np.argwhere(qs != rq)
    assert bad.size == 0, f"{what}: {len(bad)} qs mismatches, first at {bad[:5].tolist()}"
    assert np.array_equal(d.view(np.uint32), rd.view(np.uint32)), f"{what}: d differs"
    assert np.array_equal(s, rs), f"{what}: s differs"
