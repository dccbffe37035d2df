"""Thin ctypes binding of libmq.so (include/mq.h), with the same entry-point names.

Argument marshalling only: torch tensors are checked for device, dtype and
contiguity, their data pointers and the current CUDA stream are passed to the
C ABI, and a non-zero status raises MQError. Every step of the computation
runs in the library's CUDA kernels; there is no other code path. If the
library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmq.so")

MQ_OK, MQ_ERR_NULL, MQ_ERR_SHAPE, MQ_ERR_ALIGN, MQ_ERR_ARCH, MQ_ERR_LAUNCH, MQ_ERR_DEVICE, MQ_ERR_SCRATCH = range(8)
MQ_GEMV_MAX_ROWS = 8   # include/mq.h

EXPORTED = ["mq_plane_bytes", "mq_q4k_row_bytes", "mq_q6k_row_bytes", "mq_q6k_packed_row_bytes", "mq_prepack_q6k",
            "mq_quantize_q8", "mq_rms_quant",
            "mq_swiglu_quant", "mq_gemm_q4k", "mq_gemm_q6k", "mq_gemv_q4k", "mq_gemv_q6k",
            "mq_q5k_row_bytes", "mq_q4_0_row_bytes", "mq_q4_1_row_bytes", "mq_gemv_q5k", "mq_gemv_q4_0",
            "mq_gemv_q4_1", "mq_gemm_q4_0", "mq_gemm_q4_1", "mq_gemv_q6k_packed", "mq_gemm_q6k_static", "mq_gemm_q4k_pair",
            "mq_device_status", "mq_status_str"]


class MQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} (status {status})")


class CPlane(ctypes.Structure):
    _fields_ = [("qs", ctypes.c_void_p), ("d", ctypes.c_void_p), ("s", ctypes.c_void_p),
                ("ah", ctypes.c_void_p), ("ax", ctypes.c_void_p), ("af", ctypes.c_void_p),
                ("M", ctypes.c_int), ("K", ctypes.c_int)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        pp = ctypes.POINTER(CPlane)
        psz = ctypes.POINTER(ctypes.c_size_t)
        sig = {
            "mq_plane_bytes": (sz, [i, i, psz, psz, psz, psz, psz, psz]),
            "mq_q4k_row_bytes": (sz, [i]),
            "mq_q6k_row_bytes": (sz, [i]),
            "mq_q6k_packed_row_bytes": (sz, [i]),
            "mq_prepack_q6k": (i, [vp, i, i, vp, vp]),
            "mq_quantize_q8": (i, [vp, i, i, pp, vp]),
            "mq_rms_quant": (i, [vp, vp, i, i, f, pp, vp]),
            "mq_swiglu_quant": (i, [vp, vp, i, i, pp, vp]),
            "mq_gemm_q4k": (i, [pp, vp, i, vp, vp]),
            "mq_gemm_q6k": (i, [pp, vp, i, vp, vp]),
            "mq_gemv_q4k": (i, [pp, vp, i, vp, vp]),
            "mq_gemv_q6k": (i, [pp, vp, i, vp, vp]),
            "mq_gemv_q6k_packed": (i, [pp, vp, i, vp, vp]),
            "mq_gemm_q6k_static": (i, [pp, vp, i, vp, vp]),
            "mq_gemm_q4k_pair": (i, [pp, vp, i, vp, vp, i, vp, vp]),
            "mq_q5k_row_bytes": (sz, [i]),
            "mq_q4_0_row_bytes": (sz, [i]),
            "mq_q4_1_row_bytes": (sz, [i]),
            "mq_gemv_q5k": (i, [pp, vp, i, vp, vp]),
            "mq_gemv_q4_0": (i, [pp, vp, i, vp, vp]),
            "mq_gemv_q4_1": (i, [pp, vp, i, vp, vp]),
            "mq_gemm_q4_0": (i, [pp, vp, i, vp, vp]),
            "mq_gemm_q4_1": (i, [pp, vp, i, vp, vp]),
            "mq_device_status": (i, [vp]),
            "mq_status_str": (ctypes.c_char_p, [i]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().mq_status_str(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status: int, where: str):
    if status != MQ_OK:
        raise MQError(status, where)


def _dev_tensor(t, dtype, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


class Plane:
    """Device activation plane (include/mq.h): the q8 arrays qs int8 [M, K],
    d f32 [M, K/32], s int32 [M, K/32] (read by the GEMV), and/or the GEMM's
    operand arrays ah f16 [M, K], ax f16 [M, K/256, 16], af f32 [K/256, Mp]
    with Mp = M rounded up to a multiple of 4. Producers fill whichever groups
    are present."""

    def __init__(self, qs=None, d=None, s=None, ah=None, ax=None, af=None, M=None, K=None):
        self.qs, self.d, self.s, self.ah, self.ax, self.af = qs, d, s, ah, ax, af
        ref = qs if qs is not None else ah
        if ref is None:
            raise ValueError("a plane needs its q8 arrays, its operand arrays, or both")
        self.M, self.K = int(ref.shape[0]), int(ref.shape[1])
        if qs is not None:
            _dev_tensor(qs, torch.int8, "plane.qs")
            _dev_tensor(d, torch.float32, "plane.d")
            _dev_tensor(s, torch.int32, "plane.s")
        if ah is not None:
            _dev_tensor(ah, torch.float16, "plane.ah")
            _dev_tensor(ax, torch.float16, "plane.ax")
            _dev_tensor(af, torch.float32, "plane.af")

    @staticmethod
    def af_stride(M: int) -> int:
        return (M + 3) // 4 * 4

    @classmethod
    def empty(cls, M: int, K: int, device="cuda", q8: bool = True, op: bool = True) -> "Plane":
        """Allocate a plane with the q8 arrays (q8=True) and/or the operand arrays (op=True)."""
        kw = {}
        if q8:
            kw.update(qs=torch.empty((M, K), dtype=torch.int8, device=device),
                      d=torch.empty((M, K // 32), dtype=torch.float32, device=device),
                      s=torch.empty((M, K // 32), dtype=torch.int32, device=device))
        if op:
            kw.update(ah=torch.empty((M, K), dtype=torch.float16, device=device),
                      ax=torch.empty((M, K // 256, 16), dtype=torch.float16, device=device),
                      af=torch.empty((K // 256, cls.af_stride(M)), dtype=torch.float32, device=device))
        return cls(**kw)

    def c(self) -> CPlane:
        def p(t):
            return t.data_ptr() if t is not None else None
        return CPlane(p(self.qs), p(self.d), p(self.s), p(self.ah), p(self.ax), p(self.af), self.M, self.K)


def mq_plane_bytes(M: int, K: int):
    """(total, qs, d, s, ah, ax, af) bytes of an M x K plane."""
    v = [ctypes.c_size_t() for _ in range(6)]
    tot = lib().mq_plane_bytes(M, K, *[ctypes.byref(x) for x in v])
    return (int(tot),) + tuple(int(x.value) for x in v)


def mq_q4k_row_bytes(K: int) -> int:
    return int(lib().mq_q4k_row_bytes(K))


def mq_q6k_row_bytes(K: int) -> int:
    return int(lib().mq_q6k_row_bytes(K))


def mq_q6k_packed_row_bytes(K: int) -> int:
    return int(lib().mq_q6k_packed_row_bytes(K))


def mq_prepack_q6k(w: torch.Tensor, N: int, K: int, out: torch.Tensor = None, stream=None) -> torch.Tensor:
    """Raw q6_K rows [N, K/256*210] (uint8) -> the prepacked layout [N, K/256*224] the GEMM reads."""
    _dev_tensor(w, torch.uint8, "w")
    if out is None:
        out = torch.empty((N, mq_q6k_packed_row_bytes(K)), dtype=torch.uint8, device=w.device)
    _dev_tensor(out, torch.uint8, "out")
    _check(lib().mq_prepack_q6k(_ptr(w), int(N), int(K), _ptr(out), _stream(stream)), "mq_prepack_q6k")
    return out


def mq_quantize_q8(x: torch.Tensor, out: Plane, stream=None) -> Plane:
    _dev_tensor(x, torch.float32, "x")
    cp = out.c()
    _check(lib().mq_quantize_q8(_ptr(x), x.shape[0], x.shape[1], ctypes.byref(cp), _stream(stream)),
           "mq_quantize_q8")
    return out


def mq_rms_quant(x: torch.Tensor, w: torch.Tensor, eps: float, out: Plane, stream=None) -> Plane:
    _dev_tensor(x, torch.float32, "x")
    _dev_tensor(w, torch.float32, "w")
    cp = out.c()
    _check(lib().mq_rms_quant(_ptr(x), _ptr(w), x.shape[0], x.shape[1], float(eps), ctypes.byref(cp),
                              _stream(stream)), "mq_rms_quant")
    return out


def mq_swiglu_quant(g: torch.Tensor, u: torch.Tensor, out: Plane, stream=None) -> Plane:
    _dev_tensor(g, torch.float32, "g")
    _dev_tensor(u, torch.float32, "u")
    if g.shape != u.shape:
        raise ValueError("g and u must have the same shape")
    cp = out.c()
    _check(lib().mq_swiglu_quant(_ptr(g), _ptr(u), g.shape[0], g.shape[1], ctypes.byref(cp), _stream(stream)),
           "mq_swiglu_quant")
    return out


def _matmul(fn_name: str, a: Plane, w: torch.Tensor, N: int, out: torch.Tensor, stream):
    _dev_tensor(w, torch.uint8, "w")
    _dev_tensor(out, torch.float32, "out")
    if out.numel() < a.M * N:
        raise ValueError(f"{fn_name}: out holds {out.numel()} floats, needs M * N = {a.M * N}")
    cp = a.c()
    _check(getattr(lib(), fn_name)(ctypes.byref(cp), _ptr(w), int(N), _ptr(out), _stream(stream)), fn_name)
    return out


def mq_gemm_q4k(a: Plane, w: torch.Tensor, N: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    return _matmul("mq_gemm_q4k", a, w, N, out, stream)


def mq_gemm_q6k(a: Plane, w: torch.Tensor, N: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    return _matmul("mq_gemm_q6k", a, w, N, out, stream)


def mq_gemv_q4k(a: Plane, w: torch.Tensor, N: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    return _matmul("mq_gemv_q4k", a, w, N, out, stream)


def mq_gemv_q6k(a: Plane, w: torch.Tensor, N: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    return _matmul("mq_gemv_q6k", a, w, N, out, stream)


def mq_gemv_q6k_packed(a: Plane, w: torch.Tensor, N: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    """q6_K GEMV on prepacked rows (mq_prepack_q6k), the form the GEMM reads too."""
    return _matmul("mq_gemv_q6k_packed", a, w, N, out, stream)


def mq_gemm_q4k_pair(a: Plane, w0: torch.Tensor, N0: int, out0: torch.Tensor, w1: torch.Tensor, N1: int,
                     out1: torch.Tensor, stream=None):
    """Two q4_K GEMMs on one plane (include/mq.h): out0 = a x w0, out1 = a x w1, in one launch
    where that pays."""
    for t, n in ((w0, "w0"), (w1, "w1")):
        _dev_tensor(t, torch.uint8, n)
    for t, n, N in ((out0, "out0", N0), (out1, "out1", N1)):
        _dev_tensor(t, torch.float32, n)
        if t.numel() < a.M * N:
            raise ValueError(f"mq_gemm_q4k_pair: {n} holds {t.numel()} floats, needs M * N = {a.M * N}")
    cp = a.c()
    _check(lib().mq_gemm_q4k_pair(ctypes.byref(cp), _ptr(w0), int(N0), _ptr(out0), _ptr(w1), int(N1), _ptr(out1),
                                  _stream(stream)), "mq_gemm_q4k_pair")
    return out0, out1


def mq_gemm_q6k_static(a: Plane, w: torch.Tensor, N: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    """mq_gemm_q6k for callers that cannot have device memory allocated for them: its scratch is
    a fixed array inside the library (see include/mq.h)."""
    return _matmul("mq_gemm_q6k_static", a, w, N, out, stream)


def mq_gemm_q4_0(a: Plane, w: torch.Tensor, N: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    return _matmul("mq_gemm_q4_0", a, w, N, out, stream)


def mq_gemm_q4_1(a: Plane, w: torch.Tensor, N: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    return _matmul("mq_gemm_q4_1", a, w, N, out, stream)


def mq_gemv_q5k(a: Plane, w: torch.Tensor, N: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    return _matmul("mq_gemv_q5k", a, w, N, out, stream)


def mq_gemv_q4_0(a: Plane, w: torch.Tensor, N: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    return _matmul("mq_gemv_q4_0", a, w, N, out, stream)


def mq_gemv_q4_1(a: Plane, w: torch.Tensor, N: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    return _matmul("mq_gemv_q4_1", a, w, N, out, stream)


def mq_q5k_row_bytes(K: int) -> int:
    return int(lib().mq_q5k_row_bytes(K))


def mq_q4_0_row_bytes(K: int) -> int:
    return int(lib().mq_q4_0_row_bytes(K))


def mq_q4_1_row_bytes(K: int) -> int:
    return int(lib().mq_q4_1_row_bytes(K))


def mq_device_status(stream=None) -> int:
    return int(lib().mq_device_status(_stream(stream)))


def gemm_weights(kind: str, w: torch.Tensor, N: int, K: int, stream=None) -> torch.Tensor:
    """The weight form the GEMM reads: q6_K rows prepacked, every other type as it is."""
    return mq_prepack_q6k(w, N, K, stream=stream) if kind == "q6k" else w


def gemm(kind: str, a: Plane, w: torch.Tensor, N: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    return {"q4k": mq_gemm_q4k, "q6k": mq_gemm_q6k, "q4_0": mq_gemm_q4_0, "q4_1": mq_gemm_q4_1}[kind](a, w, N, out,
                                                                                                 stream)


def gemv(kind: str, a: Plane, w: torch.Tensor, N: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    return {"q4k": mq_gemv_q4k, "q6k": mq_gemv_q6k, "q5k": mq_gemv_q5k, "q4_0": mq_gemv_q4_0,
            "q4_1": mq_gemv_q4_1}[kind](a, w, N, out, stream)
