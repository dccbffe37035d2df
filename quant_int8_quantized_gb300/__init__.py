"""GB300-native block-quantized matmul hot path: q8 activation planes, fused
RMSNorm/SwiGLU producers, q4_K/q6_K prefill GEMM and decode GEMV.

The compute lives in libmq.so (C ABI, include/mq.h); `mq` is its ctypes
binding and `synth` the seeded synthetic-input generator.
"""
from . import synth  # noqa: F401

__all__ = ["synth", "mq", "build"]
