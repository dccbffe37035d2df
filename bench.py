"""Benchmark of the block-quantized matmul hot path on one GB300 (or N replicas).

Step = one pass of the 7B-shaped full matmul stack at M = 3314 tokens:
28 layers of {RMSNorm->q8 plane; Q, K (q4_K), V (q6_K) GEMMs; attention
stand-in -> q8 plane (standalone quantize); O (q4_K) GEMM; RMSNorm->q8 plane;
gate, up (q4_K) GEMMs; SwiGLU->q8 plane; down (q6_K) GEMM}, then RMSNorm->q8 of
the last token and the q6_K lm_head GEMV (152064 x 3584). Weights are distinct
per layer (4.6 GB in total, far above the 129 MB L2, so every step streams
them from HBM). value = tokens/s = 3314 / step time.

Also measured in the same run (separately timed):
  * decode: the 14B-shaped 48-layer M = 1 sweep (rms->q8, attn_q/k/v/o,
    gate/up GEMVs, SwiGLU->q8, down GEMV; k|v and gate|up stored stacked and
    run as one GEMV each; the k|v GEMV on a second stream beside attn_q, both
    reading the rms plane), GB/s of algorithmic bytes;
  * e2e: the same prefill step with its inputs copied from pinned host memory
    and the logits copied back inside the timed region;
  * roofline: the q4_K GEMM launches (the dominant kernel), timed with CUDA
    events on their stream, against the measured f16/bf16 tensor peak;
  * cpu_baseline: the CPU oracle on a bounded sample of the same workload.

`--impl reference` times the CPU oracle alone (the reference arm).
Multi-GPU: replicas only (one process per GPU, each its own full workload).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M_TOK = 3314
HID, FFN, KVD, VOCAB, LAYERS = 3584, 18944, 512, 152064, 28
D_HID, D_FFN, D_KV, D_LAYERS = 5120, 13824, 1024, 48
EPS = 1e-6
METRIC = "prefill effective int8 TOPS & tok/s (7B-shaped stack, M=3314); decode GEMV GB/s"

# (name, kind, N, K, input) per layer; input: "rms" (rms plane), "attn" (stand-in plane), "swiglu"
PREFILL_MATS = [("q", "q4k", HID, HID, "rms"), ("k", "q4k", KVD, HID, "rms"), ("v", "q6k", KVD, HID, "rms"),
                ("o", "q4k", HID, HID, "attn"), ("gate", "q4k", FFN, HID, "rms2"), ("up", "q4k", FFN, HID, "rms2"),
                ("down", "q6k", HID, FFN, "swiglu")]
DECODE_MATS = [("q", "q4k", D_HID, D_HID), ("k", "q6k", D_KV, D_HID), ("v", "q6k", D_KV, D_HID),
               ("o", "q4k", D_HID, D_HID), ("gate", "q4k", D_FFN, D_HID), ("up", "q4k", D_FFN, D_HID),
               ("down", "q6k", D_HID, D_FFN)]
# Decode storage: projections that read the same plane and share a quant type are stored as one
# stacked matrix and run as one GEMV (k|v, gate|up); the rows, bytes and products are the same.
DECODE_STACKS = [("q", ("q",)), ("kv", ("k", "v")), ("o", ("o",)), ("gate_up", ("gate", "up")), ("down", ("down",))]
BYTES_PER_SB = {"q4k": 144, "q6k": 210, "q5k": 176, "q4_0": 8 * 18, "q4_1": 8 * 20}   # bytes per 256 weights

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one gemm_kernel<q4_K> launch at
# 3314 x 18944 x 3584, from one ncu capture (summary under profiles/). It describes the device code
# with these SHA-256 digests (gemm.cu up to its host-side section, and tc.cuh) and is reported as
# null once either changes.
GEMM_Q4K_TRAFFIC = {"bytes": 67058432 + 204712960,
                    "sha256": {"gemm.cu": "c5a12fc9c911e518b926dfbcfb3fc2ecbb646a65af2637e6ff5c2390560f8581",
                               "tc.cuh": "77627d374b6dc4619249b40701e93050c782a7d46494b273d5b7a343462067e1"}}
HOST_SECTION = b"// ------------------------------------------------------------------ host side"


def device_code_digest(fn):
    import hashlib
    with open(os.path.join(ROOT, "quant_int8_quantized_gb300", "csrc", fn), "rb") as f:
        src = f.read()
    return hashlib.sha256(src.split(HOST_SECTION)[0]).hexdigest()


def gemm_q4k_traffic():
    for fn, digest in GEMM_Q4K_TRAFFIC["sha256"].items():
        if device_code_digest(fn) != digest:
            return None
    return GEMM_Q4K_TRAFFIC["bytes"]


def gemm_launches(kind, M, N, K, sms):
    """Kernel launches one GEMM call makes: two for a q6_K GEMM whose output tiles (192 tokens x
    128 rows) leave the persistent grid's last round partly idle and whose split pays (the library
    then runs those tiles as ordered K slices in a second launch), else one. Mirrors the library's
    rule (order_slices in csrc/gemm.cu); the launch list under profiles/ shows the count."""
    if kind != "q6k" or M <= 64:
        return 1
    bt = 192 if M >= 192 else (M + 15) // 16 * 16
    tiles = -(-M // bt) * -(-N // 128)
    S = K // 256
    if tiles <= sms or tiles % sms == 0:
        return 1
    rest = tiles % sms
    best_cost = S
    for ts in range(2, min(sms // rest, 15) + 1):
        best_cost = min(best_cost, -(-S // ts) + 2 * (ts - 1) + 10)
    return 2 if best_cost < S else 1


def wbytes(kind, N, K):
    return N * (K // 256) * BYTES_PER_SB[kind]


def plane_bytes(M, K, q8=True, op=False):
    """Bytes of a plane: the q8 arrays qs (1 B/elem), d and s (4 B per 32-block each), and the
    GEMM operand arrays ah (2 B/elem), ax (32 B per super-block) and af (4 B per super-block)."""
    n = 0
    if q8:
        n += M * K + M * (K // 32) * 8
    if op:
        n += 2 * M * K + M * (K // 256) * 36
    return n


def gemm_act_bytes(kind, M, K):
    """Activation bytes a GEMM reads: the operand arrays ah, af and (the min terms of q4_K and
    q4_1) ax."""
    return 2 * M * K + M * (K // 256) * (36 if kind in ("q4k", "q4_1") else 4)


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- workload

class Stack:
    """Device-resident 7B-shaped prefill stack and 14B-shaped decode sweep."""

    def __init__(self, dev, seed=0, decode=True):
        from quant_int8_quantized_gb300 import mq, synth
        self.mq, self.dev = mq, dev
        S = synth
        self.x = S.normal((M_TOK, HID), seed, "x", device=dev)
        self.attn = S.normal((M_TOK, HID), seed, "attn", device=dev)
        self.rms_w = [S.normal((HID,), seed, f"L{l}.rms1", 1.0, 0.1, device=dev) for l in range(LAYERS)]
        self.rms2_w = [S.normal((HID,), seed, f"L{l}.rms2", 1.0, 0.1, device=dev) for l in range(LAYERS)]
        self.final_w = S.normal((HID,), seed, "final_norm", 1.0, 0.1, device=dev)
        # q6_K weights are prepacked once, as at weight registration (the GEMM's weight form)
        self.W = [{n: mq.gemm_weights(kind, S.weights(kind, N, K, seed, f"L{l}.{n}", device=dev), N, K)
                   for n, kind, N, K, _ in PREFILL_MATS} for l in range(LAYERS)]
        self.lm_head = mq.mq_prepack_q6k(S.q6k_weights(VOCAB, HID, seed, "lm_head", device=dev), VOCAB, HID)
        f32 = dict(dtype=torch.float32, device=dev)
        self.out = {n: torch.empty((M_TOK, N), **f32) for n, _, N, _, _ in PREFILL_MATS}
        # prefill planes feed only GEMMs: the producers write the operand arrays alone
        self.p_rms = mq.Plane.empty(M_TOK, HID, dev, q8=False)
        self.p_rms2 = mq.Plane.empty(M_TOK, HID, dev, q8=False)
        self.p_attn = mq.Plane.empty(M_TOK, HID, dev, q8=False)
        self.p_ffn = mq.Plane.empty(M_TOK, FFN, dev, q8=False)
        self.p_last = mq.Plane.empty(1, HID, dev, op=False)
        self.logits = torch.empty((VOCAB,), **f32)
        self.q4_events = []
        if decode:
            self.dx = S.normal((1, D_HID), seed, "d.x", device=dev)
            self.dattn = S.normal((1, D_HID), seed, "d.attn", device=dev)
            self.dg = S.normal((1, D_FFN), seed, "d.g", device=dev)
            self.du = S.normal((1, D_FFN), seed, "d.u", device=dev)
            self.drms = [S.normal((D_HID,), seed, f"D{l}.rms", 1.0, 0.1, device=dev) for l in range(D_LAYERS)]
            mats = {n: (kind, N, K) for n, kind, N, K in DECODE_MATS}
            self.dstack = {}
            for name, parts in DECODE_STACKS:
                kinds, Ks = {mats[p][0] for p in parts}, {mats[p][2] for p in parts}
                assert len(kinds) == 1 and len(Ks) == 1
                self.dstack[name] = (kinds.pop(), sum(mats[p][1] for p in parts), Ks.pop())
            # q6_K matrices prepacked, as for the prefill GEMM: one registered form serves both
            self.DW = [{n: mq.gemm_weights(kind, S.weights(kind, N, K, seed, f"D{l}.{n}", device=dev), N, K)
                        for n, (kind, N, K) in self.dstack.items()} for l in range(D_LAYERS)]
            self.dout = {n: torch.empty((N,), **f32) for n, (_, N, _) in self.dstack.items()}
            self.dp_h = mq.Plane.empty(1, D_HID, dev, op=False)
            self.dp_a = mq.Plane.empty(1, D_HID, dev, op=False)
            self.dp_f = mq.Plane.empty(1, D_FFN, dev, op=False)
            # q and k|v only read the rms plane: k|v runs on a second stream, joined before the
            # attention stand-in, so the two GEMVs overlap (inside the captured graph too)
            self.side = torch.cuda.Stream(device=dev)
            self.ev_h = torch.cuda.Event()
            self.ev_kv = torch.cuda.Event()

    # launches per prefill step: 28 * (2 rms + 1 quantize + 1 swiglu + the GEMMs' launches) + rms + gemv;
    # attn_q and attn_k are one paired call (one launch when their tiles fill a round, as here)
    @staticmethod
    def launches_per_step(sms):
        mats = {name: (kind, N, K) for name, kind, N, K, _ in PREFILL_MATS}
        tiles = lambda N: -(-M_TOK // 192) * -(-N // 128)
        qk = 1 if tiles(mats["q"][1]) + tiles(mats["k"][1]) >= sms else 2
        gemms = qk + sum(gemm_launches(kind, M_TOK, N, K, sms) for name, (kind, N, K) in mats.items()
                         if name not in ("q", "k"))
        return LAYERS * (4 + gemms) + 2
    LAUNCHES_PER_DECODE = D_LAYERS * 8   # rms, q, k|v, quantize, o, gate|up, swiglu, down

    def step(self, time_q4=False):
        mq = self.mq
        planes = {"rms": self.p_rms, "rms2": self.p_rms2, "attn": self.p_attn, "swiglu": self.p_ffn}
        for l in range(LAYERS):
            W = self.W[l]
            mq.mq_rms_quant(self.x, self.rms_w[l], EPS, self.p_rms)
            mq.mq_quantize_q8(self.attn, self.p_attn)
            mq.mq_rms_quant(self.x, self.rms2_w[l], EPS, self.p_rms2)
            for name, kind, N, K, src in PREFILL_MATS:
                if name == "k":
                    continue   # with q, below
                if name == "q":   # attn_q and attn_k read the same plane: one paired call
                    mq.mq_gemm_q4k_pair(planes[src], W["q"], N, self.out["q"], W["k"], KVD, self.out["k"])
                    continue
                if name == "down":
                    mq.mq_swiglu_quant(self.out["gate"], self.out["up"], self.p_ffn)
                if time_q4 and name in ("gate", "up"):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    mq.gemm(kind, planes[src], W[name], N, self.out[name])
                    e1.record()
                    self.q4_events.append((e0, e1, 2.0 * M_TOK * N * K))
                else:
                    mq.gemm(kind, planes[src], W[name], N, self.out[name])
        mq.mq_rms_quant(self.out["down"][-1:], self.final_w, EPS, self.p_last)
        mq.mq_gemv_q6k_packed(self.p_last, self.lm_head, VOCAB, self.logits)

    def decode_step(self):
        mq = self.mq
        main = torch.cuda.current_stream()
        for l in range(D_LAYERS):
            W = self.DW[l]
            mq.mq_rms_quant(self.dx, self.drms[l], EPS, self.dp_h)
            self.ev_h.record(main)
            self.side.wait_event(self.ev_h)
            mq.mq_gemv_q6k_packed(self.dp_h, W["kv"], 2 * D_KV, self.dout["kv"], stream=self.side)
            self.ev_kv.record(self.side)
            mq.mq_gemv_q4k(self.dp_h, W["q"], D_HID, self.dout["q"])
            main.wait_event(self.ev_kv)
            mq.mq_quantize_q8(self.dattn, self.dp_a)
            mq.mq_gemv_q4k(self.dp_a, W["o"], D_HID, self.dout["o"])
            mq.mq_gemv_q4k(self.dp_h, W["gate_up"], 2 * D_FFN, self.dout["gate_up"])
            mq.mq_swiglu_quant(self.dg, self.du, self.dp_f)
            mq.mq_gemv_q6k_packed(self.dp_f, W["down"], D_HID, self.dout["down"])

    @staticmethod
    def prefill_flops():
        per_layer = sum(2.0 * M_TOK * N * K for _, _, N, K, _ in PREFILL_MATS)
        return LAYERS * per_layer + 2.0 * VOCAB * HID

    LAUNCHES_PER_DECODE_UNSTACKED = D_LAYERS * 10   # rms, q, k, v, quantize, o, gate, up, swiglu, down

    def decode_step_unstacked(self):
        """The decode layer as config 4 names it: seven GEMVs a layer, one stream. k, v, gate
        and up are row slices of the stacked matrices (the same bytes, no copy)."""
        mq = self.mq
        for l in range(D_LAYERS):
            W = self.DW[l]
            mq.mq_rms_quant(self.dx, self.drms[l], EPS, self.dp_h)
            mq.mq_gemv_q4k(self.dp_h, W["q"], D_HID, self.dout["q"])
            mq.mq_gemv_q6k_packed(self.dp_h, W["kv"][:D_KV], D_KV, self.dout["kv"][:D_KV])
            mq.mq_gemv_q6k_packed(self.dp_h, W["kv"][D_KV:], D_KV, self.dout["kv"][D_KV:])
            mq.mq_quantize_q8(self.dattn, self.dp_a)
            mq.mq_gemv_q4k(self.dp_a, W["o"], D_HID, self.dout["o"])
            mq.mq_gemv_q4k(self.dp_h, W["gate_up"][:D_FFN], D_FFN, self.dout["gate_up"][:D_FFN])
            mq.mq_gemv_q4k(self.dp_h, W["gate_up"][D_FFN:], D_FFN, self.dout["gate_up"][D_FFN:])
            mq.mq_swiglu_quant(self.dg, self.du, self.dp_f)
            mq.mq_gemv_q6k_packed(self.dp_f, W["down"], D_HID, self.dout["down"])

    @staticmethod
    def decode_bytes():
        per_layer = sum(wbytes(kind, N, K) + 4 * N for _, kind, N, K in DECODE_MATS)
        per_layer += 4 * D_HID * 2 + plane_bytes(1, D_HID) * 2 + 8 * D_FFN + plane_bytes(1, D_FFN)  # producers
        per_layer += 4 * D_HID                                                                        # rms weight
        return D_LAYERS * per_layer


# Single-kernel timings put a short GPU spin (torch.cuda._sleep, ~0.25 ms at 2 GHz) in front
# of the first event: the binding's host work (argument checks, tensor-map encoding) then
# overlaps the spin instead of leaving the GPU idle inside the timed region.
GPU_HOLD_CYCLES = 500_000


def producer_rates(st, dev, stream, reps=20):
    """Each prefill producer alone at the stack's shapes, writing the GEMM operand arrays, its
    inputs rotated over buffers that together exceed L2. Rates are counted in the method's
    bytes (the f32 input, 4 or 8 B per element, and the q8 plane, 1.25 B per element); the
    operand arrays the GEMM reads instead (2.14 B per element) are listed beside them."""
    from quant_int8_quantized_gb300 import mq, synth as S
    hbm = load_peaks()[2]
    out = {}
    xs = [S.normal((M_TOK, HID), 0, f"pr.x{i}", device=dev) for i in range(4)]          # 4 x 47.5 MB
    gs = [S.normal((M_TOK, FFN), 0, f"pr.g{i}", device=dev) for i in range(2)]          # 2 x 251 MB
    us = [S.normal((M_TOK, FFN), 0, f"pr.u{i}", device=dev) for i in range(2)]
    w = S.normal((HID,), 0, "pr.w", 1.0, 0.1, device=dev)
    ph, pf = mq.Plane.empty(M_TOK, HID, dev, q8=False), mq.Plane.empty(M_TOK, FFN, dev, q8=False)
    cases = [("rms_quant", HID, 4, lambda i: mq.mq_rms_quant(xs[i % 4], w, EPS, ph)),
             ("quantize_q8", HID, 4, lambda i: mq.mq_quantize_q8(xs[i % 4], ph)),
             ("swiglu_quant", FFN, 8, lambda i: mq.mq_swiglu_quant(gs[i % 2], us[i % 2], pf))]
    for name, K, in_b, fn in cases:
        for i in range(4):
            fn(i)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(GPU_HOLD_CYCLES * 4)   # the GPU is busy while the host enqueues the calls
        a.record(stream)
        for i in range(reps):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize()
        t = a.elapsed_time(b) * 1e-3 / reps
        n = M_TOK * K
        method = n * in_b + n * 1.25
        actual = n * in_b + plane_bytes(M_TOK, K, q8=False, op=True)
        out[f"{name} {M_TOK}x{K}"] = {"us": t * 1e6, "method_bytes": method, "GBps_method": method / t / 1e9,
                                      "hbm_frac_method": method / t / 1e9 / hbm, "written_operand_bytes": actual - n * in_b,
                                      "GBps_actual": actual / t / 1e9, "hbm_frac_actual": actual / t / 1e9 / hbm}
    del xs, gs, us
    return out


def capture_graph(fn):
    """Capture fn's launches (all on the current stream) into a CUDA graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


# ----------------------------------------------------------------------------- CPU oracle sample

def oracle_sample_tok_s(frac=8, prod_frac=16, seed=0):
    """Time the CPU oracle on a bounded sample of the prefill stack at M = 3314 and
    extrapolate to tok/s.

    The oracle's matmul cost is linear in output rows (it dequantizes exactly the weight
    rows it computes), not in tokens, so the sample keeps all 3314 tokens: one layer's 7
    matmuls on 1 in `frac` of their output rows (x frac), the layer's 4 producers on 1 in
    `prod_frac` of the tokens (x prod_frac), times 28 layers, plus the last-token lm_head on
    1 in 8*frac of its rows. Input generation is not timed.
    """
    from oracle import mq_oracle as O
    from quant_int8_quantized_gb300 import synth as S
    mp = M_TOK // prod_frac
    x = S.normal((mp, HID), seed, "x").numpy()
    attn = S.normal((mp, HID), seed, "attn").numpy()
    w1 = S.normal((HID,), seed, "L0.rms1", 1.0, 0.1).numpy()
    w2 = S.normal((HID,), seed, "L0.rms2", 1.0, 0.1).numpy()
    g = S.normal((mp, FFN), seed, "L0.g").numpy()
    u = S.normal((mp, FFN), seed, "L0.u").numpy()
    Ws = {n: S.weights(kind, N // frac, K, seed, f"L0.{n}").numpy() for n, kind, N, K, _ in PREFILL_MATS}
    lm_rows = VOCAB // (8 * frac)
    lm = S.q6k_weights(lm_rows, HID, seed, "lm_head").numpy()
    t0 = time.perf_counter()
    planes = {"rms": O.rms_quant(x, w1, EPS), "attn": O.quantize_q8(attn), "rms2": O.rms_quant(x, w2, EPS),
              "swiglu": O.swiglu_quant(g, u)}
    t_prod = (time.perf_counter() - t0) * (M_TOK / mp)
    # the matmuls read full-height planes (3314 rows; the sampled producer rows repeated)
    full = {k: (np.resize(qs, (M_TOK, qs.shape[1])), np.resize(d, (M_TOK, d.shape[1]))) for k, (qs, d, _) in planes.items()}
    t0 = time.perf_counter()
    last = None
    for name, kind, N, K, src in PREFILL_MATS:
        qs, d = full[src]
        last, _ = O.gemm_rows(qs, d, Ws[name], kind, N // frac, K)
    t_mat = (time.perf_counter() - t0) * frac
    t0 = time.perf_counter()
    qs, d, _ = O.rms_quant(np.resize(last[-1:], (1, HID)).astype(np.float32), w1, EPS)
    O.gemm_rows(qs, d, lm, "q6k", lm_rows, HID)
    t_lm = (time.perf_counter() - t0) * (VOCAB / lm_rows)
    est = LAYERS * (t_prod + t_mat) + t_lm
    sample = (f"M={M_TOK}: one layer's 7 matmuls on 1/{frac} of their output rows (x{frac}) and its 4 producers "
              f"on 1/{prod_frac} of the tokens (x{prod_frac}), x{LAYERS} layers; lm_head on {lm_rows} of {VOCAB} "
              f"rows (x{VOCAB / lm_rows:.1f})")
    return M_TOK / est, est, sample


def oracle_one_core(frac, prod_frac):
    """The same sample in a child process whose numpy may use one thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = (f"import sys, json; sys.path.insert(0, {ROOT!r}); import bench; "
            f"v, est, s = bench.oracle_sample_tok_s(frac={frac}, prod_frac={prod_frac}); print(json.dumps([v, est]))")
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
        v, est = json.loads(r.stdout.strip().splitlines()[-1])
        return {"value": v, "unit": "tok/s", "cores": 1, "kind": "oracle", "sample": f"as above, 1/{frac} rows"}
    except Exception as e:   # a baseline figure, not the measurement: report why it is missing
        return {"value": None, "unit": "tok/s", "cores": 1, "kind": "oracle", "error": str(e)[:200]}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ----------------------------------------------------------------------------- main

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("bf16_tflops_sustained"), d.get("bf16_tflops"), d.get("hbm_gbs"), "measured"
    return 1700.0, 1900.0, 6800.0, "fallback"


def dist_setup(backend: str = "nccl"):
    """Read RANK / LOCAL_RANK / WORLD_SIZE; for more than one rank join the process group
    (NCCL on the GPU box; the multi-process tests pass "gloo" and stay on the CPU)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if backend == "nccl":
        torch.cuda.set_device(local if ws > 1 else 0)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, ws, device="cuda"):
    """The largest of every rank's v (each rank times its own replica; the job takes the slowest)."""
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tok_s(ws, t_ms):
    """Whole-job throughput of ws replicas of the prefill step, each M_TOK tokens, that took at
    most t_ms per step (weak scaling: the work per GPU is fixed)."""
    return ws * M_TOK / (t_ms * 1e-3)


def run_reference(args):
    ws, rank = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        oracle_sample_tok_s(frac=64, prod_frac=64)
    vals, ests = [], []
    for _ in range(args.steps):
        v, est, sample = oracle_sample_tok_s(frac=64, prod_frac=64)
        vals.append(v)
        ests.append(est)
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * statistics.median(ests),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic", "config": {"workload": "7B-shaped matmul stack prefill (28 layers + lm_head), M=3314",
                                            "oracle_sample": "each step a bounded sample of the step, extrapolated"},
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- the shape/token sweep

SWEEP_M = [1, 2, 3, 8, 15, 16, 64, 512, 3314, 8192]   # M in [2, 16): the small-batch paths
MQ_GEMV_ROWS = 8   # the GEMV takes up to 8 activation rows; M in [2, 8] is timed through both calls
SWEEP_NK = [(1024, 5120), (3584, 3584), (18944, 3584), (3584, 18944), (13824, 5120)]


def run_sweep(steps: int, warmup: int):
    """Time every (M, N, K, type) case of the sweep (activations with 1% x50 outliers), M <= 8
    through the GEMV, M >= 2 through the GEMM (both for M in [2, 8]), with a 256 MB L2 flush before each timed
    launch (a read, so that L2 holds no dirty lines whose write-back the timed kernel would pay). Each case's roofline is whichever of the tensor time (2MNK / measured bf16 burst peak)
    and the stream time (algorithmic bytes / measured HBM bandwidth) is larger; `frac` is that
    time over the measured one."""
    import __graft_entry__
    __graft_entry__.build()
    from quant_int8_quantized_gb300 import mq, synth as S
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _, peak_burst, hbm, _ = load_peaks()
    flush = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    for kind in ("q4k", "q6k"):
        for N, K in SWEEP_NK:
            w = S.weights(kind, N, K, 0, f"sweep.{kind}.{N}x{K}", device=dev)
            wg = mq.gemm_weights(kind, w, N, K)
            for M in SWEEP_M:
                x = S.with_outliers(S.normal((M, K), 0, f"sweep.x.{M}x{K}", device=dev), 0, f"sweep.o.{M}x{K}")
                p = mq.Plane.empty(M, K, dev, op=M > 1)
                mq.mq_quantize_q8(x, p)
                out = torch.empty((M, N), dtype=torch.float32, device=dev)
                paths = (["gemv"] if M <= MQ_GEMV_ROWS else []) + (["gemm"] if M > 1 else [])
                for path in paths:
                    if path == "gemv":   # q6_K: the GEMV on the prepacked rows the GEMM reads
                        fn = ((lambda: mq.gemv(kind, p, w, N, out)) if kind == "q4k" else
                              (lambda: mq.mq_gemv_q6k_packed(p, wg, N, out)))
                        act = M * (plane_bytes(1, K, op=False) - (0 if kind == "q4k" else K // 32 * 4))
                    else:
                        fn = lambda: mq.gemm(kind, p, wg, N, out)
                        act = gemm_act_bytes(kind, M, K)
                    nbytes = wbytes(kind, N, K) + act + 4 * M * N
                    for _ in range(max(1, warmup)):
                        fn()
                    ts = []
                    for _ in range(steps):
                        flush.sum()
                        torch.cuda._sleep(GPU_HOLD_CYCLES)
                        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        a.record()
                        fn()
                        b.record()
                        torch.cuda.synchronize()
                        ts.append(a.elapsed_time(b) * 1e-3)
                    t = statistics.median(ts)
                    t_tensor = 2.0 * M * N * K / (peak_burst * 1e12)
                    t_stream = nbytes / (hbm * 1e9)
                    label = "q6kp" if path == "gemv" and kind == "q6k" else kind
                    line = {"case": f"{path}_{label}:{M}x{N}x{K}", "us": t * 1e6,
                            "TFLOPs": 2.0 * M * N * K / t / 1e12, "GBps": nbytes / t / 1e9,
                            "bound": "tensor" if t_tensor >= t_stream else "hbm",
                            "frac": max(t_tensor, t_stream) / t}
                    print(json.dumps(line))
                del x, p, out
    # the other block types on the 14B decode shapes: the GEMV at M = 1, 2, 8; q4_0 / q4_1 also
    # through the GEMM at M = 16 and 3314
    for kind in ("q5k", "q4_0", "q4_1"):
        for N, K in [(5120, 5120), (1024, 5120), (13824, 5120), (5120, 13824)]:
            w = S.weights(kind, N, K, 0, f"sweep.{kind}.{N}x{K}", device=dev)
            cases = [("gemv", M) for M in (1, 2, 8)] + ([("gemm", M) for M in (16, 3314)] if kind != "q5k" else [])
            for path, M in cases:
                x = S.normal((M, K), 0, f"sweep.x.{M}x{K}", device=dev)
                p = mq.Plane.empty(M, K, dev, op=path == "gemm")
                mq.mq_quantize_q8(x, p)
                out = torch.empty((M, N), dtype=torch.float32, device=dev)
                if path == "gemv":
                    fn = lambda: mq.gemv(kind, p, w, N, out)
                    nbytes = wbytes(kind, N, K) + M * plane_bytes(1, K, op=False) + 4 * M * N
                else:
                    fn = lambda: mq.gemm(kind, p, w, N, out)
                    nbytes = wbytes(kind, N, K) + gemm_act_bytes(kind, M, K) + 4 * M * N
                for _ in range(max(1, warmup)):
                    fn()
                ts = []
                for _ in range(steps):
                    flush.sum()
                    torch.cuda._sleep(GPU_HOLD_CYCLES)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    fn()
                    b.record()
                    torch.cuda.synchronize()
                    ts.append(a.elapsed_time(b) * 1e-3)
                t = statistics.median(ts)
                t_tensor = 2.0 * M * N * K / (peak_burst * 1e12)
                t_stream = nbytes / (hbm * 1e9)
                print(json.dumps({"case": f"{path}_{kind}:{M}x{N}x{K}", "us": t * 1e6, "GBps": nbytes / t / 1e9,
                                  "TFLOPs": 2.0 * M * N * K / t / 1e12,
                                  "bound": "tensor" if t_tensor >= t_stream else "hbm",
                                  "frac": max(t_tensor, t_stream) / t}))
                del x, p, out
    if mq.mq_device_status() != mq.MQ_OK:
        raise RuntimeError("device status")
    return 0


# ----------------------------------------------------------------------------- decode alone

def run_decode_only(steps: int, warmup: int):
    """The 14B decode token launched eagerly: `warmup` tokens, then `steps` timed ones (384
    launches each). Without graph replay the host's launch cost shows in the time; the mode
    exists for launch lists (ncu -s 384*warmup -c 384)."""
    import __graft_entry__
    __graft_entry__.build()
    from quant_int8_quantized_gb300 import mq
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    st = Stack(dev)
    for _ in range(warmup):
        st.decode_step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        st.decode_step()
    b.record()
    torch.cuda.synchronize()
    if mq.mq_device_status() != mq.MQ_OK:
        raise RuntimeError("device status")
    t = a.elapsed_time(b) * 1e-3 / max(1, steps)
    print(json.dumps({"decode_eager_ms_per_token": t * 1e3, "GBps": Stack.decode_bytes() / t / 1e9}))
    return 0


# ----------------------------------------------------------------------------- single-kernel cases

def run_case(spec: str, steps: int, warmup: int):
    """Time one kernel on seeded inputs: `kind:MxNxK` (gemm_q4k, gemm_q6k, gemv_q4k, gemv_q6k, gemv_q6kp:
    the q6_K GEMV on prepacked rows, and the other block types)
    or `kind:MxK` (quantize, rms, swiglu). Prints one JSON line with its roofline figure."""
    import __graft_entry__
    __graft_entry__.build()
    from quant_int8_quantized_gb300 import mq, synth as S
    kind, shape = spec.split(":")
    dims = [int(v) for v in shape.lower().split("x")]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak_sus, peak_burst, hbm, peak_kind = load_peaks()
    if kind.startswith("gemm") or kind.startswith("gemv"):
        M, N, K = dims
        wk = kind.split("_", 1)[1]
        packed = wk == "q6kp"   # the q6_K GEMV on prepacked rows
        wk = "q6k" if packed else wk
        x = S.normal((M, K), 0, "case.x", device=dev)
        w = S.weights(wk, N, K, 0, "case.w", device=dev)
        p = mq.Plane.empty(M, K, dev)
        mq.mq_quantize_q8(x, p)
        out = torch.empty((M, N), dtype=torch.float32, device=dev)
        wg = mq.gemm_weights(wk, w, N, K) if kind.startswith("gemm") or packed else w
        fn = ((lambda: mq.gemm(wk, p, wg, N, out)) if kind.startswith("gemm") else
              (lambda: mq.mq_gemv_q6k_packed(p, wg, N, out)) if packed else (lambda: mq.gemv(wk, p, w, N, out)))
        flops = 2.0 * M * N * K
        act = gemm_act_bytes(wk, M, K) if kind.startswith("gemm") else plane_bytes(M, K) - (0 if wk != "q6k" else M * (K // 32) * 4)
        nbytes = wbytes(wk, N, K) + act + 4 * M * N
    else:
        M, K = dims
        x = S.normal((M, K), 0, "case.x", device=dev)
        p = mq.Plane.empty(M, K, dev)
        flops = 0.0
        if kind == "quantize":
            fn = lambda: mq.mq_quantize_q8(x, p)
            nbytes = 4 * M * K + plane_bytes(M, K, op=True)
        elif kind == "rms":
            w = S.normal((K,), 0, "case.rmsw", 1.0, 0.1, device=dev)
            fn = lambda: mq.mq_rms_quant(x, w, EPS, p)
            nbytes = 4 * M * K + 4 * K + plane_bytes(M, K, op=True)
        elif kind == "swiglu":
            u = S.normal((M, K), 0, "case.u", device=dev)
            fn = lambda: mq.mq_swiglu_quant(x, u, p)
            nbytes = 8 * M * K + plane_bytes(M, K, op=True)
        else:
            raise ValueError(kind)
    flush = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)   # 256 MB > L2, read
    for _ in range(max(1, warmup)):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        flush.sum()
        torch.cuda._sleep(GPU_HOLD_CYCLES)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e-3)
    if mq.mq_device_status() != mq.MQ_OK:
        raise RuntimeError("device status")
    t = statistics.median(ts)
    line = {"case": spec, "us": t * 1e6, "GBps": nbytes / t / 1e9, "hbm_frac": nbytes / t / 1e9 / hbm,
            "algorithmic_bytes": nbytes}
    if flops:
        line.update({"TFLOPs": flops / t / 1e12, "tensor_frac_burst": flops / t / 1e12 / peak_burst})
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--case", default=None, help="time one kernel, e.g. gemm_q4k:3314x18944x3584")
    ap.add_argument("--decode-only", action="store_true",
                    help="run the decode token alone, eagerly (W warm-up tokens, then K timed), for launch lists")
    ap.add_argument("--sweep", action="store_true",
                    help="time the 60-case shape/token sweep; one JSON line per case with its roofline fraction")
    args = ap.parse_args()
    if args.case:
        return run_case(args.case, args.steps, args.warmup)
    if args.sweep:
        return run_sweep(args.steps, args.warmup)
    if args.decode_only:
        return run_decode_only(args.steps, args.warmup)
    if args.impl == "reference":
        return run_reference(args)
    ws, rank, local = dist_setup()
    import __graft_entry__
    __graft_entry__.build()
    from quant_int8_quantized_gb300 import mq

    dev = torch.device("cuda", torch.cuda.current_device())
    st = Stack(dev, decode=not args.no_decode)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        st.step()
        if not args.no_decode:
            st.decode_step()
    torch.cuda.synchronize()

    # ---- prefill, inputs resident in HBM
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            st.step(time_q4=True)
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(ws)
    t_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws)
    status = mq.mq_device_status()
    if status != mq.MQ_OK:
        raise RuntimeError(f"device status {status}")
    q4_t = sum(a.elapsed_time(b) for a, b, _ in st.q4_events) * 1e-3
    q4_f = sum(f for _, _, f in st.q4_events)
    q4_launches = len(st.q4_events)

    # ---- decode sweep: 384 small launches per token, replayed from a CUDA graph so that the
    #      host's per-launch cost does not stand in for the kernels' time
    dec = None
    if not args.no_decode:
        graph = capture_graph(st.decode_step)
        for _ in range(3):
            graph.replay()
        barrier(ws)
        torch.cuda.synchronize()
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        d1.record(stream)
        torch.cuda.synchronize()
        dt = max_over_ranks(d0.elapsed_time(d1) / args.steps, ws) * 1e-3
        if mq.mq_device_status() != mq.MQ_OK:
            raise RuntimeError("device status after the decode sweep")
        dec = {"workload": "14B-shaped decode sweep, 48 layers, M=1", "GBps": ws * Stack.decode_bytes() / dt / 1e9,
               "ms_per_token": dt * 1e3, "bytes_per_token": Stack.decode_bytes(),
               "hbm_frac": Stack.decode_bytes() / dt / 1e9 / load_peaks()[2],
               "launches_per_token": Stack.LAUNCHES_PER_DECODE, "launch": "CUDA graph replay",
               "stacked": "k|v and gate|up weights stored as one matrix each, one GEMV per pair",
               "streams": "the k|v GEMV runs on a second stream beside attn_q (both read only the rms plane)"}

    # ---- decode as config 4 writes it: seven GEMVs a layer on one stream
    dec_u = None
    if not args.no_decode:
        graph_u = capture_graph(st.decode_step_unstacked)
        for _ in range(3):
            graph_u.replay()
        torch.cuda.synchronize()
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for _ in range(args.steps):
            graph_u.replay()
        d1.record(stream)
        torch.cuda.synchronize()
        dtu = max_over_ranks(d0.elapsed_time(d1) / args.steps, ws) * 1e-3
        dec_u = {"workload": "14B-shaped decode sweep, 48 layers, M=1, seven GEMVs a layer on one stream",
                 "GBps": ws * Stack.decode_bytes() / dtu / 1e9, "ms_per_token": dtu * 1e3,
                 "hbm_frac": Stack.decode_bytes() / dtu / 1e9 / load_peaks()[2],
                 "launches_per_token": Stack.LAUNCHES_PER_DECODE_UNSTACKED, "launch": "CUDA graph replay"}

    # ---- the prefill producers alone, at the stack's shapes
    prod = producer_rates(st, dev, stream) if rank == 0 else None

    # ---- end to end: inputs from pinned host memory, logits back to the host
    host_x = st.x.cpu().pin_memory()
    host_attn = st.attn.cpu().pin_memory()
    host_logits = torch.empty((VOCAB,), dtype=torch.float32).pin_memory()
    barrier(ws)
    torch.cuda.synchronize()
    h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    h0.record(stream)
    for _ in range(args.steps):
        st.x.copy_(host_x, non_blocking=True)
        st.attn.copy_(host_attn, non_blocking=True)
        st.step()
        host_logits.copy_(st.logits, non_blocking=True)
    h1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(h0.elapsed_time(h1) / args.steps, ws)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        v, est, sample = oracle_sample_tok_s()
        cpu = {"value": v, "unit": "tok/s", "cores": cpu_cores(), "kind": "oracle", "sample": sample,
               "one_core": oracle_one_core(32, 64)}

    peak_sus, peak_burst, hbm, peak_kind = load_peaks()
    achieved = q4_f / q4_t / 1e12
    if rank == 0:
        line = {
            "metric": METRIC, "value": job_tok_s(ws, t_ms), "unit": "tok/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "q8 activations as binary16 operands (2^-11) x exact 4/6-bit weight operands, f16 tensor pipe, f32 accumulate",
            "data": "synthetic",
            "config": {"workload": "7B-shaped matmul stack prefill (28 layers + lm_head), M=3314",
                       "hidden": HID, "ffn": FFN, "kv": KVD, "vocab": VOCAB, "layers": LAYERS,
                       "weights_bytes": sum(wbytes(k, N, K) for _, k, N, K, _ in PREFILL_MATS) * LAYERS
                       + wbytes("q6k", VOCAB, HID),
                       "l2": "weights per step (4.6 GB) far exceed L2; no flush",
                       "parallelism": f"replicas x{ws}"},
            "effective_tops": ws * Stack.prefill_flops() / (t_ms * 1e-3) / 1e12,
            "decode": dec,
            "decode_unstacked": dec_u,
            "producers": prod,
            "e2e": {"value": job_tok_s(ws, e2e_ms), "unit": "tok/s",
                    "h2d_bytes_per_step": host_x.numel() * 4 + host_attn.numel() * 4,
                    "d2h_bytes_per_step": VOCAB * 4},
            "roofline": {"kernel": "gemm q4_K 3314x18944x3584 (gate and up launches of the timed steps)",
                         "bound": "tensor",
                         "achieved": achieved, "peak": peak_sus, "unit": "TFLOP/s", "frac": achieved / peak_sus,
                         "peak_kind": f"{peak_kind} bf16 sustained (f16 runs at the bf16 rate)",
                         "launches": q4_launches, "traffic": gemm_q4k_traffic(), "traffic_unit": "bytes per launch"},
            "gpu_launches": Stack.launches_per_step(torch.cuda.get_device_properties(dev).multi_processor_count) * args.steps,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
