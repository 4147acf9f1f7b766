"""A second, independent restatement of the method from library routines.

The pytorch/ao PR pages benchmark their Triton kernels against a "torch loop"
(#2668 benchmark tables, column torch_time_us; #2863 Benchmarks, column
torch_loop_time_us): a Python loop over token groups of plain tensor ops.  This
module is that formulation, on the CPU, built only from numpy / torch
primitives -- numpy's fp32 abs/max/divide/multiply and torch's fp32 ->
float8_e4m3fn conversion (round-to-nearest-even, applied after clamping to
[-448, 448] because torch's own cast is not saturating).  It shares nothing
with ``oracle/gq_oracle.c`` and is used to pin the oracle on small inputs.
"""
import numpy as np
import torch

FP8_MAX = np.float32(448.0)
EPS = np.float32(1e-12)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def cast_e4m3(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, np.float32))
    t = torch.clamp(t, -448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def bounds(offs, extent):
    out, prev = [], 0
    for o in np.asarray(offs, np.int64).tolist():
        e = min(max(o, prev), extent)
        out.append((prev, e))
        prev = e
    return out


def colwise(x_bits, offs, fill=0):
    xf = bf16_bits_to_f32(x_bits)
    M, K = xf.shape
    q = np.full((M, K), fill, np.uint8)
    scales = []
    for s, e in bounds(offs, M):
        blk = xf[s:e]
        amax = np.abs(blk).max(axis=0) if e > s else np.zeros(K, np.float32)
        sc = FP8_MAX / np.maximum(amax.astype(np.float32), EPS)
        q[s:e] = cast_e4m3(blk * sc[None, :])
        scales.append(sc.astype(np.float32))
    return q, np.stack(scales).astype(np.float32)


def rowwise_t(a_bits, offs, fill=0):
    af = bf16_bits_to_f32(a_bits)
    N, Mg = af.shape
    qt = np.full((Mg, N), fill, np.uint8)
    scales = []
    for s, e in bounds(offs, Mg):
        blk = af[:, s:e]
        amax = np.abs(blk).max(axis=1) if e > s else np.zeros(N, np.float32)
        sc = FP8_MAX / np.maximum(amax.astype(np.float32), EPS)
        qt[s:e] = cast_e4m3(blk * sc[:, None]).T
        scales.append(sc.astype(np.float32))
    return qt, np.stack(scales, axis=1).astype(np.float32)
