"""CPU oracle for per-token-group fp8 e4m3 quantization -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never does, and this package imports nothing from it.

The arithmetic lives in ``gq_oracle.c`` (plain C, compiled with gcc); this
module compiles it on demand and exposes numpy-level wrappers.  bf16 tensors
travel as their raw ``uint16`` bit patterns, e4m3 results as ``uint8`` codes.

Method source: pytorch/ao pull-request pages #2668 ("use smaller block sizes
for per group scaling kernels", intro and the kernel arguments in its
torch.compile failure report; its MoE fp8 training test for the grouped
grad_weight product), #2863 ("test and bench new faster method for per group
rowwise scaling", Summary; its PR stack for the expert weights along dim1)
and #3114 ("fix mxfp8 a2a bench script; set mxfp8 a2a scaling type to
RCEIL", Summary: the mxfp8 cast along dim0 and its two scaling types).

Functions: the e4m3 encoder and decoder, the scale (plain and rounded to a
power of two), colwise, rowwise_t, expert_dim1, mxfp8_dim0 and
grouped_wgrad.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "gq_oracle.c")
_LIB = os.path.join(_HERE, "libgq_oracle.so")
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra"]


def compile_source(src: str, out: str) -> str:
    """Compile an oracle C source file into a shared library at ``out``."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``gq_oracle.c`` into ``libgq_oracle.so`` when it is stale."""
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE))
    if force or stale:
        compile_source(SOURCE, _LIB)
    return _LIB


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


class Oracle:
    """numpy-level view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        lib.gqo_colwise.argtypes = [p, i64, i64, p, i32, p, p]
        lib.gqo_colwise.restype = ctypes.c_int
        lib.gqo_rowwise_t.argtypes = [p, i64, i64, p, i32, p, p]
        lib.gqo_rowwise_t.restype = ctypes.c_int
        lib.gqo_colwise_ex.argtypes = [p, i64, i64, p, i32, ctypes.c_int, p, p]
        lib.gqo_colwise_ex.restype = ctypes.c_int
        lib.gqo_rowwise_t_ex.argtypes = [p, i64, i64, p, i32, ctypes.c_int, p, p]
        lib.gqo_rowwise_t_ex.restype = ctypes.c_int
        lib.gqo_mxfp8_dim0.argtypes = [p, i64, i64, ctypes.c_int, p, p]
        lib.gqo_mxfp8_dim0.restype = ctypes.c_int
        lib.gqo_expert_dim1.argtypes = [p, i64, i64, i64, ctypes.c_int, p, p]
        lib.gqo_expert_dim1.restype = ctypes.c_int
        lib.gqo_expert_rowwise.argtypes = [p, i64, i64, i64, ctypes.c_int, p, p]
        lib.gqo_expert_rowwise.restype = ctypes.c_int
        lib.gqo_scale_pow2_array.argtypes = [p, i64, p]
        lib.gqo_grouped_wgrad.argtypes = [p, p, p, p, i64, i64, i64, p, i32, p, p]
        lib.gqo_scale_pow2_array.restype = None
        lib.gqo_e4m3_encode_array.argtypes = [p, i64, p]
        lib.gqo_e4m3_decode_array.argtypes = [p, i64, p]
        lib.gqo_scale_array.argtypes = [p, i64, p]
        lib.gqo_quant_array.argtypes = [p, p, i64, p]
        for f in ("gqo_e4m3_encode_array", "gqo_e4m3_decode_array",
                  "gqo_scale_array", "gqo_quant_array"):
            getattr(lib, f).restype = None
        self.lib = lib
        self.path = path

    # ---------------------------------------------------------- elementwise
    def e4m3_encode(self, v) -> np.ndarray:
        """Saturating round-to-nearest-even fp32 -> e4m3 codes (uint8)."""
        v = _c(v, np.float32)
        out = np.empty(v.shape, np.uint8)
        self.lib.gqo_e4m3_encode_array(v.ctypes.data, v.size, out.ctypes.data)
        return out

    def e4m3_decode(self, codes) -> np.ndarray:
        """e4m3 codes -> float64 values (NaN for S.1111.111)."""
        c = _c(codes, np.uint8)
        out = np.empty(c.shape, np.float64)
        self.lib.gqo_e4m3_decode_array(c.ctypes.data, c.size, out.ctypes.data)
        return out

    def scale_of(self, amax) -> np.ndarray:
        """fp32 scale = 448 / max(amax, 1e-12) for an array of fp32 amax."""
        a = _c(amax, np.float32)
        out = np.empty(a.shape, np.float32)
        self.lib.gqo_scale_array(a.ctypes.data, a.size, out.ctypes.data)
        return out

    def scale_pow2_of(self, amax) -> np.ndarray:
        """2^floor(log2(448 / max(amax, 1e-12))) for an array of fp32 amax."""
        a = _c(amax, np.float32)
        out = np.empty(a.shape, np.float32)
        self.lib.gqo_scale_pow2_array(a.ctypes.data, a.size, out.ctypes.data)
        return out

    def quant(self, x_bf16_bits, scale) -> np.ndarray:
        """Elementwise e4m3(fp32(x * scale)); x as bf16 bit patterns."""
        x = _c(x_bf16_bits, np.uint16)
        s = _c(np.broadcast_to(np.asarray(scale, np.float32), x.shape),
               np.float32)
        out = np.empty(x.shape, np.uint8)
        self.lib.gqo_quant_array(x.ctypes.data, s.ctypes.data, x.size,
                                 out.ctypes.data)
        return out

    # ---------------------------------------------------------------- paths
    def colwise(self, x_bf16_bits, offs, out=None, pow2=False):
        """Per-group scaling along dim0.

        x: uint16 (M, K) bf16 bits, row-major.  offs: int32 end offsets.
        Returns (q uint8 (M, K), scales float32 (n_groups, K)).  Rows outside
        every group keep the value of ``out`` (zeros when ``out`` is None).
        ``pow2`` rounds every scale down to a power of two.
        """
        x = _c(x_bf16_bits, np.uint16)
        assert x.ndim == 2
        o = _c(offs, np.int32).reshape(-1)
        M, K = x.shape
        q = np.zeros((M, K), np.uint8) if out is None else _c(out, np.uint8).copy()
        s = np.empty((o.size, K), np.float32)
        rc = self.lib.gqo_colwise_ex(x.ctypes.data, M, K, o.ctypes.data, o.size,
                                     int(bool(pow2)), q.ctypes.data, s.ctypes.data)
        if rc != 0:
            raise ValueError("oracle colwise: invalid arguments")
        return q, s

    def rowwise_t(self, a_bf16_bits, offs, out=None, pow2=False):
        """Per-group scaling along dim1 with transposed output (``pow2``:
        scales rounded down to powers of two).

        a: uint16 (N, Mg) bf16 bits, row-major.  offs: int32 end offsets
        along Mg.  Returns (qt uint8 (Mg, N) = q(a)^T, scales float32
        (N, n_groups)).  Token rows of qt outside every group keep ``out``.
        """
        a = _c(a_bf16_bits, np.uint16)
        assert a.ndim == 2
        o = _c(offs, np.int32).reshape(-1)
        N, Mg = a.shape
        qt = np.zeros((Mg, N), np.uint8) if out is None else _c(out, np.uint8).copy()
        s = np.empty((N, o.size), np.float32)
        rc = self.lib.gqo_rowwise_t_ex(a.ctypes.data, N, Mg, o.ctypes.data,
                                       o.size, int(bool(pow2)), qt.ctypes.data,
                                       s.ctypes.data)
        if rc != 0:
            raise ValueError("oracle rowwise_t: invalid arguments")
        return qt, s


    def expert_dim1(self, w_bf16_bits, pow2=False):
        """Stacked expert weights (E, K, N) scaled per (expert, column), the
        amax over each expert's K rows.  Returns (q uint8 (E, K, N), scales
        float32 (E, N))."""
        w = _c(w_bf16_bits, np.uint16)
        assert w.ndim == 3
        E, K, N = w.shape
        q = np.zeros((E, K, N), np.uint8)
        s = np.empty((E, N), np.float32)
        rc = self.lib.gqo_expert_dim1(w.ctypes.data, E, K, N, int(bool(pow2)),
                                      q.ctypes.data, s.ctypes.data)
        if rc != 0:
            raise ValueError("oracle expert_dim1: invalid arguments")
        return q, s


    def expert_rowwise(self, w_bf16_bits, pow2=False):
        """Stacked expert weights (E, N, K) scaled per (expert, row), the
        amax over the row's K elements.  Returns (q uint8 (E, N, K), scales
        float32 (E, N))."""
        w = _c(w_bf16_bits, np.uint16)
        assert w.ndim == 3
        E, N, K = w.shape
        q = np.zeros((E, N, K), np.uint8)
        s = np.empty((E, N), np.float32)
        rc = self.lib.gqo_expert_rowwise(w.ctypes.data, E, N, K, int(bool(pow2)),
                                         q.ctypes.data, s.ctypes.data)
        if rc != 0:
            raise ValueError("oracle expert_rowwise: invalid arguments")
        return q, s

    def mxfp8_dim0(self, x_bf16_bits, mode):
        """mxfp8 cast along dim0: blocks of 32 consecutive elements of a row
        share a power-of-two scale.  mode 0 = FLOOR, 1 = RCEIL.  Returns
        (q uint8 (M, K) e4m3 codes, scales uint8 (M, K / 32) e8m0 bytes)."""
        x = _c(x_bf16_bits, np.uint16)
        assert x.ndim == 2
        M, K = x.shape
        q = np.zeros((M, K), np.uint8)
        s = np.zeros((M, K // 32), np.uint8)
        rc = self.lib.gqo_mxfp8_dim0(x.ctypes.data, M, K, int(mode), q.ctypes.data,
                                     s.ctypes.data)
        if rc != 0:
            raise ValueError("oracle mxfp8_dim0: invalid arguments")
        return q, s


    def grouped_wgrad(self, qa_t, sa, qx, sx, offs):
        """grad_weight per token group from the quantized operands: qa_t e4m3
        codes (T, N), sa fp32 (N, G), qx e4m3 codes (T, K), sx fp32 (G, K).
        Returns (out float64 (G, N, K), absum float64 (G, N, K)): the exact
        sum of products divided by sa * sx, and the same for |products|."""
        qa = _c(qa_t, np.uint8)
        qxx = _c(qx, np.uint8)
        o = _c(offs, np.int32)
        T, N = qa.shape
        T2, K = qxx.shape
        assert T == T2
        G = o.shape[0]
        a_s = _c(sa, np.float32).reshape(N, G)
        x_s = _c(sx, np.float32).reshape(G, K)
        out = np.zeros((G, N, K), np.float64)
        absum = np.zeros((G, N, K), np.float64)
        rc = self.lib.gqo_grouped_wgrad(qa.ctypes.data, a_s.ctypes.data, qxx.ctypes.data,
                                        x_s.ctypes.data, T, N, K, o.ctypes.data, G,
                                        out.ctypes.data, absum.ctypes.data)
        if rc != 0:
            raise ValueError("oracle grouped_wgrad: invalid arguments")
        return out, absum


_lock = threading.Lock()
_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from ``gq_oracle.c``."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def e4m3_encode(v):
    return get().e4m3_encode(v)


def e4m3_decode(codes):
    return get().e4m3_decode(codes)


def scale_of(amax):
    return get().scale_of(amax)


def quant(x_bf16_bits, scale):
    return get().quant(x_bf16_bits, scale)


def scale_pow2_of(amax):
    return get().scale_pow2_of(amax)


def colwise(x_bf16_bits, offs, out=None, pow2=False):
    return get().colwise(x_bf16_bits, offs, out, pow2)


def rowwise_t(a_bf16_bits, offs, out=None, pow2=False):
    return get().rowwise_t(a_bf16_bits, offs, out, pow2)


def expert_dim1(w_bf16_bits, pow2=False):
    return get().expert_dim1(w_bf16_bits, pow2)


def expert_rowwise(w_bf16_bits, pow2=False):
    return get().expert_rowwise(w_bf16_bits, pow2)


def mxfp8_dim0(x_bf16_bits, mode):
    return get().mxfp8_dim0(x_bf16_bits, mode)


def grouped_wgrad(qa_t, sa, qx, sx, offs):
    return get().grouped_wgrad(qa_t, sa, qx, sx, offs)


def threads_used() -> int:
    """The oracle is single-threaded."""
    return 1
