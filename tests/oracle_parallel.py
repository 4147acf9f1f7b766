"""The C oracle over every host core, for full-size comparisons.

Colwise scaling treats every column on its own (a column's amax, scale and
codes depend on that column alone), and rowwise_t every row of A, so the
oracle's result for the whole tensor is the union of its results on
independent column slices (colwise) or row slices (rowwise_t), each with
the same offsets.  Threads call the C oracle, which runs without the
interpreter lock.  Nothing here computes anything itself: it slices,
calls ``oracle``, and places the pieces.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

import oracle

SLICE = 256  # columns (colwise) or rows (rowwise_t) per oracle call


def _threads() -> int:
    return max(1, os.cpu_count() or 1)


def colwise(x: np.ndarray, offs: np.ndarray, out=None, pow2: bool = False):
    """oracle.colwise on the whole of x (M, K), in column slices."""
    M, K = x.shape
    G = int(np.asarray(offs).size)
    q = np.zeros((M, K), np.uint8) if out is None else np.array(out, np.uint8, copy=True)
    s = np.empty((G, K), np.float32)

    def one(c0):
        c1 = min(K, c0 + SLICE)
        xs = np.ascontiguousarray(x[:, c0:c1])
        qs, ss = oracle.colwise(xs, offs, out=np.ascontiguousarray(q[:, c0:c1]), pow2=pow2)
        q[:, c0:c1] = qs
        s[:, c0:c1] = ss

    with cf.ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(0, K, SLICE)))
    return q, s


def rowwise_t(a: np.ndarray, offs: np.ndarray, out=None, pow2: bool = False):
    """oracle.rowwise_t on the whole of A (N, Mg), in row slices; returns
    (qt (Mg, N), scales (N, G))."""
    N, Mg = a.shape
    G = int(np.asarray(offs).size)
    qt = np.zeros((Mg, N), np.uint8) if out is None else np.array(out, np.uint8, copy=True)
    s = np.empty((N, G), np.float32)

    def one(r0):
        r1 = min(N, r0 + SLICE)
        qs, ss = oracle.rowwise_t(a[r0:r1], offs, out=np.ascontiguousarray(qt[:, r0:r1]),
                                  pow2=pow2)
        qt[:, r0:r1] = qs
        s[r0:r1] = ss

    with cf.ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(0, N, SLICE)))
    return qt, s


def expert_dim1(w: np.ndarray, pow2: bool = False):
    """oracle.expert_dim1 on the whole of W (E, K, N), in column slices
    (every (expert, column) is independent)."""
    E, K, N = w.shape
    q = np.zeros((E, K, N), np.uint8)
    s = np.empty((E, N), np.float32)

    def one(c0):
        c1 = min(N, c0 + SLICE)
        qs, ss = oracle.expert_dim1(np.ascontiguousarray(w[:, :, c0:c1]), pow2=pow2)
        q[:, :, c0:c1] = qs
        s[:, c0:c1] = ss

    with cf.ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(0, N, SLICE)))
    return q, s


def expert_rowwise(w: np.ndarray, pow2: bool = False):
    """oracle.expert_rowwise on the whole of W (E, N, K), in slices of rows
    (dim 1); returns (q (E, N, K), scales (E, N))."""
    E, N, K = w.shape
    q = np.zeros((E, N, K), np.uint8)
    s = np.empty((E, N), np.float32)

    def one(n0):
        n1 = min(N, n0 + SLICE)
        qs, ss = oracle.expert_rowwise(np.ascontiguousarray(w[:, n0:n1]), pow2=pow2)
        q[:, n0:n1] = qs
        s[:, n0:n1] = ss

    with cf.ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(0, N, SLICE)))
    return q, s


def mxfp8_dim0(x: np.ndarray, mode: int):
    """oracle.mxfp8_dim0 on the whole of X (M, K), in row slices (every
    32-element row block is independent)."""
    M, K = x.shape
    q = np.zeros((M, K), np.uint8)
    s = np.zeros((M, K // 32), np.uint8)
    rows = 4 * SLICE

    def one(r0):
        r1 = min(M, r0 + rows)
        qs, ss = oracle.mxfp8_dim0(np.ascontiguousarray(x[r0:r1]), mode)
        q[r0:r1] = qs
        s[r0:r1] = ss

    with cf.ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(0, M, rows)))
    return q, s
