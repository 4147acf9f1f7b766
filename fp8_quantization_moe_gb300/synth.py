"""Seeded synthetic inputs for per-token-group fp8 quantization.

This module only draws inputs: bf16 tensors (as ``uint16`` bit patterns) and
int32 end offsets.  It holds none of the quantization arithmetic and imports
neither the CUDA binding nor the oracle, so both sides can be fed from it.

Shapes and value mixes follow the workloads of the pytorch/ao PR pages:
the colwise (dim0) benchmark shapes (256, 4096), (4096, 4096) and
(65536, 4096) with 4/8/16 groups ("use smaller block sizes for per group
scaling kernels", benchmark tables), and the rowwise shape (Mg, N) =
(16640, 8192) with 1/16/64 groups ("test and bench new faster method for per
group rowwise scaling", Benchmarks), stored here as A (N=8192, Mg=16640).
Token groups are cut at multiples of 16 tokens, the alignment the MoE fp8
training test sets (``set_token_group_alignment_size_m(16)``, same page as the
dim0 kernel).

Random numbers come from numpy's PCG64 generator, whose streams are identical
on x86-64 and aarch64; fp32 samples are rounded to bf16 by torch's
round-to-nearest-even conversion.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

ALIGN = 16  # token-group alignment (tokens)


@dataclass
class Case:
    """One seeded workload.

    kind: "colwise" (x is (M, K), groups along rows) or "rowwise_t"
    (x is (N, Mg), groups along columns).
    x: uint16 bf16 bit patterns.  offs: int32 end offsets.
    """

    name: str
    kind: str
    x: np.ndarray
    offs: np.ndarray
    seed: int
    notes: dict = field(default_factory=dict)

    @property
    def n_groups(self) -> int:
        return int(self.offs.size)

    @property
    def shape(self):
        return tuple(self.x.shape)


def to_bf16_bits(f32: np.ndarray) -> np.ndarray:
    """Round an fp32 array to bf16 (RNE) and return its uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def random_partition(rng: np.random.Generator, total: int, n_groups: int,
                     n_empty: int = 0, align: int = ALIGN) -> np.ndarray:
    """End offsets of a random partition of ``total`` tokens.

    ``n_groups - n_empty`` positive parts, each a multiple of ``align``
    tokens: distinct cut points drawn uniformly without replacement from the
    interior unit positions, then sorted.  ``n_empty`` zero-length groups are
    inserted at seeded interior positions.  ``total`` must be a multiple of
    ``align``.
    """
    assert total % align == 0 and n_groups >= 1 and 0 <= n_empty < n_groups
    units = total // align
    n_pos = n_groups - n_empty
    assert n_pos <= max(units, 1)
    if n_pos > 1:
        cuts = np.sort(rng.choice(np.arange(1, units), size=n_pos - 1,
                                  replace=False))
        ends = list((cuts * align).astype(np.int64)) + [total]
    else:
        ends = [total]
    for _ in range(n_empty):
        # duplicate an end offset at an interior position -> one empty group
        pos = int(rng.integers(1, len(ends)))
        ends.insert(pos, ends[pos - 1])
    return np.asarray(ends, dtype=np.int32)


def _normal(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


# --------------------------------------------------------------- workloads --

def colwise_small(seed: int = 1104) -> Case:
    """X (256, 4096) ~ N(0,1), 4 groups."""
    rng = np.random.default_rng(seed)
    x = _normal(rng, (256, 4096))
    offs = random_partition(rng, 256, 4)
    return Case("colwise_256x4096_g4", "colwise", to_bf16_bits(x), offs, seed)


def colwise_outliers(seed: int = 1216) -> Case:
    """X (4096, 4096) ~ N(0,1); 1% of rows x100; one all-zero column;
    16 groups, one of them empty."""
    rng = np.random.default_rng(seed)
    M, K = 4096, 4096
    x = _normal(rng, (M, K))
    n_out = int(round(0.01 * M))
    rows = rng.choice(M, size=n_out, replace=False)
    x[rows] *= 100.0
    zcol = int(rng.integers(0, K))
    x[:, zcol] = 0.0
    offs = random_partition(rng, M, 16, n_empty=1)
    return Case("colwise_4096x4096_g16_outliers", "colwise", to_bf16_bits(x),
                offs, seed, {"outlier_rows": np.sort(rows), "zero_col": zcol})


def colwise_large(n_groups: int = 16, seed: int | None = None,
                  rows: int = 65536, cols: int = 4096) -> Case:
    """X (65536, 4096), row r ~ N(0,1) * 10^u_r with u_r ~ U(-2, 2)."""
    seed = 1300 + n_groups if seed is None else seed
    rng = np.random.default_rng(seed)
    x = _normal(rng, (rows, cols))
    u = rng.uniform(-2.0, 2.0, size=(rows, 1)).astype(np.float32)
    x *= np.power(np.float32(10.0), u)
    offs = random_partition(rng, rows, n_groups)
    return Case(f"colwise_{rows}x{cols}_g{n_groups}", "colwise",
                to_bf16_bits(x), offs, seed)


def rowwise_g16(seed: int = 1416, N: int = 8192, Mg: int = 16640) -> Case:
    """A (8192, 16640) ~ N(0,1), 16 groups along the token columns."""
    rng = np.random.default_rng(seed)
    a = _normal(rng, (N, Mg))
    offs = random_partition(rng, Mg, 16)
    return Case(f"rowwise_t_{N}x{Mg}_g16", "rowwise_t", to_bf16_bits(a),
                offs, seed)


def rowwise_outliers(n_groups: int = 64, seed: int | None = None,
                     N: int = 8192, Mg: int = 16640) -> Case:
    """A (8192, 16640) ~ N(0,1); 0.5% of token columns x1000;
    1 group, or 64 groups of which two are empty."""
    seed = 1500 + n_groups if seed is None else seed
    rng = np.random.default_rng(seed)
    a = _normal(rng, (N, Mg))
    n_out = int(round(0.005 * Mg))
    cols = rng.choice(Mg, size=n_out, replace=False)
    a[:, cols] *= 1000.0
    n_empty = 2 if n_groups >= 3 else 0
    offs = random_partition(rng, Mg, n_groups, n_empty=n_empty)
    return Case(f"rowwise_t_{N}x{Mg}_g{n_groups}_outliers", "rowwise_t",
                to_bf16_bits(a), offs, seed, {"outlier_cols": np.sort(cols)})


def past_int32(kind: str, rows: int, cols: int, n_groups: int, seed: int,
               period: int = 4096, uncovered: int = 32) -> Case:
    """An input of more than 2^31 elements, cheap to draw at 4 GB: a seeded
    N(0,1) block of ``period`` rows (colwise: rows of X, shape (rows, cols);
    rowwise_t: token columns of A, shape (cols, rows)) repeated along the
    grouped dimension, repetition j scaled by 2^(j mod 8) -- an add to the
    bf16 exponent field of the block's normal values, so exact -- so that a
    result read or written at the wrong repetition differs.  The last
    ``uncovered`` rows (tokens) lie past the last group."""
    assert kind in ("colwise", "rowwise_t") and rows % ALIGN == 0
    rng = np.random.default_rng(seed)
    base = to_bf16_bits(_normal(rng, (period, cols)))
    expo = base & np.uint16(0x7F80)
    normal = (expo >= 0x0080) & (expo <= 0x7B80)  # room for +7 below inf
    x = np.empty((rows, cols) if kind == "colwise" else (cols, rows), np.uint16)
    for j in range((rows + period - 1) // period):
        r0 = j * period
        n = min(period, rows - r0)
        blk = base[:n].copy()
        blk[normal[:n]] += np.uint16((j % 8) << 7)
        if kind == "colwise":
            x[r0:r0 + n] = blk
        else:
            x[:, r0:r0 + n] = blk.T
    offs = random_partition(rng, rows - uncovered, n_groups)
    return Case(f"{kind}_{x.shape[0]}x{x.shape[1]}_g{n_groups}_past_int32", kind,
                x, offs, seed)


def workload(idx: int, n_groups: int | None = None) -> Case:
    """The five workloads, numbered 1..5 in the order listed above."""
    if idx == 1:
        return colwise_small()
    if idx == 2:
        return colwise_outliers()
    if idx == 3:
        return colwise_large(16 if n_groups is None else n_groups)
    if idx == 4:
        return rowwise_g16()
    if idx == 5:
        return rowwise_outliers(64 if n_groups is None else n_groups)
    raise ValueError(f"no workload {idx}")


WORKLOAD_GROUPS = {1: [4], 2: [16], 3: [4, 8, 16], 4: [16], 5: [1, 64]}


def random_case(kind: str, rows: int, cols: int, n_groups: int, seed: int,
                n_empty: int = 0, align: int = ALIGN, scale_mix: bool = False,
                uncovered: int = 0) -> Case:
    """A small random case for parity tests.

    kind "colwise": x (rows, cols), groups along rows;
    kind "rowwise_t": x (rows, cols) = (N, Mg), groups along cols.
    ``uncovered`` tokens at the end belong to no group (offs[-1] < extent).
    ``scale_mix`` multiplies each token by 10^U(-3, 3) and plants a few
    subnormal, zero and negative-zero values.
    """
    rng = np.random.default_rng(seed)
    x = _normal(rng, (rows, cols))
    extent = rows if kind == "colwise" else cols
    if scale_mix:
        if kind == "colwise":
            x *= np.power(np.float32(10.0),
                          rng.uniform(-3, 3, size=(rows, 1)).astype(np.float32))
        else:
            x *= np.power(np.float32(10.0),
                          rng.uniform(-3, 3, size=(1, cols)).astype(np.float32))
        flat = x.reshape(-1)
        k = max(1, flat.size // 64)
        idx = rng.choice(flat.size, size=3 * k, replace=False)
        flat[idx[:k]] = rng.uniform(-1e-39, 1e-39, size=k).astype(np.float32)
        flat[idx[k:2 * k]] = 0.0
        flat[idx[2 * k:]] = -0.0
    covered = extent - uncovered
    assert covered >= 0
    if covered % align == 0 and n_groups - n_empty <= max(covered // align, 1):
        offs = random_partition(rng, covered, n_groups, n_empty, align)
    else:
        # unaligned extents: cut anywhere (the kernels must not rely on 16)
        n_pos = n_groups - n_empty
        cuts = (np.sort(rng.choice(np.arange(1, max(covered, 2)),
                                   size=max(n_pos - 1, 0), replace=False))
                if n_pos > 1 else np.zeros(0, np.int64))
        ends = list(cuts.astype(np.int64)) + [covered]
        for _ in range(n_empty):
            pos = int(rng.integers(1, len(ends))) if len(ends) > 1 else 0
            ends.insert(pos, ends[pos - 1] if pos > 0 else 0)
        offs = np.asarray(ends, dtype=np.int32)
    return Case(f"{kind}_{rows}x{cols}_g{n_groups}_s{seed}", kind,
                to_bf16_bits(x), offs, seed)


@dataclass
class WgradCase:
    """Operands of the grouped grad_weight product: e4m3 codes qa_t (T, N)
    and qx (T, K) as uint8, their fp32 scales sa (N, G) and sx (G, K), and
    int32 end offsets along T."""
    name: str
    qa_t: np.ndarray
    sa: np.ndarray
    qx: np.ndarray
    sx: np.ndarray
    offs: np.ndarray


# every e4m3 code but the two NaN codes (S.1111.111)
_FINITE_E4M3 = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)


def wgrad_case(T: int, N: int, K: int, offs, seed: int) -> WgradCase:
    """Codes drawn uniformly from the finite e4m3 codes (magnitudes 2^-9 to
    448, both signs, zeros), scales 2^U{-12..12} * U(1, 2) -- the ranges the
    two quantizers produce, without their arithmetic."""
    rng = np.random.default_rng(seed)
    offs = np.asarray(offs, np.int32)
    G = offs.shape[0]
    qa_t = rng.choice(_FINITE_E4M3, size=(T, N))
    qx = rng.choice(_FINITE_E4M3, size=(T, K))
    sa = (np.exp2(rng.integers(-12, 13, (N, G))) * rng.uniform(1, 2, (N, G))).astype(np.float32)
    sx = (np.exp2(rng.integers(-12, 13, (G, K))) * rng.uniform(1, 2, (G, K))).astype(np.float32)
    return WgradCase(f"wgrad_{T}x{N}x{K}_g{G}", qa_t, sa, qx, sx, offs)
