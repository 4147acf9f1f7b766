"""Pins that tie the CPU oracle to facts outside itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with what the pages, the e4m3 format definition, the
mathematics or an independent library routine fix.  ``test_oracle_pins.py``
runs them on the real oracle; ``test_oracle_mutants.py`` runs them on copies
of the oracle with a planted mistake and requires each copy to fail one.
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np
import torch

import ref_loop
from fp8_quantization_moe_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f32_from_bits(u):
    return np.asarray(u, np.uint32).view(np.float32)


def _torch_e4m3(v):
    return ref_loop.cast_e4m3(np.asarray(v, np.float32))


# ------------------------------------------------------------ the format --

def pin_decode_landmarks(o):
    """Decode agrees with the OCP E4M3 table's landmark codes."""
    g = _golden("e4m3_landmarks.json")
    for code, val in g["codes"].items():
        got = o.e4m3_decode([int(code, 16)])[0]
        assert got == val and np.signbit(got) == np.signbit(val), (code, got, val)
    for code in g["nan_codes"]:
        assert np.isnan(o.e4m3_decode([int(code, 16)])[0]), code


def pin_decode_vs_torch(o):
    """All 256 codes decode as torch.float8_e4m3fn does."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = o.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def pin_encode_roundtrip(o):
    """encode(decode(c)) == c for every finite code, signed zeros included."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = o.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(o.e4m3_encode(vals), codes)


def pin_encode_midpoints(o):
    """Exact midpoints between neighbouring codes go to the even code; one
    fp32 ulp either side goes to the nearer code."""
    pos = o.e4m3_decode(np.arange(0, 127, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)
    for c in range(126):
        lo, hi = pos[c], pos[c + 1]
        mid = np.float32((lo + hi) / 2)  # exact: at most 5 significant bits
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(np.inf))
        got = o.e4m3_encode(np.array([mid, below, above, -mid], np.float32))
        assert list(got) == [even, c, c + 1, even | 0x80], (c, got)


def pin_encode_boundaries(o):
    """Saturation at +-448 (the pages' fp8_dtype_max / min) and underflow."""
    k = _golden("pages_constants.json")
    cases = [
        (k["fp8_dtype_max"], 0x7E), (k["fp8_dtype_min"], 0xFE),
        (463.99, 0x7E), (464.0, 0x7E), (480.0, 0x7E), (1e30, 0x7E),
        (-1e30, 0xFE), (float(np.finfo(np.float32).max), 0x7E),
        (float("inf"), 0x7E),
        (2.0 ** -10, 0x00), (-(2.0 ** -10), 0x80), (2.0 ** -12, 0x00),
        (float(np.nextafter(np.float32(2.0 ** -10), np.float32(1))), 0x01),
        (0.0, 0x00), (-0.0, 0x80),
    ]
    vals = np.array([v for v, _ in cases], np.float32)
    got = o.e4m3_encode(vals)
    for (v, want), g in zip(cases, got):
        assert g == want, (v, hex(g), hex(want))
    assert o.e4m3_decode([0x7E])[0] == k["fp8_dtype_max"]
    assert o.e4m3_decode([0xFE])[0] == k["fp8_dtype_min"]


def pin_encode_vs_torch(o, exp_lo=116, exp_hi=135, stride=1, neg_stride=97):
    """Every positive fp32 with biased exponent in [exp_lo, exp_hi] (2^-11 up
    to 2^9) encodes as torch's RNE cast after clamping; negatives on a strided
    sample must mirror with the sign bit; below 2^-11 everything is a signed
    zero and at or above 448 everything saturates."""
    mant = np.arange(0, 1 << 23, stride, dtype=np.uint32)
    for e in range(exp_lo, exp_hi + 1):
        v = _f32_from_bits((np.uint32(e) << 23) | mant)
        got = o.e4m3_encode(v)
        ref = _torch_e4m3(v)
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, (e, v[bad[:4]], got[bad[:4]], ref[bad[:4]])
        vn = -v[::neg_stride]
        assert np.array_equal(o.e4m3_encode(vn), ref[::neg_stride] | 0x80), e
    rng = np.random.default_rng(5)
    tiny = _f32_from_bits(rng.integers(0, 116 << 23, size=100_000,
                                       dtype=np.uint32))
    assert np.all(o.e4m3_encode(tiny) == 0) and np.all(o.e4m3_encode(-tiny) == 0x80)
    big = _f32_from_bits(rng.integers(0x43E00000, 0x7F800000, size=100_000,
                                      dtype=np.uint32))
    assert np.all(o.e4m3_encode(big) == 0x7E) and np.all(o.e4m3_encode(-big) == 0xFE)


# ---------------------------------------------------------------- scale --

def _is_rn_f32(s: np.float32, exact: Fraction) -> bool:
    fs = Fraction(float(s))
    lo = Fraction(float(np.nextafter(s, np.float32(0))))
    hi = Fraction(float(np.nextafter(s, np.float32(np.inf))))
    d, dl, dh = abs(exact - fs), abs(exact - lo), abs(exact - hi)
    if d < dl and d < dh:
        return True
    if d == dl or d == dh:  # a tie: the kept value must have an even mantissa
        return int(np.float32(s).view(np.uint32)) % 2 == 0
    return False


def pin_scale_exact(o):
    """For every finite non-negative bf16 amax (|x| of a bf16 is a bf16), the
    scale is the correctly rounded fp32 of 448 / max(amax, fp32(1e-12)),
    checked in exact rational arithmetic."""
    k = _golden("pages_constants.json")
    bits = np.arange(0, 0x7F80, dtype=np.uint32)  # +0 .. largest finite bf16
    amax = _f32_from_bits(bits << 16)
    got = o.scale_of(amax)
    eps = Fraction(float(np.float32(k["EPS"])))
    num = Fraction(k["fp8_dtype_max"])
    for a, s in zip(amax.tolist(), got):
        d = max(Fraction(a), eps)
        assert _is_rn_f32(np.float32(s), num / d), (a, s)


def pin_quant_single_rounding(o):
    """q(x, s) = e4m3(RN_fp32(x * s)): the exact product (8 x 24 significant
    bits fits a double) is rounded once to fp32, then cast by torch.  Half the
    samples are random; the other half put x * s within a few fp32 ulps of an
    e4m3 rounding midpoint, where a second rounding or a reassociated product
    would flip the code."""
    rng = np.random.default_rng(11)
    n = 200_000
    xb = rng.integers(0, 1 << 16, size=n, dtype=np.uint32).astype(np.uint16)
    xb = xb[((xb & 0x7F80) != 0x7F80) & ((xb & 0x7FFF) > 0x0100)]
    xf = ref_loop.bf16_bits_to_f32(xb)
    with np.errstate(over="ignore"):
        amax = np.abs(xf) * rng.uniform(1.0, 4.0, size=xf.size).astype(np.float32)
    s_rand = ref_loop.FP8_MAX / np.maximum(amax, ref_loop.EPS)
    # near-tie samples: target an e4m3 midpoint t, take s = RN(t / x) +- k ulp
    mags = o.e4m3_decode(np.arange(0, 127, dtype=np.uint8))
    mids = (mags[:-1] + mags[1:]) / 2
    t = mids[rng.integers(0, mids.size, size=xf.size)]
    with np.errstate(over="ignore"):
        s0 = (t / np.abs(xf.astype(np.float64))).astype(np.float32)
    k = rng.integers(-3, 4, size=xf.size).astype(np.int32)
    s_tie = (s0.view(np.int32) + k).view(np.float32)
    ok = np.isfinite(s_tie) & (s_tie > 0)
    for xs, ss in ((xb, s_rand), (xb[ok], s_tie[ok])):
        xs_f = ref_loop.bf16_bits_to_f32(xs).astype(np.float64)
        v = (xs_f * ss.astype(np.float64)).astype(np.float32)
        assert np.array_equal(o.quant(xs, ss), _torch_e4m3(v))


def pin_hand_examples(o):
    """Hand-worked single-group columns."""
    g = _golden("hand_examples.json")
    for col in g["columns"]:
        x = np.array(col["x"], np.float32)
        xb = synth.to_bf16_bits(x)
        assert np.array_equal(ref_loop.bf16_bits_to_f32(xb), x)  # bf16-exact
        q, s = o.colwise(xb.reshape(-1, 1), np.array([x.size], np.int32))
        want = [int(c, 16) for c in col["q"]]
        assert q.reshape(-1).tolist() == want, (col["x"], q.reshape(-1), want)
        if "scale" in col:
            assert s[0, 0] == np.float32(col["scale"]), (s[0, 0], col["scale"])
        else:
            assert hex(int(s[0, 0:1].view(np.uint32)[0])) == col["scale_bits"]


# ------------------------------------------------------ whole-path pins --

SMALL_CASES = [
    # (kind, rows, cols, n_groups, seed, n_empty, align, scale_mix, uncovered)
    ("colwise", 64, 48, 3, 1, 0, 16, False, 0),
    ("colwise", 96, 32, 5, 2, 2, 16, True, 0),
    ("colwise", 80, 16, 4, 3, 1, 16, True, 16),
    ("colwise", 37, 24, 4, 4, 1, 1, True, 5),
    ("colwise", 1, 16, 1, 5, 0, 1, False, 0),
    ("rowwise_t", 48, 64, 3, 6, 0, 16, False, 0),
    ("rowwise_t", 32, 96, 5, 7, 2, 16, True, 0),
    ("rowwise_t", 16, 80, 4, 8, 1, 16, True, 16),
    ("rowwise_t", 24, 41, 4, 9, 1, 1, True, 3),
]


def _small_cases():
    for k, r, c, g, s, ne, al, mix, unc in SMALL_CASES:
        yield synth.random_case(k, r, c, g, seed=s, n_empty=ne, align=al,
                                scale_mix=mix, uncovered=unc)


def pin_paths_vs_library_loop(o):
    """Both paths equal the torch-loop restatement bit for bit on small cases
    with empty groups, uncovered tail tokens, subnormals and signed zeros;
    untouched elements keep a sentinel."""
    for case in _small_cases():
        fill = np.full((case.x.shape if case.kind == "colwise"
                        else case.x.shape[::-1]), 0x5A, np.uint8)
        if case.kind == "colwise":
            q, s = o.colwise(case.x, case.offs, out=fill)
            rq, rs = ref_loop.colwise(case.x, case.offs, fill=0x5A)
        else:
            q, s = o.rowwise_t(case.x, case.offs, out=fill)
            rq, rs = ref_loop.rowwise_t(case.x, case.offs, fill=0x5A)
        assert np.array_equal(q, rq), case.name
        assert np.array_equal(s.view(np.uint32), rs.view(np.uint32)), case.name


def pin_out_of_contract_offsets(o):
    """Decreasing and out-of-range offsets are read as the running maximum
    clamped to the extent (the library's documented reading)."""
    case = synth.random_case("colwise", 64, 16, 4, seed=21)
    bad = np.array([32, 16, 80, -5], np.int32)  # -> ends 32, 32, 64, 64
    q, s = o.colwise(case.x, bad)
    rq, rs = ref_loop.colwise(case.x, np.array([32, 32, 64, 64], np.int32))
    assert np.array_equal(q, rq) and np.array_equal(s, rs)


def pin_transpose_identity(o):
    """rowwise_t(A) == colwise(A^T) with the scales transposed -- the
    transpose method of the #2863 page, as an identity between the paths."""
    for seed in (31, 32):
        case = synth.random_case("rowwise_t", 40, 112, 6, seed=seed, n_empty=1,
                                 scale_mix=True)
        qt, s_r = o.rowwise_t(case.x, case.offs)
        q, s_c = o.colwise(np.ascontiguousarray(case.x.T), case.offs)
        assert np.array_equal(qt, q)
        assert np.array_equal(s_r, s_c.T)


def pin_max_code_invariant(o):
    """Every group column with amax >= 1e-12 contains a +-448 code; no NaN
    codes appear; all-zero columns give zero codes and the empty-group scale."""
    case = synth.colwise_outliers()
    x = case.x[:, :512].copy()
    q, s = o.colwise(x, case.offs)
    xf = ref_loop.bf16_bits_to_f32(x)
    empty_scale = np.float32(448.0) / np.float32(1e-12)
    assert not np.any((q & 0x7F) == 0x7F)
    for (a, b), g in zip(ref_loop.bounds(case.offs, x.shape[0]),
                         range(case.n_groups)):
        if b == a:
            assert np.all(s[g] == empty_scale)
            continue
        amax = np.abs(xf[a:b]).max(axis=0)
        nz = amax >= np.float32(1e-12)
        hit = np.any((q[a:b] & 0x7F) == 0x7E, axis=0)
        assert np.array_equal(hit[nz], np.ones(nz.sum(), bool)), g
        assert np.all(q[a:b][:, amax == 0] & 0x7F == 0)
        assert np.all(s[g][amax == 0] == empty_scale)


def pin_dequant_bound(o):
    """decode(q) / scale is within half an e4m3 ulp of x: relative 2^-4 in
    the normal range, absolute 2^-10 / scale below it."""
    case = synth.random_case("colwise", 256, 64, 4, seed=41, scale_mix=True)
    q, s = o.colwise(case.x, case.offs)
    xf = ref_loop.bf16_bits_to_f32(case.x).astype(np.float64)
    for (a, b), g in zip(ref_loop.bounds(case.offs, xf.shape[0]),
                         range(case.n_groups)):
        if b == a:
            continue
        deq = o.e4m3_decode(q[a:b]) / s[g].astype(np.float64)
        err = np.abs(deq - xf[a:b])
        lim = np.maximum(np.abs(xf[a:b]) * 2.0 ** -4,
                         2.0 ** -10 / s[g].astype(np.float64))
        assert np.all(err <= lim * (1 + 1e-6)), g


def pin_scale_pow2(o):
    """round_scales_to_power_of_2 (the kernel argument in #2668's failure
    report): for every finite non-negative bf16 amax the rounded scale is an
    exact power of two, at or below the plain scale and above half of it --
    that is, 2^floor(log2(scale)), checked without restating the formula."""
    bits = np.arange(0, 0x7F80, dtype=np.uint32)
    amax = _f32_from_bits(bits << 16)
    s = o.scale_of(amax).astype(np.float64)
    s2 = o.scale_pow2_of(amax).astype(np.float64)
    mant, _ = np.frexp(s2)
    assert np.all(mant == 0.5), "not a power of two"
    assert np.all(s2 <= s) and np.all(s < 2 * s2)


def pin_pow2_paths(o):
    """Both paths with power-of-two scales: every scale is the pinned
    rounding of its amax's plain scale; each element is the e4m3 code of the
    exact product x * 2^k (a bf16 times a power of two is exact in fp32 for
    these magnitudes); in a group column with amax >= 1e-12 the largest code
    lies in [224, 448]; and rowwise_t(A) == colwise(A^T) still holds."""
    case = synth.random_case("colwise", 300, 48, 5, seed=47, n_empty=1, align=1,
                             scale_mix=True)
    q, s = o.colwise(case.x, case.offs, pow2=True)
    qp, sp = o.colwise(case.x, case.offs)
    s64, sp64 = s.astype(np.float64), sp.astype(np.float64)
    mant, _ = np.frexp(s64)
    assert np.all(mant == 0.5)
    assert np.all((s64 <= sp64) & (sp64 < 2 * s64))
    xf = ref_loop.bf16_bits_to_f32(case.x).astype(np.float64)
    for (a, b), g in zip(ref_loop.bounds(case.offs, xf.shape[0]), range(case.n_groups)):
        if b == a:
            continue
        exact = xf[a:b] * s[g].astype(np.float64)[None, :]
        assert np.array_equal(q[a:b], o.e4m3_encode(exact.astype(np.float32))), g
        mag = np.abs(o.e4m3_decode(q[a:b])).max(axis=0)
        col = np.abs(xf[a:b]).max(axis=0) >= 1e-12
        assert np.all((mag[col] >= 224) & (mag[col] <= 448)), g
    qt, st = o.rowwise_t(np.ascontiguousarray(case.x.T), case.offs, pow2=True)
    assert np.array_equal(qt, q) and np.array_equal(st, s.T)


def pin_expert_dim1(o):
    """Stacked expert weights along dim1: a numpy / torch restatement of the
    definition (per expert and column: amax over the expert's K rows, fp32
    scale, torch's RNE-saturating e4m3 cast of the fp32 product) on ragged
    small shapes with per-row magnitudes over six decades, K = 0 included;
    and the identity with colwise on the (E * K, N) stack with E groups of
    K rows."""
    rng = np.random.default_rng(49)
    for E, K, N in ((1, 5, 16), (3, 50, 32), (4, 0, 16), (2, 33, 48)):
        x = rng.standard_normal((E, K, N)).astype(np.float32)
        x *= np.power(np.float32(10), rng.uniform(-3, 3, size=(E, K, 1))).astype(np.float32)
        w = synth.to_bf16_bits(x)
        q, s = o.expert_dim1(w)
        wf = ref_loop.bf16_bits_to_f32(w)
        for e in range(E):
            amax = np.abs(wf[e]).max(axis=0) if K else np.zeros(N, np.float32)
            se = np.float32(448.0) / np.maximum(amax, np.float32(1e-12))
            assert np.array_equal(s[e], se.astype(np.float32)), (E, K, N, e)
            if K:
                v = (wf[e] * se[None, :]).astype(np.float32)
                assert np.array_equal(q[e], _torch_e4m3(np.clip(v, -448, 448))), (E, K, N, e)
        if K:
            offs = (np.arange(1, E + 1) * K).astype(np.int32)
            qc, sc = o.colwise(w.reshape(E * K, N), offs)
            assert np.array_equal(qc, q.reshape(E * K, N)) and np.array_equal(sc, s)


def pin_expert_rowwise(o):
    """Stacked expert weights per row: a numpy / torch restatement of the
    definition (per expert and row: amax over the row's K elements, fp32
    scale, torch's RNE-saturating e4m3 cast of the fp32 product) on ragged
    small shapes with per-row magnitudes over six decades, K = 0 and N = 0
    included, plain and power-of-two scales; and the identity with rowwise_t
    on each expert's (N, K) matrix as one group of K tokens, whose output is
    the transpose."""
    rng = np.random.default_rng(53)
    for E, N, K in ((1, 5, 16), (3, 7, 40), (2, 4, 0), (2, 0, 8), (2, 9, 33)):
        x = rng.standard_normal((E, N, K)).astype(np.float32)
        x *= np.power(np.float32(10), rng.uniform(-3, 3, size=(E, N, 1))).astype(np.float32)
        if N > 1 and K:
            x[0, 1] = 0.0  # an all-zero row: scale 448 / 1e-12
        w = synth.to_bf16_bits(x)
        wf = ref_loop.bf16_bits_to_f32(w)
        amax = np.abs(wf).max(axis=2) if K else np.zeros((E, N), np.float32)
        se = (np.float32(448.0) / np.maximum(amax, np.float32(1e-12))).astype(np.float32)
        for pow2 in (False, True):
            q, s = o.expert_rowwise(w, pow2=pow2)
            assert q.shape == (E, N, K) and s.shape == (E, N)
            if pow2:  # a power of two at or below the plain scale, above half of it
                mant, _ = np.frexp(s.astype(np.float64))
                assert np.all(mant == 0.5) and np.all(s <= se) and np.all(se < 2 * s), (E, N, K)
            else:
                assert np.array_equal(s, se), (E, N, K)
            if K and N:
                v = (wf * s[:, :, None]).astype(np.float32)
                assert np.array_equal(q, _torch_e4m3(np.clip(v, -448, 448))), (E, N, K, pow2)
        if K and N:
            q, s = o.expert_rowwise(w)
            for e in range(E):
                qt, st = o.rowwise_t(np.ascontiguousarray(w[e]), np.array([K], np.int32))
                assert np.array_equal(qt.T, q[e]) and np.array_equal(st[:, 0], s[e])


def _mx_input(rng, M, K):
    """Rows of blocks with magnitudes from 2^-140 to 2^120, zero blocks,
    bf16 subnormals, signed zeros and exact powers of two."""
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= np.power(np.float32(2), rng.integers(-140, 121, size=(M, K // 32, 1)).astype(np.float32)
                  ).repeat(32, axis=2).reshape(M, K)
    bits = synth.to_bf16_bits(x)
    special = [
        np.zeros(32, np.uint16),                                      # a zero block
        np.full(32, 0x8000, np.uint16),                               # negative zeros
        np.arange(1, 33, dtype=np.uint16),                            # bf16 subnormals
        0x4000 | np.arange(0, 32, dtype=np.uint16) % 2 * 0x0080,      # 2 and 4
    ]
    per_row = 2 if K >= 64 else 1          # two special blocks a row where they fit
    for i, blk in enumerate(special):
        r, c = divmod(i, per_row)
        if r < M:
            bits[r, 32 * c:32 * c + 32] = blk
    return bits


def pin_mxfp8_dim0(o):
    """mxfp8 along dim0, checked block by block without restating the
    exponent rule: zero blocks get byte 0 and zero codes; otherwise, with
    E = byte - 127 and E not clamped, amax * 2^-E lies in [256, 512) under
    FLOOR and in (224, 448] under RCEIL (up to the rounding of amax / 448),
    and every element is torch's saturating RNE e4m3 cast of the fp32
    product x * 2^-E."""
    rng = np.random.default_rng(53)
    bits = _mx_input(rng, 24, 256)
    xf = ref_loop.bf16_bits_to_f32(bits)
    for mode in (0, 1):
        q, s = o.mxfp8_dim0(bits, mode)
        E = s.astype(np.int64) - 127
        for r in range(bits.shape[0]):
            for b in range(bits.shape[1] // 32):
                xb = xf[r, 32 * b:32 * b + 32]
                amax = float(np.abs(xb).max())
                if amax == 0.0:
                    assert s[r, b] == 0 and not np.any(q[r, 32 * b:32 * b + 32] & 0x7F)
                    continue
                e = int(E[r, b])
                t = amax * 2.0 ** -e
                if -127 < e < 127:
                    if mode == 0:
                        assert 256 <= t < 512, (r, b, amax, e)
                    else:
                        assert 224 * (1 - 2 ** -23) < t <= 448 * (1 + 2 ** -23), (r, b, amax, e)
                f = np.float32(np.ldexp(1.0, -e))
                want = _torch_e4m3(np.clip((xb * f).astype(np.float32), -448, 448))
                assert np.array_equal(q[r, 32 * b:32 * b + 32], want), (mode, r, b)



def _torch_decode_f64(codes):
    """torch's own e4m3 decode, in float64 (independent of the oracle's)."""
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()


def pin_wgrad_hand(o):
    """grad_weight per token group worked by hand: 4 tokens, groups [0, 1),
    [1, 1) (empty) and [1, 3); token 3 belongs to no group.  Codes 0x38 = 1,
    0x40 = 2, 0x30 = 0.5, 0xC8 = -4, 0xC0 = -2; the scales are powers of two,
    so every quotient below is exact."""
    qa = np.array([[0x38, 0x40], [0x30, 0xC8], [0x38, 0x38], [0x7E, 0x7E]], np.uint8)
    qx = np.array([[0x40, 0x30], [0x38, 0x38], [0xC0, 0x38], [0x7E, 0xFE]], np.uint8)
    sa = np.array([[2, 64, 4], [0.5, 64, 1]], np.float32)        # (N, G)
    sx = np.array([[1, 8], [64, 64], [0.25, 2]], np.float32)      # (G, K)
    out, absum = o.grouped_wgrad(qa, sa, qx, sx, np.array([1, 1, 3], np.int32))
    # group 0: token 0 alone, a = (1, 2), x = (2, 0.5)
    want0 = [[2 / (2 * 1), 0.5 / (2 * 8)], [4 / (0.5 * 1), 1 / (0.5 * 8)]]
    # group 2: tokens 1 and 2: sums (-1.5, 1.5; -6, -3), |sums| (2.5, 1.5; 6, 5)
    want2 = [[-1.5 / (4 * 0.25), 1.5 / (4 * 2)], [-6 / (1 * 0.25), -3 / (1 * 2)]]
    abs2 = [[2.5 / (4 * 0.25), 1.5 / (4 * 2)], [6 / (1 * 0.25), 5 / (1 * 2)]]
    assert np.array_equal(out[0], np.array(want0)), out[0]
    assert np.array_equal(out[1], np.zeros((2, 2))), out[1]
    assert np.array_equal(out[2], np.array(want2)), out[2]
    assert np.array_equal(absum[2], np.array(abs2)), absum[2]


def pin_wgrad_vs_matmul(o):
    """Each group's result times sa * sx is the plain matrix product of the
    decoded operands over the group's tokens (numpy's float64 matmul of
    torch-decoded values: every product and sum is exact, so any summation
    order gives the same numbers), with empty groups, ragged sizes and
    uncovered tokens; the same for |products|."""
    rng = np.random.default_rng(59)
    T, N, K = 150, 40, 24
    offs = np.array([13, 13, 61, 100, 141], np.int32)   # an empty group; 9 tokens uncovered
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    qa = rng.choice(finite, size=(T, N))
    qx = rng.choice(finite, size=(T, K))
    G = offs.shape[0]
    sa = (np.exp2(rng.integers(-10, 11, (N, G))) * rng.uniform(1, 2, (N, G))).astype(np.float32)
    sx = (np.exp2(rng.integers(-10, 11, (G, K))) * rng.uniform(1, 2, (G, K))).astype(np.float32)
    out, absum = o.grouped_wgrad(qa, sa, qx, sx, offs)
    da, dx = _torch_decode_f64(qa), _torch_decode_f64(qx)
    s0 = 0
    for g in range(G):
        e = int(offs[g])
        d = sa[:, g].astype(np.float64)[:, None] * sx[g].astype(np.float64)[None, :]
        want = da[s0:e].T @ dx[s0:e]
        wabs = np.abs(da[s0:e]).T @ np.abs(dx[s0:e])
        assert np.allclose(out[g] * d, want, rtol=2.0 ** -50, atol=0), g
        assert np.allclose(absum[g] * d, wabs, rtol=2.0 ** -50, atol=0), g
        s0 = e


ALL_PINS = [
    pin_decode_landmarks, pin_decode_vs_torch, pin_encode_roundtrip,
    pin_encode_midpoints, pin_encode_boundaries, pin_encode_vs_torch,
    pin_scale_exact, pin_quant_single_rounding, pin_hand_examples,
    pin_paths_vs_library_loop, pin_out_of_contract_offsets,
    pin_transpose_identity, pin_max_code_invariant, pin_dequant_bound,
    pin_scale_pow2, pin_pow2_paths, pin_expert_dim1, pin_expert_rowwise, pin_mxfp8_dim0,
    pin_wgrad_hand, pin_wgrad_vs_matmul,
]
