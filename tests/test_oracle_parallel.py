"""The sliced, multi-threaded oracle driver gives the same bytes as one
oracle call on the whole tensor (no GPU needed)."""
import numpy as np

import oracle
import oracle_parallel
from fp8_quantization_moe_gb300 import synth


def test_colwise_slices_equal_whole():
    c = synth.random_case("colwise", 300, 1000 - 1000 % 16, 7, seed=11, n_empty=1,
                          align=1, scale_mix=True, uncovered=9)
    fill = np.full(c.x.shape, 0x5A, np.uint8)
    for pow2 in (False, True):
        q1, s1 = oracle.colwise(c.x, c.offs, out=fill, pow2=pow2)
        q2, s2 = oracle_parallel.colwise(c.x, c.offs, out=fill, pow2=pow2)
        assert np.array_equal(q1, q2)
        assert np.array_equal(s1.view(np.uint32), s2.view(np.uint32))


def test_rowwise_slices_equal_whole():
    r = synth.random_case("rowwise_t", 600, 720, 9, seed=12, n_empty=2, align=1,
                          scale_mix=True, uncovered=5)
    fill = np.full(r.x.shape[::-1], 0x5A, np.uint8)
    for pow2 in (False, True):
        q1, s1 = oracle.rowwise_t(r.x, r.offs, out=fill, pow2=pow2)
        q2, s2 = oracle_parallel.rowwise_t(r.x, r.offs, out=fill, pow2=pow2)
        assert np.array_equal(q1, q2)
        assert np.array_equal(s1.view(np.uint32), s2.view(np.uint32))


def test_expert_and_mxfp8_slices_equal_whole():
    rng = np.random.default_rng(13)
    w = synth.to_bf16_bits(rng.standard_normal((3, 40, 600)).astype(np.float32))
    q1, s1 = oracle.expert_dim1(w)
    q2, s2 = oracle_parallel.expert_dim1(w)
    assert np.array_equal(q1, q2) and np.array_equal(s1.view(np.uint32), s2.view(np.uint32))
    w = synth.to_bf16_bits(rng.standard_normal((3, 600, 40)).astype(np.float32))
    q1, s1 = oracle.expert_rowwise(w)
    q2, s2 = oracle_parallel.expert_rowwise(w)
    assert np.array_equal(q1, q2) and np.array_equal(s1.view(np.uint32), s2.view(np.uint32))
    x = synth.to_bf16_bits(rng.standard_normal((2100, 96)).astype(np.float32))
    for mode in (0, 1):
        q1, s1 = oracle.mxfp8_dim0(x, mode)
        q2, s2 = oracle_parallel.mxfp8_dim0(x, mode)
        assert np.array_equal(q1, q2) and np.array_equal(s1, s2)
