"""The grouped grad_weight GEMM on the tensor cores against the oracle.

The oracle's result is the exact per-group sum of e4m3 products divided by
sa * sx (double); the kernel accumulates in fp32 on the tensor cores, in an
order of its own, then multiplies by the two reciprocals and rounds to bf16.
Per element the bound is
    |gpu - exact| <= 2^-8 |exact| + 2^-12 S,
S = the same quotient of the sum of |products| (the oracle's absum): the
first term covers the bf16 rounding (half an ulp, 2^-9 relative) and the
three fp32 roundings of the epilogue; the second covers an fp32 accumulation
of up to 2^11 partial sums, each rounding at most 2^-24 of a partial sum no
larger than S.  A dropped or extra token, a transposed operand or a wrong
scale moves an element by a sizeable fraction of S and fails it.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_quantization_moe_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    import __graft_entry__

    __graft_entry__.build()
    import fp8_quantization_moe_gb300 as m

    return m


def run_gpu(gq, case):
    dev = torch.device("cuda")
    qa = torch.from_numpy(case.qa_t).to(dev).view(torch.float8_e4m3fn)
    qx = torch.from_numpy(case.qx).to(dev).view(torch.float8_e4m3fn)
    sa = torch.from_numpy(case.sa).to(dev)
    sx = torch.from_numpy(case.sx).to(dev)
    offs = torch.from_numpy(case.offs).to(dev)
    out = gq.grouped_wgrad(qa, sa, qx, sx, offs)
    gq.check_device_error()
    return out.float().cpu().numpy().astype(np.float64)


def check(got, want, absum, what):
    err = np.abs(got - want)
    bound = 2.0 ** -8 * np.abs(want) + 2.0 ** -12 * absum
    bad = err > bound
    assert not bad.any(), (
        f"{what}: {int(bad.sum())} of {bad.size} elements out of bound; first at "
        f"{np.argwhere(bad)[0]}: got {got[bad][0]}, want {want[bad][0]}, S {absum[bad][0]}")
    return float((err / np.maximum(absum, 1e-300)).max())


CASES = [
    # T, N, K, offs
    (300, 128, 256, [100, 228, 300]),                 # one tile per group, ragged chunks
    (1000, 256, 512, [160, 160, 480, 800, 960]),      # an empty group, 40 tokens uncovered
    (77, 48, 80, [33, 77]),                           # N, K below one tile: zero fill
    (4096, 128, 256, [4096]),                         # 32 token chunks in one accumulation
    (600, 384, 768, [0, 1, 16, 31, 64, 97, 128, 129, 161, 600]),  # tiny and odd groups
    (520, 272, 400, [130, 260, 390, 520]),            # ragged N and K tails
]


@pytest.mark.parametrize("T,N,K,offs", CASES)
def test_grouped_wgrad(gq, T, N, K, offs):
    case = synth.wgrad_case(T, N, K, offs, seed=900 + T + N + K)
    got = run_gpu(gq, case)
    want, absum = oracle.grouped_wgrad(case.qa_t, case.sa, case.qx, case.sx, case.offs)
    worst = check(got, want, absum, case.name)
    print(f"{case.name}: max |err| / S = {worst:.3g}")
    s0 = 0
    for g, e in enumerate(offs):  # empty groups: exact zeros
        if e <= s0:
            assert not got[g].any(), g
        s0 = max(s0, e)


def test_grouped_wgrad_output_16_byte_aligned(gq):
    """An output that is 16- but not 32-byte aligned (the contract asks for
    16) takes 16-byte stores; the bytes before it are left alone."""
    T, N, K, offs = 520, 272, 400, [130, 260, 390, 520]
    case = synth.wgrad_case(T, N, K, offs, seed=907)
    G = len(offs)
    dev = torch.device("cuda")
    buf = torch.full((G * N * K + 8,), 3.0, dtype=torch.bfloat16, device=dev)
    out = buf[8:].view(G, N, K)
    assert out.data_ptr() % 32 == 16
    gq.grouped_wgrad(torch.from_numpy(case.qa_t).to(dev), torch.from_numpy(case.sa).to(dev),
                     torch.from_numpy(case.qx).to(dev), torch.from_numpy(case.sx).to(dev),
                     torch.from_numpy(case.offs).to(dev), out=out)
    gq.check_device_error()
    assert (buf[:8].float() == 3.0).all()
    want, absum = oracle.grouped_wgrad(case.qa_t, case.sa, case.qx, case.sx, case.offs)
    check(out.float().cpu().numpy().astype(np.float64), want, absum, "16-byte aligned output")


def test_grouped_wgrad_no_tokens(gq):
    case = synth.wgrad_case(0, 32, 48, [0, 0], seed=901)
    dev = torch.device("cuda")
    out = torch.full((2, 32, 48), 7.0, dtype=torch.bfloat16, device=dev)
    gq.grouped_wgrad(torch.empty((0, 32), dtype=torch.uint8, device=dev),
                     torch.from_numpy(case.sa).to(dev),
                     torch.empty((0, 48), dtype=torch.uint8, device=dev),
                     torch.from_numpy(case.sx).to(dev),
                     torch.from_numpy(case.offs).to(dev), out=out)
    torch.cuda.synchronize()
    assert not out.float().any()


def test_grouped_wgrad_full_size_sampled(gq):
    """The benchmark shape -- 16640 tokens in 16 groups, N = 8192, K = 4096 --
    checked on 64 sampled rows n x 64 sampled columns k of every group (the
    oracle on the matching slices of the operands is exact there)."""
    T, N, K, G = 16640, 8192, 4096, 16
    rng = np.random.default_rng(902)
    offs = synth.random_partition(rng, T, G)
    case = synth.wgrad_case(T, N, K, offs, seed=903)
    dev = torch.device("cuda")
    out = gq.grouped_wgrad(torch.from_numpy(case.qa_t).to(dev), torch.from_numpy(case.sa).to(dev),
                           torch.from_numpy(case.qx).to(dev), torch.from_numpy(case.sx).to(dev),
                           torch.from_numpy(case.offs).to(dev))
    gq.check_device_error()
    ns = np.sort(np.concatenate([[0, 127, 128, N - 1], rng.choice(N, 60, replace=False)]))
    ks = np.sort(np.concatenate([[0, 255, 256, K - 1], rng.choice(K, 60, replace=False)]))
    ns, ks = np.unique(ns), np.unique(ks)
    got = out.index_select(1, torch.from_numpy(ns).cuda()).index_select(
        2, torch.from_numpy(ks).cuda()).float().cpu().numpy().astype(np.float64)
    want, absum = oracle.grouped_wgrad(np.ascontiguousarray(case.qa_t[:, ns]),
                                       np.ascontiguousarray(case.sa[ns]),
                                       np.ascontiguousarray(case.qx[:, ks]),
                                       np.ascontiguousarray(case.sx[:, ks]), case.offs)
    worst = check(got, want, absum, case.name)
    print(f"{case.name} sampled: max |err| / S = {worst:.3g}")


def test_grouped_wgrad_out_of_contract_offsets(gq):
    """Decreasing and out-of-range end offsets are read as the running
    maximum clamped to [0, T], as in the quantization calls."""
    T, N, K = 200, 128, 256
    offs = np.array([60, 40, 150, 500], np.int32)   # -> ends 60, 60, 150, 200
    case = synth.wgrad_case(T, N, K, offs, seed=905)
    got = run_gpu(gq, case)
    want, absum = oracle.grouped_wgrad(case.qa_t, case.sa, case.qx, case.sx, case.offs)
    check(got, want, absum, "out-of-contract offsets")
    assert not got[1].any()


def test_grouped_wgrad_timeout_is_reported_not_hung(gq):
    """A withheld accumulator release makes block 0's MMA warp give up after
    the (shortened) limit; every role leaves its loop, the TMEM is freed and
    the call reports GQ_ERR_TIMEOUT; the next call is fine."""
    T, N, K = 256, 1024, 2048          # 8 x 8 tiles per group: block 0 gets 4 tiles
    offs = np.arange(32, T + 1, 32, dtype=np.int32)
    case = synth.wgrad_case(T, N, K, offs, seed=906)
    try:
        gq.debug_set(skip_arrival=True, wait_timeout_ns=5_000_000)
        dev = torch.device("cuda")
        gq.grouped_wgrad(torch.from_numpy(case.qa_t).to(dev), torch.from_numpy(case.sa).to(dev),
                         torch.from_numpy(case.qx).to(dev), torch.from_numpy(case.sx).to(dev),
                         torch.from_numpy(case.offs).to(dev))
        with pytest.raises(gq.GQError) as e:
            gq.check_device_error()
        assert e.value.status == 4
    finally:
        gq.debug_set(False, 0)
    got = run_gpu(gq, case)
    want, absum = oracle.grouped_wgrad(case.qa_t, case.sa, case.qx, case.sx, case.offs)
    check(got, want, absum, "after a timeout")
