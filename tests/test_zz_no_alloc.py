"""gq_fp8_colwise_noalloc, through the C ABI (needs an sm_103 GPU).

This entry point serves callers that cannot allocate device memory where they
quantize (a plugin inside a runtime that owns the whole device heap, or a hot
path that must not call cudaMalloc because it can synchronise the device).
Its scratch is a fixed array inside the library, so the test checks that two
calls in a row -- the second with much smaller magnitudes, which would expose
amax words left over from the first -- give the same bytes as gq_fp8_colwise
with a caller workspace and as the CPU oracle, and that a call too large for
the array is refused.

The file name makes pytest collect it last.
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

    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    return m


def _dev(case):
    x = torch.from_numpy(case.x.view(np.int16)).view(torch.bfloat16).cuda()
    return x, torch.from_numpy(case.offs).cuda()


def _noalloc(lib, x, offs, out, scales, stream):
    M, K = x.shape
    return lib.gq_fp8_colwise_noalloc(x.data_ptr(), M, K, offs.data_ptr(),
                                      offs.numel(), out.data_ptr(),
                                      scales.data_ptr(), stream)


def _with_workspace(lib, gq, x, offs, out, scales, stream):
    M, K = x.shape
    G = offs.numel()
    need = gq.workspace_bytes(gq.GQ_KIND_COLWISE, M, K, G)
    ws = torch.empty(need + 256, dtype=torch.uint8, device=x.device)
    p = (ws.data_ptr() + 255) & ~255
    st = lib.gq_fp8_colwise(x.data_ptr(), M, K, offs.data_ptr(), G,
                            out.data_ptr(), scales.data_ptr(), p,
                            ws.numel() - (p - ws.data_ptr()), stream)
    return st, ws


def test_noalloc_matches_workspace_path_twice(gq):
    lib = gq.lib()
    stream = torch.cuda.current_stream().cuda_stream
    big = synth.random_case("colwise", 2048, 4096, 16, seed=901, n_empty=1,
                            scale_mix=True)
    small = synth.random_case("colwise", 1500, 4096, 60, seed=902, n_empty=3,
                              align=1)
    # second call: magnitudes in [2^-7, 2^-6) instead of up to ~10^3, so any
    # amax word left over from the first call would change its scales
    small.x = (small.x & np.uint16(0x807F)) | np.uint16(120 << 7)
    for case in (big, small):
        x, offs = _dev(case)
        M, K = x.shape
        G = offs.numel()
        assert gq.workspace_bytes(gq.GQ_KIND_COLWISE, M, K, G) <= (1 << 20)
        q1 = torch.full((M, K), 0x5A, dtype=torch.uint8, device="cuda")
        s1 = torch.empty((G, K), dtype=torch.float32, device="cuda")
        q2 = q1.clone()
        s2 = torch.empty_like(s1)
        assert _noalloc(lib, x, offs, q1, s1, stream) == 0
        st, ws = _with_workspace(lib, gq, x, offs, q2, s2, stream)
        assert st == 0
        torch.cuda.synchronize()
        assert lib.gq_check_device_error(stream) == 0
        assert torch.equal(q1, q2), case.name
        assert torch.equal(s1.view(torch.int32), s2.view(torch.int32)), case.name
        # and the oracle, byte for byte (rows past the last group keep 0x5A)
        rq, rs = oracle.colwise(case.x, case.offs,
                                out=np.full((M, K), 0x5A, np.uint8))
        assert np.array_equal(q1.cpu().numpy(), rq), case.name
        assert np.array_equal(s1.cpu().numpy().view(np.uint32), rs.view(np.uint32)), case.name
        del ws


def test_noalloc_refuses_calls_beyond_the_scratch(gq):
    lib = gq.lib()
    M, K, G = 64, 4096, 64  # 64 * 4096 amax words: just over 1 MiB
    assert gq.workspace_bytes(gq.GQ_KIND_COLWISE, M, K, G) > (1 << 20)
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    offs = torch.full((G,), M, dtype=torch.int32, device="cuda")
    q = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    s = torch.empty((G, K), dtype=torch.float32, device="cuda")
    st = _noalloc(lib, x, offs, q, s, torch.cuda.current_stream().cuda_stream)
    assert st == gq._binding.GQ_ERR_UNSUPPORTED
    assert b"GQ_NOALLOC_SCRATCH_BYTES" in lib.gq_last_error()
