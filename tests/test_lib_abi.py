"""The C ABI without a GPU: the library builds, loads, exports every symbol
the header declares, and rejects bad arguments on the host before touching
CUDA (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gq_fp8.h")


@pytest.fixture(scope="module")
def gq():
    import __graft_entry__

    __graft_entry__.build()
    import fp8_quantization_moe_gb300 as m

    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for need in ("gq_fp8_colwise", "gq_fp8_rowwise_t", "gq_workspace_bytes",
                 "gq_check_device_error", "gq_status_string"):
        assert need in names


def test_library_exports_every_declared_symbol(gq):
    lib = ctypes.CDLL(gq.library_path())
    for name in declared_functions():
        assert hasattr(lib, name), name
    from fp8_quantization_moe_gb300 import _binding
    assert set(_binding.SIGNATURES) == set(declared_functions())


def test_constants_match_header(gq):
    text = open(HEADER).read()
    assert f"#define GQ_MAX_GROUPS {gq.GQ_MAX_GROUPS}" in text
    assert f"#define GQ_KIND_COLWISE {gq.GQ_KIND_COLWISE}" in text
    assert f"#define GQ_KIND_ROWWISE_T {gq.GQ_KIND_ROWWISE_T}" in text


def test_status_strings(gq):
    assert gq.status_string(0) == "ok"
    assert gq.status_string(4) == "device wait timed out"
    assert gq.version() >= 100


def test_workspace_bytes(gq):
    # colwise 65536x4096, 16 groups: 256 B header + 16 x 32 strip counters
    # (2 KiB) + 16*4096 amax words
    assert gq.workspace_bytes(0, 65536, 4096, 16) == 256 + 2048 + 16 * 4096 * 4
    # regions padded to 256 bytes: 3 groups x 2 slabs (K = 144), 3 x 144
    # amax words
    assert gq.workspace_bytes(0, 100, 144, 3) == 256 + 256 + 1792
    # rowwise_t: a unit counter and a finished-blocks counter, padded
    # rowwise_t: 256 B header + 68 words per (band, group) unit that may be
    # split (groups of 4090 tokens or more: at most 16640 // 4090 = 4)
    assert gq.workspace_bytes(1, 8192, 16640, 64) == 256 + 128 * 4 * 68 * 4
    assert gq.workspace_bytes(1, 8192, 16640, 2) == 256 + 128 * 2 * 68 * 4
    assert gq.workspace_bytes(1, 64, 4089, 8) == 256
    assert gq.workspace_bytes(0, 0, 4096, 4) == 0
    assert gq.workspace_bytes(1, 16, 0, 4) == 0
    assert gq.workspace_bytes(0, 16, 16, 0) == 0
    assert gq.workspace_bytes(0, 16, 16, gq.GQ_MAX_GROUPS + 1) == 0
    assert gq.workspace_bytes(7, 16, 16, 1) == 0


# Fake device addresses: the host-side checks return before any CUDA call,
# so these are never dereferenced.
A16 = 0x10000
BAD = 0x10008


@pytest.mark.parametrize("args,status", [
    # x, M, K, offs, G, out, scales, ws, ws_bytes
    ((A16, -1, 16, A16, 1, A16, A16, A16, 1 << 20), 1),
    ((A16, 16, 16, None, 1, A16, A16, A16, 1 << 20), 1),
    ((A16, 16, 16, A16, 0, A16, A16, A16, 1 << 20), 1),
    ((A16, 16, 16, A16, 1025, A16, A16, A16, 1 << 20), 2),
    ((None, 16, 16, A16, 1, A16, A16, A16, 1 << 20), 1),
    ((BAD, 16, 16, A16, 1, A16, A16, A16, 1 << 20), 1),
    ((A16, 16, 16, A16, 1, BAD, A16, A16, 1 << 20), 1),
    ((A16, 16, 24, A16, 1, A16, A16, A16, 1 << 20), 2),
    ((A16, 16, 16, A16, 1, A16, None, A16, 1 << 20), 1),
    ((A16, 16, 16, A16, 1, A16, A16, None, 0), 1),
    ((A16, 16, 16, A16, 1, A16, A16, A16, 16), 1),
    ((A16, 16, 16, A16, 1, A16, A16, A16 + 16, 1 << 20), 1),
    ((A16, 1 << 31, 16, A16, 1, A16, A16, A16, 1 << 40), 2),
])
def test_colwise_host_validation(gq, args, status):
    lib = gq.lib()
    assert lib.gq_fp8_colwise(*args, None) == status
    assert lib.gq_last_error() != b""


@pytest.mark.parametrize("args,status", [
    # a, N, Mg, offs, G, out_t, scales, ws, ws_bytes
    ((A16, 24, 64, A16, 1, A16, A16, A16, 1 << 20), 2),   # N % 16
    ((A16, 16, 20, A16, 1, A16, A16, A16, 1 << 20), 2),   # Mg % 8
    ((A16, 16, 64, A16, 1, A16, BAD + 2, A16, 1 << 20), 1),
    ((A16, -16, 64, A16, 1, A16, A16, A16, 1 << 20), 1),
    ((A16, 16, 64, A16, 1, None, A16, A16, 1 << 20), 1),
    ((A16, 16, 64, A16, 1, A16, A16, A16, 100), 1),
])
def test_rowwise_host_validation(gq, args, status):
    lib = gq.lib()
    assert lib.gq_fp8_rowwise_t(*args, None) == status


def test_debug_set_rejects_negative_timeout(gq):
    assert gq.lib().gq_debug_set(0, -1) == 1
    assert gq.lib().gq_debug_set(4, 0) == 1   # unknown flag bit
    assert gq.lib().gq_debug_set(3, 0) == 0
    assert gq.lib().gq_debug_set(0, 0) == 0


def test_set_lag_validation(gq):
    lib = gq.lib()
    assert lib.gq_set_lag(7, 1) == 1          # unknown kind
    assert lib.gq_set_lag(0, -1) == 1         # negative lag
    assert lib.gq_set_lag(0, 3) == 0
    assert lib.gq_set_lag(1, 0) == 0
    assert lib.gq_set_lag(0, 0) == 0          # back to automatic


def test_binding_rejects_cpu_tensors(gq):
    import torch
    x = torch.zeros((16, 16), dtype=torch.bfloat16)
    o = torch.tensor([16], dtype=torch.int32)
    with pytest.raises(ValueError):
        gq.colwise(x, o)
    with pytest.raises(ValueError):
        gq.rowwise_t(x, o)


def test_ex_calls_reject_unknown_flags(gq):
    """The _ex calls check their flags before anything else (no GPU needed)."""
    lib = gq.lib()
    assert gq.GQ_SCALE_POW2 == 1
    assert gq.GQ_WORKSPACE_ZEROED == 2
    assert gq.GQ_TWO_PHASE == 4
    for bad in (8, 0x80000000, 15):
        assert lib.gq_fp8_colwise_ex(A16, 16, 16, A16, 1, A16, A16, bad, A16, 1 << 20, None) == 1
    for bad in (4, 0x80000000, 7):   # GQ_TWO_PHASE is colwise's alone
        assert lib.gq_fp8_rowwise_t_ex(A16, 16, 16, A16, 1, A16, A16, bad, A16, 1 << 20, None) == 1


@pytest.mark.parametrize("args,status", [
    # w, E, K, N, out, scales, flags, ws, ws_bytes
    ((A16, 0, 16, 16, A16, A16, 0, A16, 1 << 20), 1),      # no experts
    ((A16, 2000, 16, 16, A16, A16, 0, A16, 1 << 20), 2),   # > GQ_MAX_GROUPS
    ((A16, 2, 16, 24, A16, A16, 0, A16, 1 << 20), 2),      # N % 16
    ((A16, 2, -1, 16, A16, A16, 0, A16, 1 << 20), 1),      # negative K
    ((A16, 2, 16, 16, A16, A16, 8, A16, 1 << 20), 1),      # unknown flag
    ((A16, 2, 16, 16, None, A16, 0, A16, 1 << 20), 1),     # NULL output
    ((A16, 2, 16, 16, A16, A16, 0, A16, 100), 1),          # workspace too small
    ((A16, 4, 1 << 30, 16, A16, A16, 0, A16, 1 << 20), 2),  # E * K >= 2^31
])
def test_expert_dim1_host_validation(gq, args, status):
    assert gq.lib().gq_fp8_expert_dim1(*args, None) == status


@pytest.mark.parametrize("args,status", [
    # x, M, K, out, scales, mode
    ((A16, 4, 32, A16, A16, 2), 1),        # unknown mode
    ((A16, 4, 48, A16, A16, 0), 2),        # K % 32
    ((A16, -4, 32, A16, A16, 0), 1),       # negative M
    ((A16, 4, 32, None, A16, 1), 1),       # NULL output
    ((BAD, 4, 32, A16, A16, 1), 1),        # misaligned input
    ((None, 0, 32, None, None, 0), 0),     # empty: nothing to do
])
def test_mxfp8_host_validation(gq, args, status):
    assert gq.lib().gq_mxfp8_dim0(*args, None) == status


@pytest.mark.parametrize("args,status", [
    # qa_t, sa, qx, sx, T, N, K, offs, G, out
    ((A16, A16, A16, A16, -1, 16, 16, A16, 1, A16), 1),    # negative T
    ((A16, A16, A16, A16, 16, 16, 16, A16, 0, A16), 1),    # no groups
    ((A16, A16, A16, A16, 16, 16, 16, A16, 1025, A16), 1),  # > GQ_MAX_GROUPS
    ((A16, A16, A16, A16, 16, 24, 16, A16, 1, A16), 2),    # N % 16
    ((A16, A16, A16, A16, 16, 16, 40, A16, 1, A16), 2),    # K % 16
    ((A16, A16, A16, A16, 16, 16, 16, A16, 1, None), 1),   # NULL output
    ((A16, A16, A16, A16, 16, 16, 16, None, 1, A16), 1),   # NULL offsets
    ((None, A16, A16, A16, 16, 16, 16, A16, 1, A16), 1),   # NULL operand
    ((BAD, A16, A16, A16, 16, 16, 16, A16, 1, A16), 1),    # misaligned operand
    ((A16, A16, A16, A16, 16, 16, 16, A16, 1, BAD), 1),    # misaligned output
    ((None, None, None, None, 16, 0, 16, None, 1, None), 0),  # N == 0: nothing to do
])
def test_grouped_wgrad_host_validation(gq, args, status):
    assert gq.lib().gq_grouped_wgrad(*args, None) == status


def test_header_compiles_as_c(tmp_path):
    """The boundary is a C ABI: the header compiles as strict C99 (and C++)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    src = tmp_path / "use.c"
    src.write_text('#include "gq_fp8.h"\n'
                   "int main(void) { return (int)gq_workspace_bytes(GQ_KIND_ROWWISE_T, 64, 64, 1) & 0; }\n")
    inc = os.path.dirname(HEADER)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", inc,
                    "-fsyntax-only", str(src)], check=True)
    if shutil.which("g++") is not None:
        subprocess.run(["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-I", inc,
                        "-fsyntax-only", "-x", "c++", str(src)], check=True)


def test_binding_rejects_bad_wgrad_and_mxfp8_args(gq):
    """The binding checks shapes, dtypes and devices on the host (no GPU)."""
    import torch
    f8 = torch.zeros((32, 16), dtype=torch.uint8)
    s = torch.zeros((16, 2), dtype=torch.float32)
    o = torch.tensor([16, 32], dtype=torch.int32)
    with pytest.raises(ValueError):   # host tensors
        gq.grouped_wgrad(f8, s, f8, torch.zeros((2, 16)), o)
    with pytest.raises(ValueError):   # host tensors
        gq.mxfp8_dim0(torch.zeros((4, 32), dtype=torch.bfloat16))
    with pytest.raises(ValueError):   # unknown mode is checked before the device
        gq.mxfp8_dim0(torch.zeros((4, 32), dtype=torch.bfloat16), "nearest")


@pytest.mark.parametrize("args,status", [
    # w, E, N, K, out, scales, flags
    ((A16, 0, 16, 16, A16, A16, 0), 1),           # no experts
    ((A16, 2, -1, 16, A16, A16, 0), 1),           # negative N
    ((A16, 2, 16, -8, A16, A16, 0), 1),           # negative K
    ((A16, 2, 16, 12, A16, A16, 0), 2),           # K % 8
    ((A16, 2, 16, 1 << 31, A16, A16, 0), 2),      # K >= 2^31
    ((A16, 2, 16, 16, A16, A16, 2), 1),           # GQ_WORKSPACE_ZEROED: no workspace here
    ((A16, 2, 16, 16, None, A16, 0), 1),          # NULL output
    ((None, 2, 16, 16, A16, A16, 0), 1),          # NULL input
    ((A16 + 8, 2, 16, 16, A16, A16, 0), 1),       # input not 16-byte aligned
    ((A16, 2, 16, 16, A16, None, 0), 1),          # NULL scales
    ((A16, 2, 0, 16, None, None, 0), 0),          # no rows: nothing to do
])
def test_expert_rowwise_host_validation(gq, args, status):
    assert gq.lib().gq_fp8_expert_rowwise(*args, None) == status
