"""GPU path against the oracle, through the C ABI (needs an sm_103 GPU).

Bit-exact comparison of every fp8 byte and every fp32 scale bit pattern: the
method is deterministic (max is order-independent, the scale is one IEEE
division, the product one IEEE multiply, the cast one RNE step), so the bar is
exact equality, and untouched output bytes must keep a sentinel.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_quantization_moe_gb300 import synth

pytestmark = pytest.mark.gpu

SENTINEL = 0x5A


@pytest.fixture(scope="module")
def gq():
    import __graft_entry__

    __graft_entry__.build()
    import fp8_quantization_moe_gb300 as m

    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    return m


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        torch.bfloat16).cuda()


def dev_i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def run_colwise(gq, x_bits, offs, fill=SENTINEL, pow2=False, two_phase=False):
    M, K = x_bits.shape
    out = torch.full((M, K), fill, dtype=torch.uint8, device="cuda")
    q, s = gq.colwise(dev_bf16(x_bits), dev_i32(offs),
                      out=out.view(torch.float8_e4m3fn), pow2_scales=pow2,
                      two_phase=two_phase)
    gq.check_device_error()
    return q.view(torch.uint8).cpu().numpy(), s.cpu().numpy()


def run_rowwise(gq, a_bits, offs, fill=SENTINEL, pow2=False):
    N, Mg = a_bits.shape
    out = torch.full((Mg, N), fill, dtype=torch.uint8, device="cuda")
    q, s = gq.rowwise_t(dev_bf16(a_bits), dev_i32(offs),
                        out=out.view(torch.float8_e4m3fn), pow2_scales=pow2)
    gq.check_device_error()
    return q.view(torch.uint8).cpu().numpy(), s.cpu().numpy()


def assert_same(q, s, rq, rs, what):
    if not np.array_equal(q, rq):
        bad = np.argwhere(q != rq)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} fp8 bytes differ; first at "
                             f"{i}: gpu {q[i]:#x} oracle {rq[i]:#x}")
    su, ru = s.view(np.uint32), rs.view(np.uint32)
    if not np.array_equal(su, ru):
        bad = np.argwhere(su != ru)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} scales differ; first at {i}: "
                             f"gpu {s[i]!r} oracle {rs[i]!r}")


def check_colwise(gq, case, pow2=False, two_phase=False):
    q, s = run_colwise(gq, case.x, case.offs, pow2=pow2, two_phase=two_phase)
    fill = np.full(case.x.shape, SENTINEL, np.uint8)
    rq, rs = oracle.colwise(case.x, case.offs, out=fill, pow2=pow2)
    assert_same(q, s, rq, rs, case.name)


def check_rowwise(gq, case, pow2=False):
    q, s = run_rowwise(gq, case.x, case.offs, pow2=pow2)
    fill = np.full(case.x.shape[::-1], SENTINEL, np.uint8)
    rq, rs = oracle.rowwise_t(case.x, case.offs, out=fill, pow2=pow2)
    assert_same(q, s, rq, rs, case.name)


# --------------------------------------------------------- small / ragged --
# Sizes span several 64x128 (colwise) or 128x64 (rowwise) tiles with ragged
# tails; groups include empty ones, unaligned boundaries and uncovered tails.
COLWISE_CASES = [
    # rows, cols, groups, seed, n_empty, align, scale_mix, uncovered
    (200, 272, 4, 1, 1, 16, True, 0),
    (1000, 384, 7, 2, 2, 1, True, 0),
    (513, 144, 3, 3, 0, 1, False, 29),
    (64, 128, 1, 4, 0, 16, False, 0),
    (1, 16, 1, 5, 0, 1, False, 0),
    (3, 16, 2, 6, 0, 1, True, 0),
    (130, 32, 40, 7, 5, 1, True, 0),      # many tiny groups, many per tile
    (4096, 256, 16, 8, 1, 16, True, 0),
    (777, 2064, 9, 9, 2, 1, True, 13),
]

ROWWISE_CASES = [
    (144, 200, 4, 11, 1, 8, True, 0),
    (256, 520, 7, 12, 2, 8, True, 0),
    (16, 8, 1, 13, 0, 8, False, 0),
    (384, 1000, 5, 14, 0, 8, False, 40),
    (128, 64, 1, 15, 0, 8, False, 0),
    (48, 392, 60, 16, 10, 1, True, 0),    # > 8 segments in a tile
    (2064, 1040, 16, 17, 1, 16, True, 0),
    (160, 2048, 33, 18, 3, 1, True, 7),
]


@pytest.mark.parametrize("spec", COLWISE_CASES, ids=lambda s: f"{s[0]}x{s[1]}g{s[2]}")
@pytest.mark.parametrize("two_phase", [False, True], ids=["auto", "two_phase"])
def test_colwise_small(gq, spec, two_phase):
    """Ragged cases, with the resident path where strips allow it and with
    every strip forced through the two phases (GQ_TWO_PHASE)."""
    r, c, g, seed, ne, al, mix, unc = spec
    check_colwise(gq, synth.random_case("colwise", r, c, g, seed, n_empty=ne,
                                        align=al, scale_mix=mix, uncovered=unc),
                  two_phase=two_phase)


@pytest.mark.parametrize("spec", ROWWISE_CASES, ids=lambda s: f"{s[0]}x{s[1]}g{s[2]}")
def test_rowwise_small(gq, spec):
    r, c, g, seed, ne, al, mix, unc = spec
    check_rowwise(gq, synth.random_case("rowwise_t", r, c, g, seed, n_empty=ne,
                                        align=al, scale_mix=mix, uncovered=unc))


# ------------------------------------------------------------ edge cases --

def test_colwise_no_tokens(gq):
    """M = 0: every group is empty; all scales are 448 / 1e-12."""
    x = np.zeros((0, 64), np.uint16)
    q, s = run_colwise(gq, x, np.array([0, 0, 0], np.int32))
    _, rs = oracle.colwise(x, np.array([0, 0, 0], np.int32))
    assert q.shape == (0, 64)
    assert np.array_equal(s.view(np.uint32), rs.view(np.uint32))


def test_rowwise_no_tokens(gq):
    a = np.zeros((32, 0), np.uint16)
    q, s = run_rowwise(gq, a, np.array([0, 0], np.int32))
    _, rs = oracle.rowwise_t(a, np.array([0, 0], np.int32))
    assert q.shape == (0, 32)
    assert np.array_equal(s.view(np.uint32), rs.view(np.uint32))


def test_empty_columns_and_rows(gq):
    q, s = run_colwise(gq, np.zeros((5, 0), np.uint16), np.array([5], np.int32))
    assert q.shape == (5, 0) and s.shape == (1, 0)
    q, s = run_rowwise(gq, np.zeros((0, 24), np.uint16), np.array([24], np.int32))
    assert q.shape == (24, 0) and s.shape == (0, 1)


@pytest.mark.parametrize("offs", [[40, 20, 100, 90], [-5, 64, 64, 300],
                                  [0, 0, 0, 0], [96, 96, 96, 96]])
def test_out_of_contract_offsets(gq, offs):
    """Offsets are read as a running maximum clamped to [0, extent]."""
    c = synth.random_case("colwise", 96, 48, 1, seed=51)
    r = synth.random_case("rowwise_t", 32, 96, 1, seed=52)
    o = np.array(offs, np.int32)
    check_colwise(gq, synth.Case("oob_c", "colwise", c.x, o, 0))
    check_rowwise(gq, synth.Case("oob_r", "rowwise_t", r.x, o, 0))


def test_single_token_groups(gq):
    o = np.arange(1, 41, dtype=np.int32)
    c = synth.random_case("colwise", 40, 32, 1, seed=53, scale_mix=True)
    check_colwise(gq, synth.Case("tok1_c", "colwise", c.x, o, 0))
    r = synth.random_case("rowwise_t", 16, 40, 1, seed=54, scale_mix=True)
    check_rowwise(gq, synth.Case("tok1_r", "rowwise_t", r.x, o, 0))


def test_max_groups(gq):
    """GQ_MAX_GROUPS groups of one or zero tokens."""
    G = gq.GQ_MAX_GROUPS
    rng = np.random.default_rng(55)
    o = np.sort(rng.integers(0, 800, size=G)).astype(np.int32)
    c = synth.random_case("colwise", 800, 16, 1, seed=56)
    check_colwise(gq, synth.Case("maxg_c", "colwise", c.x, o, 0))
    r = synth.random_case("rowwise_t", 16, 800, 1, seed=57)
    check_rowwise(gq, synth.Case("maxg_r", "rowwise_t", r.x, o, 0))


@pytest.mark.parametrize("n_groups,tokens", [(65, 3000), (200, 6000), (1000, 20000)])
def test_many_groups(gq, n_groups, tokens):
    """More than 32 groups: the tile header is searched block by block over
    the group-end table; tiles hold several segments, some more than the
    stage carries amax words for, and group starts fall in every block."""
    seed = 70 + n_groups
    check_colwise(gq, synth.random_case("colwise", tokens, 144, n_groups, seed,
                                        n_empty=n_groups // 10, align=1,
                                        scale_mix=True, uncovered=5))
    check_rowwise(gq, synth.random_case("rowwise_t", 144, tokens, n_groups,
                                        seed + 1, n_empty=n_groups // 10,
                                        align=1, scale_mix=True, uncovered=5))


@pytest.mark.parametrize("lag", [1, 2, 5, 1000])
def test_results_do_not_depend_on_lag(gq, lag):
    """The phase interleave is a schedule choice: every lag, from the
    shortest lead to all phase-A tiles before any phase-B tile, gives the
    oracle's bytes."""
    c = synth.random_case("colwise", 3000, 1040, 9, seed=80 + lag, n_empty=1,
                          align=1, scale_mix=True, uncovered=3)
    r = synth.random_case("rowwise_t", 1040, 3000, 9, seed=90 + lag, n_empty=1,
                          align=1, scale_mix=True, uncovered=3)
    try:
        gq.set_lag(gq.GQ_KIND_COLWISE, lag)
        gq.set_lag(gq.GQ_KIND_ROWWISE_T, lag)
        check_colwise(gq, c)
        check_rowwise(gq, r)
    finally:
        gq.set_lag(gq.GQ_KIND_COLWISE, 0)
        gq.set_lag(gq.GQ_KIND_ROWWISE_T, 0)


@pytest.mark.parametrize("widths,lead", [
    ((768, 760, 776, 768), 0),        # 12, 12, 13 (straddles), 12 windows
    ((764, 772, 8, 1540, 64), 4),     # starts off the 8-token grid
    ((5000, 3, 1, 1100), 1),          # long groups and one-token groups
    ((800, 700, 900, 640, 1000), 0),  # long and resident units alternate
])
def test_rowwise_resident_and_long_units(gq, widths, lead):
    """Groups around the number of windows a unit may keep in shared memory
    between its two passes (12 windows of 64 tokens): units just inside,
    just past (a group whose first window starts below it, rounded down to 8
    tokens) and far past it, which stream twice; plus groups of one token."""
    widths = list(widths)
    Mg = lead + sum(widths)
    Mg += (-Mg) % 8
    offs = np.cumsum([lead + widths[0]] + widths[1:]).astype(np.int32)
    base = synth.random_case("rowwise_t", 80, Mg, 1, seed=300 + len(widths),
                             align=8, scale_mix=True)
    check_rowwise(gq, synth.Case("resident_" + "_".join(map(str, widths)),
                                 "rowwise_t", base.x, offs, 0))


@pytest.mark.parametrize("rows,widths,lead", [
    (64, (16640,), 0),                       # one band: 22 parts of one unit
    (208, (100, 900, 5000, 0, 4992), 4),     # short, long, split, empty, split
    (144, (4091, 4089, 4097, 3, 9000), 5),   # around the split limit (64 windows)
])
def test_rowwise_split_units(gq, rows, widths, lead):
    """Groups of more than 64 windows are cut into parts of at most 12
    windows that other blocks take; the parts' row maxima meet in the
    workspace before any part is cast.  Mixed with resident, long (13-64
    windows, read twice) and empty groups."""
    widths = list(widths)
    Mg = lead + sum(widths)
    Mg += (-Mg) % 8
    offs = np.cumsum([lead + widths[0]] + widths[1:]).astype(np.int32)
    base = synth.random_case("rowwise_t", rows, Mg, 1, seed=400 + rows, align=8,
                             scale_mix=True)
    case = synth.Case("split_" + "_".join(map(str, widths)), "rowwise_t", base.x, offs, 0)
    check_rowwise(gq, case)
    check_rowwise(gq, case, pow2=True)  # the split units' scales, rounded down


@pytest.mark.parametrize("rows,widths,lead", [(64, (16640,), 0),
                                               (208, (100, 900, 5000, 0, 4992), 4)])
def test_rowwise_split_build_without_splitting(gq, rows, widths, lead):
    """The build that can split units, told not to (the path it takes when
    it does not find every block resident): those units run whole, read
    twice, and give the same bytes."""
    widths = list(widths)
    Mg = lead + sum(widths)
    Mg += (-Mg) % 8
    offs = np.cumsum([lead + widths[0]] + widths[1:]).astype(np.int32)
    base = synth.random_case("rowwise_t", rows, Mg, 1, seed=410 + rows, align=8,
                             scale_mix=True)
    try:
        gq.debug_set(no_split=True)
        check_rowwise(gq, synth.Case("nosplit_" + "_".join(map(str, widths)), "rowwise_t",
                                     base.x, offs, 0))
    finally:
        gq.debug_set(False, 0)


def test_rowwise_split_timeout_is_reported_not_hung(gq):
    """A part that never reports its maxima makes the other parts' scale
    waits give up after the (shortened) limit: GQ_ERR_TIMEOUT, and the
    workspace is left zeroed for the next call."""
    r = synth.random_case("rowwise_t", 128, 8192, 1, seed=64)
    try:
        gq.debug_set(skip_arrival=True, wait_timeout_ns=5_000_000)
        gq.rowwise_t(dev_bf16(r.x), dev_i32(r.offs))
        with pytest.raises(gq.GQError) as e:
            gq.check_device_error()
        assert e.value.status == 4
    finally:
        gq.debug_set(False, 0)
    check_rowwise(gq, r)


@pytest.mark.parametrize("widths,K", [
    ((319, 320, 321, 1, 16, 0, 300, 256), 400),       # around the resident limit
    ((767, 768, 769, 1536, 1537, 40), 272),           # around the tile size
    ((256, 3000, 128, 0, 2305, 255, 17, 768), 1040),  # resident and long strips alternate
])
def test_colwise_resident_and_two_phase_strips(gq, widths, K):
    """Group strips of at most 320 rows are folded and cast by one block out
    of shared memory; longer ones go through the two phases in 768-row
    tiles.  Groups just inside and past both sizes, empty and one-row
    groups, mixed in one call, over several column slabs (the last one
    partial)."""
    offs = np.cumsum(widths).astype(np.int32)
    M = int(offs[-1]) + 5  # uncovered tail rows keep the sentinel
    base = synth.random_case("colwise", M, K, 1, seed=310 + len(widths), scale_mix=True)
    check_colwise(gq, synth.Case("strips_" + "_".join(map(str, widths)), "colwise",
                                 base.x, offs, 0))
    check_colwise(gq, synth.Case("strips_pow2", "colwise", base.x, offs, 0), pow2=True)


@pytest.mark.parametrize("widths", [
    # 11271 x 4096: 512-row phase-A tiles, read again as 256-row phase-B tiles
    (511, 512, 513, 1023, 1024, 1025, 255, 256, 257, 0, 1, 3000, 2889),
    # 17005 x 4096: 768-row phase-A tiles, read again as 384-row phase-B tiles
    (383, 384, 385, 767, 768, 769, 1151, 1152, 1153, 1536, 1537, 0, 2000, 4000, 1015),
])
def test_colwise_split_phase_b_tiles(gq, widths):
    """Sizes at which a 152-SM GB300 cuts long strips into 512- or 768-row
    tiles, whose second read comes in halves: strips just inside and past a
    half tile, a tile and one and a half tiles, empty, one-row and resident
    strips mixed in one call, every column against the oracle."""
    K = 4096
    offs = np.cumsum(widths).astype(np.int32)
    M = int(offs[-1]) + 5  # uncovered tail rows keep the sentinel
    base = synth.random_case("colwise", M, K, 1, seed=400 + len(widths), scale_mix=True)
    check_colwise(gq, synth.Case("split_" + str(M), "colwise", base.x, offs, 0))


def test_short_super_tiles_many_tickets(gq):
    """Many short pieces of work: 512 column slabs of five short strips
    (colwise), or 1024 row bands of short groups (rowwise_t), so that every
    block takes many items whose stages do not reach every consumer warp --
    a warp must still read each context before releasing it."""
    c = synth.random_case("colwise", 320, 65536, 5, seed=81, n_empty=1, align=1,
                          scale_mix=True)
    check_colwise(gq, c)
    check_colwise(gq, c, two_phase=True)
    check_rowwise(gq, synth.random_case("rowwise_t", 65536, 320, 5, seed=82,
                                        n_empty=1, align=1, scale_mix=True))


def test_element_map_exhaustive_amax(gq):
    """Every finite non-negative bf16 value as a column amax, each with 127
    elements of magnitude at most that amax (both signs, zeros, subnormals,
    the amax itself): the elementwise map (x, amax) -> q, and every scale,
    against the oracle -- through both paths."""
    rng = np.random.default_rng(58)
    amax = np.arange(0, 0x7F80, dtype=np.uint16)  # 32640 columns
    K = amax.size
    R = 128
    mag = rng.integers(0, 1 << 15, size=(R, K), dtype=np.uint32).astype(np.uint16)
    mag = np.minimum(mag, amax[None, :])
    mag[1] = amax            # the amax itself
    mag[2] = 0               # zero
    mag[3] = amax // 2       # half the bit pattern: spans binades
    mag[4] = np.minimum(amax, rng.integers(0, 0x80, size=K).astype(np.uint16))  # subnormals
    sign = (rng.integers(0, 2, size=(R, K)) << 15).astype(np.uint16)
    x = mag | sign
    x[0] = amax              # row 0 carries the amax, positive
    case = synth.Case("elemmap_c", "colwise", x, np.array([R], np.int32), 0)
    check_colwise(gq, case)
    caseT = synth.Case("elemmap_r", "rowwise_t", np.ascontiguousarray(x.T),
                       np.array([R], np.int32), 0)
    check_rowwise(gq, caseT)


def test_deterministic_and_stream(gq):
    """Two calls, on a side stream, give identical bytes."""
    c = synth.random_case("colwise", 2048, 512, 8, seed=59, scale_mix=True)
    x, o = dev_bf16(c.x), dev_i32(c.offs)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        q1, s1 = gq.colwise(x, o, stream=s)
        q2, s2 = gq.colwise(x, o, stream=s)
    s.synchronize()
    gq.check_device_error(stream=s)
    assert torch.equal(q1.view(torch.uint8), q2.view(torch.uint8))
    assert torch.equal(s1, s2)


def test_guard_bytes_untouched(gq):
    """Outputs placed inside a larger buffer: the bytes around them stay."""
    c = synth.random_case("colwise", 300, 160, 3, seed=60)
    M, K = c.x.shape
    buf = torch.full((M * K + 512,), 0xA5, dtype=torch.uint8, device="cuda")
    out = buf[256:256 + M * K].view(M, K)
    sbuf = torch.full((3 * K + 128,), -7.0, dtype=torch.float32, device="cuda")
    sc = sbuf[64:64 + 3 * K].view(3, K)
    gq.colwise(dev_bf16(c.x), dev_i32(c.offs), out=out.view(torch.float8_e4m3fn),
               scales=sc)
    gq.check_device_error()
    b = buf.cpu().numpy()
    assert np.all(b[:256] == 0xA5) and np.all(b[256 + M * K:] == 0xA5)
    sb = sbuf.cpu().numpy()
    assert np.all(sb[:64] == -7.0) and np.all(sb[64 + 3 * K:] == -7.0)
    rq, rs = oracle.colwise(c.x, c.offs)
    assert np.array_equal(b[256:256 + M * K].reshape(M, K), rq)


def test_timeout_is_reported_not_hung(gq):
    """A withheld completion signal makes the waiting blocks give up after
    the (shortened) limit and report GQ_ERR_TIMEOUT; the next call is fine."""
    c = synth.random_case("colwise", 1024, 256, 4, seed=61)
    r = synth.random_case("rowwise_t", 256, 512, 4, seed=62)
    try:
        gq.debug_set(skip_arrival=True, wait_timeout_ns=5_000_000)
        gq.colwise(dev_bf16(c.x), dev_i32(c.offs))
        with pytest.raises(gq.GQError) as e:
            gq.check_device_error()
        assert e.value.status == 4
        gq.rowwise_t(dev_bf16(r.x), dev_i32(r.offs))
        with pytest.raises(gq.GQError) as e:
            gq.check_device_error()
        assert e.value.status == 4
    finally:
        gq.debug_set(False, 0)
    check_colwise(gq, c)
    check_rowwise(gq, r)


def test_host_buffer_calls(gq):
    """The end-to-end host-buffer entry points."""
    c = synth.random_case("colwise", 640, 256, 5, seed=63)
    xh = torch.from_numpy(c.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    oh = torch.from_numpy(c.offs).pin_memory()
    q, s = gq.colwise_host(xh, oh)
    torch.cuda.synchronize()
    rq, rs = oracle.colwise(c.x, c.offs)
    assert_same(q.view(torch.uint8).numpy(), s.numpy(), rq, rs, "colwise_host")
    r = synth.random_case("rowwise_t", 256, 640, 5, seed=64)
    ah = torch.from_numpy(r.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    oh = torch.from_numpy(r.offs).pin_memory()
    q, s = gq.rowwise_t_host(ah, oh)
    torch.cuda.synchronize()
    rq, rs = oracle.rowwise_t(r.x, r.offs)
    assert_same(q.view(torch.uint8).numpy(), s.numpy(), rq, rs, "rowwise_t_host")


@pytest.mark.parametrize("idx", range(4))
def test_pow2_scales(gq, idx):
    """round_scales_to_power_of_2 through both kernels: ragged cases with
    empty groups, unaligned boundaries, uncovered tails and magnitudes over
    six decades, a resident and a long rowwise unit, and empty extents."""
    seed = 400 + idx
    if idx == 0:
        check_colwise(gq, synth.random_case("colwise", 777, 400, 9, seed, n_empty=2,
                                            align=1, scale_mix=True, uncovered=7), pow2=True)
        check_rowwise(gq, synth.random_case("rowwise_t", 144, 2000, 9, seed, n_empty=2,
                                            align=1, scale_mix=True, uncovered=7), pow2=True)
    elif idx == 1:
        check_colwise(gq, synth.random_case("colwise", 4096, 256, 16, seed, n_empty=1,
                                            scale_mix=True), pow2=True)
        check_rowwise(gq, synth.random_case("rowwise_t", 80, 6112, 3, seed,
                                            align=8, scale_mix=True), pow2=True)
    elif idx == 2:  # every finite bf16 amax as a column / row maximum
        amax = np.arange(0, 0x7F80, dtype=np.uint16)
        rng = np.random.default_rng(seed)
        mag = rng.integers(0, 1 << 15, size=(64, amax.size), dtype=np.uint32).astype(np.uint16)
        x = np.minimum(mag, amax[None, :])
        x[0] = amax
        check_colwise(gq, synth.Case("pow2_map_c", "colwise", x, np.array([64], np.int32), 0),
                      pow2=True)
        check_rowwise(gq, synth.Case("pow2_map_r", "rowwise_t", np.ascontiguousarray(x.T),
                                     np.array([64], np.int32), 0), pow2=True)
    else:  # empty extents: only scales, all the empty group's
        z = np.zeros((0, 32), np.uint16)
        check_colwise(gq, synth.Case("pow2_m0", "colwise", z, np.array([0, 0], np.int32), 0),
                      pow2=True)
        z = np.zeros((32, 0), np.uint16)
        check_rowwise(gq, synth.Case("pow2_mg0", "rowwise_t", z, np.array([0], np.int32), 0),
                      pow2=True)


@pytest.mark.parametrize("E,K,N,pow2", [
    (1, 64, 16, False), (3, 100, 48, False), (8, 333, 272, False), (5, 257, 4112, True),
    (2, 1, 16, False), (5, 0, 32, False), (4, 17, 0, False), (64, 40, 32, True),
])
def test_expert_dim1(gq, E, K, N, pow2):
    """Stacked expert weights scaled along dim1, against the oracle, bit for
    bit: ragged K and N over several tiles, one-row experts, K = 0 (scales
    only), N = 0 (nothing), many experts."""
    rng = np.random.default_rng(600 + E + K + N)
    x = rng.standard_normal((E, K, N)).astype(np.float32)
    x *= np.power(np.float32(10), rng.uniform(-3, 3, size=(E, K, 1))).astype(np.float32)
    w = synth.to_bf16_bits(x)
    out = torch.full((E, K, N), SENTINEL, dtype=torch.uint8, device="cuda")
    wd = torch.from_numpy(np.ascontiguousarray(w).view(np.int16)).view(torch.bfloat16).cuda()
    q, s = gq.expert_dim1(wd, out=out.view(torch.float8_e4m3fn), pow2_scales=pow2)
    gq.check_device_error()
    rq, rs = oracle.expert_dim1(w, pow2=pow2)
    assert_same(q.view(torch.uint8).cpu().numpy(), s.cpu().numpy(), rq, rs,
                f"expert_dim1_{E}x{K}x{N}")


@pytest.mark.parametrize("E,N,K,pow2", [
    (1, 1, 8, False), (3, 37, 40, False), (2, 129, 4096, False), (2, 65, 4104, False),
    (1, 3, 8192, True), (8, 300, 264, False), (6, 1000, 520, True), (4, 0, 16, False),
    (5, 7, 0, False), (5, 7, 0, True),
])
def test_expert_rowwise(gq, E, N, K, pow2):
    """Stacked expert weights scaled per row, against the oracle, bit for
    bit: rows shorter than a warp's first load, rows held in registers (up
    to 4096 elements) and longer rows read twice, an all-zero row, many rows
    per warp, N = 0 (nothing) and K = 0 (scales only)."""
    rng = np.random.default_rng(620 + E + N + K)
    x = rng.standard_normal((E, N, K)).astype(np.float32)
    x *= np.power(np.float32(10), rng.uniform(-3, 3, size=(E, N, 1))).astype(np.float32)
    if N > 2 and K:
        x[E - 1, 2] = 0.0
    w = synth.to_bf16_bits(x)
    out = torch.full((E, N, K), SENTINEL, dtype=torch.uint8, device="cuda")
    sc = torch.full((E, N), -1.0, dtype=torch.float32, device="cuda")
    wd = torch.from_numpy(np.ascontiguousarray(w).view(np.int16)).view(torch.bfloat16).cuda()
    q, s = gq.expert_rowwise(wd, out=out.view(torch.float8_e4m3fn), scales=sc, pow2_scales=pow2)
    gq.check_device_error()
    rq, rs = oracle.expert_rowwise(w, pow2=pow2)
    assert_same(q.view(torch.uint8).cpu().numpy(), s.cpu().numpy(), rq, rs,
                f"expert_rowwise_{E}x{N}x{K}")


@pytest.mark.parametrize("M,K,mode", [
    (1, 32, "floor"), (1, 32, "rceil"), (24, 256, "floor"), (24, 256, "rceil"),
    (333, 4096, "floor"), (333, 4096, "rceil"), (4097, 96, "rceil"), (0, 64, "floor"),
])
def test_mxfp8_dim0(gq, M, K, mode):
    """mxfp8 along dim0 against the oracle, bit for bit (codes and e8m0
    bytes): block magnitudes from 2^-140 to 2^120 (clamped exponents at both
    ends), zero and negative-zero blocks, bf16 subnormals, exact powers of
    two, ragged M and a chunk count that is not a multiple of the grid's."""
    import oracle_pins
    rng = np.random.default_rng(700 + M + K)
    bits = oracle_pins._mx_input(rng, M, K)
    x = dev_bf16(bits) if M else torch.empty((0, K), dtype=torch.bfloat16, device="cuda")
    q, s = gq.mxfp8_dim0(x, mode)
    torch.cuda.synchronize()
    rq, rs = oracle.mxfp8_dim0(bits, 0 if mode == "floor" else 1)
    gq_q, gq_s = q.view(torch.uint8).cpu().numpy(), s.cpu().numpy()
    assert np.array_equal(gq_s, rs), f"{mode} scales: {np.argwhere(gq_s != rs)[:3]}"
    assert np.array_equal(gq_q, rq), f"{mode} codes: {np.argwhere(gq_q != rq)[:3]}"


def test_rowwise_workspace_left_zeroed(gq):
    """Every rowwise_t launch returns its counters and split words to zero,
    so calls given GQ_WORKSPACE_ZEROED on one workspace (zero-filled once)
    stay exact -- across shapes and group counts (split units included), and
    after a call without the flag."""
    cases = [synth.random_case("rowwise_t", 144, 520, 6, seed=70, n_empty=1, scale_mix=True),
             synth.random_case("rowwise_t", 1040, 3000, 9, seed=71, n_empty=1, align=1, uncovered=3),
             synth.random_case("rowwise_t", 64, 16, 1, seed=72),
             synth.random_case("rowwise_t", 192, 12000, 2, seed=73, scale_mix=True)]
    nws = max(gq.workspace_bytes(gq.GQ_KIND_ROWWISE_T, c.x.shape[0], c.x.shape[1], len(c.offs))
              for c in cases)
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for c in cases:
            a, o = dev_bf16(c.x), dev_i32(c.offs)
            qt = torch.full((c.x.shape[1], c.x.shape[0]), SENTINEL, dtype=torch.uint8, device="cuda")
            s = torch.empty((c.x.shape[0], len(c.offs)), dtype=torch.float32, device="cuda")
            st = gq.lib().gq_fp8_rowwise_t_ex(
                a.data_ptr(), c.x.shape[0], c.x.shape[1], o.data_ptr(), len(c.offs),
                qt.data_ptr(), s.data_ptr(), gq.GQ_WORKSPACE_ZEROED if rep == 0 else 0,
                ws.data_ptr(), nws, torch.cuda.current_stream().cuda_stream)
            assert st == 0
            gq.check_device_error()
            assert not ws.any().item(), "counters or split words not returned to zero"
            rq, rs = oracle.rowwise_t(c.x, c.offs, out=np.full((c.x.shape[1], c.x.shape[0]), SENTINEL, np.uint8))
            assert_same(qt.cpu().numpy(), s.cpu().numpy(), rq, rs, c.name)


def test_graph_capture_and_replay(gq):
    """Both calls captured into one CUDA graph on a fresh stream (so the
    workspaces are created during the capture) and replayed: each replay
    gives the oracle's bytes."""
    c = synth.random_case("colwise", 700, 272, 5, seed=81, n_empty=1, align=1, scale_mix=True)
    r = synth.random_case("rowwise_t", 144, 520, 6, seed=82, n_empty=1, scale_mix=True)
    x, xo, a, ao = dev_bf16(c.x), dev_i32(c.offs), dev_bf16(r.x), dev_i32(r.offs)
    q = torch.full(c.x.shape, SENTINEL, dtype=torch.uint8, device="cuda")
    qs = torch.empty((len(c.offs), c.x.shape[1]), dtype=torch.float32, device="cuda")
    qt = torch.full(r.x.shape[::-1], SENTINEL, dtype=torch.uint8, device="cuda")
    ts = torch.empty((r.x.shape[0], len(r.offs)), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gq.colwise(x, xo, out=q.view(torch.float8_e4m3fn), scales=qs, stream=s)
        gq.rowwise_t(a, ao, out=qt.view(torch.float8_e4m3fn), scales=ts, stream=s)
    rq, rs = oracle.colwise(c.x, c.offs, out=np.full(c.x.shape, SENTINEL, np.uint8))
    tq, trs = oracle.rowwise_t(r.x, r.offs, out=np.full(r.x.shape[::-1], SENTINEL, np.uint8))
    for _ in range(2):
        q.fill_(SENTINEL)
        qt.fill_(SENTINEL)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        gq.check_device_error()
        assert_same(q.cpu().numpy(), qs.cpu().numpy(), rq, rs, "colwise in a graph")
        assert_same(qt.cpu().numpy(), ts.cpu().numpy(), tq, trs, "rowwise_t in a graph")


def test_host_calls_back_to_back(gq):
    """Host-buffer calls queued back to back on one stream: each call's
    host->device copy runs on a side stream and may overlap the previous
    call's kernel and copies; every result still matches the oracle."""
    c = synth.random_case("colwise", 1024, 512, 5, seed=91, n_empty=1, align=1, scale_mix=True)
    r = synth.random_case("rowwise_t", 256, 1040, 6, seed=92, n_empty=1, scale_mix=True)
    xh = torch.from_numpy(c.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    ah = torch.from_numpy(r.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    xo, ao = torch.from_numpy(c.offs).pin_memory(), torch.from_numpy(r.offs).pin_memory()
    rq, rs = oracle.colwise(c.x, c.offs)
    tq, trs = oracle.rowwise_t(r.x, r.offs)
    s = torch.cuda.Stream()
    outs = []
    for _ in range(3):
        outs.append(("colwise", gq.colwise_host(xh, xo, stream=s)))
        outs.append(("rowwise_t", gq.rowwise_t_host(ah, ao, stream=s)))
    s.synchronize()
    gq.check_device_error()
    for kind, (q, sc) in outs:
        if kind == "colwise":
            assert_same(q.view(torch.uint8).numpy(), sc.numpy(), rq, rs, "colwise_host")
        else:
            assert_same(q.view(torch.uint8).numpy(), sc.numpy(), tq, trs, "rowwise_t_host")
