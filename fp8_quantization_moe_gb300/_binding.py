"""ctypes binding over the C ABI of libgqfp8 (include/gq_fp8.h).

Argument marshalling only: every step of the quantization runs in the
library's CUDA kernels.  torch supplies device memory and streams.  There is
no CPU fallback: without the compiled library or a CUDA device the calls
raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

GQ_OK = 0
GQ_ERR_INVALID_ARG = 1
GQ_ERR_UNSUPPORTED = 2
GQ_ERR_CUDA = 3
GQ_ERR_TIMEOUT = 4
GQ_KIND_COLWISE = 0
GQ_KIND_ROWWISE_T = 1
GQ_MAX_GROUPS = 1024
GQ_SCALE_POW2 = 1
GQ_WORKSPACE_ZEROED = 2
GQ_TWO_PHASE = 4
GQ_MX_FLOOR = 0
GQ_MX_RCEIL = 1

# Every symbol the header declares, with its ctypes signature.
_P, _I64, _I32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
SIGNATURES = {
    "gq_workspace_bytes": (_SZ, [ctypes.c_int, _I64, _I64, _I32]),
    "gq_fp8_colwise": (ctypes.c_int, [_P, _I64, _I64, _P, _I32, _P, _P, _P, _SZ, _P]),
    "gq_fp8_rowwise_t": (ctypes.c_int, [_P, _I64, _I64, _P, _I32, _P, _P, _P, _SZ, _P]),
    "gq_fp8_colwise_noalloc": (ctypes.c_int, [_P, _I64, _I64, _P, _I32, _P, _P, _P]),
    "gq_fp8_colwise_ex": (ctypes.c_int, [_P, _I64, _I64, _P, _I32, _P, _P, ctypes.c_uint32, _P, _SZ, _P]),
    "gq_fp8_expert_dim1": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, ctypes.c_uint32, _P, _SZ, _P]),
    "gq_fp8_expert_rowwise": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, ctypes.c_uint32, _P]),
    "gq_mxfp8_dim0": (ctypes.c_int, [_P, _I64, _I64, _P, _P, ctypes.c_int, _P]),
    "gq_grouped_wgrad": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _P, _I32, _P, _P]),
    "gq_fp8_rowwise_t_ex": (ctypes.c_int, [_P, _I64, _I64, _P, _I32, _P, _P, ctypes.c_uint32, _P, _SZ, _P]),
    "gq_check_device_error": (ctypes.c_int, [_P]),
    "gq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "gq_last_error": (ctypes.c_char_p, []),
    "gq_version": (ctypes.c_int, []),
    "gq_debug_set": (ctypes.c_int, [ctypes.c_int, _I64]),
    "gq_set_lag": (ctypes.c_int, [ctypes.c_int, ctypes.c_int32]),
}


class GQError(RuntimeError):
    """A non-OK status from libgqfp8."""

    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({detail})")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded library.  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libgqfp8 is not built ({path} missing); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            handle = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def _check(status: int, where: str):
    if status != GQ_OK:
        L = lib()
        detail = (L.gq_status_string(status) or b"").decode()
        msg = (L.gq_last_error() or b"").decode()
        raise GQError(status, where, f"{detail}: {msg}" if msg else detail)


def status_string(status: int) -> str:
    return lib().gq_status_string(status).decode()


def version() -> int:
    return lib().gq_version()


def workspace_bytes(kind: int, rows: int, cols: int, n_groups: int) -> int:
    return int(lib().gq_workspace_bytes(kind, rows, cols, n_groups))


# ----------------------------------------------------------- workspaces --
_ws_cache: dict = {}
_ws_lock = threading.Lock()


def _workspace(nbytes: int, device: torch.device, stream_handle: int, kind: int = 0):
    """(buffer, zeroed): a cached device workspace per (device, stream, kind),
    zero-filled when it is allocated.  Calls on one stream run in order, so
    reuse is safe, and every colwise or rowwise_t launch leaves the part of
    its workspace it used at zero when it ends (also after a bounded wait
    expired), so calls on a cached buffer pass GQ_WORKSPACE_ZEROED and skip
    the clear.  While the stream is being captured into a CUDA graph a
    missing buffer is not created in the cache (that would synchronise the
    device): the call gets a fresh one, not known to be zero."""
    if nbytes == 0:
        return None, False
    key = (device.index, stream_handle, kind)
    with _ws_lock:
        buf = _ws_cache.get(key)
        if buf is None or buf.numel() < nbytes:
            if torch.cuda.is_current_stream_capturing():
                return torch.empty(nbytes + 256, dtype=torch.uint8, device=device), False
            buf = torch.zeros(nbytes + 256, dtype=torch.uint8, device=device)
            torch.cuda.synchronize(device)  # zero before work on any stream uses it
            _ws_cache[key] = buf
    return buf, True


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_handle(stream, device):
    s = torch.cuda.current_stream(device) if stream is None else stream
    return s.cuda_stream


def _ws_ptr(buf):
    if buf is None:
        return None, 0
    p = buf.data_ptr()
    aligned = (p + 255) & ~255
    return aligned, buf.numel() - (aligned - p)


def _check_in(x, offs, name):
    if not (isinstance(x, torch.Tensor) and x.is_cuda):
        raise ValueError(f"{name}: input must be a CUDA tensor")
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_contiguous():
        raise ValueError(f"{name}: input must be a contiguous 2-D bf16 tensor")
    if not (isinstance(offs, torch.Tensor) and offs.is_cuda
            and offs.dtype == torch.int32 and offs.dim() == 1
            and offs.is_contiguous() and offs.device == x.device):
        raise ValueError(f"{name}: offs must be a contiguous 1-D int32 tensor "
                         "on the input's device")


# ---------------------------------------------------------------- paths --

def colwise(x: torch.Tensor, offs: torch.Tensor, *, out=None, scales=None,
            stream=None, workspace=None, pow2_scales: bool = False,
            two_phase: bool = False):
    """Colwise per-token-group scaling (groups along dim0).

    ``pow2_scales`` rounds every scale down to a power of two
    (GQ_SCALE_POW2); ``two_phase`` sends every strip through the two-phase
    path (GQ_TWO_PHASE; same results).

    x: bf16 (M, K) CUDA tensor; offs: int32 (n_groups,) end offsets on the
    same device.  Returns (q float8_e4m3fn (M, K), scales float32
    (n_groups, K)).  Rows outside every group keep the contents of ``out``
    (uninitialised when ``out`` is None).  Asynchronous on ``stream`` (default:
    the current stream).
    """
    _check_in(x, offs, "colwise")
    M, K = x.shape
    G = offs.numel()
    dev = x.device
    if out is None:
        out = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=dev)
    if scales is None:
        scales = torch.empty((G, K), dtype=torch.float32, device=dev)
    if out.shape != (M, K) or out.element_size() != 1 or not out.is_contiguous():
        raise ValueError("colwise: out must be a contiguous 1-byte (M, K) tensor")
    if scales.shape != (G, K) or scales.dtype != torch.float32 or not scales.is_contiguous():
        raise ValueError("colwise: scales must be a contiguous float32 (G, K) tensor")
    sh = _stream_handle(stream, dev)
    need = workspace_bytes(GQ_KIND_COLWISE, M, K, G)
    flags = (GQ_SCALE_POW2 if pow2_scales else 0) | (GQ_TWO_PHASE if two_phase else 0)
    if workspace is None:
        ws, zeroed = _workspace(need, dev, sh, GQ_KIND_COLWISE)
        flags |= GQ_WORKSPACE_ZEROED if zeroed else 0
    else:
        ws = workspace
    wp, wn = _ws_ptr(ws)
    with torch.cuda.device(dev):
        st = lib().gq_fp8_colwise_ex(_ptr(x), M, K, _ptr(offs), G, _ptr(out),
                                     _ptr(scales), flags, wp, wn, sh)
    _check(st, "gq_fp8_colwise")
    return out, scales


def rowwise_t(a: torch.Tensor, offs: torch.Tensor, *, out=None, scales=None,
              stream=None, workspace=None, pow2_scales: bool = False):
    """Rowwise per-token-group scaling with transposed output (groups along
    dim1 of A).  ``pow2_scales`` rounds every scale down to a power of two.

    a: bf16 (N, Mg) CUDA tensor; offs: int32 (n_groups,) end offsets along
    Mg.  Returns (qt float8_e4m3fn (Mg, N) = q(a)^T, scales float32
    (N, n_groups)).  Token rows of qt outside every group keep ``out``.
    """
    _check_in(a, offs, "rowwise_t")
    N, Mg = a.shape
    G = offs.numel()
    dev = a.device
    if out is None:
        out = torch.empty((Mg, N), dtype=torch.float8_e4m3fn, device=dev)
    if scales is None:
        scales = torch.empty((N, G), dtype=torch.float32, device=dev)
    if out.shape != (Mg, N) or out.element_size() != 1 or not out.is_contiguous():
        raise ValueError("rowwise_t: out must be a contiguous 1-byte (Mg, N) tensor")
    if scales.shape != (N, G) or scales.dtype != torch.float32 or not scales.is_contiguous():
        raise ValueError("rowwise_t: scales must be a contiguous float32 (N, G) tensor")
    sh = _stream_handle(stream, dev)
    need = workspace_bytes(GQ_KIND_ROWWISE_T, N, Mg, G)
    flags = GQ_SCALE_POW2 if pow2_scales else 0
    if workspace is None:
        ws, zeroed = _workspace(need, dev, sh, GQ_KIND_ROWWISE_T)
        flags |= GQ_WORKSPACE_ZEROED if zeroed else 0
    else:
        ws = workspace
    wp, wn = _ws_ptr(ws)
    with torch.cuda.device(dev):
        st = lib().gq_fp8_rowwise_t_ex(_ptr(a), N, Mg, _ptr(offs), G, _ptr(out),
                                       _ptr(scales), flags, wp, wn, sh)
    _check(st, "gq_fp8_rowwise_t")
    return out, scales


def expert_dim1(w: torch.Tensor, *, out=None, scales=None, stream=None, workspace=None,
                pow2_scales: bool = False):
    """Stacked expert weights scaled along dim1: w bf16 (E, K, N) CUDA tensor;
    one scale per (expert, column), the amax over the expert's K rows.
    Returns (q float8_e4m3fn (E, K, N), scales float32 (E, N))."""
    if not (isinstance(w, torch.Tensor) and w.is_cuda and w.dtype == torch.bfloat16
            and w.dim() == 3 and w.is_contiguous()):
        raise ValueError("expert_dim1: w must be a contiguous 3-D bf16 CUDA tensor")
    E, K, N = w.shape
    dev = w.device
    if out is None:
        out = torch.empty((E, K, N), dtype=torch.float8_e4m3fn, device=dev)
    if scales is None:
        scales = torch.empty((E, N), dtype=torch.float32, device=dev)
    if out.shape != (E, K, N) or out.element_size() != 1 or not out.is_contiguous():
        raise ValueError("expert_dim1: out must be a contiguous 1-byte (E, K, N) tensor")
    if scales.shape != (E, N) or scales.dtype != torch.float32 or not scales.is_contiguous():
        raise ValueError("expert_dim1: scales must be a contiguous float32 (E, N) tensor")
    sh = _stream_handle(stream, dev)
    need = workspace_bytes(GQ_KIND_COLWISE, E * K, N, E)
    flags = GQ_SCALE_POW2 if pow2_scales else 0
    if workspace is None:  # the colwise kernel: the colwise cache
        ws, zeroed = _workspace(need, dev, sh, GQ_KIND_COLWISE)
        flags |= GQ_WORKSPACE_ZEROED if zeroed else 0
    else:
        ws = workspace
    wp, wn = _ws_ptr(ws)
    with torch.cuda.device(dev):
        st = lib().gq_fp8_expert_dim1(_ptr(w), E, K, N, _ptr(out), _ptr(scales),
                                      flags, wp, wn, sh)
    _check(st, "gq_fp8_expert_dim1")
    return out, scales


def expert_rowwise(w: torch.Tensor, *, out=None, scales=None, stream=None,
                   pow2_scales: bool = False):
    """Stacked expert weights scaled per row: w bf16 (E, N, K) CUDA tensor,
    K % 8 == 0; one scale per (expert, row), the amax over the row's K
    elements.  Returns (q float8_e4m3fn (E, N, K), scales float32 (E, N))."""
    if not (isinstance(w, torch.Tensor) and w.is_cuda and w.dtype == torch.bfloat16
            and w.dim() == 3 and w.is_contiguous()):
        raise ValueError("expert_rowwise: w must be a contiguous 3-D bf16 CUDA tensor")
    E, N, K = w.shape
    dev = w.device
    if out is None:
        out = torch.empty((E, N, K), dtype=torch.float8_e4m3fn, device=dev)
    if scales is None:
        scales = torch.empty((E, N), dtype=torch.float32, device=dev)
    if out.shape != (E, N, K) or out.element_size() != 1 or not out.is_contiguous():
        raise ValueError("expert_rowwise: out must be a contiguous 1-byte (E, N, K) tensor")
    if scales.shape != (E, N) or scales.dtype != torch.float32 or not scales.is_contiguous():
        raise ValueError("expert_rowwise: scales must be a contiguous float32 (E, N) tensor")
    sh = _stream_handle(stream, dev)
    flags = GQ_SCALE_POW2 if pow2_scales else 0
    with torch.cuda.device(dev):
        st = lib().gq_fp8_expert_rowwise(_ptr(w), E, N, K, _ptr(out), _ptr(scales), flags, sh)
    _check(st, "gq_fp8_expert_rowwise")
    return out, scales


def mxfp8_dim0(x: torch.Tensor, mode: str = "floor", *, out=None, scales=None, stream=None):
    """mxfp8 cast along dim0: blocks of 32 consecutive elements of a row share
    a power-of-two scale.  x bf16 (M, K) CUDA tensor, K % 32 == 0; mode
    "floor" or "rceil".  Returns (q float8_e4m3fn (M, K), scales uint8
    (M, K // 32) e8m0 bytes)."""
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.bfloat16
            and x.dim() == 2 and x.is_contiguous()):
        raise ValueError("mxfp8_dim0: x must be a contiguous 2-D bf16 CUDA tensor")
    modes = {"floor": GQ_MX_FLOOR, "rceil": GQ_MX_RCEIL}
    if mode not in modes:
        raise ValueError("mxfp8_dim0: mode must be 'floor' or 'rceil'")
    M, K = x.shape
    dev = x.device
    if out is None:
        out = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=dev)
    if scales is None:
        scales = torch.empty((M, K // 32), dtype=torch.uint8, device=dev)
    if out.shape != (M, K) or out.element_size() != 1 or not out.is_contiguous():
        raise ValueError("mxfp8_dim0: out must be a contiguous 1-byte (M, K) tensor")
    if scales.shape != (M, K // 32) or scales.element_size() != 1 or not scales.is_contiguous():
        raise ValueError("mxfp8_dim0: scales must be a contiguous 1-byte (M, K // 32) tensor")
    sh = _stream_handle(stream, dev)
    with torch.cuda.device(dev):
        st = lib().gq_mxfp8_dim0(_ptr(x), M, K, _ptr(out), _ptr(scales), modes[mode], sh)
    _check(st, "gq_mxfp8_dim0")
    return out, scales


def grouped_wgrad(qa_t: torch.Tensor, sa: torch.Tensor, qx: torch.Tensor, sx: torch.Tensor,
                  offs: torch.Tensor, *, out=None, stream=None):
    """grad_weight per token group from the quantized operands: qa_t e4m3
    (T, N) (the rowwise_t output), sa float32 (N, G), qx e4m3 (T, K) (the
    colwise output), sx float32 (G, K), offs int32 (G,) end offsets along T.
    Returns out bf16 (G, N, K) = the per-group sum of products divided by
    sa * sx."""
    for name, t, nd in (("qa_t", qa_t, 2), ("qx", qx, 2)):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.element_size() == 1
                and t.dim() == nd and t.is_contiguous()):
            raise ValueError(f"grouped_wgrad: {name} must be a contiguous 2-D 1-byte CUDA tensor")
    T, N = qa_t.shape
    T2, K = qx.shape
    if T2 != T:
        raise ValueError("grouped_wgrad: qa_t and qx must have the same number of tokens")
    if not (offs.is_cuda and offs.dtype == torch.int32 and offs.dim() == 1 and offs.is_contiguous()):
        raise ValueError("grouped_wgrad: offs must be a contiguous 1-D int32 CUDA tensor")
    G = offs.shape[0]
    for name, t, shape in (("sa", sa, (N, G)), ("sx", sx, (G, K))):
        if not (t.is_cuda and t.dtype == torch.float32 and tuple(t.shape) == shape
                and t.is_contiguous()):
            raise ValueError(f"grouped_wgrad: {name} must be a contiguous float32 {shape} CUDA tensor")
    dev = qa_t.device
    if out is None:
        out = torch.empty((G, N, K), dtype=torch.bfloat16, device=dev)
    if out.shape != (G, N, K) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("grouped_wgrad: out must be a contiguous bf16 (G, N, K) tensor")
    sh = _stream_handle(stream, dev)
    with torch.cuda.device(dev):
        st = lib().gq_grouped_wgrad(_ptr(qa_t), _ptr(sa), _ptr(qx), _ptr(sx), T, N, K,
                                    _ptr(offs), G, _ptr(out), sh)
    _check(st, "gq_grouped_wgrad")
    return out


def colwise_noalloc(x: torch.Tensor, offs: torch.Tensor, *, out=None,
                    scales=None, stream=None):
    """colwise() for callers that cannot allocate device memory: the library
    uses its own fixed scratch array instead of a workspace.  Limited to
    problems whose workspace would fit GQ_NOALLOC_SCRATCH_BYTES; calls that
    may overlap on the GPU must not be issued (they share the scratch).
    The outputs must be passed in by such callers; when omitted, torch
    allocates them here as a convenience."""
    _check_in(x, offs, "colwise_noalloc")
    M, K = x.shape
    G = offs.numel()
    dev = x.device
    if out is None:
        out = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=dev)
    if scales is None:
        scales = torch.empty((G, K), dtype=torch.float32, device=dev)
    if out.shape != (M, K) or out.element_size() != 1 or not out.is_contiguous():
        raise ValueError("colwise_noalloc: out must be a contiguous 1-byte (M, K) tensor")
    if scales.shape != (G, K) or scales.dtype != torch.float32 or not scales.is_contiguous():
        raise ValueError("colwise_noalloc: scales must be a contiguous float32 (G, K) tensor")
    sh = _stream_handle(stream, dev)
    with torch.cuda.device(dev):
        st = lib().gq_fp8_colwise_noalloc(_ptr(x), M, K, _ptr(offs), G,
                                          _ptr(out), _ptr(scales), sh)
    _check(st, "gq_fp8_colwise_noalloc")
    return out, scales


def check_device_error(stream=None, device=None):
    """Synchronises the stream and raises GQError on a recorded device-side
    timeout (or a CUDA error)."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    sh = _stream_handle(stream, dev)
    with torch.cuda.device(dev):
        _check(lib().gq_check_device_error(sh), "gq_check_device_error")


def debug_set(skip_arrival: bool = False, wait_timeout_ns: int = 0, no_split: bool = False):
    """Test hooks: see gq_debug_set in include/gq_fp8.h (skip_arrival is
    flag bit 0, no_split bit 1)."""
    flags = int(bool(skip_arrival)) | (2 if no_split else 0)
    _check(lib().gq_debug_set(flags, int(wait_timeout_ns)), "gq_debug_set")


def set_lag(kind: int, lag: int = 0):
    """Tuning knob: see gq_set_lag in include/gq_fp8.h (0 = automatic)."""
    _check(lib().gq_set_lag(int(kind), int(lag)), "gq_set_lag")


# ------------------------------------------------------ host-buffer calls --

_h2d_streams: dict = {}  # (device, stream) -> side stream for host->device copies


def _to_device(t, device, s, name):
    """Copies a host tensor to the device on a side stream, so that the copy
    can run while the work already queued on ``s`` (the previous call's
    kernel and device->host copies) finishes; ``s`` waits for the copy.  The
    device buffer is allocated on the side stream and recorded on ``s``, so
    the allocator reuses it only after the side stream's copy and ``s``'s use
    of it are both done."""
    if t.is_cuda:
        raise ValueError(f"{name}: expected a host tensor")
    key = (device.index, s.cuda_stream)
    with _ws_lock:
        cs = _h2d_streams.get(key)
        if cs is None:
            cs = torch.cuda.Stream(device)
            _h2d_streams[key] = cs
    with torch.cuda.stream(cs):
        d = t.to(device, non_blocking=True)
    ev = torch.cuda.Event()
    ev.record(cs)
    s.wait_event(ev)
    d.record_stream(s)
    return d


def colwise_host(x_host, offs_host, out_host=None, scales_host=None, *,
                 device="cuda", stream=None, pow2_scales: bool = False):
    """End-to-end colwise call on host buffers: host->device copies of x and
    offs (on a side stream that ``stream`` waits for, so that they overlap
    the work already queued), the kernel and the device->host copies of q
    and scales on ``stream``.  Pinned host tensors make the copies
    asynchronous; the caller synchronises ``stream`` before reading the
    results and keeps the host inputs unchanged until then."""
    dev = torch.device(device)
    M, K = x_host.shape
    G = offs_host.numel()
    if out_host is None:
        out_host = torch.empty((M, K), dtype=torch.float8_e4m3fn, pin_memory=True)
    if scales_host is None:
        scales_host = torch.empty((G, K), dtype=torch.float32, pin_memory=True)
    s = torch.cuda.current_stream(dev) if stream is None else stream
    x = _to_device(x_host, dev, s, "colwise_host")
    o = _to_device(offs_host, dev, s, "colwise_host")
    with torch.cuda.stream(s):
        q, sc = colwise(x, o, stream=s, pow2_scales=pow2_scales)
        out_host.copy_(q, non_blocking=True)
        scales_host.copy_(sc, non_blocking=True)
    return out_host, scales_host


def rowwise_t_host(a_host, offs_host, out_host=None, scales_host=None, *,
                   device="cuda", stream=None, pow2_scales: bool = False):
    """End-to-end rowwise_t call on host buffers (see colwise_host)."""
    dev = torch.device(device)
    N, Mg = a_host.shape
    G = offs_host.numel()
    if out_host is None:
        out_host = torch.empty((Mg, N), dtype=torch.float8_e4m3fn, pin_memory=True)
    if scales_host is None:
        scales_host = torch.empty((N, G), dtype=torch.float32, pin_memory=True)
    s = torch.cuda.current_stream(dev) if stream is None else stream
    a = _to_device(a_host, dev, s, "rowwise_t_host")
    o = _to_device(offs_host, dev, s, "rowwise_t_host")
    with torch.cuda.stream(s):
        qt, sc = rowwise_t(a, o, stream=s, pow2_scales=pow2_scales)
        out_host.copy_(qt, non_blocking=True)
        scales_host.copy_(sc, non_blocking=True)
    return out_host, scales_host
