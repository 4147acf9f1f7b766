"""GB300-native per-token-group fp8 e4m3 quantization for MoE grouped GEMMs.

Two paths, both in hand-written sm_103a CUDA kernels behind the C ABI of
``include/gq_fp8.h``:

* ``colwise(x, offs)``   -- groups along dim0: one scale per (group, column);
* ``rowwise_t(a, offs)`` -- groups along dim1: one scale per (row, group), fp8
  output written transposed;
* ``expert_dim1(w)``     -- stacked expert weights (E, K, N): one scale per
  (expert, column), reduced along dim1;
* ``expert_rowwise(w)``  -- stacked expert weights (E, N, K): one scale per
  (expert, row);
* ``mxfp8_dim0(x, mode)`` -- mxfp8: 32-element row blocks with e8m0 scales
  (FLOOR or RCEIL);
* ``grouped_wgrad(qa_t, sa, qx, sx, offs)`` -- the consumer of the two
  paths: grad_weight per token group on the tensor cores, bf16 out.

scale = 448 / max(amax, 1e-12) in IEEE fp32; q = saturating round-to-nearest-
even e4m3 cast of fp32(x * scale); ``pow2_scales=True`` rounds every scale
down to a power of two first.  ``offs`` are int32 end offsets of the
token groups.  This package is argument marshalling over the library; torch
supplies device memory and streams.  ``synth`` draws seeded inputs.
"""
from ._binding import (GQ_KIND_COLWISE, GQ_KIND_ROWWISE_T, GQ_MAX_GROUPS,
                       GQ_SCALE_POW2, GQ_TWO_PHASE, GQ_WORKSPACE_ZEROED, GQError, check_device_error, colwise, colwise_host,
                       colwise_noalloc, expert_dim1, expert_rowwise, mxfp8_dim0,
                       grouped_wgrad, debug_set, lib, library_path, rowwise_t,
                       rowwise_t_host, set_lag, status_string, version,
                       workspace_bytes)
from ._build import build

__all__ = [
    "GQ_KIND_COLWISE", "GQ_KIND_ROWWISE_T", "GQ_MAX_GROUPS", "GQ_SCALE_POW2", "GQ_TWO_PHASE",
    "GQ_WORKSPACE_ZEROED", "GQError",
    "build", "check_device_error", "colwise", "colwise_host",
    "colwise_noalloc", "debug_set", "expert_dim1", "expert_rowwise", "grouped_wgrad",
    "mxfp8_dim0",
    "lib", "library_path", "rowwise_t", "rowwise_t_host", "set_lag",
    "status_string",
    "version", "workspace_bytes",
]
