"""GB300-native (sm_103a) Mamba-1 selective-SSM mixer core.

C-ABI entry points (include/mamba_ssm.h), each backed by hand-written CUDA kernels:
  mamba_conv1d_silu_prefill     causal depthwise conv1d + SiLU over T tokens
  mamba_conv1d_silu_step        T=1 conv step on a [n_layers][B*Di*K] state
  mamba_selective_scan_prefill  selective scan + SiLU(z) gate, state in/out
  mamba_ssm_step_batched        T=1 SSM step on a [n_layers][B*Di*N] state
  mamba_mixer_step_batched      both T=1 steps fused in one kernel
  mamba_mixer_prefill           conv1d + SiLU and the selective scan in one pass
  mamba_decode_graph_*          n_steps x n_layers fused steps recorded as one CUDA graph
  mamba3_siso_step_batched      T=1 step of the Mamba-3 SISO (trapezoidal) recurrence
  mamba3_siso_step_prepare      its inputs: angle state advanced, k and q rotated, alpha/beta/gamma
  mamba3_siso_step_fused_batched  both in one launch (k and q never leave the SM)
  mamba3_decode_graph_create    n_steps x n_layers such tokens recorded once as a CUDA graph
  mamba_linear_bf16             a projection of the layer on the tensor cores (tcgen05)
  mamba_rmsnorm                 RMSNorm of the f32 residual stream
  mamba_layer_prefill / _step   the whole Mamba-1 block (norm, projections, mixer, residual)
  mamba_layer_decode_graph_create  one decode token through n_layers blocks as one CUDA graph
  mamba_selective_scan_prefill_noalloc  the scan prefill with a static scratch
  mamba_selective_scan_workspace_bytes  scratch size of the prefill's balanced routes
This package is the thin Python binding (argument marshalling over ctypes);
`synth` holds the seeded synthetic inputs used by the tests and the benchmark.
"""
from ._binding import (  # noqa: F401
    ABI_SYMBOLS,
    DecodeGraph,
    LayerDecodeGraph,
    Mamba3DecodeGraph,
    LIB_PATH,
    MAMBA_BF16,
    MAMBA_ERR_CUDA,
    MAMBA_ERR_INVALID_ARG,
    MAMBA_ERR_UNSUPPORTED,
    MAMBA_F32,
    MAMBA_FAULT_RING_WAIT,
    MAMBA_FAULT_SCAN_WAIT,
    MAMBA_FAULT_GEMM_WAIT,
    MAMBA_MAX_FUSED_D_CONV,
    MAMBA_NOALLOC_SCRATCH_BYTES,
    MAMBA_OK,
    MambaError,
    load,
    mamba3_siso_step_batched,
    mamba3_siso_step_prepare,
    mamba3_siso_step_fused_batched,
    mamba_conv1d_silu_prefill,
    mamba_conv1d_silu_step,
    mamba_device_faults,
    mamba_last_error,
    mamba_layer_prefill,
    mamba_layer_step,
    mamba_layer_workspace_bytes,
    mamba_linear_bf16,
    mamba_rmsnorm,
    layer_struct,
    LAYER_WEIGHTS,
    mamba_mixer_prefill,
    mamba_mixer_step_batched,
    mamba_selective_scan_prefill,
    mamba_selective_scan_prefill_noalloc,
    mamba_selective_scan_workspace_bytes,
    mamba_selftest_bounded_wait,
    mamba_ssm_step_batched,
    mamba_version,
)

__version__ = "0.1.0"
