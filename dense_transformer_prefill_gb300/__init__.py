"""GB300 (sm_103a) dense-transformer prefill: Python binding of the C-ABI library.

Every step of the forward pass runs in the CUDA kernels of `libdtp.so`; this
package only marshals arguments (torch tensors are used for device memory and
streams) and raises `DtpError` on a non-zero status.  There is no CPU fallback:
importing the binding without the built library raises.
"""
from .build import build  # noqa: F401
from ._binding import (  # noqa: F401
    DTP_BF16,
    DTP_F32,
    DTP_TF32,
    DTP_PREC_BF16,
    DTP_PREC_E4M3,
    DTP_PREC_F32,
    DTP_PREC_TF32,
    KERNEL_KINDS,
    DtpError,
    Model,
    check,
    config_from,
    fwd_prefill,
    fwd_prefill_chunk,
    fwd_prefill_ex,
    fwd_prefill_host,
    fwd_prefill_host_batch,
    fwd_prefill_varlen,
    gate_up_swiglu,
    kv_state_size,
    last_error,
    launch_count,
    linear,
    linear_e4m3,
    lib,
    pack_globals,
    pack_layer,
    packed_size,
    qk_norm_rope_neox,
    quantize_rows_e4m3,
    qkv_norm_rope,
    rms_norm,
    rms_norm_e4m3,
    sdpa_causal_gqa,
    sdpa_workspace_size,
    selftest_wait_timeout,
    swiglu,
    timer_disable,
    timer_enable,
    timer_read,
    workspace_size,
    workspace_size_host,
    workspace_size_host_batch,
    workspace_size_varlen,
)
