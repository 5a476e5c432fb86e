"""Mamba-3 SSM layer core on NVIDIA B300 (sm_103a).

The computation lives in ``libm3ssm.so`` (CUDA; C ABI in ``include/m3_ssm.h``):
a chunked tcgen05/TMA prefill, a CUDA-core recurrent prefill for fp32, and a
bandwidth-bound decode step, plus the Mamba-2 special case of both (lambda = 1,
theta = 0) for the Mamba-2 versus Mamba-3 comparison.  This package is the thin Python binding.
"""
from ._binding import (  # noqa: F401
    M3_BF16,
    M3_ERR_RANGE,
    M3_ERR_TIMEOUT,
    M3_ERR_UNSUPPORTED,
    M3_ERR_WORKSPACE,
    M3_F32,
    M3_OK,
    BCNorm,
    M3BcNorm,
    M3Dims,
    M3Error,
    M3State,
    State,
    library_path,
    load,
    m3_ssd_decode_step,
    m3_ssd_prefill,
    m3_ssm_decode_step,
    m3_ssm_decode_step_bcnorm,
    m3_ssm_device_status,
    m3_ssm_prefill,
    m3_ssm_prefill_backward,
    m3_ssm_prefill_bcnorm,
    m3_ssm_prefill_noalloc,
    m3_ssm_prefill_workspace,
    prefill_workspace,
    status_str,
    workspace_for,
)
