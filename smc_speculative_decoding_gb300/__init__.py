"""SMC speculative decoding (SMC-SD) per-step particle update on NVIDIA GB300.

The compute lives in libsmcsd.so (hand-written CUDA for sm_103a, C ABI in
include/smcsd.h).  ``binding`` exposes its entry points to Python with the
same names; ``workloads`` draws seeded synthetic inputs; ``build`` compiles
the library in-tree.
"""
from .binding import (  # noqa: F401
    SmcError, smc_params, smc_kv, make_params, make_kv, alloc_workspace,
    smc_abi_version, smc_strerror, smc_workspace_bytes, smc_workspace_init,
    smc_device_status, status_names, smc_step, smc_resample, kv_blocktable_remap,
    sps_verify, sps_verify_ex, smc_set_row_timing_events, smc_set_step_clock,
    smc_selftest_bounded_wait, smc_step_ex,
    smc_draft_sample,
    smc_kv_usage,
    smc_step_opts, SMC_F32, SMC_BF16,
)

__all__ = [
    "SmcError", "smc_params", "smc_kv", "make_params", "make_kv", "alloc_workspace",
    "smc_abi_version", "smc_strerror", "smc_workspace_bytes", "smc_workspace_init",
    "smc_device_status", "status_names", "smc_step", "smc_resample", "kv_blocktable_remap",
    "sps_verify", "sps_verify_ex", "smc_set_row_timing_events", "smc_set_step_clock",
    "smc_selftest_bounded_wait",
    "smc_step_ex", "smc_draft_sample",
    "smc_kv_usage", "smc_step_opts", "SMC_F32", "SMC_BF16",
]
