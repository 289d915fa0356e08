"""Exact tiled attention on one GB300 (sm_103a).

Python binding of the C ABI in ``include/fa.h`` (``libfa.so``). See
:mod:`exact_tiled_attention_28_gb300.binding`.
"""

from .binding import (  # noqa: F401
    FA_DQ_ATOMIC,
    FA_DQ_AUTO,
    FA_DQ_SEPARATE,
    FA_ERR_CUDA,
    FA_ERR_DEVICE_CHECK,
    FA_ERR_INVALID_ARG,
    FA_ERR_TIMEOUT,
    FA_ERR_UNSUPPORTED,
    FA_ERR_WORKSPACE,
    FA_OK,
    FaError,
    fa_bwd,
    fa_bwd_stages,
    fa_bwd_varlen,
    fa_bwd_varlen_workspace_size,
    fa_bwd_workspace_size,
    fa_decode,
    fa_decode_workspace_size,
    fa_fwd,
    fa_fwd_varlen,
    fa_last_device_status,
    fa_measure_unit_rates,
    fa_selftest_exp2,
    fa_selftest_wait_timeout,
    fa_set_wait_limit_ns,
    fa_is_debug_build,
    fa_selftest_index_check,
    use_library,
    fa_status_string,
    library_path,
    load,
)
