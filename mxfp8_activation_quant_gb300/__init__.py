"""GB300 (sm_103a) MXFP8 activation chain: standalone quantizer, the fused `_o_proj` pair
(wo_a einsum writing MXFP8 z, wo_b MXFP8 GEMM consuming it) and the RMSNorm dual-output
producer, behind the C ABI in include/mxq.h. The Python layer only marshals arguments."""
from ._lib import (  # noqa: F401
    MXFP8,
    SF_PACKED_I32_MN,
    SF_ROWMAJOR_U8,
    SF_TILED_128X4,
    MxqError,
    abi_version,
    check_status,
    empty_sf,
    gemm_mxfp8_bf16,
    load,
    mxfp8_quantize,
    new_status,
    o_proj_mxfp8,
    o_proj_mxfp8_from_bf16,
    o_proj_mxfp8_noalloc,
    quantize,
    rmsnorm_dual_out,
    selftest_hold_sms,
    selftest_wait_timeout,
    sf_bytes,
    status_bytes,
    wo_a_einsum_mxfp8,
    workspace_bytes,
    workspace_for,
)
