"""LSH-sampled decode attention (MagicPIG) on one GB300: Python binding of libmagicpig.

Every step of the path runs in the library's CUDA kernels; this module only checks tensor
arguments, allocates outputs and workspaces with PyTorch, and calls the C ABI declared in
include/magicpig.h. There is no CPU fallback: without the built library every call raises.
"""
from .binding import (  # noqa: F401
    MP_BF16,
    MP_F32,
    MP_FLAG_CROSS_POLYTOPE,
    MP_FLAG_MIPS,
    MP_LOGU_TABLE_ENTRIES,
    MagicPIGError,
    Params,
    abi_version,
    build_buckets,
    build_tables,
    buckets_bytes,
    check_report,
    codes_bytes,
    codes_unpack,
    cp_codes_bytes,
    cp_logu_table,
    debug_log_inclusion,
    debug_select,
    debug_select_buckets,
    debug_wait_expiry,
    debug_workspace_bytes,
    decode_attention,
    decode_workspace_bytes,
    device_status,
    encode_keys,
    encode_keys_cp,
    encode_keys_mips,
    encode_query,
    key_mean,
    key_radius,
    key_mean_workspace_bytes,
    lib,
    library_path,
    sampled_attention,
    sampled_attention_buckets,
)
