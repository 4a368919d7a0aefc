"""GB300 (sm_103a) fused EXL3 routed-expert MoE layer.

The compute runs in the CUDA library built from csrc/ (see include/exl3.h);
this package holds its build script and a thin ctypes binding.
"""
from .binding import (  # noqa: F401
    DeviceExperts, DeviceProjection, DeviceStages, Exl3Error,
    exl3_abi_version, exl3_linear, exl3_linear_workspace_bytes, exl3_moe_additive,
    exl3_moe_forward, exl3_moe_workspace_bytes, exl3_route_pack, exl3_route_pack_max_tiles,
    exl3_workspace_error, EXL3_F16, EXL3_BF16, EXL3_F32, EXL3_I32, EXL3_I64,
)
