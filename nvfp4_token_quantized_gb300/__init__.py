"""GB300 (sm_103a) routed-MoE forward with online per-token NVFP4 activations.

The product is the CUDA library ``_lib/libmoe_nvfp4.so`` (C ABI in
``include/moe_nvfp4.h``); this package builds it (``build``) and binds it
(``binding``).  There is no CPU path: if the library is missing or no sm_103a
device is present, the calls fail.
"""

from .builder import build, LIB_PATH  # noqa: F401
from .binding import (  # noqa: F401
    EXPORTED,
    MOE_FLAG_DETERMINISTIC,
    MOE_FLAG_STATIC_ACT_SCALES,
    MoE,
    MoEError,
    load_library,
    moe_create,
    moe_debug_block_scaled_gemm,
    moe_debug_convert,
    moe_destroy,
    moe_forward,
    moe_forward_ex,
    moe_forward_host,
    moe_get_last_error,
    moe_get_status,
    moe_get_workspace_bytes,
    moe_load_weights,
    moe_refresh_scales_inplace,
    moe_route_noalloc,
    moe_set_static_scales,
)
