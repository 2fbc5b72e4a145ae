"""GB300 (sm_103a) WNA16 routed-expert MoE forward.

The compute lives in ``libwna16_moe.so`` (hand-written CUDA kernels behind the
C ABI of ``include/wna16_moe.h``); this package only builds it
(``build.build()``) and binds it (``binding``).
"""
from .binding import (ERR_BAD_ROUTING, ERR_CUDA, ERR_DEVICE_TIMEOUT, ERR_INVALID_ARG, ERR_UNSUPPORTED,  # noqa: F401
                      ERR_WORKSPACE_TOO_SMALL, OK, Wna16Error, alloc_workspace, check_wait_timeout, combine, forward,
                      forward_noalloc, forward_partial, launches_last_forward, load_library, pack, profile, profile_read,
                      quantize, read_status, route, route_topk, w2, w13, workspace_size)
