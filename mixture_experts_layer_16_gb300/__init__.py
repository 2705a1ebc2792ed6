"""A fused mixture-of-experts layer (forward + backward) for one NVIDIA GB300.

The compute runs in libmm_moe.so (hand-written sm_103a CUDA behind a C ABI,
include/mm_moe.h); `binding` marshals torch tensors into it.  The library is
loaded on first use and every call raises if it is missing.
"""
from .binding import (Shape, Workspace, MoEError, make_shape, mm_moe_workspace_size,  # noqa: F401
                      mm_moe_forward, mm_moe_backward, mm_moe_get_routing, mm_moe_read_status,
                      mm_moe_last_launch_count, mm_moe_profile_start, mm_moe_profile_stop,
                      mm_moe_kernel_name, mm_moe_kernel_count)
from .layer import MoELayer, MoERouter  # noqa: F401,E402
