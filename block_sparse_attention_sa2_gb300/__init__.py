"""GB300 (sm_103a) hot path of SpargeAttention2: hybrid Top-k + Top-p block mask and
trainable block-sparse attention, behind the C ABI of include/sa2.h.

The Python surface is a thin ctypes binding (``sa2.py``); the library is built in-tree by
``build_lib.build()``.  Mask diagnostics, off the attention path, are in ``diagnostics``.
"""
from .sa2 import (  # noqa: F401
    BlockMask,
    Sa2Error,
    attn_bwd,
    attn_fwd,
    blocks,
    build_mask,
    check_device,
    debug_set_wait_limit,
    device_status,
    load_library,
    make_shape,
    profiler_collect,
    profiler_enable,
    vd_loss,
    workspace,
)
