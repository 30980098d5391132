"""GB300-native (sm_103a) binary low-rank (blr) linear layer: forward, backward and sign gradients.

The compute path is the CUDA library ``_lib/libblr.so`` (C ABI in
``include/blr.h``); this package is its thin Python binding plus the seeded
synthetic workloads used by the tests and the benchmark.
"""
from ._binding import (  # noqa: F401
    BLR_ERR_ALIGN,
    BLR_ERR_ARG,
    BLR_ERR_CUDA,
    BLR_ERR_DEVICE_CHECK,
    BLR_ERR_SHAPE,
    BLR_ERR_STATE,
    BLR_ERR_UNSUPPORTED_DEVICE,
    BLR_ERR_WORKSPACE,
    BLR_OK,
    BlrError,
    adam,
    alloc_paths_workspace,
    alloc_plane_workspace,
    alloc_sign_workspace,
    alloc_workspace,
    backward,
    backward_paths,
    check_status,
    forward,
    forward_paths,
    forward_noalloc,
    load,
    pack_signs,
    path_workspace,
    paths_workspace_bytes,
    plane_linear,
    plane_workspace_bytes,
    sign_grads,
    sign_workspace_bytes,
    trace_begin,
    trace_end,
    unpack_signs,
    words_per_row,
    workspace_bytes,
)
