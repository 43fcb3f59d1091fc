"""TriAttention periodic KV-cache compression step on B300 (sm_103a).

The compute path is libtri.so (CUDA kernels behind the C ABI in include/tri.h);
`tri` is its ctypes binding.  There is no CPU fallback.
"""
from .tri import (  # noqa: F401
    KVCache,
    Params,
    Stats,
    TriError,
    tri_calibrate_stats,
    tri_clear_device_status,
    tri_compact_kv,
    tri_compress_step,
    tri_compress_step_static_scratch,
    tri_get_device_status,
    tri_score,
    tri_select_topb,
    tri_version,
    tri_workspace_bytes,
    workspace,
    tri_append_kv,
    tri_decode_attention,
    tri_decode_workspace_bytes,
)
from .decode import DecodeLoop  # noqa: F401
