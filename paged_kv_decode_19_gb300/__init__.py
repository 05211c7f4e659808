"""GB300-native paged-KV decode attention (libpageddecode).

Python front of the C-ABI library ``include/pageddecode.h``: ``batch_decode_paged_kv``,
``merge_state_inplace`` and ``append_paged_kv`` run hand-written sm_103a CUDA kernels.
PyTorch supplies device memory and streams only.
"""
from ._lib import (  # noqa: F401
    PDError,
    append_paged_kv,
    append_paged_kv_rope,
    batch_decode_paged_kv,
    batch_decode_paged_kv_noalloc,
    batch_decode_paged_kv_mq,
    check_device_errors,
    host_meta_of,
    last_decode_variant,
    make_desc,
    merge_state_inplace,
    merge_states,
    merge_states_packed,
    cp_shard_plan,
    plan,
    release_stream_workspace,
    version,
    workspace_init,
    workspace_size,
)
