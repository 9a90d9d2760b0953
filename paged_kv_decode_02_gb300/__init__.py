"""Paged-KV single-token decode attention for GB300 (sm_103a).

The compute runs in ``libpagedkv.so`` (hand-written CUDA behind a C ABI, declared in
``include/pagedkv.h``); :mod:`.pagedkv` is a thin ctypes binding over it. The binding
is loaded on first use of one of its names, so ``workloads`` (the seeded input
generator) can be imported without the library.
"""

_API = (
    "paged_kv_append", "paged_kv_append_int8", "paged_kv_append_fp8",
    "paged_decode_attention", "paged_decode_attention_int8", "paged_decode_attention_fp8",
    "paged_decode_attention_cascade", "paged_decode_attention_multi",
    "paged_decode_attention_multi_q8", "paged_decode_attention_cascade_q8",
    "cascade_q8_workspace_bytes",
    "cascade_workspace_bytes", "multi_workspace_bytes", "multi_q8_workspace_bytes",
    "copy_blocks", "swap_out", "swap_in",
    "decode_workspace_bytes", "library_path", "load_library", "PagedKVError",
    "Status", "Dims",
)

__all__ = list(_API)


def __getattr__(name):
    if name in _API:
        from . import pagedkv
        return getattr(pagedkv, name)
    raise AttributeError(name)
