"""GB300 (sm_103a) NVFP4 paged KV cache: append, A4Q paged prefill, paged decode.

The compute path is the CUDA library libnvfp4kv.so (C ABI in include/nvfp4kv.h);
``nvfp4_paged_kv_append_gb300.binding`` is its thin Python binding.  Build it
with ``__graft_entry__.build()`` (or ``python -m nvfp4_paged_kv_append_gb300.build``).
"""
__version__ = "0.1.0"


def load_binding():
    """Import and return the binding module (raises if the library is missing)."""
    from . import binding as _b
    return _b
