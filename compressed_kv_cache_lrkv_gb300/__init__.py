"""GB300-native attention over an LRKV-compressed KV cache.

The product is the C-ABI library ``liblrkv.so`` (declared in ``include/lrkv.h``)
built from ``csrc/`` for sm_103a; ``compressed_kv_cache_lrkv_gb300.binding`` is a
thin ctypes layer with the same entry-point names.  Nothing here falls back to a
CPU implementation: if the CUDA library cannot be loaded, every call raises.
"""
from . import accounting  # noqa: F401
