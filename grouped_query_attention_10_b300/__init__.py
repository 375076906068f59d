"""B300-native (sm_103a) grouped-query attention forward: prefill, decode and
KV-cache append behind a C interface (include/gqa.h).

The functions below are thin ctypes bindings; every step of the computation
runs in the CUDA kernels of ``libgqa_b300.so``. A missing library raises on
first use; there is no CPU fallback.
"""

from .binding import (  # noqa: F401
    GQAError,
    gqa_decode_fwd,
    gqa_decode_workspace_bytes,
    gqa_prefill_fwd,
    gqa_prefill_kvcache_fwd,
    gqa_status_string,
    kv_cache_append,
    kv_cache_append_paged_rope,
    kv_cache_append_rope,
    load_library,
)
