"""GB300 (sm_103a) paged decode / step attention.

The product is the C-ABI library ``liblnk.so`` (declared in ``include/lnk.h``);
this package holds its CUDA sources (``csrc/``), the build step (``build.py``)
and a thin ctypes binding with the C names (``binding.py``).
"""
from .binding import (  # noqa: F401
    DEV_TIMEOUT,
    EXPORTED,
    KV_BF16,
    KV_E4M3,
    LIBRARY_PATH,
    AttnDesc,
    LnkError,
    Pager,
    RopeDesc,
    attn_desc,
    lnk_paged_append_rope,
    lnk_paged_copy_pages,
    lnk_paged_decode_attn,
    lnk_paged_decode_step,
    lnk_paged_decode_step_launches,
    lnk_paged_decode_attn_static,
    lnk_paged_step_attn,
    lnk_paged_workspace_size,
    lnk_rope_inv_freq,
    lnk_selftest_wait_timeout,
    lnk_status_string,
    rope_desc,
)
