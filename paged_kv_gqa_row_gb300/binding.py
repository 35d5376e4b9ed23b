"""Thin ctypes binding of liblnk's C ABI (include/lnk.h).

Argument marshalling only: torch tensors (or raw integer addresses) become
pointers, Python numbers become the C descriptor structs, and a non-OK status
raises LnkError.  Every computation runs in the library's CUDA kernels; there
is no other code path.  Importing this module fails if liblnk.so has not been
built (``python -c "import __graft_entry__ as g; g.build()"``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_HERE, "liblnk.so")

if not os.path.exists(LIBRARY_PATH):
    raise ImportError(f"liblnk.so is not built ({LIBRARY_PATH}); run paged_kv_gqa_row_gb300/build.py")
_lib = ctypes.CDLL(LIBRARY_PATH)

c_i32, c_f32, c_f64, c_size, c_vp = ctypes.c_int32, ctypes.c_float, ctypes.c_double, ctypes.c_size_t, ctypes.c_void_p

LNK_OK = 0
STATUS_NAMES = {0: "LNK_OK", 1: "LNK_EINVAL", 2: "LNK_ERANGE", 3: "LNK_ECUDA",
                4: "LNK_EUNSUPPORTED", 5: "LNK_EWORKSPACE", 6: "LNK_ENOSPACE"}
DEV_BAD_ROW, DEV_BAD_POSITION, DEV_BAD_PAGE, DEV_BAD_SLOT = 0x01, 0x02, 0x04, 0x08
DEV_SEGMENT, DEV_BAD_LAST, DEV_TIMEOUT = 0x10, 0x20, 0x40

EXPORTED = ["lnk_status_string", "lnk_rope_inv_freq", "lnk_paged_workspace_size",
            "lnk_paged_append_rope", "lnk_paged_decode_attn", "lnk_paged_decode_step",
            "lnk_paged_decode_step_launches", "lnk_paged_step_attn",
            "lnk_paged_decode_attn_static", "lnk_pager_create", "lnk_pager_destroy", "lnk_pager_reserve",
            "lnk_pager_fork", "lnk_pager_prepare_append", "lnk_pager_release", "lnk_pager_table",
            "lnk_pager_free_pages", "lnk_pager_refcount", "lnk_paged_copy_pages",
            "lnk_selftest_wait_timeout"]


class LnkError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.lnk_status_string(status).decode()
        super().__init__(f"{where}: {msg}")


KV_BF16, KV_E4M3 = 0, 1


class AttnDesc(ctypes.Structure):
    _fields_ = [("num_q_heads", c_i32), ("num_kv_heads", c_i32), ("head_dim", c_i32),
                ("page_size", c_i32), ("num_pages", c_i32), ("num_rows", c_i32),
                ("pages_per_row", c_i32), ("window", c_i32), ("scale", c_f32),
                ("kv_dtype", c_i32), ("k_scale", c_f32), ("v_scale", c_f32)]


class RopeDesc(ctypes.Structure):
    _fields_ = [("theta", c_f64), ("llama3", c_i32), ("factor", c_f64),
                ("low_freq_factor", c_f64), ("high_freq_factor", c_f64),
                ("original_max_position", c_f64)]


_lib.lnk_status_string.restype = ctypes.c_char_p
_lib.lnk_status_string.argtypes = [ctypes.c_int]
_lib.lnk_rope_inv_freq.restype = ctypes.c_int
_lib.lnk_rope_inv_freq.argtypes = [ctypes.POINTER(RopeDesc), c_i32, ctypes.POINTER(c_f32)]
_lib.lnk_paged_workspace_size.restype = c_size
_lib.lnk_paged_workspace_size.argtypes = [ctypes.POINTER(AttnDesc), c_i32]
_lib.lnk_paged_append_rope.restype = ctypes.c_int
_lib.lnk_paged_append_rope.argtypes = [ctypes.POINTER(AttnDesc), ctypes.POINTER(RopeDesc),
                                       c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_f32,
                                       c_vp, c_vp, c_vp, c_i32, c_vp, c_vp]
_lib.lnk_paged_decode_attn.restype = ctypes.c_int
_lib.lnk_paged_decode_attn.argtypes = [ctypes.POINTER(AttnDesc), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                       c_i32, c_vp, c_size, c_vp, c_vp]
_lib.lnk_paged_decode_step.restype = ctypes.c_int
_lib.lnk_paged_decode_step.argtypes = [ctypes.POINTER(AttnDesc), ctypes.POINTER(RopeDesc),
                                       c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_f32,
                                       c_vp, c_vp, c_vp, c_vp, c_i32, c_vp, c_size, c_vp, c_vp]
_lib.lnk_paged_decode_step_launches.restype = c_i32
_lib.lnk_paged_decode_step_launches.argtypes = [ctypes.POINTER(AttnDesc), c_i32]
_lib.lnk_paged_decode_attn_static.restype = ctypes.c_int
_lib.lnk_paged_decode_attn_static.argtypes = [ctypes.POINTER(AttnDesc), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                              c_i32, c_vp, c_vp]
_lib.lnk_paged_step_attn.restype = ctypes.c_int
_lib.lnk_paged_step_attn.argtypes = [ctypes.POINTER(AttnDesc), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                     c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_vp, c_size,
                                     c_vp, c_vp]
_i32p = ctypes.POINTER(c_i32)
_lib.lnk_pager_create.restype = ctypes.c_int
_lib.lnk_pager_create.argtypes = [c_i32, c_i32, c_i32, ctypes.POINTER(c_vp)]
_lib.lnk_pager_destroy.restype = None
_lib.lnk_pager_destroy.argtypes = [c_vp]
_lib.lnk_pager_reserve.restype = ctypes.c_int
_lib.lnk_pager_reserve.argtypes = [c_vp, c_i32, c_i32]
_lib.lnk_pager_fork.restype = ctypes.c_int
_lib.lnk_pager_fork.argtypes = [c_vp, c_i32, c_i32, c_i32]
_lib.lnk_pager_prepare_append.restype = ctypes.c_int
_lib.lnk_pager_prepare_append.argtypes = [c_vp, _i32p, _i32p, c_i32, _i32p, _i32p, _i32p]
_lib.lnk_pager_release.restype = ctypes.c_int
_lib.lnk_pager_release.argtypes = [c_vp, c_i32]
_lib.lnk_pager_table.restype = ctypes.c_int
_lib.lnk_pager_table.argtypes = [c_vp, _i32p]
_lib.lnk_pager_free_pages.restype = c_i32
_lib.lnk_pager_free_pages.argtypes = [c_vp]
_lib.lnk_pager_refcount.restype = c_i32
_lib.lnk_pager_refcount.argtypes = [c_vp, c_i32]
_lib.lnk_paged_copy_pages.restype = ctypes.c_int
_lib.lnk_paged_copy_pages.argtypes = [ctypes.POINTER(AttnDesc), c_vp, c_vp, c_vp, c_vp, c_i32, c_vp, c_vp]
_lib.lnk_selftest_wait_timeout.restype = ctypes.c_int
_lib.lnk_selftest_wait_timeout.argtypes = [c_vp, ctypes.c_uint64, c_vp]


def attn_desc(num_q_heads, num_kv_heads, head_dim, num_pages, num_rows, pages_per_row,
              window=0, scale=0.0, page_size=64, kv_dtype=KV_BF16, k_scale=1.0, v_scale=1.0) -> AttnDesc:
    return AttnDesc(num_q_heads, num_kv_heads, head_dim, page_size, num_pages, num_rows,
                    pages_per_row, window, scale, kv_dtype, k_scale, v_scale)


def rope_desc(theta, llama3=None) -> RopeDesc:
    if llama3 is None:
        return RopeDesc(theta, 0, 0.0, 0.0, 0.0, 0.0)
    factor, low, high, orig = llama3
    return RopeDesc(theta, 1, factor, low, high, orig)


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != LNK_OK:
        raise LnkError(status, where)


def lnk_status_string(status: int) -> str:
    return _lib.lnk_status_string(status).decode()


def lnk_rope_inv_freq(rope: RopeDesc, head_dim: int):
    out = (c_f32 * (head_dim // 2))()
    _check(_lib.lnk_rope_inv_freq(ctypes.byref(rope), head_dim, out), "lnk_rope_inv_freq")
    return [float(x) for x in out]


def lnk_paged_workspace_size(desc: AttnDesc, max_rows: int) -> int:
    return int(_lib.lnk_paged_workspace_size(ctypes.byref(desc), max_rows))


def lnk_paged_append_rope(desc, rope, q, k, v, positions, rows, slots, table, q_norm_w, k_norm_w,
                          norm_eps, k_pool, v_pool, q_out, T, dev_status=None, stream=None):
    st = _lib.lnk_paged_append_rope(ctypes.byref(desc), ctypes.byref(rope), _ptr(q), _ptr(k), _ptr(v),
                                    _ptr(positions), _ptr(rows), _ptr(slots), _ptr(table),
                                    _ptr(q_norm_w), _ptr(k_norm_w), norm_eps, _ptr(k_pool),
                                    _ptr(v_pool), _ptr(q_out), T, _ptr(dev_status), _stream(stream))
    _check(st, "lnk_paged_append_rope")


def lnk_paged_decode_attn(desc, q_roped, positions, table, k_pool, v_pool, out, B, workspace,
                          ws_bytes, dev_status=None, stream=None):
    st = _lib.lnk_paged_decode_attn(ctypes.byref(desc), _ptr(q_roped), _ptr(positions), _ptr(table),
                                    _ptr(k_pool), _ptr(v_pool), _ptr(out), B, _ptr(workspace),
                                    ws_bytes, _ptr(dev_status), _stream(stream))
    _check(st, "lnk_paged_decode_attn")


def lnk_paged_decode_step(desc, rope, q, k, v, positions, table, q_norm_w, k_norm_w, norm_eps, k_pool,
                          v_pool, q_out, out, B, workspace, ws_bytes, dev_status=None, stream=None):
    st = _lib.lnk_paged_decode_step(ctypes.byref(desc), ctypes.byref(rope), _ptr(q), _ptr(k), _ptr(v),
                                    _ptr(positions), _ptr(table), _ptr(q_norm_w), _ptr(k_norm_w), norm_eps,
                                    _ptr(k_pool), _ptr(v_pool), _ptr(q_out), _ptr(out), B, _ptr(workspace),
                                    ws_bytes, _ptr(dev_status), _stream(stream))
    _check(st, "lnk_paged_decode_step")


def lnk_paged_decode_step_launches(desc, B) -> int:
    """Kernels lnk_paged_decode_step enqueues for B rows (1 or 2; 0 for B = 0; -1: rejected)."""
    return int(_lib.lnk_paged_decode_step_launches(ctypes.byref(desc), B))


def lnk_paged_decode_attn_static(desc, q_roped, positions, table, k_pool, v_pool, out, B,
                                 dev_status=None, stream=None):
    """lnk_paged_decode_attn with the library's own static scratch (no workspace)."""
    st = _lib.lnk_paged_decode_attn_static(ctypes.byref(desc), _ptr(q_roped), _ptr(positions), _ptr(table),
                                           _ptr(k_pool), _ptr(v_pool), _ptr(out), B, _ptr(dev_status),
                                           _stream(stream))
    _check(st, "lnk_paged_decode_attn_static")


def lnk_paged_step_attn(desc, q_roped, rows, positions, segments, step_positions, table, k_pool,
                        v_pool, out, last, last_out, P, B, M, workspace, ws_bytes, dev_status=None,
                        stream=None):
    st = _lib.lnk_paged_step_attn(ctypes.byref(desc), _ptr(q_roped), _ptr(rows), _ptr(positions),
                                  _ptr(segments), _ptr(step_positions), _ptr(table), _ptr(k_pool),
                                  _ptr(v_pool), _ptr(out), _ptr(last), _ptr(last_out), P, B, M,
                                  _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(st, "lnk_paged_step_attn")


def lnk_paged_copy_pages(desc, k_pool, v_pool, src_pages, dst_pages, n, dev_status=None, stream=None):
    st = _lib.lnk_paged_copy_pages(ctypes.byref(desc), _ptr(k_pool), _ptr(v_pool), _ptr(src_pages),
                                   _ptr(dst_pages), n, _ptr(dev_status), _stream(stream))
    _check(st, "lnk_paged_copy_pages")


def lnk_selftest_wait_timeout(dev_status, limit_ns, stream=None):
    st = _lib.lnk_selftest_wait_timeout(_ptr(dev_status), int(limit_ns), _stream(stream))
    _check(st, "lnk_selftest_wait_timeout")


def _i32_array(values):
    import numpy as np
    a = np.ascontiguousarray(values, dtype=np.int32)
    return a, a.ctypes.data_as(_i32p)


class Pager:
    """The host page allocator (lnk_pager_*): calls marshalled to the C ABI."""

    def __init__(self, num_pages: int, num_rows: int, pages_per_row: int):
        h = c_vp()
        _check(_lib.lnk_pager_create(num_pages, num_rows, pages_per_row, ctypes.byref(h)), "lnk_pager_create")
        self._h = h
        self.num_pages, self.num_rows, self.pages_per_row = num_pages, num_rows, pages_per_row

    def close(self):
        if self._h:
            _lib.lnk_pager_destroy(self._h)
            self._h = c_vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reserve(self, row: int, length: int):
        _check(_lib.lnk_pager_reserve(self._h, row, length), "lnk_pager_reserve")

    def fork(self, src_row: int, dst_row: int, length: int):
        _check(_lib.lnk_pager_fork(self._h, src_row, dst_row, length), "lnk_pager_fork")

    def prepare_append(self, rows, positions):
        """Returns the (old, new) page copies the append needs, in order."""
        r, rp = _i32_array(rows)
        q, qp = _i32_array(positions)
        n = len(r)
        src, srcp = _i32_array([0] * max(1, n))
        dst, dstp = _i32_array([0] * max(1, n))
        nc = c_i32(0)
        _check(_lib.lnk_pager_prepare_append(self._h, rp, qp, n, srcp, dstp, ctypes.byref(nc)),
               "lnk_pager_prepare_append")
        return [(int(src[i]), int(dst[i])) for i in range(nc.value)]

    def release(self, row: int):
        _check(_lib.lnk_pager_release(self._h, row), "lnk_pager_release")

    def table(self):
        import numpy as np
        t = np.empty((self.num_rows, self.pages_per_row), dtype=np.int32)
        _check(_lib.lnk_pager_table(self._h, t.ctypes.data_as(_i32p)), "lnk_pager_table")
        return t

    def free_pages(self) -> int:
        return int(_lib.lnk_pager_free_pages(self._h))

    def refcount(self, page: int) -> int:
        return int(_lib.lnk_pager_refcount(self._h, page))


def raw_status(fn_name: str, *args) -> int:
    """Calls a C entry point with already-marshalled arguments and returns its
    status without raising (used to test argument checking)."""
    return getattr(_lib, fn_name)(*args)
