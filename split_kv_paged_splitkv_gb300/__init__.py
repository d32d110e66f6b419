"""Python binding of libsplitkv (split-KV paged decode attention, sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libsplitkv.so``.  The functions keep the C names of
``include/splitkv.h``.  Device buffers may be passed as torch tensors (their
``data_ptr()`` is used) or as integer addresses; streams as
``torch.cuda.Stream`` or integer handles (``None`` = torch's current stream).

Importing this package loads the library and fails loudly if it has not been
built (``python -c "import __graft_entry__ as g; g.build()"``); there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsplitkv.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "splitkv.h")

SPLITKV_OK, SPLITKV_EINVAL, SPLITKV_EUNSUPPORTED, SPLITKV_ECUDA, SPLITKV_EWORKSPACE, SPLITKV_EDEVICE = range(6)
SPLITKV_BF16, SPLITKV_FP8_E4M3 = 0, 1
SPLITKV_COMBINE_FUSED, SPLITKV_COMBINE_SEPARATE = 0, 1
SPLITKV_LAYOUT_HND, SPLITKV_LAYOUT_NHD = 0, 1
SPLITKV_ITEM_FIELDS = 8
SPLITKV_RANGE_FIELDS = 5
SPLITKV_DEVERR_TIMEOUT, SPLITKV_DEVERR_SEQLEN, SPLITKV_DEVERR_PAGE = 1, 2, 4
ITEM_FIELD_NAMES = ("b", "h_kv", "split", "num_splits", "page_begin", "page_end", "slot", "group")


class splitkv_desc_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "q_tokens", "num_q_heads", "num_kv_heads", "qk_dim", "v_dim", "page_size",
        "max_pages_per_seq", "num_pages_total", "kv_dtype", "v_shares_k", "combine_mode",
        "kv_layout")]


class SplitKVError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"splitkv status {status}: {message}")
        self.status = status


_vp, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
_SIGNATURES = {
    "splitkv_plan": (_i32, [ctypes.POINTER(splitkv_desc_t), _vp, _i32, _i32, ctypes.POINTER(_vp)]),
    "splitkv_plan_fixed": (_i32, [ctypes.POINTER(splitkv_desc_t), _i32, ctypes.POINTER(_vp)]),
    "splitkv_plan_refresh": (_i32, [_vp, _vp, _vp, _vp]),
    "splitkv_read_items": (_i32, [_vp, _vp, _vp, _i32, _vp]),
    "splitkv_plan_destroy": (None, [_vp]),
    "splitkv_plan_get_items": (_i32, [_vp, _vp, _i32, ctypes.POINTER(_i32)]),
    "splitkv_plan_get_ranges": (_i32, [_vp, _vp, _i32, ctypes.POINTER(_i32)]),
    "splitkv_plan_num_items": (_i32, [_vp]),
    "splitkv_plan_num_ctas": (_i32, [_vp]),
    "splitkv_plan_heads_per_item": (_i32, [_vp]),
    "splitkv_plan_launches_per_call": (_i32, [_vp]),
    "splitkv_workspace_size": (_sz, [_vp]),
    "splitkv_plan_upload": (_i32, [_vp, _vp, _sz, _vp]),
    "splitkv_decode": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _f32, _f32, _vp, _vp, _vp]),
    "splitkv_decode_kv_scales": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _f32, _vp, _vp, _vp,
                                        _vp, _vp]),
    "splitkv_decode_noalloc": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _f32, _f32, _vp, _vp, _vp]),
    "splitkv_noalloc_read_stats": (_i32, [_vp, _vp, _i32, _vp, _vp]),
    "splitkv_decode_partials": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _f32, _f32, _vp, _vp,
                                       _vp]),
    "splitkv_combine_workspace": (_i32, [_vp, _vp, _vp, _vp, _vp]),
    "splitkv_combine": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp]),
    "splitkv_read_stats": (_i32, [_vp, _vp, _vp, _i32, _vp, _vp]),
    "splitkv_debug_gather": (_i32, [ctypes.POINTER(splitkv_desc_t), _vp, _i32, _vp, _i32, _i32,
                                    _i32, _vp, _vp]),
    "splitkv_last_error": (ctypes.c_char_p, []),
}


def header_functions() -> list:
    """Names of the functions ``include/splitkv.h`` declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(splitkv_[a-z_]+)\s*\(", text)))


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int):
    if status != SPLITKV_OK:
        raise SplitKVError(status, _lib.splitkv_last_error().decode())


def make_desc(batch, q_tokens, num_q_heads, num_kv_heads, qk_dim, v_dim, page_size,
              max_pages_per_seq, num_pages_total, kv_dtype=SPLITKV_BF16, v_shares_k=0,
              combine_mode=SPLITKV_COMBINE_SEPARATE, kv_layout=SPLITKV_LAYOUT_HND) -> splitkv_desc_t:
    return splitkv_desc_t(batch, q_tokens, num_q_heads, num_kv_heads, qk_dim, v_dim, page_size,
                          max_pages_per_seq, num_pages_total, kv_dtype, int(v_shares_k), combine_mode,
                          kv_layout)


class Plan:
    """Owns a ``splitkv_plan_t*``; frees it when collected."""

    def __init__(self, handle: int, desc: splitkv_desc_t, num_splits: int):
        self.handle = handle
        self.desc = desc
        self.num_splits = num_splits

    def __del__(self):
        if getattr(self, "handle", None):
            _lib.splitkv_plan_destroy(self.handle)
            self.handle = None

    @property
    def num_items(self) -> int:
        return _lib.splitkv_plan_num_items(self.handle)

    @property
    def workspace_size(self) -> int:
        return splitkv_workspace_size(self)


def splitkv_plan(desc: splitkv_desc_t, seq_lens_host, num_splits: int = 0, num_sms: int = 0) -> Plan:
    lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
    h = _vp()
    _check(_lib.splitkv_plan(ctypes.byref(desc), lens.ctypes.data, num_splits, num_sms, ctypes.byref(h)))
    return Plan(h.value, desc, num_splits)


def splitkv_plan_fixed(desc: splitkv_desc_t, num_splits: int) -> Plan:
    """Capacity plan whose work list splitkv_plan_refresh rewrites on the device."""
    h = _vp()
    _check(_lib.splitkv_plan_fixed(ctypes.byref(desc), num_splits, ctypes.byref(h)))
    return Plan(h.value, desc, num_splits)


def splitkv_plan_refresh(plan: Plan, workspace, seq_lens, stream=None):
    _check(_lib.splitkv_plan_refresh(plan.handle, _ptr(workspace), _ptr(seq_lens), _stream(stream)))


def splitkv_read_items(plan: Plan, workspace, stream=None) -> np.ndarray:
    """The work list currently in `workspace` (synchronises the stream)."""
    n = plan.num_items
    out = np.zeros((n, SPLITKV_ITEM_FIELDS), dtype=np.int32)
    _check(_lib.splitkv_read_items(plan.handle, _ptr(workspace), out.ctypes.data, n, _stream(stream)))
    return out


def splitkv_plan_get_items(plan: Plan) -> np.ndarray:
    n = _i32()
    _check(_lib.splitkv_plan_get_items(plan.handle, None, 0, ctypes.byref(n)))
    out = np.zeros((n.value, SPLITKV_ITEM_FIELDS), dtype=np.int32)
    _check(_lib.splitkv_plan_get_items(plan.handle, out.ctypes.data if n.value else None,
                                       n.value, ctypes.byref(n)))
    return out


def splitkv_plan_get_ranges(plan: Plan) -> np.ndarray:
    """The split table per KV head: rows (b, h_kv, s, page_begin, page_end)."""
    n = _i32()
    _check(_lib.splitkv_plan_get_ranges(plan.handle, None, 0, ctypes.byref(n)))
    out = np.zeros((n.value, SPLITKV_RANGE_FIELDS), dtype=np.int32)
    _check(_lib.splitkv_plan_get_ranges(plan.handle, out.ctypes.data if n.value else None,
                                        n.value, ctypes.byref(n)))
    return out


def splitkv_workspace_size(plan: Plan) -> int:
    return int(_lib.splitkv_workspace_size(plan.handle))


def splitkv_plan_upload(plan: Plan, workspace, workspace_bytes: int, stream=None):
    _check(_lib.splitkv_plan_upload(plan.handle, _ptr(workspace), workspace_bytes, _stream(stream)))


def splitkv_decode(plan: Plan, workspace, q, k_pages, v_pages, block_table, seq_lens,
                   num_splits: int, scale: float, kv_scale: float, out, lse, stream=None):
    _check(_lib.splitkv_decode(plan.handle, _ptr(workspace), _ptr(q), _ptr(k_pages), _ptr(v_pages),
                               _ptr(block_table), _ptr(seq_lens), num_splits, scale, kv_scale,
                               _ptr(out), _ptr(lse), _stream(stream)))


def splitkv_decode_partials(plan: Plan, workspace, q, k_pages, v_pages, block_table, seq_lens,
                            num_splits: int, scale: float, kv_scale: float, out, lse, stream=None):
    """The split-KV kernel of splitkv_decode alone (partials stay in the workspace)."""
    _check(_lib.splitkv_decode_partials(plan.handle, _ptr(workspace), _ptr(q), _ptr(k_pages),
                                        _ptr(v_pages), _ptr(block_table), _ptr(seq_lens),
                                        num_splits, scale, kv_scale, _ptr(out), _ptr(lse),
                                        _stream(stream)))


def splitkv_combine_workspace(plan: Plan, workspace, out, lse, stream=None):
    """The merge of the partials splitkv_decode_partials left in the workspace."""
    _check(_lib.splitkv_combine_workspace(plan.handle, _ptr(workspace), _ptr(out), _ptr(lse),
                                          _stream(stream)))


def splitkv_decode_kv_scales(plan: Plan, workspace, q, k_pages, v_pages, block_table, seq_lens,
                             num_splits: int, scale: float, k_scale, v_scale, out, lse,
                             stream=None):
    """splitkv_decode over an e4m3 cache with per-KV-head K and V scales
    (``k_scale``, ``v_scale``: fp32 [Hkv] device tensors)."""
    _check(_lib.splitkv_decode_kv_scales(plan.handle, _ptr(workspace), _ptr(q), _ptr(k_pages),
                                         _ptr(v_pages), _ptr(block_table), _ptr(seq_lens),
                                         num_splits, scale, _ptr(k_scale), _ptr(v_scale), _ptr(out),
                                         _ptr(lse), _stream(stream)))


def splitkv_decode_noalloc(plan: Plan, q, k_pages, v_pages, block_table, seq_lens,
                           num_splits: int, scale: float, kv_scale: float, out, lse, stream=None):
    """splitkv_decode without a caller workspace (the library's 16 MiB device
    array is used instead); for callers that cannot allocate device memory."""
    _check(_lib.splitkv_decode_noalloc(plan.handle, _ptr(q), _ptr(k_pages), _ptr(v_pages),
                                       _ptr(block_table), _ptr(seq_lens), num_splits, scale,
                                       kv_scale, _ptr(out), _ptr(lse), _stream(stream)))


def splitkv_combine(o_part, lse_part, n_parts: int, rows: int, dv: int, out_bf16=None,
                    out_f32=None, lse_out=None, stream=None):
    _check(_lib.splitkv_combine(_ptr(o_part), _ptr(lse_part), n_parts, rows, dv, _ptr(out_bf16),
                                _ptr(out_f32), _ptr(lse_out), _stream(stream)))


def splitkv_plan_launches_per_call(plan: Plan) -> int:
    return int(_lib.splitkv_plan_launches_per_call(plan.handle))


def splitkv_plan_num_ctas(plan: Plan) -> int:
    return int(_lib.splitkv_plan_num_ctas(plan.handle))


def splitkv_plan_heads_per_item(plan: Plan) -> int:
    return int(_lib.splitkv_plan_heads_per_item(plan.handle))


def splitkv_read_stats(plan: Plan, workspace, stream=None):
    """Returns (cta_log [n_ctas][4] int32, status int)."""
    n = splitkv_plan_num_ctas(plan)
    log = np.zeros((max(n, 1), 4), dtype=np.int32)
    st = np.zeros(1, dtype=np.int32)
    _check(_lib.splitkv_read_stats(plan.handle, _ptr(workspace), log.ctypes.data, log.shape[0],
                                   st.ctypes.data, _stream(stream)))
    return log[:n], int(st[0])


def splitkv_noalloc_read_stats(plan: Plan, stream=None):
    """(cta_log [n_ctas][4] int32, status int) of the last splitkv_decode_noalloc
    call on the current device (synchronises the stream)."""
    n = splitkv_plan_num_ctas(plan)
    log = np.zeros((max(n, 1), 4), dtype=np.int32)
    st = np.zeros(1, dtype=np.int32)
    _check(_lib.splitkv_noalloc_read_stats(plan.handle, log.ctypes.data, log.shape[0],
                                           st.ctypes.data, _stream(stream)))
    return log[:n], int(st[0])


def splitkv_debug_gather(desc: splitkv_desc_t, pages, row_elems: int, block_table, b: int,
                         h_kv: int, n_keys: int, dst, stream=None):
    _check(_lib.splitkv_debug_gather(ctypes.byref(desc), _ptr(pages), row_elems, _ptr(block_table),
                                     b, h_kv, n_keys, _ptr(dst), _stream(stream)))


def splitkv_last_error() -> str:
    return _lib.splitkv_last_error().decode()
