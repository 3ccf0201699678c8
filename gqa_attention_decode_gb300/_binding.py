"""ctypes binding of libgqa_attn.so: argument checks and marshalling, nothing else.

Function names and argument order follow include/gqa_attn.h.  Tensors are torch
tensors (device memory and streams come from PyTorch); sizes are read from
their shapes.  Every non-zero status raises GQAError.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

GQA_OK = 0
GQA_ERR_INVALID_ARG = 1
GQA_ERR_UNSUPPORTED = 2
GQA_ERR_CUDA = 3
GQA_ERR_WORKSPACE = 4
GQA_ERR_TIMEOUT = 5
GQA_ERR_OUT_OF_BOUNDS = 6

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libgqa_attn.so"
_lock = threading.Lock()
_lib = None

_c_int, _c_size, _c_float, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p
_ip = ctypes.POINTER(ctypes.c_int)

_SIGNATURES = {
    "gqa_status_string": (ctypes.c_char_p, [_c_int]),
    "gqa_attn_abi_version": (_c_int, []),
    "gqa_attn_decode_plan": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _ip, _ip]),
    "gqa_attn_decode_workspace_size": (_c_size, [_c_int] * 7),
    "gqa_attn_decode": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                 _c_float, _c_int, _vp, _vp, _vp, _c_size, _vp]),
    "gqa_attn_decode_paged": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                       _c_int, _c_int, _c_int, _c_float, _c_int, _vp, _vp, _vp,
                                       _c_size, _vp]),
    "gqa_attn_decode_paged_multi": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                                             _c_int, _c_int, _c_int, _c_int, _c_int, _c_float,
                                             _c_int, _vp, _vp, _vp, _c_size, _vp]),
    "gqa_attn_decode_multi_workspace_size": (_c_size, [_c_int] * 8),
    "gqa_attn_decode_multi": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                       _c_int, _c_float, _c_int, _vp, _vp, _vp, _c_size, _vp]),
    "gqa_attn_decode_kernel_count": (_c_int, [_c_int] * 6 + [_ip]),
    "gqa_attn_decode_split": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                       _c_int, _c_float, _c_int, _vp, _c_size, _vp]),
    "gqa_attn_decode_merge": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                       _vp, _vp, _vp, _c_size, _vp]),
    "gqa_attn_decode_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                         _c_int, _c_float, _c_int, _vp, _vp, _vp]),
    "gqa_attn_prefill_causal": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                         _c_int, _c_int, _c_float, _vp, _vp, _vp]),
    "gqa_attn_prefill_causal_workspace_size": (_c_size, [_c_int] * 8),
    "gqa_attn_prefill_causal_ws": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                            _c_int, _c_int, _c_int, _c_float, _vp, _vp, _vp,
                                            _c_size, _vp]),
    "gqa_attn_prefill_causal_kernel_count": (_c_int, [_c_int] * 7 + [_c_size, _ip]),
    "gqa_attn_prefill_causal_paged": (_c_int, [_vp, _vp, _vp, _vp] + [_c_int] * 10 +
                                      [_c_float, _vp, _vp, _vp, _c_size, _vp]),
    "gqa_attn_prefill_causal_plan": (_c_int, [_c_int] * 8 + [_c_size, _ip, _ip, _ip]),
    "gqa_attn_decode_from_host_arena_size": (_c_size, [_c_int] * 7),
    "gqa_attn_decode_from_host": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                           _c_int, _c_float, _c_int, _vp, _vp, _vp, _c_size,
                                           _vp]),
    "gqa_attn_prefill_causal_from_host_arena_size": (_c_size, [_c_int] * 6),
    "gqa_attn_prefill_causal_from_host": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int,
                                                   _c_int, _c_int, _c_int, _c_int, _c_float,
                                                   _vp, _vp, _vp, _c_size, _vp]),
    "gqa_attn_merge_states": (_c_int, [_vp, _vp, _c_int, ctypes.c_longlong, _c_int, _vp, _vp,
                                       _vp]),
    "gqa_attn_device_status": (_c_int, [_vp, _ip]),
    "gqa_attn_selftest_bounded_wait": (_c_int, [_c_int, _vp]),
    "gqa_attn_bounds_checked": (_c_int, []),
    "gqa_attn_selftest_bounds": (_c_int, [_vp]),
    "gqa_attn_debug_s_tile_count": (_c_int, [_vp, ctypes.POINTER(ctypes.c_ulonglong)]),
}


class GQAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gqa_status_string(status)} (status {status})")


def lib_path() -> str:
    return os.environ.get("GQA_ATTN_LIB", os.path.join(_PKG_DIR, _LIB_NAME))


def load_library() -> ctypes.CDLL:
    """Loads libgqa_attn.so once; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with "
                    "`python -m gqa_attention_decode_gb300.build` (needs nvcc)")
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def gqa_status_string(status: int) -> str:
    return load_library().gqa_status_string(int(status)).decode()


def gqa_attn_abi_version() -> int:
    return load_library().gqa_attn_abi_version()


def _check(status: int, where: str) -> None:
    if status != GQA_OK:
        raise GQAError(status, where)


def _stream_handle(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return _vp(stream.cuda_stream)


def _num_sms(device) -> int:
    return torch.cuda.get_device_properties(device).multi_processor_count


def _need(t: torch.Tensor, name: str, dtype, ndim: int, device=None, cuda=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if cuda and t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if not cuda and t.device.type != "cpu":
        raise ValueError(f"{name} must be a CPU tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _ptr(t):
    return _vp(t.data_ptr()) if t is not None else _vp(0)


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------

def gqa_attn_decode_plan(B: int, H_kv: int, S_max: int, num_sms: int, num_splits: int = 0):
    """(num_splits, chunk) the library will use; host only."""
    s, c = ctypes.c_int(), ctypes.c_int()
    _check(load_library().gqa_attn_decode_plan(B, H_kv, S_max, num_sms, num_splits,
                                               ctypes.byref(s), ctypes.byref(c)),
           "gqa_attn_decode_plan")
    return s.value, c.value


def gqa_attn_decode_workspace_size(B, H_q, H_kv, S_max, d, num_sms, num_splits=0) -> int:
    return int(load_library().gqa_attn_decode_workspace_size(B, H_q, H_kv, S_max, d, num_sms,
                                                             num_splits))


def gqa_attn_decode(q, k_cache, v_cache, seqlens, scale, num_splits=0, o=None, lse=None,
                    workspace=None, stream=None):
    """Split-KV GQA decode.  q [B,H_q,d] bf16; k_cache, v_cache [B,H_kv,S_max,d] bf16;
    seqlens [B] int32 (device).  Returns (o [B,H_q,d] bf16, lse [B,H_q] fp32)."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 3)
    dev = q.device
    _need(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _need(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _need(seqlens, "seqlens", torch.int32, 1, dev)
    B, H_q, d = q.shape
    _, H_kv, S_max, _ = k_cache.shape
    if tuple(k_cache.shape) != (B, H_kv, S_max, d) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError(f"k_cache/v_cache must be [B,H_kv,S_max,d] = [{B},H_kv,S_max,{d}]")
    if seqlens.shape[0] != B:
        raise ValueError("seqlens must have B entries")
    if o is None:
        o = torch.empty((B, H_q, d), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=dev)
    _need(o, "o", torch.bfloat16, 3, dev)
    _need(lse, "lse", torch.float32, 2, dev)
    if workspace is None:
        nbytes = gqa_attn_decode_workspace_size(B, H_q, H_kv, S_max, d, _num_sms(dev), num_splits)
        workspace = torch.empty((max(nbytes, 1),), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, 1, dev)
    with torch.cuda.device(dev):
        rc = lib.gqa_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), B, H_q,
                                 H_kv, S_max, d, float(scale), int(num_splits), _ptr(o),
                                 _ptr(lse), _ptr(workspace), workspace.numel(),
                                 _stream_handle(stream, dev))
    _check(rc, "gqa_attn_decode")
    return o, lse


def gqa_attn_decode_paged(q, k_pages, v_pages, block_table, seqlens, scale, num_splits=0,
                          o=None, lse=None, workspace=None, stream=None):
    """Decode over a paged cache.  k_pages, v_pages [num_pages, H_kv, page_size, d] bf16;
    block_table [B, max_pages_per_seq] int32; seqlens [B] int32 (all on the device)."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 3)
    dev = q.device
    _need(k_pages, "k_pages", torch.bfloat16, 4, dev)
    _need(v_pages, "v_pages", torch.bfloat16, 4, dev)
    _need(block_table, "block_table", torch.int32, 2, dev)
    _need(seqlens, "seqlens", torch.int32, 1, dev)
    B, H_q, d = q.shape
    num_pages, H_kv, page_size, _ = k_pages.shape
    if tuple(v_pages.shape) != tuple(k_pages.shape) or k_pages.shape[3] != d:
        raise ValueError("k_pages/v_pages must be [num_pages, H_kv, page_size, d]")
    if block_table.shape[0] != B or seqlens.shape[0] != B:
        raise ValueError("block_table and seqlens need B rows")
    max_pages = block_table.shape[1]
    if o is None:
        o = torch.empty((B, H_q, d), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=dev)
    if workspace is None:
        nbytes = gqa_attn_decode_workspace_size(B, H_q, H_kv, max_pages * page_size, d,
                                                _num_sms(dev), num_splits)
        workspace = torch.empty((max(nbytes, 1),), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = lib.gqa_attn_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                       _ptr(seqlens), B, H_q, H_kv, num_pages, page_size,
                                       max_pages, d, float(scale), int(num_splits), _ptr(o),
                                       _ptr(lse), _ptr(workspace), workspace.numel(),
                                       _stream_handle(stream, dev))
    _check(rc, "gqa_attn_decode_paged")
    return o, lse


def gqa_attn_decode_paged_multi(q, k_pages, v_pages, block_table, seqlens, scale, num_splits=0,
                                o=None, lse=None, workspace=None, stream=None):
    """Multi-token decode over a paged cache.  q [B,H_q,T_q,d] bf16 (token t at position
    seqlens[b]-T_q+t); k_pages, v_pages [num_pages,H_kv,page_size,d] bf16; block_table
    [B, max_pages_per_seq] int32; seqlens [B] int32.  Returns (o, lse)."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 4)
    dev = q.device
    _need(k_pages, "k_pages", torch.bfloat16, 4, dev)
    _need(v_pages, "v_pages", torch.bfloat16, 4, dev)
    _need(block_table, "block_table", torch.int32, 2, dev)
    _need(seqlens, "seqlens", torch.int32, 1, dev)
    B, H_q, T_q, d = q.shape
    num_pages, H_kv, page_size, _ = k_pages.shape
    if tuple(v_pages.shape) != tuple(k_pages.shape) or k_pages.shape[3] != d:
        raise ValueError("k_pages/v_pages must be [num_pages, H_kv, page_size, d]")
    if block_table.shape[0] != B or seqlens.shape[0] != B:
        raise ValueError("block_table and seqlens need B rows")
    max_pages = block_table.shape[1]
    if o is None:
        o = torch.empty((B, H_q, T_q, d), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H_q, T_q), dtype=torch.float32, device=dev)
    if workspace is None:
        nbytes = gqa_attn_decode_multi_workspace_size(B, H_q, H_kv, T_q, max_pages * page_size, d,
                                                      _num_sms(dev), num_splits)
        workspace = torch.empty((max(nbytes, 1),), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = lib.gqa_attn_decode_paged_multi(_ptr(q), _ptr(k_pages), _ptr(v_pages),
                                             _ptr(block_table), _ptr(seqlens), B, H_q, H_kv, T_q,
                                             num_pages, page_size, max_pages, d, float(scale),
                                             int(num_splits), _ptr(o), _ptr(lse),
                                             _ptr(workspace), workspace.numel(),
                                             _stream_handle(stream, dev))
    _check(rc, "gqa_attn_decode_paged_multi")
    return o, lse


def gqa_attn_decode_multi_workspace_size(B, H_q, H_kv, T_q, S_max, d, num_sms,
                                         num_splits=0) -> int:
    return int(load_library().gqa_attn_decode_multi_workspace_size(B, H_q, H_kv, T_q, S_max, d,
                                                                   num_sms, num_splits))


def gqa_attn_decode_multi(q, k_cache, v_cache, seqlens, scale, num_splits=0, o=None, lse=None,
                          workspace=None, stream=None):
    """Multi-token decode.  q [B,H_q,T_q,d] bf16 (token t at position seqlens[b]-T_q+t);
    k_cache, v_cache [B,H_kv,S_max,d] bf16; seqlens [B] int32.  Returns (o, lse)."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 4)
    dev = q.device
    _need(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _need(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _need(seqlens, "seqlens", torch.int32, 1, dev)
    B, H_q, T_q, d = q.shape
    _, H_kv, S_max, _ = k_cache.shape
    if tuple(v_cache.shape) != tuple(k_cache.shape) or k_cache.shape[0] != B:
        raise ValueError("k_cache/v_cache must be [B,H_kv,S_max,d]")
    if o is None:
        o = torch.empty((B, H_q, T_q, d), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H_q, T_q), dtype=torch.float32, device=dev)
    _need(o, "o", torch.bfloat16, 4, dev)
    _need(lse, "lse", torch.float32, 3, dev)
    if workspace is None:
        nbytes = gqa_attn_decode_multi_workspace_size(B, H_q, H_kv, T_q, S_max, d, _num_sms(dev),
                                                      num_splits)
        workspace = torch.empty((max(nbytes, 1),), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = lib.gqa_attn_decode_multi(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), B,
                                       H_q, H_kv, T_q, S_max, d, float(scale), int(num_splits),
                                       _ptr(o), _ptr(lse), _ptr(workspace), workspace.numel(),
                                       _stream_handle(stream, dev))
    _check(rc, "gqa_attn_decode_multi")
    return o, lse


def gqa_attn_decode_kernel_count(B, H_q, H_kv, S_max, d, num_splits=0, device=None) -> int:
    """Kernels gqa_attn_decode launches for these sizes on the device (1 or 2)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    out = ctypes.c_int(-1)
    with torch.cuda.device(dev):
        _check(load_library().gqa_attn_decode_kernel_count(B, H_q, H_kv, S_max, d, num_splits,
                                                           ctypes.byref(out)),
               "gqa_attn_decode_kernel_count")
    return out.value


def gqa_attn_decode_split(q, k_cache, v_cache, seqlens, scale, num_splits, workspace,
                          stream=None):
    """First phase of gqa_attn_decode: per-split partials into `workspace`."""
    lib = load_library()
    dev = q.device
    B, H_q, d = q.shape
    _, H_kv, S_max, _ = k_cache.shape
    for t, n, dt, nd in ((q, "q", torch.bfloat16, 3), (k_cache, "k_cache", torch.bfloat16, 4),
                         (v_cache, "v_cache", torch.bfloat16, 4), (seqlens, "seqlens", torch.int32, 1),
                         (workspace, "workspace", torch.uint8, 1)):
        _need(t, n, dt, nd, dev)
    with torch.cuda.device(dev):
        rc = lib.gqa_attn_decode_split(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), B,
                                       H_q, H_kv, S_max, d, float(scale), int(num_splits),
                                       _ptr(workspace), workspace.numel(),
                                       _stream_handle(stream, dev))
    _check(rc, "gqa_attn_decode_split")


def gqa_attn_decode_merge(seqlens, H_kv, S_max, num_splits, o, lse, workspace, stream=None):
    """Second phase of gqa_attn_decode: merge the partials into o and lse."""
    lib = load_library()
    dev = o.device
    B, H_q, d = o.shape
    for t, n, dt, nd in ((seqlens, "seqlens", torch.int32, 1), (o, "o", torch.bfloat16, 3),
                         (lse, "lse", torch.float32, 2), (workspace, "workspace", torch.uint8, 1)):
        _need(t, n, dt, nd, dev)
    with torch.cuda.device(dev):
        rc = lib.gqa_attn_decode_merge(_ptr(seqlens), B, H_q, H_kv, S_max, d, int(num_splits),
                                       _ptr(o), _ptr(lse), _ptr(workspace), workspace.numel(),
                                       _stream_handle(stream, dev))
    _check(rc, "gqa_attn_decode_merge")


GQA_NOALLOC_SCRATCH_BYTES = 48 << 20


def gqa_attn_decode_noalloc(q, k_cache, v_cache, seqlens, scale, num_splits=0, o=None, lse=None,
                            stream=None):
    """gqa_attn_decode for callers that cannot allocate device memory: the split
    partials go to the library's fixed static scratch (GQA_NOALLOC_SCRATCH_BYTES)
    instead of a workspace.  Calls that overlap on the GPU race on that scratch.
    o and lse must be given (this function allocates nothing)."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 3)
    dev = q.device
    _need(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _need(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _need(seqlens, "seqlens", torch.int32, 1, dev)
    _need(o, "o", torch.bfloat16, 3, dev)
    _need(lse, "lse", torch.float32, 2, dev)
    B, H_q, d = q.shape
    _, H_kv, S_max, _ = k_cache.shape
    with torch.cuda.device(dev):
        rc = lib.gqa_attn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), B,
                                         H_q, H_kv, S_max, d, float(scale), int(num_splits),
                                         _ptr(o), _ptr(lse), _stream_handle(stream, dev))
    _check(rc, "gqa_attn_decode_noalloc")
    return o, lse


# ---------------------------------------------------------------------------
# causal prefill
# ---------------------------------------------------------------------------

def gqa_attn_prefill_causal_workspace_size(B, H_q, H_kv, T_q, S_kv, d, q_offset, num_sms) -> int:
    return int(load_library().gqa_attn_prefill_causal_workspace_size(B, H_q, H_kv, T_q, S_kv, d,
                                                                      q_offset, num_sms))


def gqa_attn_prefill_causal_plan(B, H_q, H_kv, T_q, S_kv, d, q_offset, num_sms, ws_bytes):
    """Host-only prefill work plan on `num_sms` SMs: (units, split units, pieces per unit)."""
    u, su, ps = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    rc = load_library().gqa_attn_prefill_causal_plan(B, H_q, H_kv, T_q, S_kv, d, q_offset,
                                                     num_sms, ws_bytes, ctypes.byref(u),
                                                     ctypes.byref(su), ctypes.byref(ps))
    _check(rc, "gqa_attn_prefill_causal_plan")
    return u.value, su.value, ps.value


def gqa_attn_prefill_causal_kernel_count(B, H_q, H_kv, T_q, S_kv, d, q_offset, ws_bytes,
                                         device=None) -> int:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    out = ctypes.c_int(0)
    with torch.cuda.device(dev):
        rc = load_library().gqa_attn_prefill_causal_kernel_count(B, H_q, H_kv, T_q, S_kv, d,
                                                                 q_offset, ws_bytes,
                                                                 ctypes.byref(out))
    _check(rc, "gqa_attn_prefill_causal_kernel_count")
    return out.value


def gqa_attn_prefill_causal(q, k, v, scale, q_offset=0, o=None, lse=None, workspace=None,
                            stream=None):
    """Causal GQA prefill.  q [B,H_q,T_q,d]; k, v [B,H_kv,S_kv,d] (bf16).
    Row i of q is at absolute position q_offset + i.  Returns (o, lse).

    workspace: CUDA uint8 scratch for key-range splitting of a partial last
    round of work; None allocates gqa_attn_prefill_causal_workspace_size bytes,
    an empty tensor runs without splitting."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 4)
    dev = q.device
    _need(k, "k", torch.bfloat16, 4, dev)
    _need(v, "v", torch.bfloat16, 4, dev)
    B, H_q, T_q, d = q.shape
    _, H_kv, S_kv, _ = k.shape
    if tuple(k.shape) != (B, H_kv, S_kv, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k/v must be [B,H_kv,S_kv,d] matching q")
    if o is None:
        o = torch.empty((B, H_q, T_q, d), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H_q, T_q), dtype=torch.float32, device=dev)
    _need(o, "o", torch.bfloat16, 4, dev)
    _need(lse, "lse", torch.float32, 3, dev)
    if workspace is None:
        nbytes = gqa_attn_prefill_causal_workspace_size(B, H_q, H_kv, T_q, S_kv, d,
                                                        int(q_offset), _num_sms(dev))
        workspace = torch.empty((nbytes,), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, 1, dev)
    ws_ptr = _ptr(workspace) if workspace.numel() > 0 else None
    with torch.cuda.device(dev):
        rc = lib.gqa_attn_prefill_causal_ws(_ptr(q), _ptr(k), _ptr(v), B, H_q, H_kv, T_q, S_kv,
                                            d, int(q_offset), float(scale), _ptr(o), _ptr(lse),
                                            ws_ptr, workspace.numel(),
                                            _stream_handle(stream, dev))
    _check(rc, "gqa_attn_prefill_causal_ws")
    return o, lse


def gqa_attn_merge_states(o_parts, lse_parts, o=None, lse=None, stream=None):
    """Combine attention states over disjoint key shards.  o_parts [P, ..., d] bf16,
    lse_parts [P, ...] fp32 (natural log), the shards stacked on the first axis.
    Returns (o [..., d] bf16, lse [...] fp32)."""
    lib = load_library()
    if not isinstance(o_parts, torch.Tensor) or not isinstance(lse_parts, torch.Tensor):
        raise TypeError("o_parts and lse_parts must be torch.Tensors")
    if o_parts.dtype != torch.bfloat16 or lse_parts.dtype != torch.float32:
        raise TypeError("o_parts must be bfloat16 and lse_parts float32")
    if not o_parts.is_cuda or lse_parts.device != o_parts.device:
        raise ValueError("o_parts and lse_parts must be CUDA tensors on one device")
    if o_parts.dim() < 2 or tuple(o_parts.shape[:-1]) != tuple(lse_parts.shape):
        raise ValueError("o_parts must be [P, ..., d] and lse_parts [P, ...]")
    if not o_parts.is_contiguous() or not lse_parts.is_contiguous():
        raise ValueError("o_parts and lse_parts must be contiguous")
    dev = o_parts.device
    P, d = o_parts.shape[0], o_parts.shape[-1]
    rows = lse_parts[0].numel() if P > 0 else 0
    if o is None:
        o = torch.empty(o_parts.shape[1:], dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(lse_parts.shape[1:], dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        rc = lib.gqa_attn_merge_states(_ptr(o_parts), _ptr(lse_parts), P, rows, d, _ptr(o),
                                       _ptr(lse), _stream_handle(stream, dev))
    _check(rc, "gqa_attn_merge_states")
    return o, lse


def gqa_attn_prefill_causal_paged(q, k_pages, v_pages, block_table, S_kv, scale, q_offset=0,
                                  o=None, lse=None, workspace=None, stream=None):
    """Causal prefill over a paged cache.  q [B,H_q,T_q,d]; k_pages, v_pages
    [num_pages,H_kv,page_size,d] bf16; block_table [B, max_pages_per_seq] int32;
    every sequence has S_kv keys.  Row i of q is at absolute position q_offset + i."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 4)
    dev = q.device
    _need(k_pages, "k_pages", torch.bfloat16, 4, dev)
    _need(v_pages, "v_pages", torch.bfloat16, 4, dev)
    _need(block_table, "block_table", torch.int32, 2, dev)
    B, H_q, T_q, d = q.shape
    num_pages, H_kv, page_size, _ = k_pages.shape
    if tuple(v_pages.shape) != tuple(k_pages.shape) or k_pages.shape[3] != d:
        raise ValueError("k_pages/v_pages must be [num_pages, H_kv, page_size, d]")
    if block_table.shape[0] != B:
        raise ValueError("block_table needs B rows")
    if o is None:
        o = torch.empty((B, H_q, T_q, d), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H_q, T_q), dtype=torch.float32, device=dev)
    if workspace is None:
        nbytes = gqa_attn_prefill_causal_workspace_size(B, H_q, H_kv, T_q, S_kv, d,
                                                        int(q_offset), _num_sms(dev))
        workspace = torch.empty((nbytes,), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, 1, dev)
    ws_ptr = _ptr(workspace) if workspace.numel() > 0 else None
    with torch.cuda.device(dev):
        rc = lib.gqa_attn_prefill_causal_paged(
            _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), B, H_q, H_kv, T_q,
            int(S_kv), num_pages, page_size, block_table.shape[1], d, int(q_offset),
            float(scale), _ptr(o), _ptr(lse), ws_ptr, workspace.numel(),
            _stream_handle(stream, dev))
    _check(rc, "gqa_attn_prefill_causal_paged")
    return o, lse


# ---------------------------------------------------------------------------
# host-buffer variants
# ---------------------------------------------------------------------------

def gqa_attn_decode_from_host_arena_size(B, H_q, H_kv, S_max, d, num_sms, num_splits=0) -> int:
    return int(load_library().gqa_attn_decode_from_host_arena_size(B, H_q, H_kv, S_max, d,
                                                                   num_sms, num_splits))


def gqa_attn_decode_from_host(q, k_cache, v_cache, seqlens, scale, num_splits, o, lse, arena,
                              stream=None):
    """Decode on CPU (ideally pinned) tensors, staged through the CUDA uint8 `arena`."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 3, cuda=False)
    _need(k_cache, "k_cache", torch.bfloat16, 4, cuda=False)
    _need(v_cache, "v_cache", torch.bfloat16, 4, cuda=False)
    _need(seqlens, "seqlens", torch.int32, 1, cuda=False)
    _need(o, "o", torch.bfloat16, 3, cuda=False)
    _need(lse, "lse", torch.float32, 2, cuda=False)
    _need(arena, "arena", torch.uint8, 1)
    B, H_q, d = q.shape
    _, H_kv, S_max, _ = k_cache.shape
    dev = arena.device
    with torch.cuda.device(dev):
        rc = lib.gqa_attn_decode_from_host(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens),
                                           B, H_q, H_kv, S_max, d, float(scale), int(num_splits),
                                           _ptr(o), _ptr(lse), _ptr(arena), arena.numel(),
                                           _stream_handle(stream, dev))
    _check(rc, "gqa_attn_decode_from_host")
    return o, lse


def gqa_attn_prefill_causal_from_host_arena_size(B, H_q, H_kv, T_q, S_kv, d) -> int:
    return int(load_library().gqa_attn_prefill_causal_from_host_arena_size(B, H_q, H_kv, T_q,
                                                                           S_kv, d))


def gqa_attn_prefill_causal_from_host(q, k, v, scale, q_offset, o, lse, arena, stream=None):
    """Causal prefill on CPU (ideally pinned) tensors, staged through the CUDA `arena`."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 4, cuda=False)
    _need(k, "k", torch.bfloat16, 4, cuda=False)
    _need(v, "v", torch.bfloat16, 4, cuda=False)
    _need(o, "o", torch.bfloat16, 4, cuda=False)
    _need(lse, "lse", torch.float32, 3, cuda=False)
    _need(arena, "arena", torch.uint8, 1)
    B, H_q, T_q, d = q.shape
    _, H_kv, S_kv, _ = k.shape
    dev = arena.device
    with torch.cuda.device(dev):
        rc = lib.gqa_attn_prefill_causal_from_host(_ptr(q), _ptr(k), _ptr(v), B, H_q, H_kv, T_q,
                                                   S_kv, d, int(q_offset), float(scale), _ptr(o),
                                                   _ptr(lse), _ptr(arena), arena.numel(),
                                                   _stream_handle(stream, dev))
    _check(rc, "gqa_attn_prefill_causal_from_host")
    return o, lse


# ---------------------------------------------------------------------------
# diagnostics
# ---------------------------------------------------------------------------

def gqa_attn_device_status(stream=None, device=None) -> int:
    """Synchronises the stream and returns (and clears) the device status word."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    out = ctypes.c_int(-1)
    with torch.cuda.device(dev):
        _check(load_library().gqa_attn_device_status(_stream_handle(stream, dev),
                                                     ctypes.byref(out)),
               "gqa_attn_device_status")
    return out.value


def gqa_attn_bounds_checked() -> bool:
    """Whether the loaded library is a bounds-checked build (libgqa_attn_debug.so)."""
    return bool(load_library().gqa_attn_bounds_checked())


def gqa_attn_selftest_bounds(stream=None, device=None) -> None:
    """Bounds-checked builds: one store past its range, recorded as
    GQA_ERR_OUT_OF_BOUNDS in the device status (raises GQAError elsewhere)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        _check(load_library().gqa_attn_selftest_bounds(_stream_handle(stream, dev)),
               "gqa_attn_selftest_bounds")


def gqa_attn_debug_s_tile_count(stream=None, device=None) -> int:
    """Bounds-checked builds: S = Q K^T tile products (per query head and 128-key
    tile) the prefill kernels issued since the previous call; the counter resets.
    Raises GQAError (GQA_ERR_UNSUPPORTED) in release builds."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    out = ctypes.c_ulonglong(0)
    with torch.cuda.device(dev):
        _check(load_library().gqa_attn_debug_s_tile_count(_stream_handle(stream, dev),
                                                          ctypes.byref(out)),
               "gqa_attn_debug_s_tile_count")
    return int(out.value)


def gqa_attn_selftest_bounded_wait(timeout_us: int, stream=None, device=None) -> None:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        _check(load_library().gqa_attn_selftest_bounded_wait(int(timeout_us),
                                                             _stream_handle(stream, dev)),
               "gqa_attn_selftest_bounded_wait")
